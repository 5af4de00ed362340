"""CPU tests of the iteration-latency estimator (ConfluxServe §6.2 Eq. 2-6,
App. D Eq. 7-11, §8.4 accuracy measure).

First the fp64 oracle (oracle/latency.py) is pinned to facts fixed outside
its own formulas: brute-force counts of causal (query, key) pairs, library
least squares and MAPE, the pages' worked dispatch example, and invariants
the text states (the linear region waits for the largest combined load, the
sequence-parallel attention term ignores how prefill tokens are spread,
alpha and beta act on one path each).  Then the native estimator behind the
C ABI is checked against the oracle on random inputs.
"""
import itertools
import math
import random

import numpy as np
import pytest

from oracle import latency as O


# --------------------------------------------------------------- oracle pins
def causal_pairs(l, c):
    """(query, key) pairs a chunk of l tokens after c cached ones scores:
    query i sits at position c + i and sees keys 0 .. c + i."""
    mask = np.arange(c + l)[None, :] <= (c + np.arange(l))[:, None]
    return int(mask.sum())


def test_chunk_workload_counts_the_causal_pairs():
    # App. D Eq. 9: l (c + (l+1)/2) is the chunk's causal attention work
    for l in range(0, 25):
        for c in (0, 1, 2, 7, 16, 33, 100):
            assert O.chunk_workload(l, c) == causal_pairs(l, c)


def test_fit_line_matches_library_least_squares():
    from scipy import stats
    rng = np.random.default_rng(7)
    for n in (2, 3, 10, 200):
        x = rng.uniform(0, 1e5, n)
        y = 3e-4 * x + 0.2 + rng.normal(0, 0.05, n)
        s, b = O.fit_line(x, y)
        r = stats.linregress(x, y)
        assert s == pytest.approx(r.slope, rel=1e-9, abs=1e-15)
        assert b == pytest.approx(r.intercept, rel=1e-9, abs=1e-12)


def test_fit_line_recovers_an_exact_line_and_rejects_constant_x():
    x = np.arange(1, 40, dtype=float) * 256
    s, b = O.fit_line(x, 2.5e-3 * x - 1.25)
    assert s == pytest.approx(2.5e-3, rel=1e-12)
    assert b == pytest.approx(-1.25, rel=1e-10)
    with pytest.raises(ValueError):
        O.fit_line([5.0, 5.0, 5.0], [1.0, 2.0, 3.0])


def test_mape_is_the_mean_absolute_percentage_error():
    assert O.mape([110.0, 90.0, 100.0, 50.0], [100.0, 100.0, 100.0, 100.0]) == pytest.approx(17.5)
    metrics = pytest.importorskip("sklearn.metrics")
    rng = np.random.default_rng(1)
    t = rng.uniform(0.1, 10, 300)
    p = t * rng.uniform(0.8, 1.2, 300)
    assert O.mape(p, t) == pytest.approx(100 * metrics.mean_absolute_percentage_error(t, p), rel=1e-12)


def unit_model(**kw):
    base = dict(gamma=0.0, gamma0=0.0, a_d=0.0, a_d0=0.0, a_p=0.0, a_p0=0.0, a_comm=0.0, a_comm0=0.0,
                alpha=1.0, beta=1.0)
    base.update(kw)
    return O.LatencyModel(**base)


def test_worked_dispatch_example_levels_the_combined_load():
    # the dispatch example on the pages: decode tokens 40 / 10 / 10 / 0 and a
    # water level of 300 leave room for 260 / 290 / 290 / 300 prefill tokens
    # (1140 in all); every rank then carries 300 tokens, so the linear region
    # costs what one rank of 300 tokens costs (§6.2 Eq. 3)
    m = unit_model(gamma=1.0, gamma0=5.0)
    dec = [40, 10, 10, 0]
    pre = [260, 290, 290, 300]
    assert sum(pre) == 1140
    ranks = [O.RankLoad(p, d, tuple([1000] * d)) for p, d in zip(pre, dec)]
    assert O.t_gemm(m, ranks) == 305.0
    # any other split of the same 1140 tokens raises the largest load
    moved = [270, 280, 290, 300]
    ranks2 = [O.RankLoad(p, d, tuple([1000] * d)) for p, d in zip(moved, dec)]
    assert O.t_gemm(m, ranks2) == 315.0


def test_prefill_attention_term_ignores_the_token_split():
    # §6.2: Ulysses-SP spreads the aggregate chunk workload evenly, so only
    # f_comm sees how prefill tokens are assigned to ranks
    chunks = [(700, 3000), (340, 0), (100, 12000)]
    w = sum(causal_pairs(l, c) for l, c in chunks)
    m = unit_model(a_p=1.0)
    splits = [(1140, 0, 0, 0), (285, 285, 285, 285), (0, 1140, 0, 0), (500, 40, 300, 300)]
    for sp in splits:
        ranks = [O.RankLoad(p, 0, ()) for p in sp]
        assert O.t_prefill(m, ranks, chunks) == pytest.approx(w / 4, rel=1e-15)
    mc = unit_model(a_comm=2.0, a_comm0=1.0)
    for sp in splits:
        ranks = [O.RankLoad(p, 0, ()) for p in sp]
        assert O.t_prefill(mc, ranks, chunks) == 2.0 * max(sp) + 1.0
    # one rank: no All-to-All
    assert O.t_prefill(mc, [O.RankLoad(1140, 0, ())], chunks) == 0.0


def test_decode_path_waits_for_the_largest_context_sum():
    m = unit_model(a_d=1.0, a_d0=0.5)
    ctx = [(8192, 100, 7), (16384,), (), (4000, 4000, 4000, 4000, 1)]
    ranks = [O.RankLoad(0, len(c), c) for c in ctx]
    mat = np.zeros((4, 5))
    for r, c in enumerate(ctx):
        mat[r, :len(c)] = c
    assert O.t_decode(m, ranks) == mat.sum(axis=1).max() + 0.5
    # a rank without decodes does not set the max through the intercept
    only_empty = [O.RankLoad(10, 0, ())]
    assert O.t_decode(unit_model(a_d0=9.0), only_empty) == 0.0


def test_contention_factors_act_on_one_path_each():
    ranks, chunks = O.one_gpu(512, 2048, [4096] * 8)
    m = unit_model(gamma=1e-3, gamma0=0.1, a_d=1e-5, a_d0=0.01, a_p=1e-7, a_p0=0.02)
    tp = O.t_prefill(m, ranks, chunks)
    td = O.t_decode(m, ranks)
    assert tp > 0 and td > 0
    for a, b in itertools.product((1.0, 1.5, 4.0), (1.0, 1.25, 7.0)):
        mm = O.LatencyModel(**{**m.__dict__, "alpha": a, "beta": b})
        r = O.t_iter(mm, ranks, chunks)
        assert r["t_attn"] == max(a * td, b * tp)
        assert r["t_prefill"] == tp and r["t_decode"] == td
    # decode only: beta plays no part; prefill only: alpha plays no part
    rd, cd = O.one_gpu(0, 0, [4096] * 8)
    rp, cp = O.one_gpu(512, 2048, [])
    for b in (1.0, 3.0):
        assert O.t_iter(O.LatencyModel(**{**m.__dict__, "beta": b}), rd, cd)["t_attn"] == td
        assert O.t_iter(O.LatencyModel(**{**m.__dict__, "alpha": b}), rp, cp)["t_attn"] == tp


def test_iteration_is_layers_times_one_layer_and_empty_paths_cost_nothing():
    m = unit_model(gamma=1e-3, gamma0=0.1, a_d=1e-5, a_d0=0.01, a_p=1e-7, a_p0=0.02, alpha=1.1, beta=1.2)
    ranks, chunks = O.one_gpu(300, 100, [1000, 2000])
    one = O.t_iter(m, ranks, chunks)
    for L in (1, 2, 32, 80):
        assert O.t_iter(m, ranks, chunks, L)["t_iter"] == pytest.approx(L * one["t_iter"], rel=1e-15)
    r0, c0 = O.one_gpu(0, 0, [])
    assert O.t_iter(m, r0, c0)["t_iter"] == 0.0
    r1, c1 = O.one_gpu(64, 0, [])
    assert O.t_decode(m, r1) == 0.0
    r2, c2 = O.one_gpu(0, 0, [5])
    assert O.t_prefill(m, r2, c2) == 0.0


def test_calibration_recovers_planted_factors_and_matches_a_brute_search():
    from scipy import optimize
    rng = np.random.default_rng(3)
    n = 40
    t_g = rng.uniform(0.1, 2.0, n)
    t_p = rng.uniform(0.0, 3.0, n)
    t_d = rng.uniform(0.0, 3.0, n)
    t_p[:5] = 0.0     # decode-only batches pin alpha
    t_d[5:10] = 0.0   # prefill-only batches pin beta
    alpha, beta = 1.37, 1.12
    meas = t_g + np.where(t_p * beta > t_d * alpha, t_p * beta, t_d * alpha)
    m, err = O.calibrate(O.LatencyModel(), t_g, t_p, t_d, meas, f_max=2.0, step=0.01)
    assert (m.alpha, m.beta) == (pytest.approx(alpha, abs=1e-12), pytest.approx(beta, abs=1e-12))
    assert err == pytest.approx(0.0, abs=1e-12)
    # noisy data: the grid search agrees with scipy's brute-force minimiser
    noisy = meas * rng.uniform(0.95, 1.05, n)
    m2, err2 = O.calibrate(O.LatencyModel(), t_g, t_p, t_d, noisy, f_max=2.0, step=0.05)

    def score(v):
        a, b = v
        pred = t_g + np.maximum(b * t_p, a * t_d)
        return float(np.mean(np.abs(pred - noisy) / noisy)) * 100

    grid = slice(1.0, 2.0 + 1e-9, 0.05)
    best = optimize.brute(score, (grid, grid), finish=None)
    assert score(best) == pytest.approx(err2, rel=1e-12)
    assert score((m2.alpha, m2.beta)) == pytest.approx(err2, rel=1e-12)


def test_factor_grid():
    g = O.factor_grid(3.0, 0.01)
    assert len(g) == 201 and g[0] == 1.0 and g[-1] == pytest.approx(3.0)
    assert list(O.factor_grid(1.0, 0.5)) == [1.0]


# --------------------------------------------------------- native vs oracle
@pytest.fixture(scope="module")
def cf():
    import co_prefill_decode_gb300 as cf
    from co_prefill_decode_gb300 import build
    build.build()
    return cf


def native_model(cf, m: O.LatencyModel):
    return cf.cf_latency_model(**m.__dict__)


def random_case(rng: random.Random):
    n_ranks = rng.choice([1, 1, 2, 4, 8])
    ranks = []
    for _ in range(n_ranks):
        nd = rng.choice([0, 1, rng.randint(1, 128)])
        ctx = tuple(rng.randint(1, 32768) for _ in range(nd))
        ranks.append(O.RankLoad(rng.choice([0, rng.randint(1, 8192)]), nd, ctx))
    chunks = [(rng.choice([0, rng.randint(1, 10240)]), rng.randint(0, 65536)) for _ in range(rng.randint(0, 4))]
    m = O.LatencyModel(gamma=rng.uniform(0, 1e-3), gamma0=rng.uniform(0, 0.2), a_d=rng.uniform(0, 1e-5),
                       a_d0=rng.uniform(0, 0.05), a_p=rng.uniform(0, 1e-7), a_p0=rng.uniform(0, 0.05),
                       a_comm=rng.uniform(0, 1e-4), a_comm0=rng.uniform(0, 0.05), alpha=rng.uniform(1, 2),
                       beta=rng.uniform(1, 2))
    return m, ranks, chunks


def test_native_prediction_matches_the_oracle(cf):
    rng = random.Random(11)
    for _ in range(500):
        m, ranks, chunks = random_case(rng)
        L = rng.choice([1, 32, 64])
        want = O.t_iter(m, ranks, chunks, L)
        got = cf.cf_latency_predict(native_model(cf, m),
                                    [(r.n_prefill, r.n_decode, float(sum(r.contexts))) for r in ranks], chunks, L)
        for k in ("t_iter", "t_gemm", "t_attn", "t_prefill", "t_decode"):
            assert got[k] == pytest.approx(want[k], rel=1e-12, abs=1e-15), k


def test_native_fit_and_calibration_match_the_oracle(cf):
    rng = np.random.default_rng(5)
    for n in (2, 5, 64):
        x = rng.uniform(0, 1e6, n)
        y = 1e-6 * x + 0.3 + rng.normal(0, 0.01, n)
        s, b = cf.cf_latency_fit_line(x, y)
        so, bo = O.fit_line(x, y)
        assert s == pytest.approx(so, rel=1e-9) and b == pytest.approx(bo, rel=1e-9, abs=1e-12)
    for trial in range(4):
        n = 30
        t_g = rng.uniform(0.1, 2.0, n)
        t_p = rng.uniform(0.0, 3.0, n)
        t_d = rng.uniform(0.0, 3.0, n)
        meas = (t_g + np.maximum(1.2 * t_p, 1.5 * t_d)) * rng.uniform(0.9, 1.1, n)
        mo, eo = O.calibrate(O.LatencyModel(), t_g, t_p, t_d, meas, f_max=2.5, step=0.01)
        mn = cf.cf_latency_model(gamma=7.0)
        en = cf.cf_latency_calibrate(mn, t_g, t_p, t_d, meas, f_max=2.5, step=0.01)
        assert (mn.alpha, mn.beta) == (mo.alpha, mo.beta)
        assert en == pytest.approx(eo, rel=1e-12)
        assert mn.gamma == 7.0   # other fields untouched


def test_native_estimator_rejects_bad_arguments(cf):
    m = cf.cf_latency_model(alpha=1.0, beta=1.0)
    with pytest.raises(cf.CfError):
        cf.cf_latency_predict(m, [], [])
    with pytest.raises(cf.CfError):
        cf.cf_latency_predict(m, [(-1, 0, 0.0)], [])
    with pytest.raises(cf.CfError):
        cf.cf_latency_predict(m, [(1, 0, 0.0)], [(-5, 0)])
    with pytest.raises(cf.CfError):
        cf.cf_latency_predict(cf.cf_latency_model(gamma=math.nan), [(1, 0, 0.0)], [])
    with pytest.raises(cf.CfError):
        cf.cf_latency_fit_line([1.0], [2.0])
    with pytest.raises(cf.CfError):
        cf.cf_latency_fit_line([3.0, 3.0], [1.0, 2.0])
    with pytest.raises(cf.CfError):
        cf.cf_latency_calibrate(m, [1.0], [1.0], [1.0], [0.0])
    with pytest.raises(cf.CfError):
        cf.cf_latency_calibrate(m, [1.0], [1.0], [1.0], [1.0], f_max=0.5)
    with pytest.raises(cf.CfError):
        cf.cf_latency_calibrate(m, [1.0], [1.0], [1.0], [1.0], step=0.0)
