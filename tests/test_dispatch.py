"""CPU tests of the waterfill prefill dispatcher (ConfluxServe §6.3, App. E
Algorithm 2).

The oracle (oracle/dispatch.py) is pinned by the worked example the
paper-daily.com summary of the paper prints (tests/golden/), by brute force
over every level and every split on tiny cases (the level is the largest
feasible one; the water-filled split minimises the largest load), and by
the single-GPU reduction (the dispatcher returns the largest chunk whose
estimated iteration fits the SLO).  The native dispatcher behind the C ABI is
then compared with the oracle on random multi-rank states.
"""
import itertools
import json
import os
import random

import pytest

from oracle import dispatch as D
from oracle import latency as L

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "waterfill_worked_example.json")


def state(n_decode, ctx=1000):
    return D.DecodeState(tuple(n_decode), tuple(tuple([ctx] * d) for d in n_decode))


def test_worked_example_from_the_pages():
    g = json.load(open(GOLDEN))
    # a latency model under which the SLO admits exactly 300 tokens per rank:
    # only the shared linear region costs, 1 unit per token (§6.2 Eq. 3, 7)
    m = L.LatencyModel(gamma=1.0)
    dec = state(g["n_decode"])
    tau = float(g["n_target"])
    r = D.waterfill(m, 1, tau, 1, dec, [0] * 4, [], None)
    assert r["n_target"] == g["n_target"] and r["budget"] == g["budget"]
    assert [g["n_target"] - d for d in g["n_decode"]] == g["capacity"]
    r = D.waterfill(m, 1, tau, 1, dec, [0] * 4, [], (g["request_remaining"], 0))
    assert r["chunk"] == g["chunk"] and r["assign"] == g["assign"]
    # the same with an alignment quantum that divides 300, and one that does not
    assert D.waterfill(m, 1, tau, 50, dec, [0] * 4, [], None)["n_target"] == 300
    r64 = D.waterfill(m, 1, tau, 64, dec, [0] * 4, [], None)
    assert r64["n_target"] == 256 and r64["budget"] == 216 + 246 + 246 + 256


def brute_assign(loads, tokens, n_target):
    """Every split of `tokens` within the level; the lexicographically
    smallest sorted-descending load vector is the water-filled one."""
    n = len(loads)
    cap = [max(0, n_target - x) for x in loads]
    best = None
    for give in itertools.product(*[range(c + 1) for c in cap]):
        if sum(give) != tokens:
            continue
        key = sorted((x + g for x, g in zip(loads, give)), reverse=True)
        if best is None or key < best[0]:
            best = (key, give)
    return best


def test_waterfill_assign_levels_the_loads():
    rng = random.Random(2)
    for _ in range(150):
        n = rng.randint(1, 4)
        loads = [rng.randint(0, 9) for _ in range(n)]
        n_target = rng.randint(0, 12)
        room = sum(max(0, n_target - x) for x in loads)
        tokens = rng.randint(0, room)
        give = D.waterfill_assign(loads, tokens, n_target)
        assert sum(give) == tokens
        assert all(0 <= g <= max(0, n_target - x) for g, x in zip(give, loads))
        key, _ = brute_assign(loads, tokens, n_target)
        assert sorted((x + g for x, g in zip(loads, give)), reverse=True) == key
        # ties: the extra token goes to the lowest rank index among equals
        final = [x + g for x, g in zip(loads, give)]
        for a in range(n):
            for b in range(a + 1, n):
                if loads[a] == loads[b] and give[a] < max(0, n_target - loads[a]):
                    assert give[a] >= give[b]
        assert max(final) <= max(max(loads), n_target)


def small_model(rng):
    return L.LatencyModel(gamma=rng.uniform(0.5, 2.0), gamma0=rng.uniform(0, 5), a_d=rng.uniform(0, 0.01),
                          a_d0=rng.uniform(0, 3), a_p=rng.uniform(0, 0.001), a_p0=rng.uniform(0, 3),
                          a_comm=rng.uniform(0, 0.5), a_comm0=rng.uniform(0, 2), alpha=rng.uniform(1, 1.5),
                          beta=rng.uniform(1, 1.5))


def random_state(rng, n):
    nd = [rng.randint(0, 12) for _ in range(n)]
    dec = D.DecodeState(tuple(nd), tuple(tuple(rng.randint(1, 300) for _ in range(d)) for d in nd))
    a_p = [rng.choice([0, rng.randint(0, 20)]) for _ in range(n)]
    chunks = [(rng.randint(1, 30), rng.randint(0, 200)) for _ in range(rng.randint(0, 2))]
    return dec, a_p, chunks


def t_of(m, L_, dec, a_p, chunks, give, req_chunk):
    ranks = [L.RankLoad(p + g, d, c) for p, g, d, c in zip(a_p, give, dec.n_decode, dec.contexts)]
    return L.t_iter(m, ranks, list(chunks) + ([req_chunk] if req_chunk and req_chunk[0] > 0 else []), L_)["t_iter"]


def test_level_is_the_largest_feasible_by_brute_force():
    rng = random.Random(4)
    for _ in range(120):
        n = rng.randint(1, 3)
        m = small_model(rng)
        dec, a_p, chunks = random_state(rng, n)
        q = rng.choice([1, 1, 4, 8])
        loads = [d + p for d, p in zip(dec.n_decode, a_p)]
        request = rng.choice([None, (rng.randint(1, 80), rng.randint(0, 300))])
        tau = rng.uniform(10, 250)
        r = D.waterfill(m, 1, tau, q, dec, a_p, chunks, request)
        # brute-force range: past the first infeasible level (the level's
        # latency grows at least with gamma > 0 per token)
        top = max(loads) + (request[0] if request else int(tau / m.gamma) + 1) + 2 * q

        def level_t(level):
            if request is None:
                give = [max(0, level - x) for x in loads]
                return t_of(m, 1, dec, a_p, chunks, give, None)
            budget = sum(max(0, level - x) for x in loads)
            li = min(request[0], budget)
            give = D.waterfill_assign(loads, li, level)
            return t_of(m, 1, dec, a_p, chunks, give, (li, request[1]))

        feas = [k for k in range(0, top // q + 1) if level_t(k * q) <= tau]
        if level_t(0) > tau:
            assert not r["feasible"] and r["budget"] == 0 and r["chunk"] == 0
            continue
        assert r["feasible"]
        # the estimator is monotone in the level, so feasible levels form a prefix
        assert feas == list(range(len(feas)))
        if request is None:
            assert r["n_target"] == feas[-1] * q
        else:
            # the search ends at the first level whose budget covers m_i
            assert r["n_target"] == min(feas[-1], -(-(max(loads) + request[0]) // q)) * q
            assert r["chunk"] == min(request[0], r["budget"])
            assert sum(r["assign"]) == r["chunk"]
        assert r["budget"] == sum(max(0, r["n_target"] - x) for x in loads)


def test_one_gpu_reduces_to_the_largest_chunk_within_the_slo():
    # on one rank the level is n_d + l: the chunk is the largest l whose
    # iteration (all layers) fits the SLO
    m = L.LatencyModel(gamma=2.5e-4, gamma0=0.08, a_d=5.4e-7, a_d0=0.06, a_p=1.4e-8, a_p0=0.1,
                       alpha=1.2, beta=1.085)
    ctx = (8192,) * 16
    dec = D.DecodeState((16,), (ctx,))
    for tau in (50.0, 100.0):
        r = D.waterfill(m, 32, tau, 1, dec, [0], [], (100000, 0))

        def t(l):
            ranks, chunks = L.one_gpu(l, 0, ctx)
            return L.t_iter(m, ranks, chunks, 32)["t_iter"]

        l = r["chunk"]
        assert t(l) <= tau < t(l + 1)
        assert r["n_target"] == 16 + l and r["assign"] == [l]


# --------------------------------------------------------- native vs oracle
@pytest.fixture(scope="module")
def cf():
    import co_prefill_decode_gb300 as cf
    from co_prefill_decode_gb300 import build
    build.build()
    return cf


def test_native_worked_example(cf):
    g = json.load(open(GOLDEN))
    m = cf.cf_latency_model(gamma=1.0, alpha=1.0, beta=1.0)
    r = cf.cf_waterfill_dispatch(m, 1, float(g["n_target"]), 1, g["n_decode"], [0.0] * 4, [0] * 4, [],
                                 (g["request_remaining"], 0))
    assert (r["n_target"], r["budget"], r["chunk"], r["assign"]) == (g["n_target"], g["budget"], g["chunk"],
                                                                     g["assign"])


def test_native_dispatch_matches_the_oracle(cf):
    rng = random.Random(9)
    for _ in range(300):
        n = rng.randint(1, 8)
        m = small_model(rng)
        dec, a_p, chunks = random_state(rng, n)
        q = rng.choice([1, 2, 16, 64])
        request = rng.choice([None, (rng.randint(0, 5000), rng.randint(0, 3000))])
        L_ = rng.choice([1, 4])
        tau = rng.uniform(5, 3000)
        want = D.waterfill(m, L_, tau, q, dec, a_p, chunks, request)
        got = cf.cf_waterfill_dispatch(cf.cf_latency_model(**m.__dict__), L_, tau, q, list(dec.n_decode),
                                       [float(sum(c)) for c in dec.contexts], a_p, chunks, request)
        for k in ("n_target", "budget", "chunk", "feasible", "assign"):
            assert got[k] == want[k], (k, got, want)
    for _ in range(300):
        n = rng.randint(1, 8)
        loads = [rng.randint(0, 500) for _ in range(n)]
        n_target = rng.randint(0, 700)
        tokens = rng.randint(0, sum(max(0, n_target - x) for x in loads))
        assert cf.cf_waterfill_assign(loads, tokens, n_target) == D.waterfill_assign(loads, tokens, n_target)


def test_native_dispatch_rejects_bad_arguments(cf):
    m = cf.cf_latency_model(gamma=1.0, alpha=1.0, beta=1.0)
    with pytest.raises(cf.CfError):
        cf.cf_waterfill_dispatch(m, 1, 10.0, 0, [1], [1.0], [0])
    with pytest.raises(cf.CfError):
        cf.cf_waterfill_dispatch(m, 1, 10.0, 1, [], [], [])
    with pytest.raises(cf.CfError):
        cf.cf_waterfill_dispatch(m, 1, 10.0, 1, [-1], [1.0], [0])
    with pytest.raises(cf.CfError):
        cf.cf_waterfill_assign([0, 0], 5, 2)
    with pytest.raises(cf.CfError):
        cf.cf_waterfill_assign([0, -1], 0, 2)
