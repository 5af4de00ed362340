"""Pins for the fp64 oracle: each check compares it with something other than
itself — brute force, closed forms, library routines, invariants.

Page references: ConfluxServe (co-batched layer, Fig. 1, Fig. 7, §4, App. D
Eq. 9), Adaptive Context Parallelism (§2.1 causal attention, §2.2 Eq. 1),
Decode Token Parallelism (§4.3 RoPE -> append -> attention, §4.4 Eq. 1).
"""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
import workload as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ bf16
def test_bf16_round_matches_torch_rne():
    g = torch.Generator().manual_seed(1)
    a = torch.randn(200_000, generator=g, dtype=torch.float32) * torch.exp(
        torch.randn(200_000, generator=g) * 6)
    ref = a.to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_round(a.to(torch.float64).numpy())
    assert np.array_equal(got, ref)


def test_bf16_round_ties_to_even_and_edges():
    # exact halfway cases between bf16 neighbours (1 + k/128 grid)
    base = 1.0 + np.arange(0, 128) / 128.0
    half = base + 1.0 / 256.0
    got = oracle.bf16_round(half)
    k = np.arange(128)
    want = np.where(k % 2 == 0, base, base + 1.0 / 128.0)
    want[-1] = 2.0  # 1 + 127/128 is odd -> rounds up to 2
    assert np.array_equal(got, want)
    assert oracle.bf16_round(np.array([0.0]))[0] == 0.0
    # near the top of the range: compare with torch's float32 -> bfloat16 (RNE)
    edge = torch.tensor([3.0e38, 3.3895e38, 3.3961e38, 3.4e38, -3.39e38], dtype=torch.float32)
    want = edge.to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_round(edge.to(torch.float64).numpy())
    assert np.array_equal(got, want) and np.isinf(got[3])
    tiny = np.array([2.0 ** -130 + 2.0 ** -140])     # subnormal range: spacing 2^-133
    assert oracle.bf16_round(tiny)[0] == 2.0 ** -130
    t = torch.tensor([2.0 ** -130 + 2.0 ** -140], dtype=torch.float32).to(torch.bfloat16)
    assert float(t.to(torch.float64)) == 2.0 ** -130


# ------------------------------------------------------------------ rmsnorm
def test_rmsnorm_unit_gain_has_unit_rms():
    x = np.random.default_rng(0).normal(size=(7, 256)) * 3.0
    y = oracle.rmsnorm(x, np.ones(256), 0.0)
    assert np.allclose(np.sqrt((y * y).mean(-1)), 1.0, rtol=0, atol=1e-13)


def test_rmsnorm_closed_form_and_gain_index():
    c, eps, H = 2.5, 1e-5, 8
    x = np.full((1, H), c)
    g = np.arange(1, H + 1, dtype=np.float64)
    y = oracle.rmsnorm(x, g, eps)
    assert np.allclose(y[0], c / math.sqrt(c * c + eps) * g, rtol=1e-15)
    # one-hot input: only that index survives, scaled by its own gain
    x = np.zeros((1, H)); x[0, 3] = 1.0
    y = oracle.rmsnorm(x, g, 0.0)
    assert np.allclose(y[0], np.eye(H)[3] * math.sqrt(H) * g[3])


# ------------------------------------------------------------------ rope
def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).normal(size=(3, 2, 64))
    assert np.array_equal(oracle.rope(x, np.zeros(3), 1e4), x)


def test_rope_closed_form_rotate_half_pairing():
    d, theta = 8, 10000.0
    for i in range(d // 2):
        e = np.zeros((1, 1, d)); e[0, 0, i] = 1.0
        for p in (1, 7, 1000):
            a = p * theta ** (-2.0 * i / d)
            y = oracle.rope(e, np.array([p]), theta)[0, 0]
            want = np.zeros(d); want[i] = math.cos(a); want[i + d // 2] = math.sin(a)
            assert np.allclose(y, want, atol=1e-12)
        e = np.zeros((1, 1, d)); e[0, 0, i + d // 2] = 1.0
        y = oracle.rope(e, np.array([3]), theta)[0, 0]
        a = 3 * theta ** (-2.0 * i / d)
        want = np.zeros(d); want[i] = -math.sin(a); want[i + d // 2] = math.cos(a)
        assert np.allclose(y, want, atol=1e-12)


def test_rope_relative_position_and_norm():
    rng = np.random.default_rng(2)
    q = rng.normal(size=(1, 1, 128)); k = rng.normal(size=(1, 1, 128))
    dots = []
    for m, n in ((5, 2), (103, 100), (40003, 40000)):
        qm = oracle.rope(q, np.array([m]), 5e5); kn = oracle.rope(k, np.array([n]), 5e5)
        dots.append(float((qm * kn).sum()))
        assert np.isclose(np.linalg.norm(qm), np.linalg.norm(q), rtol=1e-13)
    assert np.allclose(dots, dots[0], rtol=1e-9)


# ------------------------------------------------------------------ silu
def test_silu_against_expit():
    z = np.linspace(-30, 30, 1001)
    assert np.allclose(oracle.silu(z), z * expit(z), rtol=1e-14, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert np.allclose(oracle.swiglu(np.array([2.0]), np.array([3.0])), 3 * 2 * expit(2.0))


# ------------------------------------------------------------------ attention
def brute_attention(q, K, V, qpos):
    """Per-query, per-head Python loops with math.exp (no numpy reductions)."""
    nq, Hq, d = q.shape
    G = Hq // K.shape[1]
    out = np.zeros_like(q)
    for r in range(nq):
        for h in range(Hq):
            kv = h // G
            logits = []
            for j in range(int(qpos[r]) + 1):
                logits.append(sum(float(q[r, h, t]) * float(K[j, kv, t]) for t in range(d)) / math.sqrt(d))
            m = max(logits)
            w = [math.exp(s - m) for s in logits]
            z = sum(w)
            for t in range(d):
                out[r, h, t] = sum(w[j] * float(V[j, kv, t]) for j in range(len(w))) / z
    return out


def test_attention_matches_brute_force_gqa_causal():
    rng = np.random.default_rng(3)
    n, Hq, Hkv, d = 21, 4, 2, 8
    K = rng.normal(size=(n, Hkv, d)); V = rng.normal(size=(n, Hkv, d))
    q = rng.normal(size=(5, Hq, d)) * 2
    qpos = np.array([0, 3, 10, 19, 20])
    got = oracle.attention(q, K, V, qpos, block=2)
    want = brute_attention(q, K, V, qpos)
    assert np.allclose(got, want, rtol=0, atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(4)
    K = rng.normal(size=(9, 1, 4)); V = rng.normal(size=(9, 1, 4))
    # q = 0: uniform weights -> mean of the visible values
    out = oracle.attention(np.zeros((1, 1, 4)), K, V, np.array([5]))
    assert np.allclose(out[0, 0], V[:6, 0].mean(0), atol=1e-14)
    # one visible key -> its value
    out = oracle.attention(rng.normal(size=(1, 1, 4)), K, V, np.array([0]))
    assert np.allclose(out[0, 0], V[0, 0], atol=1e-15)
    # one dominant logit -> that value row
    Kd = np.zeros((9, 1, 4)); Kd[4, 0, 0] = 1.0
    out = oracle.attention(np.array([[[1e4, 0, 0, 0]]]), Kd, V, np.array([8]))
    assert np.allclose(out[0, 0], V[4, 0], atol=1e-12)


def test_attention_gqa_groups_are_contiguous():
    # KV head 0 values are -5, KV head 1 values are +5: with G = 2 query heads
    # 0,1 must read head 0 and 2,3 head 1.
    n, d = 6, 4
    K = np.random.default_rng(5).normal(size=(n, 2, d))
    V = np.stack([np.full((n, d), -5.0), np.full((n, d), 5.0)], axis=1)
    q = np.random.default_rng(6).normal(size=(1, 4, d))
    out = oracle.attention(q, K, V, np.array([n - 1]))
    assert np.allclose(out[0, :2], -5.0) and np.allclose(out[0, 2:], 5.0)


def test_attention_mask_hides_future_keys():
    n, d = 8, 4
    K = np.zeros((n, 1, d)); V = np.zeros((n, 1, d)); V[5:] = 1e6
    out = oracle.attention(np.ones((3, 1, d)), K, V, np.array([0, 2, 4]))
    assert np.abs(out).max() == 0.0


def test_chunk_workload_brute_force():
    for R, P in ((1, 0), (5, 0), (64, 128), (17, 33), (3, 1000)):
        count = sum(1 for i in range(R) for j in range(P + R) if j <= P + i)
        assert oracle.chunk_workload(R, P) == count


# ------------------------------------------------------------------ paging
def test_slot_and_gather_match_contiguous_cache():
    rng = np.random.default_rng(7)
    ps, Hkv, d, n = 16, 3, 8, 83
    npg = (n + ps - 1) // ps
    pages = rng.permutation(np.arange(11))[:npg]
    pool = np.full((11, Hkv, ps, d), np.nan)
    contiguous = rng.normal(size=(n, Hkv, d))
    for p in range(n):                             # brute-force placement
        page, off = pages[p // ps], p % ps
        pool[page, :, off, :] = contiguous[p]
        assert oracle.slot_of(pages, p, ps) == page * ps + off
    got = oracle.gather_request_kv(pool, pages, n, ps)
    assert np.array_equal(got, contiguous)
    # append then gather sees the new rows; other slots untouched
    k = rng.normal(size=(2, Hkv, d)); v = rng.normal(size=(2, Hkv, d))
    pool_v = pool.copy()
    before = pool.copy()
    slots = oracle.slot_of(np.concatenate([pages, [10]]), np.array([n, n + 1]), ps)
    oracle.kv_append(pool, pool_v, k, v, slots, ps)
    full = np.concatenate([pages, [10]]) if (n + 1) // ps >= npg else pages
    g2 = oracle.gather_request_kv(pool, full, n + 2, ps)
    assert np.array_equal(g2[:n], contiguous) and np.array_equal(g2[n:], k)
    changed = ~np.isclose(np.nan_to_num(pool, nan=-99), np.nan_to_num(before, nan=-99))
    assert changed.sum() == 2 * Hkv * d


# several prefill chunks of different requests in one step (ConfluxServe
# §6.2 Eq. 6: the scheduled prefill batch P), plus decodes
TINY_MC = wl.Workload("tiny-mc", wl.TINY, 3, (5, 40, 200), 64, 128,
                      more_chunks=((37, 0), (130, 300), (1, 17)), description="tiny, four chunks")


def test_workload_pages_cover_each_request_once():
    for name in ("tiny", "mix", "mchunk"):
        w = wl.WORKLOADS[name]
        b = wl.make_batch(w)
        used = []
        for l, c, p in b.chunks:
            assert len(p) == (l + c + 15) // 16
            used += list(p)
        for j in range(b.n_decode):
            npg = (int(b.dec_ctx[j]) + 1 + 15) // 16
            assert (b.dec_pages[j, :npg] >= 0).all() and (b.dec_pages[j, npg:] == -1).all()
            used += list(b.dec_pages[j, :npg])
        assert len(used) == len(set(used)) and max(used) < b.num_pages


def test_pool_generation_places_tokens_by_page_table():
    w = wl.WORKLOADS["tiny"]
    b = wl.make_batch(w)
    kp, vp = wl.make_pools(w, b)
    # a request's cached KV is drawn position-major, independent of paging:
    # gathering through the table must give finite values for cached slots and
    # NaN for the slot the new token will take.
    for j in range(b.n_decode):
        c = int(b.dec_ctx[j])
        Kg = oracle.gather_request_kv(kp, b.dec_pages[j], c + 1, 16)
        assert np.isfinite(Kg[:c]).all() and np.isnan(Kg[c]).all()
    Kp = oracle.gather_request_kv(kp, b.pre_pages, b.prefill_prefix + b.prefill_len, 16)
    assert np.isfinite(Kp[:b.prefill_prefix]).all() and np.isnan(Kp[b.prefill_prefix:]).all()
    b = wl.make_batch(TINY_MC)
    kp, vp = wl.make_pools(TINY_MC, b)
    for l, c, p in b.chunks:
        Kp = oracle.gather_request_kv(kp, p, c + l, 16)
        assert np.isfinite(Kp[:c]).all() and np.isnan(Kp[c:]).all()


def test_extra_chunks_leave_the_first_requests_draws_unchanged():
    # the extra chunks' prefixes are drawn after every other request, so a
    # one-chunk batch's cached KV, pages and x rows do not move
    one = wl.Workload("one", wl.TINY, 3, (5, 40, 200), 64, 128)
    b1, bm = wl.make_batch(one), wl.make_batch(TINY_MC)
    assert np.array_equal(b1.dec_ctx, bm.dec_ctx)
    k1, _ = wl.make_pools(one, b1)
    km, _ = wl.make_pools(TINY_MC, bm)
    for j in range(b1.n_decode):
        c = int(b1.dec_ctx[j])
        assert torch.equal(torch.as_tensor(oracle.gather_request_kv(k1, b1.dec_pages[j], c, 16)),
                           torch.as_tensor(oracle.gather_request_kv(km, bm.dec_pages[j], c, 16)))


# ------------------------------------------------------------------ layer
def _tiny(seed=0, unit=False, **kw):
    w = wl.WORKLOADS["tiny"]
    if kw:
        w = wl.reduced(w, kw.get("dec", w.dec_ctx), kw.get("l", w.prefill_len), kw.get("cp", w.prefill_prefix))
    b = wl.make_batch(w, seed)
    x = oracle.to_f64(wl.make_x(w, b, seed))
    W = oracle.LayerWeights64.from_torch(wl.make_weights(w, seed, unit_gains=unit))
    kp, vp = wl.make_pools(w, b, seed)
    return w, b, x, W, oracle.to_f64(kp), oracle.to_f64(vp)


def test_layer_with_zero_projections_is_identity():
    w, b, x, W, kp, vp = _tiny()
    W.w_o[:] = 0.0
    W.w_down[:] = 0.0
    r = oracle.layer_step(x, W, w.shape, b, kp, vp)
    assert np.array_equal(r["out"], x)      # bf16 inputs round to themselves
    assert np.array_equal(r["h"], x)


def test_layer_rows_subset_matches_full():
    w, b, x, W, kp, vp = _tiny()
    full = oracle.layer_step(x, W, w.shape, b, kp, vp)
    rows = [0, 5, 63, 64, 67]
    sub = oracle.layer_step(x, W, w.shape, b, kp, vp, rows=rows)
    for key in ("out", "q", "k", "v", "attn", "h", "slots"):
        assert np.array_equal(sub[key], full[key][rows]), key


def test_layer_cobatched_rows_equal_separate_rows():
    """ConfluxServe §4: co-batching needs only shared weights and feature dim."""
    w, b, x, W, kp, vp = _tiny()
    full = oracle.layer_step(x, W, w.shape, b, kp, vp)
    l = b.prefill_len
    b_pre = wl.Batch(w, b.dec_ctx[:0], l, b.prefill_prefix, b.dec_pages[:0], b.pre_pages, b.num_pages)
    b_dec = wl.Batch(w, b.dec_ctx, 0, 0, b.dec_pages, b.pre_pages[:0], b.num_pages)
    pre = oracle.layer_step(x[:l], W, w.shape, b_pre, kp, vp)
    dec = oracle.layer_step(x[l:], W, w.shape, b_dec, kp, vp)
    assert np.allclose(full["out"][:l], pre["out"], rtol=0, atol=0)
    assert np.allclose(full["out"][l:], dec["out"], rtol=0, atol=0)


def test_multi_chunk_rows_equal_each_chunk_alone():
    """Each chunk of a multi-chunk step (ConfluxServe §6.2 Eq. 6: several
    requests' chunks in one iteration) computes exactly what it computes as
    the only chunk of a step: same positions, own prefix, own pages; and the
    decode rows are unaffected."""
    w = TINY_MC
    b = wl.make_batch(w)
    x = oracle.to_f64(wl.make_x(w, b))
    W = oracle.LayerWeights64.from_torch(wl.make_weights(w))
    kp, vp = (oracle.to_f64(t) for t in wl.make_pools(w, b))
    full = oracle.layer_step(x, W, w.shape, b, kp, vp)
    assert full["out"].shape[0] == 64 + 37 + 130 + 1 + 3
    r0 = 0
    for l, c, p in b.chunks:
        alone = wl.Batch(w, b.dec_ctx[:0], l, c, b.dec_pages[:0], p, b.num_pages)
        r = oracle.layer_step(x[r0:r0 + l], W, w.shape, alone, kp, vp)
        for key in ("out", "q", "k", "v", "attn", "slots"):
            assert np.array_equal(full[key][r0:r0 + l], r[key]), key
        # slot of chunk row i: position c + i through the chunk's own table
        pos = c + np.arange(l)
        assert np.array_equal(full["slots"][r0:r0 + l], p[pos // 16].astype(np.int64) * 16 + pos % 16)
        r0 += l
    dec = wl.Batch(w, b.dec_ctx, 0, 0, b.dec_pages, b.pre_pages[:0], b.num_pages)
    r = oracle.layer_step(x[r0:], W, w.shape, dec, kp, vp)
    assert np.array_equal(full["out"][r0:], r["out"])
    # a row subset spanning several chunks matches the full step
    rows = [0, 63, 64, 100, 101, 230, 231, 232, 234]
    sub = oracle.layer_step(x, W, w.shape, b, kp, vp, rows=rows)
    for key in ("out", "attn", "slots"):
        assert np.array_equal(sub[key], full[key][rows]), key


def _append_rows(r, b, kp, vp):
    kp, vp = kp.copy(), vp.copy()
    oracle.kv_append(kp, vp, r["k"], r["v"], r["slots"], b.page_size)
    return kp, vp


def test_chunked_prefill_equals_one_shot():
    """Adaptive Context Parallelism §2.1: split execution equals single-rank causal attention."""
    w, b, x, W, kp, vp = _tiny()
    l, cp = b.prefill_len, b.prefill_prefix
    one = wl.Batch(w, b.dec_ctx[:0], l, cp, b.dec_pages[:0], b.pre_pages, b.num_pages)
    ref = oracle.layer_step(x[:l], W, w.shape, one, kp, vp)
    c1 = 16
    b1 = wl.Batch(w, b.dec_ctx[:0], c1, cp, b.dec_pages[:0], b.pre_pages, b.num_pages)
    r1 = oracle.layer_step(x[:c1], W, w.shape, b1, kp, vp)
    kp2, vp2 = _append_rows(r1, b1, kp, vp)
    b2 = wl.Batch(w, b.dec_ctx[:0], l - c1, cp + c1, b.dec_pages[:0], b.pre_pages, b.num_pages)
    r2 = oracle.layer_step(x[c1:l], W, w.shape, b2, kp2, vp2)
    assert np.allclose(np.concatenate([r1["out"], r2["out"]]), ref["out"], rtol=0, atol=1e-12)
    assert np.array_equal(np.concatenate([r1["k"], r2["k"]]), ref["k"])


def test_decode_row_equals_last_prefill_row():
    """A decode token's output equals the matching row of causal prefill."""
    w, b, x, W, kp, vp = _tiny()
    cp, l = b.prefill_prefix, b.prefill_len
    # prefill the first l-1 chunk tokens, then decode the last one
    b1 = wl.Batch(w, b.dec_ctx[:0], l - 1, cp, b.dec_pages[:0], b.pre_pages, b.num_pages)
    r1 = oracle.layer_step(x[:l - 1], W, w.shape, b1, kp, vp)
    kp2, vp2 = _append_rows(r1, b1, kp, vp)
    stride = b.dec_pages.shape[1]
    table = np.full((1, max(stride, len(b.pre_pages))), -1, np.int32)
    table[0, :len(b.pre_pages)] = b.pre_pages
    bd = wl.Batch(w, np.array([cp + l - 1], np.int32), 0, 0, table, b.pre_pages[:0], b.num_pages)
    rd = oracle.layer_step(x[l - 1:l], W, w.shape, bd, kp2, vp2)
    one = wl.Batch(w, b.dec_ctx[:0], l, cp, b.dec_pages[:0], b.pre_pages, b.num_pages)
    ref = oracle.layer_step(x[:l], W, w.shape, one, kp, vp)
    assert np.allclose(rd["out"][0], ref["out"][l - 1], rtol=0, atol=1e-12)
    assert rd["slots"][0] == ref["slots"][l - 1]


def test_decode_with_empty_context_returns_its_own_value():
    """A decode with c_j = 0 attends only to the key it appends (RoPE -> append -> attention)."""
    w, b, x, W, kp, vp = _tiny(dec=(0, 5), l=0, cp=0)
    r = oracle.layer_step(x, W, w.shape, b, kp, vp)
    G = w.shape.group
    for h in range(w.shape.n_q_heads):
        assert np.array_equal(r["attn"][0, h], oracle.bf16_round(r["v"][0, h // G]))


def test_layer_golden_tiny():
    """Regression pin: values written by tests/golden/make_golden.py (oracle only)."""
    path = os.path.join(GOLDEN, "tiny_layer_out.txt")
    rows, cols, vals = [], [], []
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            r, c, v = line.split()
            rows.append(int(r)); cols.append(int(c)); vals.append(float.fromhex(v))
    w, b, x, W, kp, vp = _tiny()
    out = oracle.layer_step(x, W, w.shape, b, kp, vp)["out"]
    assert np.array_equal(out[rows, cols], np.array(vals))


def test_qk_norm_is_per_head_over_head_dim():
    """Per-head QK-RMSNorm (Qwen3 shape): at position 0 RoPE is the identity, so
    with unit gains every (row, head) vector of q and k has unit rms up to bf16
    rounding, while a norm over the whole row would not."""
    base = wl.WORKLOADS["q14b"]
    w = wl.reduced(base, (3,), 2, 0)
    b = wl.make_batch(w)
    x = oracle.to_f64(wl.make_x(w, b))
    W = oracle.LayerWeights64.from_torch(wl.make_weights(w, unit_gains=True))
    kp, vp = wl.make_pools(w, b)
    r = oracle.layer_step(x, W, w.shape, b, kp, vp, rows=[0])
    for t in (r["q"][0], r["k"][0]):
        rms = np.sqrt((t * t).mean(-1))
        assert np.allclose(rms, 1.0, atol=4e-3)


def test_oracle_chain_sensitivity(monkeypatch):
    """How far two correct bf16-boundary implementations of the layer can drift
    apart when compared end to end: perturbing only the attention output by a
    relative 2^-17 (far below one bf16 ulp) moves the final output by up to
    ~1e-2 of max(1, |ref|), because each later bf16 rounding turns the
    difference into ulp flips that the FFN amplifies.  This is why the GPU
    layer is gated stage by stage and the chained comparison gets a wider
    bound (tests/test_gpu_layer.py)."""
    from oracle import layer as L
    w = wl.reduced(wl.WORKLOADS["l8b"], (5, 300, 17, 1), 130, 0)
    b = wl.make_batch(w)
    x = oracle.to_f64(wl.make_x(w, b))
    W = oracle.LayerWeights64.from_torch(wl.make_weights(w))
    kp, vp = wl.make_pools(w, b)
    kp, vp = oracle.to_f64(kp), oracle.to_f64(vp)
    ref = L.layer_step(x, W, w.shape, b, kp, vp)
    orig = L.attention
    rng = np.random.default_rng(0)

    def perturbed(*a, **k):
        o = orig(*a, **k)
        return o * (1.0 + rng.uniform(-1, 1, o.shape) * 2.0 ** -17)

    monkeypatch.setattr(L, "attention", perturbed)
    got = L.layer_step(x, W, w.shape, b, kp, vp)
    e = np.abs(got["out"] - ref["out"]) / np.maximum(1.0, np.abs(ref["out"]))
    assert 2e-3 < e.max() < 0.1 and e.mean() < 1e-2



# ------------------------------------------------------------------ attention over paged caches
def _place_requests(rng, n_keys, Hkv, d, ps, spare_pages=3):
    """Contiguous per-request caches [n, Hkv, d] and the same values placed
    token by token (brute force) through shuffled page tables into NaN-filled
    pools [num_pages, Hkv, ps, d]; slots no request owns stay NaN, so a
    gather that reads one key too many poisons the result."""
    need = [(n + ps - 1) // ps for n in n_keys]
    num_pages = sum(need) + spare_pages
    perm = rng.permutation(num_pages)
    stride = max(need + [1])
    tables = np.full((len(n_keys), stride), -1, np.int64)
    kpool = np.full((num_pages, Hkv, ps, d), np.nan)
    vpool = np.full((num_pages, Hkv, ps, d), np.nan)
    Ks, Vs, at = [], [], 0
    for j, n in enumerate(n_keys):
        tables[j, :need[j]] = perm[at:at + need[j]]
        at += need[j]
        K = rng.normal(size=(n, Hkv, d))
        V = rng.normal(size=(n, Hkv, d))
        for p in range(n):
            page, off = tables[j, p // ps], p % ps
            kpool[page, :, off, :] = K[p]
            vpool[page, :, off, :] = V[p]
        Ks.append(K)
        Vs.append(V)
    return Ks, Vs, kpool, vpool, tables


def test_decode_attention_equals_brute_force_over_placed_cache():
    """oracle.decode_attention (request j's single query at position n_j - 1
    over its n_j keys, read through its page table) equals brute-force
    attention over the contiguous cache.  Tiny-layer sizes (4/2 heads, d 64,
    page 16); key counts cover one key (c = 0), a page-crossing context
    (17 = one page + 1), a context ending exactly on a page (64), the next
    page's first slot (65) and a full 16-page request (256)."""
    rng = np.random.default_rng(11)
    Hq, Hkv, d, ps = 4, 2, 64, 16
    n_keys = [1, 17, 64, 65, 100, 256]
    Ks, Vs, kpool, vpool, tables = _place_requests(rng, n_keys, Hkv, d, ps)
    q = rng.normal(size=(len(n_keys), Hq, d))
    got = oracle.decode_attention(q, kpool, vpool, np.array(n_keys), tables, ps)
    assert np.isfinite(got).all()
    for j, n in enumerate(n_keys):
        want = brute_attention(q[j:j + 1], Ks[j], Vs[j], [n - 1])
        assert np.allclose(got[j:j + 1], want, rtol=0, atol=1e-12), j
    # one key: the output is that key's value row, for every query head
    G = Hq // Hkv
    for h in range(Hq):
        assert np.array_equal(got[0, h], Vs[0][0, h // G])


def test_prefill_attention_equals_brute_force_over_placed_cache():
    """oracle.prefill_attention: chunk query i at position prefix + i sees
    keys 0..prefix + i of its request, read through the page table.  The
    tiny layer's own chunk (64 on a 128-token prefix) and chunks whose prefix
    or end is not page-aligned, with no prefix, and of one token."""
    rng = np.random.default_rng(12)
    Hq, Hkv, d, ps = 4, 2, 64, 16
    for prefix, l in ((128, 64), (37, 11), (0, 20), (16, 16), (250, 1)):
        (K,), (V,), kpool, vpool, tables = _place_requests(rng, [prefix + l], Hkv, d, ps)
        q = rng.normal(size=(l, Hq, d))
        got = oracle.prefill_attention(q, kpool, vpool, prefix, tables[0], ps)
        want = brute_attention(q, K, V, prefix + np.arange(l))
        assert np.isfinite(got).all()
        assert np.allclose(got, want, rtol=0, atol=1e-12), (prefix, l)


# ------------------------------------------------------------------ layer wiring
# A layer shape whose projections are not square: Hq d = 512 != H = 256 and
# F = 512 != H, so a transposed W_o or W_down either fails to multiply or
# moves a one-hot entry to another index.
NONSQUARE = wl.LayerShape(256, 8, 2, 64, 512, 1.0e4, 1e-5, False)
NONSQUARE_W = wl.Workload("nonsquare", NONSQUARE, 2, (5, 40), 24, 16, description="non-square projections")


def _nonsquare(constant_x=None):
    w = NONSQUARE_W
    b = wl.make_batch(w)
    x = oracle.to_f64(wl.make_x(w, b))
    if constant_x is not None:
        x[:] = constant_x
    W = oracle.LayerWeights64.from_torch(wl.make_weights(w, unit_gains=True))
    kp, vp = (oracle.to_f64(t) for t in wl.make_pools(w, b))
    return w, b, x, W, kp, vp


def test_oproj_orientation_on_a_non_square_layer():
    """h = x + O_cat W_o^T with W_o in nn.Linear layout [H][Hq d]: a one-hot
    W_o[i, j] adds attention feature j (head j // d, dim j % d) to hidden
    feature i of every row and leaves every other feature of h equal to x.
    j >= H, so W_o used untransposed cannot reach it."""
    w, b, x, W, kp, vp = _nonsquare()
    d = NONSQUARE.head_dim
    i, j = 5, 300
    W.w_o[:] = 0.0
    W.w_o[i, j] = 1.0
    r = oracle.layer_step(x, W, w.shape, b, kp, vp)
    a = r["attn"][:, j // d, j % d]
    assert np.abs(a).max() > 0.1
    assert np.allclose(r["h"][:, i] - x[:, i], a, rtol=0, atol=1e-12)
    others = np.arange(NONSQUARE.hidden) != i
    assert np.array_equal(r["h"][:, others], x[:, others])


def test_ffn_gate_and_up_roles_closed_form():
    """out = h + (silu(hn W_gate^T) * (hn W_up^T)) W_down^T with the roles
    fixed: with W_o = 0 (h = x), constant rows x = 1 and unit gains, hn is
    exactly 1; a gate row of a / H and an up row of b / H then give gate
    a and up b on unit f, whose activation silu(a) b reaches hidden feature
    i through W_down[i, f] = 1 (nn.Linear layout [H][F], f >= H).  With
    a = -8, b = 4 the activation is silu(-8) 4 ~ -0.011; swapping the roles
    would give silu(4) (-8) ~ -31."""
    w, b, x, W, kp, vp = _nonsquare(constant_x=1.0)
    H, F = NONSQUARE.hidden, NONSQUARE.ffn_dim
    f, i, a, bb = 300, 7, -8.0, 4.0
    W.w_o[:] = 0.0
    W.w_gate[:] = 0.0
    W.w_up[:] = 0.0
    W.w_down[:] = 0.0
    W.w_gate[f, :] = a / H
    W.w_up[f, :] = bb / H
    W.w_down[i, f] = 1.0
    r = oracle.layer_step(x, W, w.shape, b, kp, vp)
    assert np.array_equal(r["hn"], np.ones_like(r["hn"]))
    act = float(oracle.bf16_round(np.array([a * expit(a) * bb]))[0])
    assert abs(act + 0.0107) < 1e-3
    want = np.zeros_like(r["act"])
    want[:, f] = act
    assert np.array_equal(r["act"], want)
    out_i = float(oracle.bf16_round(np.array([1.0 + act]))[0])
    assert np.array_equal(r["out"][:, i], np.full(r["out"].shape[0], out_i))
    others = np.arange(H) != i
    assert np.array_equal(r["out"][:, others], x[:, others])


def test_qkv_split_order_q_then_k_then_v():
    """The fused projection's rows are the Q heads, then the K heads, then the
    V heads (Decode Token Parallelism §4.4, Eq. 1).  With constant rows x = 1
    and unit gains xn is exactly 1, so a W_qkv that is zero except row t
    (value v / H) makes output feature t equal v and every other zero; at
    position 0 (the first row of a chunk with no prefix) RoPE is the
    identity, so exactly one element of q, k or v is non-zero, at the head
    and dimension that row t names."""
    s = NONSQUARE
    w = wl.Workload("nonsquare-p0", s, 0, (), 8, 0)
    b = wl.make_batch(w)
    x = np.ones((b.n_tokens, s.hidden))
    W = oracle.LayerWeights64.from_torch(wl.make_weights(w, unit_gains=True))
    kp, vp = (oracle.to_f64(t) for t in wl.make_pools(w, b))
    Hq, Hkv, d, H = s.n_q_heads, s.n_kv_heads, s.head_dim, s.hidden
    cases = [("q", 3 * d + 5, (3, 5)), ("k", Hq * d + 1 * d + 7, (1, 7)), ("v", (Hq + Hkv) * d + 9, (0, 9)),
             ("v", (Hq + Hkv) * d + d + 63, (1, 63))]
    for name, t, (head, dim) in cases:
        W.w_qkv[:] = 0.0
        W.w_qkv[t, :] = 2.0 / H
        r = oracle.layer_step(x, W, w.shape, b, kp, vp, rows=[0])
        for key in ("q", "k", "v"):
            want = np.zeros_like(r[key][0])
            if key == name:
                want[head, dim] = 2.0
            assert np.array_equal(r[key][0], want), (name, key)
