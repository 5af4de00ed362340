"""GPU parity of the co-batched layer step against the fp64 oracle.

Three kinds of checks:

* stage-isolated parity (the gate): every stage of the layer runs through
  the C ABI on the oracle's own bf16 inputs for that stage, and its output is
  compared element by element with the oracle's output of the same stage, at
  the layer tolerance (max e <= 2e-2, mean e <= 2e-3 with e = |gpu - ref| /
  max(1, |ref|));
* composition: cf_layer_step runs exactly those stage kernels — its
  intermediate tensors equal the stage calls chained on the GPU bit for bit;
* chained parity: cf_layer_step end to end against the oracle, with the
  wider bound that the oracle's own sensitivity to last-bit differences
  implies (each bf16 rounding between stages turns a last-bit difference
  into an ulp flip that the random-weight FFN amplifies; see
  tests/test_oracle.py::test_oracle_chain_sensitivity).
"""
import numpy as np
import pytest
import torch

import oracle
import workload as wl
from helpers import TOL_MAX, TOL_MEAN, LayerSetup, assert_close, errors, f64

pytestmark = pytest.mark.gpu

# chained bound: 5x the stage tolerance (the oracle itself moves `out` by up to
# ~0.025 when one stage is perturbed by 2^-17 relative)
CHAIN_MAX, CHAIN_MEAN = 0.1, 1e-2


@pytest.fixture(scope="module")
def cf():
    import co_prefill_decode_gb300 as cf
    cf.load_library()
    return cf


def bf16_dev(a):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=torch.float64).to(torch.bfloat16).cuda()


def slots_of_rows(b, rows):
    out = []
    P = b.prefill_rows
    for r in rows:
        if r < P:
            r0 = 0
            for l, c, pages in b.chunks:
                if r < r0 + l:
                    out.append(int(oracle.slot_of(pages, c + r - r0, 16)))
                    break
                r0 += l
        else:
            j = r - P
            out.append(int(oracle.slot_of(b.dec_pages[j], int(b.dec_ctx[j]), 16)))
    return np.asarray(out, np.int64)


def read_slots(kp, vp, slots):
    sl = torch.as_tensor(slots, device=kp.device)
    return kp[sl // 16, :, sl % 16, :], vp[sl // 16, :, sl % 16, :]


def stage_isolated(cf, S, rows=None):
    """Runs each layer stage through the C ABI on the oracle's inputs."""
    b, s, eng, W = S.b, S.s, S.eng, S.W
    T, l = S.T, b.prefill_rows
    Hq, d, H = s.n_q_heads, s.head_dim, s.hidden
    W64 = S.oracle_weights()
    x64 = f64(S.x)
    k0, v0 = S.kp.clone(), S.vp.clone()          # the cache before the step
    ref = oracle.layer_step(x64, W64, s, b, k0, v0, rows=rows)
    rr = ref["rows"]
    res = {}

    # a1: RMSNorm of x (all rows)
    xn = torch.empty_like(S.x)
    eng.cf_rmsnorm(S.x, W["g_attn"], xn)
    xn_ref = oracle.bf16_round(oracle.rmsnorm(x64, W64.g_attn, s.rms_eps))
    res["xn"] = errors(xn, xn_ref)

    # a2: fused QKV on the oracle's xn (all rows), appending into a copy of the cache
    kq, vq = k0.clone(), v0.clone()
    q = torch.empty((T, Hq, d), dtype=torch.bfloat16, device="cuda")
    eng.cf_qkv(S.batch, bf16_dev(xn_ref), cf.pool_of(kq, vq), q)
    need = ref["need_rows"]
    res["q"] = errors(q[need], ref["q_need"])
    kn, vn = read_slots(kq, vq, slots_of_rows(b, need))
    res["k"] = errors(kn, ref["k_need"])
    res["v"] = errors(vn, ref["v_need"])

    # a3 || a4: attention on the oracle's q, over a cache holding the oracle's k, v
    ka, va = k0.clone(), v0.clone()
    sl = torch.as_tensor(slots_of_rows(b, need), device="cuda")
    ka[sl // 16, :, sl % 16, :] = bf16_dev(ref["k_need"])
    va[sl // 16, :, sl % 16, :] = bf16_dev(ref["v_need"])
    pool_a = cf.pool_of(ka, va)
    q_need = bf16_dev(ref["q_need"])
    attn_rows = []
    npre = int(np.sum(need < l))
    if npre:
        # every chunk's rows at their stacked positions (the rows the oracle
        # skipped hold zeros: their outputs are not compared)
        pre_need = torch.as_tensor(need[:npre], device="cuda")
        qp = torch.zeros((l, Hq, d), dtype=torch.bfloat16, device="cuda")
        qp[pre_need] = q_need[:npre]
        op = torch.zeros_like(qp)
        if S.multi:
            eng.cf_prefill_attn_varlen(qp, pool_a, S.chunk_len, S.chunk_prefix, S.chunk_pages, op)
        else:
            eng.cf_prefill_attn(qp, pool_a, l, b.prefill_prefix, S.pre_pages, op)
        attn_rows.append(op[pre_need])
    dec_sel = need[need >= l] - l
    if len(dec_sel):
        ds = torch.as_tensor(dec_sel, device="cuda")
        keys = (S.dec_ctx[ds] + 1).contiguous()
        od = torch.zeros((len(dec_sel), Hq, d), dtype=torch.bfloat16, device="cuda")
        eng.cf_decode_attn(q_need[npre:].contiguous(), Hq * d, pool_a, len(dec_sel), keys,
                           S.dec_pages[ds].contiguous(), b.dec_stride, od, Hq * d)
        attn_rows.append(od)
    attn_need = torch.cat(attn_rows)
    where = np.searchsorted(need, rr)
    res["attn"] = errors(attn_need[torch.as_tensor(where, device="cuda")], ref["attn"])

    # a6: O-proj + residual on the oracle's attention output (selected rows)
    a_o = bf16_dev(ref["attn"].reshape(len(rr), Hq * d))
    h = torch.empty((len(rr), H), dtype=torch.float32, device="cuda")
    eng.cf_gemm(a_o, W["w_o"], h, cf.CF_EPI_RESID_F32, aux=S.x[torch.as_tensor(rr, device="cuda")].contiguous())
    res["h"] = errors(h, ref["h"])
    # a7: RMSNorm of the oracle's h
    h_o = torch.as_tensor(ref["h"], dtype=torch.float32).cuda()
    hn = torch.empty((len(rr), H), dtype=torch.bfloat16, device="cuda")
    eng.cf_rmsnorm(h_o, W["g_ffn"], hn)
    res["hn"] = errors(hn, ref["hn"])
    # a8: gate/up + SwiGLU on the oracle's hn
    act = torch.empty((len(rr), s.ffn_dim), dtype=torch.bfloat16, device="cuda")
    eng.cf_gemm(bf16_dev(ref["hn"]), W["w_gate"], act, cf.CF_EPI_SWIGLU, aux=W["w_up"])
    res["act"] = errors(act, ref["act"])
    # a9: down + residual on the oracle's act and h
    out = torch.empty((len(rr), H), dtype=torch.bfloat16, device="cuda")
    eng.cf_gemm(bf16_dev(ref["act"]), W["w_down"], out, cf.CF_EPI_RESID_BF16, aux=h_o)
    res["out"] = errors(out, ref["out"])
    torch.cuda.synchronize()
    assert eng.cf_get_error()[0] == 0
    report = "; ".join(f"{k}: max {m:.3g} mean {a:.3g}" for k, (m, a, _) in res.items())
    bad = [k for k, (m, a, _) in res.items() if m > TOL_MAX or a > TOL_MEAN]
    assert not bad, f"{bad} out of tolerance -- {report}"
    return res


def chained(S, rows=None):
    """cf_layer_step end to end against the oracle chain."""
    W64 = S.oracle_weights()
    ref = oracle.layer_step(f64(S.x), W64, S.s, S.b, S.kp.cpu(), S.vp.cpu(), rows=rows)
    out = S.step()
    rr = ref["rows"]
    T, Hq, d = S.T, S.s.n_q_heads, S.s.head_dim
    kn, vn = read_slots(S.kp, S.vp, slots_of_rows(S.b, rr))
    got = {
        "q": (S.eng.buffer("q", T).view(T, Hq, d)[rr], ref["q"], TOL_MAX, TOL_MEAN),
        "k": (kn, ref["k"], TOL_MAX, TOL_MEAN),
        "v": (vn, ref["v"], TOL_MAX, TOL_MEAN),
        "attn": (S.eng.buffer("attn", T)[rr], ref["attn"].reshape(len(rr), -1), TOL_MAX, TOL_MEAN),
        "h": (S.eng.buffer("h", T)[rr], ref["h"], TOL_MAX, TOL_MEAN),
        "out": (out[rr], ref["out"], CHAIN_MAX, CHAIN_MEAN),
    }
    res = {k: errors(g, r) for k, (g, r, _, _) in got.items()}
    report = "; ".join(f"{k}: max {m:.3g} mean {a:.3g}" for k, (m, a, _) in res.items())
    bad = [k for k, (g, r, tm, ta) in got.items() if res[k][0] > tm or res[k][1] > ta]
    assert not bad, f"{bad} out of bound -- {report}"
    return res


SLICES = [
    ("tiny", wl.WORKLOADS["tiny"]),
    ("l8b", wl.reduced(wl.WORKLOADS["l8b"], (5, 300, 17, 1), 130, 0)),
    ("q14b", wl.reduced(wl.WORKLOADS["q14b"], (40, 600), 200, 77)),
    ("q32b", wl.reduced(wl.WORKLOADS["q32b"], (1000,), 64, 500)),
    ("mix-decode-only", wl.reduced(wl.WORKLOADS["mix"], (700, 20, 3333), 0, 0)),
    ("l8b-prefill-only", wl.reduced(wl.WORKLOADS["l8b"], (), 257, 31)),
    # several chunks of different requests in one step (ConfluxServe §6.2 Eq. 6)
    ("tiny-chunks", wl.Workload("tiny-chunks", wl.TINY, 3, (5, 40, 200), 64, 128,
                                more_chunks=((37, 0), (130, 300), (1, 17)))),
    ("l8b-chunks", wl.Workload("l8b-chunks", wl.LLAMA8B, 4, (5, 300, 17, 1), 300, 0,
                               more_chunks=((130, 2000), (129, 700), (1, 5)))),
    ("q14b-chunks-only", wl.Workload("q14b-chunks-only", wl.QWEN14B, 0, (), 200, 77,
                                     more_chunks=((64, 0), (257, 1000)))),
]


@pytest.mark.parametrize("name,w", SLICES, ids=[s[0] for s in SLICES])
def test_layer_stages_full_parity(cf, name, w):
    """Every stage, every row and element, at sizes the oracle finishes in seconds."""
    stage_isolated(cf, LayerSetup(w))


@pytest.mark.parametrize("name,w", SLICES, ids=[s[0] for s in SLICES])
def test_layer_chained_parity(cf, name, w):
    chained(LayerSetup(w))


FULL = ["l8b", "q14b", "mix", "q32b", "mchunk"]


def sample_rows(b):
    nd = b.n_decode
    rng = np.random.default_rng(0)
    rows, r0 = [], 0
    for l, _, _ in b.chunks:   # each chunk's first rows, a tile edge, its last row
        rows += [r0, r0 + 1, r0 + min(127, l - 1), r0 + min(128, l - 1), r0 + l - 1]
        rows += list(r0 + rng.integers(0, l, 2))
        r0 += l
    return sorted(set(int(r) for r in rows + [r0, r0 + nd - 1] + list(r0 + rng.integers(0, nd, 3))))


@pytest.mark.parametrize("name", FULL)
def test_layer_full_size_stages_sampled(cf, name):
    """The measured workloads at full size; the oracle computes a sample of rows."""
    S = LayerSetup(wl.WORKLOADS[name], gen_device="cuda")
    stage_isolated(cf, S, rows=sample_rows(S.b))


@pytest.mark.parametrize("name", FULL)
def test_layer_full_size_chained_sampled(cf, name):
    S = LayerSetup(wl.WORKLOADS[name], gen_device="cuda")
    chained(S, rows=sample_rows(S.b))


def test_layer_step_composes_the_stage_kernels(cf):
    """cf_layer_step's intermediates equal the stage calls chained on the GPU."""
    w = wl.reduced(wl.WORKLOADS["q14b"], (300, 45, 2000), 150, 60)
    S = LayerSetup(w)
    k0, v0 = S.kp.clone(), S.vp.clone()
    out = S.step()
    eng, W, T, s = S.eng, S.W, S.T, S.s
    xn = torch.empty_like(S.x)
    eng.cf_rmsnorm(S.x, W["g_attn"], xn)
    assert torch.equal(xn, eng.buffer("xn", T))
    q = torch.empty((T, s.n_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
    eng.cf_qkv(S.batch, xn, cf.pool_of(k0, v0), q)
    torch.cuda.synchronize()
    assert torch.equal(q.view(T, -1), eng.buffer("q", T))
    # same bits in every slot (the pools hold NaN sentinels, so compare the bit patterns)
    assert torch.equal(k0.view(torch.int16), S.kp.view(torch.int16))
    assert torch.equal(v0.view(torch.int16), S.vp.view(torch.int16))
    l, nd = S.b.prefill_len, S.b.n_decode
    attn = torch.empty((T, s.n_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
    att_p = torch.empty((l, s.n_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
    eng.cf_prefill_attn(q[:l].contiguous(), S.pool, l, S.b.prefill_prefix, S.pre_pages, att_p)
    keys = (S.dec_ctx + 1).contiguous()
    od = torch.empty((nd, s.n_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
    eng.cf_decode_attn(q[l:].contiguous(), s.n_q_heads * s.head_dim, S.pool, nd, keys, S.dec_pages,
                       S.b.dec_stride, od, s.n_q_heads * s.head_dim, eng.cf_engine_decode_sms())
    attn[:l] = att_p
    attn[l:] = od
    assert torch.equal(attn.view(T, -1), eng.buffer("attn", T))
    h = torch.empty((T, s.hidden), dtype=torch.float32, device="cuda")
    eng.cf_gemm(attn.view(T, -1), W["w_o"], h, cf.CF_EPI_RESID_F32, aux=S.x)
    assert torch.equal(h, eng.buffer("h", T))
    hn = torch.empty_like(S.x)
    eng.cf_rmsnorm(h, W["g_ffn"], hn)
    assert torch.equal(hn, eng.buffer("hn", T))
    act = torch.empty((T, s.ffn_dim), dtype=torch.bfloat16, device="cuda")
    eng.cf_gemm(hn, W["w_gate"], act, cf.CF_EPI_SWIGLU, aux=W["w_up"])
    assert torch.equal(act, eng.buffer("act", T))
    o2 = torch.empty_like(S.x)
    eng.cf_gemm(act, W["w_down"], o2, cf.CF_EPI_RESID_BF16, aux=h)
    torch.cuda.synchronize()
    assert torch.equal(o2, out)


def test_layer_tiny_untouched_slots(cf):
    """The step writes exactly the T appended slots of the pool."""
    S = LayerSetup(wl.WORKLOADS["tiny"])
    before = S.kp.view(torch.int16).clone()
    S.step()
    changed = (S.kp.view(torch.int16) != before).any(dim=-1)
    expect = np.zeros(changed.shape, bool)
    for sl in slots_of_rows(S.b, range(S.T)):
        expect[sl // 16, :, sl % 16] = True
    assert np.array_equal(changed.cpu().numpy(), expect)


def test_layer_page_permutation_invariance(cf):
    """Moving the same KV to other pages (and the tables with it) gives
    bit-identical outputs."""
    w = wl.reduced(wl.WORKLOADS["l8b"], (200, 1000, 33), 100, 50)
    S1 = LayerSetup(w)
    out1 = S1.step().clone()
    S2 = LayerSetup(w)
    perm = np.random.default_rng(9).permutation(S2.b.num_pages)
    pt = torch.as_tensor(perm, device="cuda")
    kp2 = torch.empty_like(S2.kp)
    vp2 = torch.empty_like(S2.vp)
    kp2[pt] = S2.kp
    vp2[pt] = S2.vp
    S2.kp.copy_(kp2)
    S2.vp.copy_(vp2)
    dp = S2.b.dec_pages.copy()
    dp[dp >= 0] = perm[dp[dp >= 0]]
    S2.dec_pages.copy_(torch.as_tensor(dp, device="cuda"))
    S2.pre_pages.copy_(torch.as_tensor(perm[S2.b.pre_pages], device="cuda"))
    out2 = S2.step()
    assert torch.equal(out1, out2)


CHUNKS_W = wl.Workload("l8b-chunks", wl.LLAMA8B, 3, (300, 64, 1000), 96, 40,
                       more_chunks=((130, 0), (1, 2000), (257, 513)))


def test_layer_chunks_match_each_chunk_run_alone(cf):
    """ConfluxServe §6.2 Eq. 6: several requests' chunks share one step.
    With the GEMMs' split-K tail off, every chunk's rows are bit-identical
    to the same chunk run as the only chunk of a step (GEMM rows and
    attention tiles do not depend on the other rows); decode rows agree
    within fp32 rounding."""
    S = LayerSetup(CHUNKS_W)
    S.eng.cf_set_split_k(1)
    S.eng.cf_set_prefill_split(1)   # key-range cuts depend on the whole launch
    for pairing in (1, 2, 3):
        S.eng.cf_set_prefill_pairing(pairing)
        out = S.step().clone()
        r0 = 0
        for i, (l, c, pages) in enumerate(S.b.chunks):
            xi = S.x[r0:r0 + l].contiguous()
            oi = torch.empty_like(xi)
            S.eng.cf_layer_step(cf.batch_of(0, None, None, l, c, torch.as_tensor(pages, device="cuda")), xi, oi,
                                S.pool)
            torch.cuda.synchronize()
            assert torch.equal(oi, out[r0:r0 + l]), (pairing, i)
            r0 += l
        xd = S.x[r0:].contiguous()
        od = torch.empty_like(xd)
        S.eng.cf_layer_step(cf.batch_of(S.b.n_decode, S.dec_ctx, S.dec_pages, 0, 0, None), xd, od, S.pool)
        torch.cuda.synchronize()
        assert S.eng.cf_get_error()[0] == 0
        assert_close(od, f64(out[r0:]), "decode rows", 1e-2, 1e-3)
    S.eng.cf_set_prefill_pairing(0)
    S.eng.cf_set_prefill_split(0)
    S.eng.cf_set_split_k(0)


def test_layer_chunk_list_of_one_equals_the_single_chunk_fields(cf):
    S = LayerSetup(wl.reduced(wl.WORKLOADS["l8b"], (300, 64), 96, 40))
    out = S.step().clone()
    lens, prefixes, table = S.b.chunk_table()
    b1 = cf.batch_of(S.b.n_decode, S.dec_ctx, S.dec_pages, 0, 0, None,
                     chunks=(lens, prefixes, torch.as_tensor(table, device="cuda")))
    o1 = torch.empty_like(out)
    S.eng.cf_layer_step(b1, S.x, o1, S.pool)
    torch.cuda.synchronize()
    assert torch.equal(o1, out)


def test_layer_rejects_bad_chunk_lists(cf):
    S = LayerSetup(CHUNKS_W)
    lens, prefixes, table = S.b.chunk_table()
    for bad in (dict(lens=[0] + list(lens[1:])), dict(prefixes=[-1] + list(prefixes[1:])),
                dict(table=S.chunk_pages[:, :2].contiguous())):
        args = (bad.get("lens", lens), bad.get("prefixes", prefixes), bad.get("table", S.chunk_pages))
        b = cf.batch_of(S.b.n_decode, S.dec_ctx, S.dec_pages, 0, 0, None, chunks=args)
        with pytest.raises(cf.CfError) as ex:
            S.eng.cf_layer_step(b, S.x, S.out, S.pool)
        assert ex.value.status == cf.CF_ERR_INVALID_ARG
    # a single chunk and a chunk list at once
    b = cf.batch_of(S.b.n_decode, S.dec_ctx, S.dec_pages, 5, 0, S.pre_pages, chunks=(lens, prefixes, S.chunk_pages))
    with pytest.raises(cf.CfError):
        S.eng.cf_layer_step(b, S.x, S.out, S.pool)


def test_layer_cobatched_rows_match_separate_batches(cf):
    """ConfluxServe §4: rows of the co-batched step equal the same rows run
    as a prefill-only and a decode-only step over the same cache.  With the
    GEMMs' split-K tail off, prefill rows are bit-identical (GEMM rows are
    independent, attention items do not depend on the grid); decode rows may
    split the keys differently, so they agree within fp32 rounding.  With it
    on, the tile cuts depend on the batch, so prefill rows agree within
    rounding too."""
    base = wl.WORKLOADS["l8b"]
    dec, l, cp = (300, 64), 96, 40
    S = LayerSetup(wl.reduced(base, dec, l, cp))
    xp, xd = S.x[:l].contiguous(), S.x[l:].contiguous()
    for split_k in (False, True):
        S.eng.cf_set_split_k(0 if split_k else 1)
        out = S.step().clone()
        op, od = torch.empty_like(xp), torch.empty_like(xd)
        S.eng.cf_layer_step(cf.batch_of(0, None, None, l, cp, S.pre_pages), xp, op, S.pool)
        S.eng.cf_layer_step(cf.batch_of(len(dec), S.dec_ctx, S.dec_pages, 0, 0, S.pre_pages), xd, od, S.pool)
        torch.cuda.synchronize()
        assert S.eng.cf_get_error()[0] == 0
        if split_k:
            assert_close(op, f64(out[:l]), "prefill rows", 1e-2, 1e-3)
        else:
            assert torch.equal(op, out[:l])
        assert_close(od, f64(out[l:]), "decode rows", 1e-2, 1e-3)


def test_layer_flags_bad_page_id(cf):
    w = wl.reduced(wl.WORKLOADS["tiny"], (17, 40), 16, 0)
    S = LayerSetup(w)
    S.dec_pages[1, 0] = S.b.num_pages + 5        # outside the pool
    S.eng.cf_layer_step(S.batch, S.x, S.out, S.pool)
    st, msg = S.eng.cf_get_error()
    assert st == cf.CF_ERR_DEVICE and "page" in msg
    # the engine stays usable
    S.dec_pages[1, 0] = int(S.b.dec_pages[1, 0])
    S.step()


def test_layer_rejects_bad_arguments(cf):
    w = wl.reduced(wl.WORKLOADS["tiny"], (17,), 8, 0)
    S = LayerSetup(w)
    big = cf.batch_of(1, S.dec_ctx, S.dec_pages, S.cfg.max_tokens + 1, 0, S.pre_pages)
    with pytest.raises(cf.CfError) as e:
        S.eng.cf_layer_step(big, S.x, S.out, S.pool)
    assert e.value.status == cf.CF_ERR_INVALID_ARG
    with pytest.raises(cf.CfError):
        S.eng.cf_layer_step(S.batch, S.x, S.x, S.pool)      # in place is not allowed


def test_empty_calls_launch_nothing(cf):
    """Degenerate batches: no decodes and no chunk (T = 0), a GEMM with no
    rows and a decode call with no requests return at once, launch no
    kernel and write nothing."""
    w = wl.reduced(wl.WORKLOADS["tiny"], (17,), 8, 0)
    S = LayerSetup(w)
    S.out.fill_(7.0)
    n0 = S.eng.cf_launch_count()
    S.eng.cf_layer_step(cf.batch_of(0, S.dec_ctx, S.dec_pages, 0, 0, S.pre_pages), S.x, S.out, S.pool)
    A = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    B = torch.randn(256, 256, device="cuda").bfloat16()
    C = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    S.eng.cf_gemm(A, B, C)
    s = S.s
    q = torch.empty(0, s.n_q_heads, s.head_dim, dtype=torch.bfloat16, device="cuda")
    S.eng.cf_decode_attn(q, s.n_q_heads * s.head_dim, S.pool, 0, S.dec_ctx, S.dec_pages, S.b.dec_stride, q,
                         s.n_q_heads * s.head_dim)
    torch.cuda.synchronize()
    assert S.eng.cf_launch_count() == n0
    assert bool((S.out.float() == 7.0).all())
    assert S.eng.cf_get_error()[0] == 0


def test_layer_step_is_deterministic_and_launch_count(cf):
    S = LayerSetup(wl.reduced(wl.WORKLOADS["q14b"], (100, 9), 50, 10))
    first = S.step().clone()          # also measures the automatic decode share
    n0 = S.eng.cf_launch_count()
    a = S.step().clone()
    assert S.eng.cf_launch_count() - n0 == 11   # 9 stages + the fork's second decode and prefill grids
    b = S.step()
    assert torch.equal(a, b) and torch.equal(a, first)


def test_bounded_wait_runs_out_and_the_engine_recovers(cf):
    """Failure detection without a fault: cf_selftest_timeout makes a GEMM's
    MMA thread wait on a barrier nothing arrives at; the 50 ms bound runs
    out, the kernel raises the timeout bit, lets its copies land, frees its
    tensor memory and returns.  The host reads the status, the word is
    cleared, and the next layer step gives the same bits as before."""
    S = LayerSetup(wl.reduced(wl.WORKLOADS["l8b"], (300, 64), 96, 40))
    k0, v0 = S.kp.clone(), S.vp.clone()
    ref = S.step().clone()
    S.eng.cf_selftest_timeout(50_000_000)
    st, msg = S.eng.cf_get_error()
    assert st == cf.CF_ERR_TIMEOUT and "bounded wait expired" in msg
    assert S.eng.cf_get_error()[0] == 0
    S.kp.copy_(k0)
    S.vp.copy_(v0)
    assert torch.equal(S.step(), ref)
    with pytest.raises(cf.CfError):
        S.eng.cf_selftest_timeout(0)


def test_layer_step_graphs_match_eager(cf):
    """Piecewise CUDA graphs (ConfluxServe §6.1, Fig. 10): the replayed
    segments give the eager step's bits; a batch with the same rows and
    buffers but another prefix and other decode contexts replays the same
    graphs (the chunk length and prefix reach them through device memory)."""
    S = LayerSetup(wl.reduced(wl.WORKLOADS["l8b"], (300, 64, 1000), 96, 40))
    k0, v0 = S.kp.clone(), S.vp.clone()

    out = torch.empty_like(S.x)   # one output buffer: the graphs are keyed by the buffers

    def run(batch, graphs):
        S.kp.copy_(k0)
        S.vp.copy_(v0)
        S.eng.cf_set_graphs(graphs)
        out.fill_(float("nan"))
        S.eng.cf_layer_step(batch, S.x, out, S.pool)
        torch.cuda.synchronize()
        assert S.eng.cf_get_error()[0] == 0
        return out.clone()

    eager = run(S.batch, False)
    n0 = S.eng.cf_graph_captures()
    g1 = run(S.batch, True)
    g2 = run(S.batch, True)
    assert S.eng.cf_graph_captures() == n0 + 1
    assert torch.equal(g1, eager) and torch.equal(g2, eager)
    # same rows and buffers, another prefix and shorter decode contexts
    ctx2 = (S.dec_ctx // 2).contiguous()
    S.dec_ctx.copy_(ctx2)
    b2 = cf.batch_of(S.b.n_decode, S.dec_ctx, S.dec_pages, S.b.prefill_len, 24, S.pre_pages)
    eager2 = run(b2, False)
    graph2 = run(b2, True)
    assert S.eng.cf_graph_captures() == n0 + 1
    assert torch.equal(graph2, eager2)
    assert not torch.equal(eager2, eager)
    S.eng.cf_set_graphs(False)


def test_layer_step_graphs_with_chunk_lists(cf):
    """Replayed linear segments read the step's chunk table from device
    memory: another split of the same rows (other prefixes) reuses the
    captured graphs and still equals the eager step."""
    S = LayerSetup(CHUNKS_W)
    out = torch.empty_like(S.x)   # one output buffer: the graphs are keyed on the buffers

    def run(b, graphs):
        S.eng.cf_set_graphs(graphs)
        S.eng.cf_layer_step(b, S.x, out, S.pool)
        torch.cuda.synchronize()
        assert S.eng.cf_get_error()[0] == 0
        return out.clone()

    eager = run(S.batch, False)
    n0 = S.eng.cf_graph_captures()
    assert torch.equal(run(S.batch, True), eager)
    lens = S.chunk_len
    prefixes = S.chunk_prefix // 2
    b2 = cf.batch_of(S.b.n_decode, S.dec_ctx, S.dec_pages, 0, 0, None, chunks=(lens, prefixes, S.chunk_pages))
    eager2 = run(b2, False)
    graph2 = run(b2, True)
    assert S.eng.cf_graph_captures() == n0 + 1
    assert torch.equal(graph2, eager2) and not torch.equal(eager2, eager)
    S.eng.cf_set_graphs(False)


@pytest.mark.gpu
def test_latency_estimator_fits_and_predicts_through_the_library(cf, tmp_path):
    # the estimator study of bench.py on a small sample: isolated profiles ->
    # fitted lines -> calibrated contention factors -> predictions; the
    # library's predictions on the measured coefficients equal the oracle's
    import argparse
    import json

    import bench
    from oracle import latency as OL
    out = tmp_path / "est.jsonl"
    args = argparse.Namespace(estimator="tiny", seed=0, decode_sms=0, est_reps=1, est_profile=5,
                              est_calibrate=5, est_validate=8, estimator_out=str(out))
    (line,) = bench.run_estimator(args)
    c = line["coeffs_ms"]
    assert c["gamma"] > 0 and c["a_d"] > 0 and c["a_p"] > 0
    assert 1.0 <= c["alpha"] <= 4.0 and 1.0 <= c["beta"] <= 4.0
    assert np.isfinite(line["mape_pct"]) and line["n_validate"] == 8
    m = OL.LatencyModel(**c)
    rec = json.loads(out.read_text().splitlines()[0])
    for v, it in zip(rec["validate"], wl.estimator_batches(0, 8, "validate")):
        assert (v["l"], v["c_p"], v["n_d"], v["ctx_sum"]) == (it[0], it[1], len(it[2]), sum(it[2]))
        ranks, chunks = OL.one_gpu(*it)
        assert v["pred_ms"] == pytest.approx(OL.t_iter(m, ranks, chunks)["t_iter"], rel=1e-12)
        assert v["meas_ms"] > 0


GRAPH_SLICES = [s for s in SLICES if s[0] in ("tiny", "l8b", "tiny-chunks")]


@pytest.mark.parametrize("name,w", GRAPH_SLICES, ids=[s[0] for s in GRAPH_SLICES])
def test_layer_graphs_chained_parity(cf, name, w):
    """The piecewise-graph step (ConfluxServe §6.1, Fig. 10: the shared linear
    segments replayed as CUDA graphs, the attention fork launched eagerly)
    against the oracle: a replayed step's q, appended k/v, attention output,
    h and out, at the same bounds as the eager step."""
    S = LayerSetup(w)
    S.eng.cf_set_graphs(True)
    S.step()                                  # captures the two segments
    assert S.eng.cf_graph_captures() == 1
    chained(S)                                # replays them
    assert S.eng.cf_graph_captures() == 1
    S.eng.cf_set_graphs(False)


FORK_SLICES = [s for s in SLICES if s[0] in ("tiny", "l8b", "q14b", "l8b-chunks")]


@pytest.mark.parametrize("name,w", FORK_SLICES, ids=[s[0] for s in FORK_SLICES])
def test_serial_attention_gives_the_fork_bits(cf, name, w):
    """The serialized execution the fork is measured against (ConfluxServe
    §8.3, Fig. 14a: decode alone on all SMs, then prefill alone on all SMs)
    runs the same work items, so it gives the concurrent fork's bits, and it
    matches the oracle."""
    S = LayerSetup(w)
    k0, v0 = S.kp.clone(), S.vp.clone()
    fork = S.step().clone()
    attn = S.eng.buffer("attn", S.T).clone()
    S.kp.copy_(k0)
    S.vp.copy_(v0)
    S.eng.cf_set_fork_mode(1)
    n0 = S.eng.cf_launch_count()
    serial = S.step().clone()
    assert torch.equal(serial, fork)
    assert torch.equal(S.eng.buffer("attn", S.T), attn)
    assert S.eng.cf_launch_count() - n0 <= 11
    S.kp.copy_(k0)
    S.vp.copy_(v0)
    chained(S)
    S.eng.cf_set_fork_mode(0)
    with pytest.raises(cf.CfError):
        S.eng.cf_set_fork_mode(2)


def test_automatic_decode_share_is_the_90_percent_rule(cf):
    """With decode_sms = 0 the library measures ConfluxServe §6.1's rule on the
    first step of a decode-batch bucket: the fewest SMs (8, 12, 16, ...) whose
    decode time is within 1/0.9 of the fastest.  A plain layer step reports
    that share, not the fallback third of the SMs, and keeps it for later
    steps of the bucket."""
    w = wl.reduced(wl.WORKLOADS["l8b"], (4096,) * 16, 256, 0)
    S = LayerSetup(w)
    sms = cf.device_sm_count()
    S.step()
    pts = S.eng.cf_calibration_points()
    assert len(pts) >= 2 and pts[-1][0] == sms and all(p[0] % 4 == 0 for p in pts[:-1])
    best = min(t for _, t in pts)
    want = next(n for n, t in pts if best / t >= 0.9)
    want = min(want, sms - 1)
    got = S.eng.cf_engine_decode_sms()
    assert got == want
    assert got % 4 == 0 or got == sms - 1     # a measured point, not the fallback sms / 3
    n0 = S.eng.cf_launch_count()
    S.step()
    assert S.eng.cf_launch_count() - n0 == 11      # measured once per bucket
    assert S.eng.cf_engine_decode_sms() == got
    # an explicit share overrides it; 0 returns to the measured one
    S.eng.cf_set_decode_sms(24)
    assert S.eng.cf_engine_decode_sms() == 24
    S.eng.cf_set_decode_sms(0)
    assert S.eng.cf_engine_decode_sms() == got
