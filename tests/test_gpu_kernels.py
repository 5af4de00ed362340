"""GPU parity of the individual C-ABI kernels against the fp64 oracle / exact
references (cf_gemm, cf_kv_append, cf_decode_attn, cf_prefill_attn)."""
import numpy as np
import pytest
import torch

import oracle
import workload as wl
from helpers import assert_close, f64, fill_positions, randn_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cf():
    import co_prefill_decode_gb300 as cf
    cf.load_library()
    return cf


def engine_for(cf, shape, max_tokens=4096, max_decode=256):
    W = {k: v.cuda() for k, v in wl.make_weights(wl.Workload("t", shape, 1, (1,), 0, 0), 7).items()}
    return cf.Engine(cf.make_config(shape, max_tokens, max_decode), W)


def int_bf16(shape, seed, lo=-4, hi=4):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g).to(torch.bfloat16).cuda()


# --------------------------------------------------------------------- GEMM
@pytest.mark.parametrize("M,N,K", [(1, 256, 64), (68, 512, 256), (200, 768, 4096), (1040, 512, 1024),
                                   (300, 256, 8192), (1040, 6144, 512), (4128, 2048, 256),
                                   (384, 4096, 14336), (1040, 6144, 4096)])
def test_gemm_exact_integers(cf, M, N, K):
    """Small integers: fp32 accumulation is exact, so the GPU equals the integer
    product bit for bit (fp32 out via the residual epilogue with zero aux) and
    its bf16 rounding (plain epilogue).  Shapes whose last wave is partial
    cut those tiles into k-chunks (see cf_gemm_schedule), also with every
    forced chunk count tried here: a k-block lost or added in the cut shows
    up here."""
    eng = engine_for(cf, wl.TINY)
    A, B = int_bf16((M, K), 1), int_bf16((N, K), 2)
    exact = f64(A) @ f64(B).T
    C32 = torch.empty(M, N, dtype=torch.float32, device="cuda")
    z = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    for mode in (0, 1, 2, 7):
        eng.cf_set_split_k(mode)
        C32.fill_(float("nan"))
        eng.cf_gemm(A, B, C32, cf.CF_EPI_RESID_F32, aux=z)
        C16 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        eng.cf_gemm(A, B, C16, cf.CF_EPI_NONE)
        torch.cuda.synchronize()
        assert np.array_equal(f64(C32), exact), mode
        assert np.array_equal(f64(C16), oracle.bf16_round(exact)), mode
    eng.cf_set_split_k(0)
    assert eng.cf_get_error()[0] == 0


@pytest.mark.parametrize("K", [1024, 8192])
def test_gemm_epilogues(cf, K):
    """Every epilogue against fp64; K = 8192 cuts each of the 6 tiles into
    k-chunks, so the split-K fix-up feeds every epilogue."""
    eng = engine_for(cf, wl.TINY)
    M, N = 333, 512
    assert (cf.cf_gemm_schedule(M, N, K)["split"] > 1) == (K == 8192)
    A, B = randn_bf16((M, K), 3), randn_bf16((N, K), 4, std=0.03)
    U = randn_bf16((N, K), 5, std=0.03)
    res16 = randn_bf16((M, N), 6)
    res32 = torch.randn(M, N, generator=torch.Generator().manual_seed(7)).cuda()
    a, b, u = f64(A), f64(B), f64(U)
    out = torch.empty(M, N, dtype=torch.float32, device="cuda")
    eng.cf_gemm(A, B, out, cf.CF_EPI_RESID_F32, aux=res16)
    o2 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    eng.cf_gemm(A, B, o2, cf.CF_EPI_RESID_BF16, aux=res32)
    o3 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    eng.cf_gemm(A, B, o3, cf.CF_EPI_SWIGLU, aux=U)
    torch.cuda.synchronize()
    # fp32 accumulation: the rounding error of a K-term dot product grows with K
    assert_close(out, f64(res16) + a @ b.T, "resid f32", 1e-5 * K / 1024, 1e-6 * K / 1024)
    assert_close(o2, oracle.bf16_round(f64(res32) + a @ b.T), "resid bf16")
    assert_close(o3, oracle.bf16_round(oracle.swiglu(a @ b.T, a @ u.T)), "swiglu")


def test_gemm_swiglu_many_tiles(cf):
    """More tiles than CTAs: each CTA walks several tiles through both TMEM
    accumulator buffers."""
    eng = engine_for(cf, wl.TINY)
    M, F, K = 300, 14336, 512
    A, G, U = int_bf16((M, K), 21, -2, 2), int_bf16((F, K), 22, -1, 1), int_bf16((F, K), 23, -1, 1)
    out = torch.empty(M, F, dtype=torch.bfloat16, device="cuda")
    eng.cf_gemm(A, G, out, cf.CF_EPI_SWIGLU, aux=U)
    torch.cuda.synchronize()
    a = f64(A)
    ref = oracle.bf16_round(oracle.swiglu(a @ f64(G).T, a @ f64(U).T))
    assert_close(out, ref, "swiglu many tiles", 8e-3, 1e-4)


def test_gemm_rows_are_independent(cf):
    """Co-batching invariance (ConfluxServe §4): with split-K off a row of
    the stacked GEMM is bit-identical to the same row computed in a smaller
    batch; with it on, tiles are cut into k-chunks depending on the batch,
    so the rows agree within fp32 accumulation rounding."""
    eng = engine_for(cf, wl.TINY)
    K, N = 2048, 768
    assert cf.cf_gemm_schedule(700, N, K, split_mode=4)["split"] == 4
    A, B = randn_bf16((700, K), 8), randn_bf16((N, K), 9, std=0.02)
    full = torch.empty(700, N, dtype=torch.bfloat16, device="cuda")
    part = torch.empty(130, N, dtype=torch.bfloat16, device="cuda")
    full32 = torch.empty(700, N, dtype=torch.float32, device="cuda")
    part32 = torch.empty(130, N, dtype=torch.float32, device="cuda")
    z = torch.zeros(700, N, dtype=torch.bfloat16, device="cuda")
    a = A[500:630].contiguous()
    eng.cf_set_split_k(4)   # the full batch's tiles cut in 4 k-chunks ...
    eng.cf_gemm(A, B, full32, cf.CF_EPI_RESID_F32, aux=z)
    eng.cf_set_split_k(1)   # ... the small batch's tiles whole
    eng.cf_gemm(a, B, part32, cf.CF_EPI_RESID_F32, aux=z[:130])
    eng.cf_gemm(A, B, full)
    eng.cf_gemm(a, B, part)
    eng.cf_set_split_k(0)
    torch.cuda.synchronize()
    assert torch.equal(full[500:630], part)
    d = (full32[500:630] - part32).abs().max().item()
    assert d <= 1e-5 * max(1.0, part32.abs().max().item())


def test_gemm_stream_k_is_deterministic(cf):
    """Chunks of a cut tile are summed in k order by whichever CTA finishes
    last, so repeated calls agree bit for bit (the 48-tile, 224-k-block FFN
    down projection of a 384-token batch)."""
    eng = engine_for(cf, wl.TINY)
    M, N, K = 384, 4096, 14336
    assert cf.cf_gemm_schedule(M, N, K, cf.CF_EPI_RESID_BF16)["split"] > 1
    A, B = randn_bf16((M, K), 11), randn_bf16((N, K), 12, std=0.02)
    res = torch.randn(M, N, generator=torch.Generator().manual_seed(13)).cuda()
    outs = []
    for _ in range(3):
        o = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        eng.cf_gemm(A, B, o, cf.CF_EPI_RESID_BF16, aux=res)
        outs.append(o)
    torch.cuda.synchronize()
    assert eng.cf_get_error()[0] == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    ref = oracle.bf16_round(f64(res) + f64(A) @ f64(B).T)
    assert_close(outs[0], ref, "stream-K down projection")


def test_gemm_rejects_bad_shapes(cf):
    eng = engine_for(cf, wl.TINY)
    A, B = randn_bf16((64, 100), 1), randn_bf16((256, 100), 2)
    C = torch.empty(64, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cf.CfError) as e:
        eng.cf_gemm(A, B, C)
    assert e.value.status == cf.CF_ERR_UNSUPPORTED


# --------------------------------------------------------------------- append
def test_kv_append_bit_exact(cf):
    eng = engine_for(cf, wl.LLAMA8B)
    pages, Hkv, d, n = 40, 8, 128, 300
    kp = torch.full((pages, Hkv, 16, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vp = kp.clone()
    slots = torch.as_tensor(np.random.default_rng(0).permutation(pages * 16)[:n].astype(np.int32), device="cuda")
    k, v = randn_bf16((n, Hkv, d), 10), randn_bf16((n, Hkv, d), 11)
    before_k = kp.view(torch.int16).cpu().numpy().copy()
    eng.cf_kv_append(k, v, slots, cf.pool_of(kp, vp))
    torch.cuda.synchronize()
    # oracle scatter on the raw bit patterns
    ref_k = before_k.copy()
    ref_v = before_k.copy()
    oracle.kv_append(ref_k, ref_v, k.view(torch.int16).cpu().numpy(), v.view(torch.int16).cpu().numpy(),
                     slots.cpu().numpy(), 16)
    assert np.array_equal(kp.view(torch.int16).cpu().numpy(), ref_k)
    assert np.array_equal(vp.view(torch.int16).cpu().numpy(), ref_v)


def test_kv_append_flags_bad_slot(cf):
    eng = engine_for(cf, wl.TINY)
    kp = torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    vp = kp.clone()
    slots = torch.tensor([3, 4 * 16 + 5], dtype=torch.int32, device="cuda")
    k, v = randn_bf16((2, 2, 64), 1), randn_bf16((2, 2, 64), 2)
    eng.cf_kv_append(k, v, slots, cf.pool_of(kp, vp))
    st, msg = eng.cf_get_error()
    assert st == cf.CF_ERR_DEVICE and "page" in msg
    assert torch.equal(kp[0, :, 3], k[0])          # the valid row still landed
    assert eng.cf_get_error()[0] == 0              # the word was cleared


# --------------------------------------------------------------------- decode
DECODE_CASES = [
    ("tiny", wl.TINY, (17, 64, 100, 255, 1, 16)),
    ("l8b", wl.LLAMA8B, (5, 16, 17, 700, 1, 2049)),
    ("q14b", wl.QWEN14B, (33, 1000, 15)),
    ("q32b", wl.QWEN32B, (3000, 31, 64)),
    ("g16", wl.LayerShape(2048, 32, 2, 64, 512, 1e4, 1e-5, False), (90, 1, 300)),
    # group sizes that leave some of the transposed products' 8 head columns unused
    ("g1", wl.LayerShape(1024, 8, 8, 128, 512, 1e4, 1e-5, False), (40, 1, 130)),
    ("g3", wl.LayerShape(768, 6, 2, 128, 512, 1e4, 1e-5, False), (77, 16, 500)),
    ("g7", wl.LayerShape(1792, 14, 2, 128, 512, 1e4, 1e-5, False), (33, 260)),
    # one long request: ~250 chunks, so the merge reads (m, l) beyond the 64 it keeps in registers
    ("long1", wl.LLAMA8B, (20000,)),
]


@pytest.mark.parametrize("name,shape,ctx", DECODE_CASES, ids=[c[0] for c in DECODE_CASES])
@pytest.mark.parametrize("num_sms", [0, 3])
def test_decode_attention_matches_oracle(cf, name, shape, ctx, num_sms):
    w = wl.Workload(name, shape, len(ctx), ctx, 0, 0)
    b = wl.make_batch(w, 1)
    kp, vp = wl.make_pools(w, b, 1, "cuda")
    n, Hq, d = len(ctx), shape.n_q_heads, shape.head_dim
    q = randn_bf16((n, Hq, d), 12)
    out = torch.zeros((n, Hq, d), dtype=torch.bfloat16, device="cuda")
    eng = engine_for(cf, shape)
    keys = torch.as_tensor(b.dec_ctx, device="cuda")        # positions 0..c_j-1 are cached
    pages = torch.as_tensor(b.dec_pages, device="cuda")
    ref = oracle.decode_attention(f64(q), kp, vp, b.dec_ctx, b.dec_pages, 16)
    eng.cf_decode_attn(q, Hq * d, cf.pool_of(kp, vp), n, keys, pages, b.dec_stride, out, Hq * d, num_sms)
    torch.cuda.synchronize()
    assert eng.cf_get_error()[0] == 0
    assert_close(out, ref, f"decode {name}")


def test_decode_split_count_and_page_order_invariance(cf):
    """Layout changes must not change results: a shuffled page table gives
    bit-identical outputs, and so does any grid size (the chunk plan is
    sized for the device, never for the launch)."""
    shape = wl.LLAMA8B
    ctx = (4000, 2500, 77)
    w = wl.Workload("inv", shape, len(ctx), ctx, 0, 0)
    b = wl.make_batch(w, 2)
    kp, vp = wl.make_pools(w, b, 2, "cuda")
    n, Hq, d = len(ctx), shape.n_q_heads, shape.head_dim
    q = randn_bf16((n, Hq, d), 13)
    eng = engine_for(cf, shape)
    keys = torch.as_tensor(b.dec_ctx, device="cuda")
    outs = {}
    # identity layout: the same KV placed on pages in order
    perm = np.argsort(np.random.default_rng(3).permutation(b.num_pages))
    kp2 = torch.empty_like(kp); vp2 = torch.empty_like(vp)
    ptab = b.dec_pages.copy()
    valid = ptab >= 0
    ptab[valid] = perm[ptab[valid]]
    kp2[torch.as_tensor(perm, device="cuda")] = kp
    vp2[torch.as_tensor(perm, device="cuda")] = vp
    for tag, (K, V, tab) in {"a": (kp, vp, b.dec_pages), "b": (kp2, vp2, ptab)}.items():
        for sms in (0, 7):
            out = torch.zeros((n, Hq, d), dtype=torch.bfloat16, device="cuda")
            eng.cf_decode_attn(q, Hq * d, cf.pool_of(K, V), n, keys, torch.as_tensor(tab, device="cuda"),
                               b.dec_stride, out, Hq * d, sms)
            outs[(tag, sms)] = out
    torch.cuda.synchronize()
    assert torch.equal(outs[("a", 0)], outs[("b", 0)])
    assert torch.equal(outs[("a", 7)], outs[("b", 7)])
    assert torch.equal(outs[("a", 7)], outs[("a", 0)])


# --------------------------------------------------------------------- prefill
PREFILL_CASES = [
    ("tiny", wl.TINY, 64, 128),
    ("tiny-ragged", wl.TINY, 77, 5),
    ("l8b", wl.LLAMA8B, 300, 0),
    ("l8b-prefix", wl.LLAMA8B, 130, 333),
    ("q14b", wl.QWEN14B, 1, 255),
    ("q32b", wl.QWEN32B, 256, 1000),
]


def pairing_modes(shape):
    """Prefill pair kinds valid for the shape: automatic, single tiles, tile
    pairs, and head pairs when the GQA group size is even."""
    return [0, 1, 2] + ([3] if (shape.n_q_heads // shape.n_kv_heads) % 2 == 0 else [])


@pytest.mark.parametrize("name,shape,l,cp", PREFILL_CASES, ids=[c[0] for c in PREFILL_CASES])
@pytest.mark.parametrize("pairing", [0, 2, 3])
@pytest.mark.parametrize("split", [0, 1, 3])
def test_prefill_attention_matches_oracle(cf, name, shape, l, cp, pairing, split):
    if pairing not in pairing_modes(shape):
        pytest.skip("head pairs need an even GQA group")
    w = wl.Workload(name, shape, 0, (), l, cp)
    b = wl.make_batch(w, 4)
    kp, vp = wl.make_pools(w, b, 4, "cuda")
    fill_positions(kp, vp, b.pre_pages, cp, l, 40)   # the chunk's own K/V (appended before attention)
    Hq, d = shape.n_q_heads, shape.head_dim
    q = randn_bf16((l, Hq, d), 14)
    out = torch.zeros((l, Hq, d), dtype=torch.bfloat16, device="cuda")
    eng = engine_for(cf, shape)
    eng.cf_set_prefill_pairing(pairing)
    eng.cf_set_prefill_split(split)       # automatic, never, or 3 key ranges where possible
    ref = oracle.prefill_attention(f64(q), kp, vp, cp, b.pre_pages, 16)
    eng.cf_prefill_attn(q, cf.pool_of(kp, vp), l, cp, torch.as_tensor(b.pre_pages, device="cuda"), out)
    torch.cuda.synchronize()
    assert eng.cf_get_error()[0] == 0
    assert_close(out, ref, f"prefill {name}")


@pytest.mark.parametrize("name,shape,l,cp", PREFILL_CASES, ids=[c[0] for c in PREFILL_CASES])
def test_prefill_pairs_change_no_bit(cf, name, shape, l, cp):
    """Items that pair two query tiles sharing each K/V tile compute every
    tile exactly as single-tile items do (same key order, same MMAs)."""
    w = wl.Workload(name, shape, 0, (), l, cp)
    b = wl.make_batch(w, 4)
    kp, vp = wl.make_pools(w, b, 4, "cuda")
    Hq, d = shape.n_q_heads, shape.head_dim
    q = randn_bf16((l, Hq, d), 41)
    fill_positions(kp, vp, b.pre_pages, cp, l, 42)
    eng = engine_for(cf, shape)
    eng.cf_set_prefill_split(1)
    pages = torch.as_tensor(b.pre_pages, device="cuda")
    outs = []
    for mode in pairing_modes(shape)[1:]:
        eng.cf_set_prefill_pairing(mode)
        o = torch.full((l, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        eng.cf_prefill_attn(q, cf.pool_of(kp, vp), l, cp, pages, o)
        outs.append(o)
    eng.cf_set_prefill_pairing(0)
    torch.cuda.synchronize()
    assert eng.cf_get_error()[0] == 0
    for o in outs[1:]:
        assert torch.equal(outs[0], o)


SPLIT_CASES = [
    ("l8b-short-after-long", wl.LLAMA8B, 123, 8082),
    ("l8b-two-tiles", wl.LLAMA8B, 256, 3000),
    ("q14b-odd-group", wl.QWEN14B, 200, 5000),
    ("tiny", wl.TINY, 77, 700),
]


@pytest.mark.parametrize("name,shape,l,cp", SPLIT_CASES, ids=[c[0] for c in SPLIT_CASES])
def test_prefill_key_range_cuts_agree_with_uncut(cf, name, shape, l, cp):
    """Items cut into key ranges (partials merged in order) agree with the
    uncut items within fp32 rounding, in every pair kind; the automatic
    policy cuts a short chunk after a long prefix; repeated runs are
    bit-identical."""
    w = wl.Workload(name, shape, 0, (), l, cp)
    b = wl.make_batch(w, 8)
    kp, vp = wl.make_pools(w, b, 8, "cuda")
    fill_positions(kp, vp, b.pre_pages, cp, l, 80)
    Hq, d = shape.n_q_heads, shape.head_dim
    q = randn_bf16((l, Hq, d), 18)
    eng = engine_for(cf, shape)
    pages = torch.as_tensor(b.pre_pages, device="cuda")
    ref = oracle.prefill_attention(f64(q), kp, vp, cp, b.pre_pages, 16)

    def run(pairing, split):
        eng.cf_set_prefill_pairing(pairing)
        eng.cf_set_prefill_split(split)
        o = torch.full((l, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        eng.cf_prefill_attn(q, cf.pool_of(kp, vp), l, cp, pages, o)
        torch.cuda.synchronize()
        assert eng.cf_get_error()[0] == 0
        return o

    for pairing in pairing_modes(shape):
        uncut = run(pairing, 1)
        for split in (0, 2, 5, 16):
            o = run(pairing, split)
            assert_close(o, f64(uncut), f"{name} pairing {pairing} split {split} vs uncut", 1e-2, 1e-3)
            assert_close(o, ref, f"{name} pairing {pairing} split {split}")
            assert torch.equal(o, run(pairing, split))
    n0 = eng.cf_launch_count()
    run(0, 0)
    cut = eng.cf_launch_count() - n0 == 2    # prefill + merge
    assert cut == (name != "tiny")   # tiny: 2 short units, nothing to balance
    eng.cf_set_prefill_pairing(0)
    eng.cf_set_prefill_split(0)


# several chunks of different requests in one launch (ConfluxServe §6.2
# Eq. 6): (shape, [(l_i, c_i)]) with ragged lengths, tile edges, empty and
# long prefixes
VARLEN_CASES = [
    ("tiny", wl.TINY, [(64, 128), (37, 0), (130, 300), (1, 17)]),
    ("l8b", wl.LLAMA8B, [(300, 0), (130, 2000), (129, 700), (1, 5), (256, 4096)]),
    ("q14b", wl.QWEN14B, [(1, 255), (128, 0), (513, 77)]),
    ("q32b-one", wl.QWEN32B, [(256, 1000)]),
]


def varlen_setup(shape, chunks, seed):
    w = wl.Workload("v", shape, 0, (), chunks[0][0], chunks[0][1], more_chunks=tuple(chunks[1:]))
    b = wl.make_batch(w, seed)
    kp, vp = wl.make_pools(w, b, seed, "cuda")
    for i, (l, c, pages) in enumerate(b.chunks):   # each chunk's own K/V (appended before attention)
        fill_positions(kp, vp, pages, c, l, 60 + 2 * i)
    lens, prefixes, table = b.chunk_table()
    return b, kp, vp, lens, prefixes, torch.as_tensor(table, device="cuda")


@pytest.mark.parametrize("name,shape,chunks", VARLEN_CASES, ids=[c[0] for c in VARLEN_CASES])
@pytest.mark.parametrize("pairing", [0, 1, 2, 3])
@pytest.mark.parametrize("split", [0, 4])
def test_prefill_varlen_matches_oracle(cf, name, shape, chunks, pairing, split):
    if pairing not in pairing_modes(shape):
        pytest.skip("head pairs need an even GQA group")
    b, kp, vp, lens, prefixes, table = varlen_setup(shape, chunks, 6)
    Hq, d = shape.n_q_heads, shape.head_dim
    P = int(lens.sum())
    q = randn_bf16((P, Hq, d), 16)
    out = torch.full((P, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    eng = engine_for(cf, shape)
    eng.cf_set_prefill_pairing(pairing)
    eng.cf_set_prefill_split(split)
    eng.cf_prefill_attn_varlen(q, cf.pool_of(kp, vp), lens, prefixes, table, out)
    torch.cuda.synchronize()
    assert eng.cf_get_error()[0] == 0
    eng.cf_set_prefill_pairing(0)
    eng.cf_set_prefill_split(0)
    r0 = 0
    for l, c, pages in b.chunks:
        ref = oracle.prefill_attention(f64(q[r0:r0 + l]), kp, vp, c, pages, 16)
        assert_close(out[r0:r0 + l], ref, f"varlen {name} chunk ({l}, {c})")
        r0 += l


@pytest.mark.parametrize("name,shape,chunks", VARLEN_CASES, ids=[c[0] for c in VARLEN_CASES])
def test_prefill_varlen_rows_equal_each_chunk_alone(cf, name, shape, chunks):
    """A chunk's rows do not depend on the other chunks sharing the launch:
    bit-identical to the chunk launched alone (same tiles, same key order)."""
    b, kp, vp, lens, prefixes, table = varlen_setup(shape, chunks, 7)
    Hq, d = shape.n_q_heads, shape.head_dim
    P = int(lens.sum())
    q = randn_bf16((P, Hq, d), 17)
    eng = engine_for(cf, shape)
    eng.cf_set_prefill_split(1)   # cuts depend on the whole launch; these rows compare bit for bit
    for mode in pairing_modes(shape)[1:]:
        eng.cf_set_prefill_pairing(mode)
        out = torch.full((P, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        eng.cf_prefill_attn_varlen(q, cf.pool_of(kp, vp), lens, prefixes, table, out)
        r0 = 0
        for i, (l, c, pages) in enumerate(b.chunks):
            alone = torch.full((l, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
            eng.cf_prefill_attn(q[r0:r0 + l].contiguous(), cf.pool_of(kp, vp), l, c,
                                torch.as_tensor(pages, device="cuda"), alone)
            torch.cuda.synchronize()
            assert torch.equal(out[r0:r0 + l], alone), (mode, i)
            r0 += l
    eng.cf_set_prefill_pairing(0)
    assert eng.cf_get_error()[0] == 0


def test_prefill_varlen_rejects_bad_chunks(cf):
    shape = wl.TINY
    eng = engine_for(cf, shape)
    kp = torch.zeros((8, shape.n_kv_heads, 16, shape.head_dim), dtype=torch.bfloat16, device="cuda")
    pool = cf.pool_of(kp, kp.clone())
    q = torch.zeros((64, shape.n_q_heads, shape.head_dim), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((33, 2), dtype=torch.int32, device="cuda")
    for lens, prefixes, tb, status in (([0, 5], [0, 0], table[:2], cf.CF_ERR_INVALID_ARG),
                                       ([5, 5], [-1, 0], table[:2], cf.CF_ERR_INVALID_ARG),
                                       ([5, 30], [0, 10], table[:2], cf.CF_ERR_INVALID_ARG),   # 3 pages > stride 2
                                       ([1] * 33, [0] * 33, table, cf.CF_ERR_UNSUPPORTED)):
        with pytest.raises(cf.CfError) as ex:
            eng.cf_prefill_attn_varlen(q, pool, lens, prefixes, tb, q)
        assert ex.value.status == status


def test_prefill_equals_decode_for_last_row(cf):
    """The last chunk row sees every key, exactly like a decode query."""
    shape = wl.LLAMA8B
    l, cp = 40, 1000
    w = wl.Workload("pd", shape, 0, (), l, cp)
    b = wl.make_batch(w, 5)
    kp, vp = wl.make_pools(w, b, 5, "cuda")
    fill_positions(kp, vp, b.pre_pages, cp, l, 50)
    Hq, d = shape.n_q_heads, shape.head_dim
    q = randn_bf16((l, Hq, d), 15)
    eng = engine_for(cf, shape)
    pages = torch.as_tensor(b.pre_pages, device="cuda")
    out_p = torch.zeros((l, Hq, d), dtype=torch.bfloat16, device="cuda")
    eng.cf_prefill_attn(q, cf.pool_of(kp, vp), l, cp, pages, out_p)
    out_d = torch.zeros((1, Hq, d), dtype=torch.bfloat16, device="cuda")
    keys = torch.tensor([cp + l], dtype=torch.int32, device="cuda")
    eng.cf_decode_attn(q[l - 1:].contiguous(), Hq * d, cf.pool_of(kp, vp), 1, keys, pages[None].contiguous(),
                       len(b.pre_pages), out_d, Hq * d)
    torch.cuda.synchronize()
    assert_close(out_p[l - 1:], f64(out_d), "prefill row vs decode", 1e-2, 1e-3)
