"""The decode-attention entry point that allocates nothing.

Callers that cannot allocate device memory (a runtime whose pool already owns
all free memory, a plugin under another framework's allocator, a loop that
must avoid cudaMalloc's device-wide synchronisation) use
cf_decode_attn_noalloc, which keeps its scratch in a fixed array inside the
library.  On all SMs it runs the same kernel with the same work plan as
cf_decode_attn, so its output must be the same bits, call after call, since
the shared array keeps the previous call's contents; it is also checked
against the fp64 oracle.  This file is collected last so that a failure here
comes after every other test has run.
"""
import numpy as np
import pytest
import torch

import oracle
import workload as wl
from helpers import assert_close, f64, randn_bf16

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20       # the array compiled into the library
ITEMS_PER_WARP, DECODE_WARPS = 4, 8


def scratch_need(n, Hq, Hkv, d, ctas):
    """Bytes of scratch a call needs, by the layout the entry point documents:
    256 bytes of words, the chunk plan, then (m, l) and O partials for every
    work item the plan may make on `ctas` CTAs."""
    a256 = lambda x: (x + 255) // 256 * 256
    G = Hq // Hkv
    items = ITEMS_PER_WARP * ctas * DECODE_WARPS + n * Hkv + 64
    off_ml = a256(256 + (n + 4) * 4)
    off_o = a256(off_ml + items * G * 2 * 4)
    return off_o + items * G * d * 4


def _case(shape, ctx, seed):
    w = wl.Workload("na", shape, len(ctx), ctx, 0, 0)
    b = wl.make_batch(w, seed)
    kp, vp = wl.make_pools(w, b, seed, "cuda")
    q = randn_bf16((len(ctx), shape.n_q_heads, shape.head_dim), 20 + seed)
    return w, b, kp, vp, q


def _oracle(b, kp, vp, q):
    return oracle.decode_attention(f64(q), kp, vp, b.dec_ctx.astype(np.int64), b.dec_pages, 16)


def test_noalloc_decode_matches_engine_decode_twice():
    import co_prefill_decode_gb300 as cf
    shape = wl.LLAMA8B
    Hq, Hkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    for call, ctx in enumerate([(3000, 17, 1, 640, 9000), (250, 4100, 33)]):
        w, b, kp, vp, q = _case(shape, ctx, 10 + call)
        n = len(ctx)
        keys = torch.as_tensor(b.dec_ctx, device="cuda")
        pages = torch.as_tensor(b.dec_pages, device="cuda")
        pool = cf.pool_of(kp, vp)
        W = {k: v.cuda() for k, v in wl.make_weights(w, 1).items()}
        eng = cf.Engine(cf.make_config(shape, 64, 64), W)
        ref = torch.zeros((n, Hq, d), dtype=torch.bfloat16, device="cuda")
        eng.cf_decode_attn(q, Hq * d, pool, n, keys, pages, b.dec_stride, ref, Hq * d)
        got = torch.full((n, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        cf.cf_decode_attn_noalloc(Hq, Hkv, d, 16, q, Hq * d, pool, n, keys, pages, b.dec_stride, got, Hq * d)
        torch.cuda.synchronize()
        assert eng.cf_get_error()[0] == 0
        # same kernel, same plan (all SMs): the same bits
        assert torch.equal(got, ref), f"no-alloc call {call} differs from cf_decode_attn"
        if call == 0:
            assert_close(got, _oracle(b, kp, vp, q), "no-alloc vs oracle")
        eng.close()


def test_noalloc_qwen32b_shape_fits_with_fewer_sms():
    """A Qwen3-32B-shaped batch (G = 8) too large for the array on all SMs is
    accepted on the largest CTA count whose plan fits, matches the oracle,
    and is rejected one CTA above it."""
    import co_prefill_decode_gb300 as cf
    shape = wl.QWEN32B
    Hq, Hkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    ctx = (32768,) + (700,) * 31
    n = len(ctx)
    sms = cf.device_sm_count()
    fits = [c for c in range(1, sms + 1) if scratch_need(n, Hq, Hkv, d, c) <= SCRATCH_BYTES]
    assert fits, "even one CTA does not fit"
    best = max(fits)
    if best == sms:
        pytest.skip("this device's SM count fits the array at this batch")
    w, b, kp, vp, q = _case(shape, ctx, 7)
    keys = torch.as_tensor(b.dec_ctx, device="cuda")
    pages = torch.as_tensor(b.dec_pages, device="cuda")
    pool = cf.pool_of(kp, vp)
    out = torch.full((n, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    for call in range(2):
        cf.cf_decode_attn_noalloc(Hq, Hkv, d, 16, q, Hq * d, pool, n, keys, pages, b.dec_stride, out, Hq * d,
                                  num_sms=best)
        torch.cuda.synchronize()
        if call == 0:
            first = out.clone()
    assert torch.equal(out, first)
    assert_close(out, _oracle(b, kp, vp, q), "q32b shape, reduced SMs")
    for c in (best + 1, 0):   # just past the boundary, and all SMs
        with pytest.raises(cf.CfError) as e:
            cf.cf_decode_attn_noalloc(Hq, Hkv, d, 16, q, Hq * d, pool, n, keys, pages, b.dec_stride, out, Hq * d,
                                      num_sms=c)
        assert e.value.status == cf.CF_ERR_INVALID_ARG
