"""The decode-attention entry point that allocates nothing.

Callers that cannot allocate device memory (a runtime whose pool already owns
all free memory, a plugin under another framework's allocator, a loop that
must avoid cudaMalloc's device-wide synchronisation) use
cf_decode_attn_noalloc, which keeps its scratch in a fixed array inside the
library.  Its output must match cf_decode_attn's on the same inputs, call
after call, since the shared array keeps the previous call's contents.
This file is collected last so that a failure here comes after every other
test has run.
"""
import numpy as np
import pytest
import torch

import workload as wl
from helpers import assert_close, f64, randn_bf16

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_engine_decode_twice():
    import co_prefill_decode_gb300 as cf
    shape = wl.LLAMA8B
    outs = []
    for call, ctx in enumerate([(3000, 17, 1, 640, 9000), (250, 4100, 33)]):
        w = wl.Workload("na", shape, len(ctx), ctx, 0, 0)
        b = wl.make_batch(w, 10 + call)
        kp, vp = wl.make_pools(w, b, 10 + call, "cuda")
        n, Hq, Hkv, d = len(ctx), shape.n_q_heads, shape.n_kv_heads, shape.head_dim
        q = randn_bf16((n, Hq, d), 30 + call)
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
        assert_close(got, f64(ref), f"no-alloc call {call}", 1e-2, 1e-3)
        outs.append(got)
        eng.close()


def test_noalloc_rejects_batches_beyond_its_scratch():
    import co_prefill_decode_gb300 as cf
    shape = wl.QWEN32B        # G = 8: the largest partials per item
    n = 2000
    q = torch.zeros((n, shape.n_q_heads, shape.head_dim), dtype=torch.bfloat16, device="cuda")
    kp = torch.zeros((4, shape.n_kv_heads, 16, shape.head_dim), dtype=torch.bfloat16, device="cuda")
    keys = torch.ones(n, dtype=torch.int32, device="cuda")
    pages = torch.zeros((n, 1), dtype=torch.int32, device="cuda")
    with pytest.raises(cf.CfError) as e:
        cf.cf_decode_attn_noalloc(shape.n_q_heads, shape.n_kv_heads, shape.head_dim, 16, q,
                                  shape.n_q_heads * shape.head_dim, cf.pool_of(kp, kp.clone()), n, keys, pages, 1,
                                  torch.empty_like(q), shape.n_q_heads * shape.head_dim)
    assert e.value.status == cf.CF_ERR_INVALID_ARG
