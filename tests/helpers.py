"""Shared helpers of the GPU parity tests (inputs, tolerance, engine set-up)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workload as wl

# Tolerance of the layer's bf16 outputs against the fp64 oracle, per element
# e = |gpu - ref| / max(1, |ref|): max e <= 2e-2 and mean e <= 2e-3.  For
# |ref| <= 1 this is the absolute bound; above 1 it scales with the value,
# because one bf16 ulp there already exceeds an absolute 2e-2.
TOL_MAX = 2e-2
TOL_MEAN = 2e-3


def f64(t) -> np.ndarray:
    return oracle.to_f64(t)


def errors(gpu, ref):
    g = f64(gpu)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.isfinite(g).all(), "non-finite GPU output"
    e = np.abs(g - r) / np.maximum(1.0, np.abs(r))
    return float(e.max()), float(e.mean()), float(np.abs(g - r).max())


def assert_close(gpu, ref, what="", tol_max=TOL_MAX, tol_mean=TOL_MEAN):
    mx, mean, ab = errors(gpu, ref)
    assert mx <= tol_max and mean <= tol_mean, f"{what}: max e {mx:.3g} mean e {mean:.3g} (max abs {ab:.3g})"
    return mx, mean


def randn_bf16(shape, seed, device="cuda", std=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16).to(device)


def fill_positions(kp, vp, pages, start, n, seed, ps=16):
    """Writes N(0,1) K/V for positions start..start+n-1 of a request (test data)."""
    Hkv, d = kp.shape[1], kp.shape[3]
    k = randn_bf16((n, Hkv, d), seed, kp.device)
    v = randn_bf16((n, Hkv, d), seed + 1, kp.device)
    pos = np.arange(start, start + n)
    pg = torch.as_tensor(np.asarray(pages)[pos // ps].astype(np.int64), device=kp.device)
    off = torch.as_tensor(pos % ps, device=kp.device)
    kp[pg, :, off, :] = k
    vp[pg, :, off, :] = v


class LayerSetup:
    """Inputs of one workload on the GPU plus an engine over its weights."""

    def __init__(self, w: wl.Workload, seed=0, gen_device="cpu", unit_gains=False, max_tokens=None,
                 max_decode=None, decode_sms=0):
        import co_prefill_decode_gb300 as cf
        self.w, self.s = w, w.shape
        self.b = wl.make_batch(w, seed)
        self.x = wl.make_x(w, self.b, seed, gen_device).cuda()
        self.W = {k: v.cuda() for k, v in wl.make_weights(w, seed, gen_device, unit_gains).items()}
        kp, vp = wl.make_pools(w, self.b, seed, gen_device)
        self.kp, self.vp = kp.cuda(), vp.cuda()
        self.T = self.b.n_tokens
        b = self.b
        self.dec_ctx = torch.as_tensor(b.dec_ctx, device="cuda")
        self.dec_pages = torch.as_tensor(b.dec_pages, device="cuda")
        self.pre_pages = torch.as_tensor(b.pre_pages if len(b.pre_pages) else np.zeros(1, np.int32), device="cuda")
        self.cfg = cf.make_config(self.s, max_tokens or max(self.T, 1), max_decode or max(b.n_decode, 1),
                                  decode_sms)
        self.eng = cf.Engine(self.cfg, self.W)
        self.pool = cf.pool_of(self.kp, self.vp)
        self.multi = len(b.chunks) > 1
        if self.multi:   # the chunk-list form of the batch
            lens, prefixes, table = b.chunk_table()
            self.chunk_len, self.chunk_prefix = lens, prefixes
            self.chunk_pages = torch.as_tensor(table, device="cuda")
            self.batch = cf.batch_of(b.n_decode, self.dec_ctx, self.dec_pages, 0, 0, None,
                                     chunks=(lens, prefixes, self.chunk_pages))
        else:
            self.batch = cf.batch_of(b.n_decode, self.dec_ctx, self.dec_pages, b.prefill_len, b.prefill_prefix,
                                     self.pre_pages)
        self.out = torch.empty_like(self.x)

    def step(self):
        self.eng.cf_layer_step(self.batch, self.x, self.out, self.pool)
        torch.cuda.synchronize()
        st, msg = self.eng.cf_get_error()
        assert st == 0, msg
        return self.out

    def oracle_weights(self):
        return oracle.LayerWeights64.from_torch({k: v.cpu() for k, v in self.W.items()})
