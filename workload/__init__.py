"""Seeded synthetic inputs for the co-batched layer step.

This module is shared by the CUDA path's tests/bench and by the CPU oracle.
It holds no arithmetic of the method: it only fixes shapes, draws random
numbers, rounds them to bf16 and lays out page tables.  Every tensor is drawn
from its own ``torch.Generator`` seeded with ``(seed, tag)`` so that any one
of them can be regenerated without the others.

Workloads (shapes from the five layer configurations the engine is measured
on; context numbers and the log-normal length mix are described in
ConfluxServe §8, Table 3 for the Mooncake-Toolagent prompt lengths, whose
P50 6,346 and spread sigma 0.86 the mix reproduces):

=====  ===========================================================
tiny   H 256, 4/2 heads, d 64, F 512; chunk 64 on prefix 128;
       decodes at contexts {17, 64, 100, 255}
l8b    Llama-3.1-8B-shaped layer; 16 decodes at 8192; chunk 1024, no prefix
q14b   Qwen3-14B-shaped layer with per-head QK-RMSNorm; 32 decodes at 8192;
       chunk 2048 on a 16384-token cached prefix
mix    Llama-3.1-8B shape; 128 decodes with log-normal contexts; chunk 256
       on a log-normal prefix; pool 1.25x the pages needed
q32b   Qwen3-32B-shaped layer; 32 decodes at 32768; chunk 4096 on 28672
=====  ===========================================================

Conventions (the pages leave them open; the readings are listed in the
design notes):

* ``c_j`` is the number of tokens already cached for decode request ``j``;
  its new token sits at position ``c_j`` and attends to ``c_j + 1`` keys.
* The prefill chunk's token ``i`` sits at position ``c_p + i``.
* Rows of the stacked token matrix are ``[prefill chunk rows; decode rows]``
  (ConfluxServe §4, Fig. 7: each rank forms ``[a3, b4]``).
* Paged KV pools are ``[num_pages, Hkv, page_size, d]`` bf16, one for K and
  one for V; the slot of position ``p`` of a request with page table ``pt``
  is ``pt[p // page_size] * page_size + p % page_size``.
* Cached slots hold i.i.d. N(0, 1) bf16 values (standing in for post-RoPE K
  and V).  Every slot that is not cached holds the bf16 NaN pattern 0x7FC1,
  so a kernel that reads a slot it should not read poisons its output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional, Tuple

import numpy as np
import torch

PAGE_SIZE = 16
# bf16 quiet-NaN bit pattern used to fill every KV slot that is not cached.
NAN_SENTINEL_BITS = 0x7FC1

# Stable tags so that each tensor has its own random stream.
_TAGS = {
    "lengths": 1, "pages": 2, "x": 3, "w_qkv": 4, "w_o": 5, "w_gate": 6,
    "w_up": 7, "w_down": 8, "g_attn": 9, "g_ffn": 10, "g_q": 11, "g_k": 12,
    "k_cache": 13, "v_cache": 14,
}


@dataclass(frozen=True)
class LayerShape:
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    rope_theta: float
    rms_eps: float
    qk_norm: bool

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def qkv_dim(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim


@dataclass(frozen=True)
class Workload:
    """One co-batched iteration: a prefill chunk plus resident decodes."""
    name: str
    shape: LayerShape
    n_decode: int
    dec_ctx: Optional[Tuple[int, ...]]        # None: drawn log-normal
    prefill_len: int                          # l (0 = no prefill chunk)
    prefill_prefix: Optional[int]             # c_p; None: drawn log-normal
    pool_slack: float = 1.0                   # pool pages / pages needed
    lognormal: Tuple[float, float, int, int] = (6346.0, 0.86, 512, 32768)
    description: str = ""
    # further prefill chunks (l_i, c_i) of other requests, stacked after the
    # first chunk's rows (the batch P of ConfluxServe §6.2 Eq. 6 / Alg. 1)
    more_chunks: Tuple[Tuple[int, int], ...] = ()


LLAMA8B = LayerShape(4096, 32, 8, 128, 14336, 5.0e5, 1e-5, False)
QWEN14B = LayerShape(5120, 40, 8, 128, 17408, 1.0e6, 1e-6, True)
QWEN32B = LayerShape(5120, 64, 8, 128, 25600, 1.0e6, 1e-6, False)
TINY = LayerShape(256, 4, 2, 64, 512, 1.0e4, 1e-5, False)

WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", TINY, 4, (17, 64, 100, 255), 64, 128,
                     description="tiny layer H256 4/2 heads d64 F512; chunk 64 on prefix 128; "
                                 "decodes {17,64,100,255}"),
    "l8b": Workload("l8b", LLAMA8B, 16, (8192,) * 16, 1024, 0,
                    description="Llama-3.1-8B-shaped layer; 16 decodes @8192 + 1024-token chunk, no prefix"),
    "q14b": Workload("q14b", QWEN14B, 32, (8192,) * 32, 2048, 16384,
                     description="Qwen3-14B-shaped layer with QK-norm; 32 decodes @8192 + 2048-token "
                                 "chunk on a 16384-token cached prefix"),
    "mix": Workload("mix", LLAMA8B, 128, None, 256, None, pool_slack=1.25,
                    description="Llama-3.1-8B shape; 128 decodes, log-normal contexts (median 6346, "
                                "sigma 0.86, clip [512,32768]) + 256-token chunk on a log-normal prefix"),
    "q32b": Workload("q32b", QWEN32B, 32, (32768,) * 32, 4096, 28672,
                     description="Qwen3-32B-shaped layer; 32 decodes @32768 + 4096-token chunk on a "
                                 "28672-token cached prefix"),
    "mchunk": Workload("mchunk", LLAMA8B, 16, (8192,) * 16, 1024, 0,
                       more_chunks=((512, 4096), (256, 12288), (128, 2048)),
                       description="Llama-3.1-8B-shaped layer; 16 decodes @8192 + four prefill chunks "
                                   "(l, c) = (1024, 0), (512, 4096), (256, 12288), (128, 2048)"),
}
# Index order of the five measured configurations.
WORKLOAD_ORDER = ("tiny", "l8b", "q14b", "mix", "q32b")


def reduced(base: Workload, dec_ctx, prefill_len, prefill_prefix, name=None) -> Workload:
    """Same layer shape as ``base`` with a smaller, explicitly given batch."""
    return Workload(name or f"{base.name}-slice", base.shape, len(dec_ctx), tuple(dec_ctx),
                    prefill_len, prefill_prefix, description=f"{base.name} shape, reduced batch")


def _gen(seed: int, tag: str, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000 + _TAGS[tag])
    return g


@dataclass
class Batch:
    """Host-side description of one iteration (all int32 numpy)."""
    workload: Workload
    dec_ctx: np.ndarray          # [n_decode] cached tokens before this step
    prefill_len: int
    prefill_prefix: int
    dec_pages: np.ndarray        # [n_decode, dec_stride] page ids (-1 padded)
    pre_pages: np.ndarray        # [ceil((c_p + l) / ps)] page ids
    num_pages: int
    page_size: int = PAGE_SIZE
    # further chunks (l_i, c_i, page ids) after the first chunk's rows
    more_chunks: Tuple[Tuple[int, int, np.ndarray], ...] = ()

    @property
    def n_decode(self) -> int:
        return int(self.dec_ctx.shape[0])

    @property
    def chunks(self):
        """Every prefill chunk as (l_i, c_i, page ids), in stacked-row order."""
        first = [(self.prefill_len, self.prefill_prefix, self.pre_pages)] if self.prefill_len > 0 else []
        return first + [(int(l), int(c), p) for l, c, p in self.more_chunks]

    @property
    def prefill_rows(self) -> int:
        return sum(l for l, _, _ in self.chunks)

    @property
    def n_tokens(self) -> int:
        return self.prefill_rows + self.n_decode

    def chunk_table(self):
        """(lengths, prefixes, page table [n_chunks, stride] -1 padded) of all chunks."""
        ch = self.chunks
        stride = max([len(p) for _, _, p in ch] + [1])
        pages = np.full((max(len(ch), 1), stride), -1, np.int32)
        for i, (_, _, p) in enumerate(ch):
            pages[i, :len(p)] = p
        return (np.array([l for l, _, _ in ch], np.int32), np.array([c for _, c, _ in ch], np.int32), pages)

    @property
    def dec_stride(self) -> int:
        return int(self.dec_pages.shape[1])


def _lognormal_lengths(w: Workload, n: int, g: torch.Generator) -> np.ndarray:
    med, sigma, lo, hi = w.lognormal
    z = torch.randn(n, generator=g, dtype=torch.float64).numpy()
    return np.clip(np.rint(np.exp(math.log(med) + sigma * z)), lo, hi).astype(np.int64)


def make_batch(w: Workload, seed: int = 0) -> Batch:
    """Context lengths and page tables (random permutation of the pool)."""
    ps = PAGE_SIZE
    if w.dec_ctx is None or w.prefill_prefix is None:
        drawn = _lognormal_lengths(w, w.n_decode + 1, _gen(seed, "lengths"))
    dec = np.asarray(w.dec_ctx if w.dec_ctx is not None else drawn[: w.n_decode], np.int64)
    cp = int(w.prefill_prefix if w.prefill_prefix is not None else drawn[-1])
    l = int(w.prefill_len)
    dec_need = (dec + 1 + ps - 1) // ps                      # pages incl. the new token
    pre_need = (cp + l + ps - 1) // ps if l > 0 else 0
    more_need = [(ml + mc + ps - 1) // ps for ml, mc in w.more_chunks]
    needed = int(dec_need.sum()) + pre_need + sum(more_need)
    num_pages = int(math.ceil(needed * w.pool_slack))
    perm = torch.randperm(num_pages, generator=_gen(seed, "pages")).numpy().astype(np.int64)
    stride = int(dec_need.max()) if len(dec) else 1
    dec_pages = np.full((len(dec), stride), -1, np.int64)
    at = 0
    pre_pages = perm[at:at + pre_need].copy()
    at += pre_need
    for j, n in enumerate(dec_need):
        dec_pages[j, :n] = perm[at:at + n]
        at += n
    more = []
    for (ml, mc), n in zip(w.more_chunks, more_need):
        more.append((int(ml), int(mc), perm[at:at + n].astype(np.int32)))
        at += n
    return Batch(w, dec.astype(np.int32), l, cp, dec_pages.astype(np.int32),
                 pre_pages.astype(np.int32), num_pages, more_chunks=tuple(more))


def _randn_bf16(shape, g, std=1.0, device="cpu", chunk=1 << 26) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 then rounded to bf16 (round-to-nearest-even)."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - s)
        t = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        flat[s:s + n] = t.to(torch.bfloat16)
    return out


def make_x(w: Workload, batch: Batch, seed: int = 0, device="cpu") -> torch.Tensor:
    """Stacked token matrix [T, H] bf16, N(0, 1)."""
    return _randn_bf16((batch.n_tokens, w.shape.hidden), _gen(seed, "x", device), device=device)


def make_weights(w: Workload, seed: int = 0, device="cpu", unit_gains: bool = False) -> Dict[str, torch.Tensor]:
    """Random-init weights of the layer, nn.Linear layout [out_features, in_features] bf16.

    w_qkv rows are the Q heads, then the K heads, then the V heads (the fused
    layout X_qkv in TKNP §4.4, Eq. 1).  Norm gains are 1 + N(0, 0.1) unless
    ``unit_gains``.
    """
    s = w.shape
    H, d, F = s.hidden, s.head_dim, s.ffn_dim
    out = {
        "w_qkv": _randn_bf16((s.qkv_dim, H), _gen(seed, "w_qkv", device), 0.02, device),
        "w_o": _randn_bf16((H, s.n_q_heads * d), _gen(seed, "w_o", device), 0.02, device),
        "w_gate": _randn_bf16((F, H), _gen(seed, "w_gate", device), 0.02, device),
        "w_up": _randn_bf16((F, H), _gen(seed, "w_up", device), 0.02, device),
        "w_down": _randn_bf16((H, F), _gen(seed, "w_down", device), 0.02, device),
    }
    def gain(n, tag):
        if unit_gains:
            return torch.ones(n, dtype=torch.bfloat16, device=device)
        return (1.0 + torch.randn(n, generator=_gen(seed, tag, device), device=device) * 0.1).to(torch.bfloat16)
    out["g_attn"] = gain(H, "g_attn")
    out["g_ffn"] = gain(H, "g_ffn")
    if s.qk_norm:
        out["g_q"] = gain(d, "g_q")
        out["g_k"] = gain(d, "g_k")
    return out


def make_pools(w: Workload, batch: Batch, seed: int = 0, device="cpu") -> Tuple[torch.Tensor, torch.Tensor]:
    """K and V pools [num_pages, Hkv, ps, d] bf16.

    Cached positions (0..c_j-1 of each decode, 0..c_i-1 of each chunk's
    request) hold N(0, 1) values; every other slot holds the NaN sentinel.
    Values are drawn request by request, position-major, so a request's
    cached KV does not depend on the page permutation.
    """
    s = w.shape
    ps = batch.page_size
    shape = (batch.num_pages, s.n_kv_heads, ps, s.head_dim)
    pools = []
    for tag in ("k_cache", "v_cache"):
        pool = torch.empty(shape, dtype=torch.bfloat16, device=device)
        pool.view(torch.int16).fill_(NAN_SENTINEL_BITS)
        g = _gen(seed, tag, device)
        reqs = [(batch.pre_pages, batch.prefill_prefix)] if batch.prefill_len > 0 else []
        reqs += [(batch.dec_pages[j], int(batch.dec_ctx[j])) for j in range(batch.n_decode)]
        reqs += [(p, c) for _, c, p in batch.more_chunks]   # after the decodes: earlier draws unchanged
        for pages, n in reqs:
            if n == 0:
                continue
            vals = _randn_bf16((n, s.n_kv_heads, s.head_dim), g, device=device)
            full, rem = divmod(n, ps)
            idx = torch.as_tensor(pages[:full].astype(np.int64), device=device)
            if full:
                pool[idx] = vals[:full * ps].view(full, ps, s.n_kv_heads, s.head_dim).transpose(1, 2)
            if rem:
                pool[int(pages[full]), :, :rem] = vals[full * ps:].transpose(0, 1)
        pools.append(pool)
    return pools[0], pools[1]


# --------------------------------------------------------------------------
# Random iterations for the latency-estimator study
# --------------------------------------------------------------------------
# Ranges of ConfluxServe §8.4 ("Latency-Estimator Accuracy"): prefill chunks
# of 32 to 10K tokens, decode batches of 1 to 128 requests, context lengths
# of 1K to 16K tokens (read as: every decode's c_j and the chunk's processed
# prefix c_p, each uniform over the range; K = 1024).
EST_CHUNK = (32, 10240)
EST_DECODES = (1, 128)
EST_CONTEXT = (1024, 16384)
_EST_KINDS = {"validate": 1, "calibrate": 2, "decode": 3, "prefill": 4}


def estimator_batches(seed: int, n: int, kind: str = "validate"):
    """``n`` random iterations as (l, c_p, dec_ctx tuple).

    ``validate`` / ``calibrate``: co-batched iterations (a chunk and decodes)
    from two independent streams; ``decode``: decodes only (l = 0);
    ``prefill``: a chunk only.  Lengths are uniform integers over the ranges
    above, inclusive."""
    rng = np.random.default_rng([int(seed), _EST_KINDS[kind]])
    out = []
    for _ in range(n):
        l = int(rng.integers(EST_CHUNK[0], EST_CHUNK[1] + 1)) if kind != "decode" else 0
        c_p = int(rng.integers(EST_CONTEXT[0], EST_CONTEXT[1] + 1)) if l else 0
        nd = int(rng.integers(EST_DECODES[0], EST_DECODES[1] + 1)) if kind != "prefill" else 0
        ctx = tuple(int(c) for c in rng.integers(EST_CONTEXT[0], EST_CONTEXT[1] + 1, size=nd))
        out.append((l, c_p, ctx))
    return out
