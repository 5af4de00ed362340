"""fp64 oracle of the co-batched layer step (test infrastructure only).

Each function cites the passage it restates.  Everything is plain numpy in
float64; the only library primitives used are matrix products and
elementwise transcendental functions.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, Iterable, Optional, Sequence

import numpy as np
import torch


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------
def to_f64(t) -> np.ndarray:
    """bf16/fp32 torch tensor (any device) or array -> exact float64 numpy."""
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits (1 implicit + 7 stored) and the float32
    exponent range; below 2^-126 its spacing is fixed at 2^-133.  The result
    is returned as float64 (exactly representable).
    """
    a = np.asarray(a, dtype=np.float64)
    m, e = np.frexp(a)                       # a = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                  # subnormal range: fixed spacing
    r = np.ldexp(np.rint(np.ldexp(a, 8 - e)), e - 8)   # np.rint: ties to even
    big = np.abs(r) > float.fromhex("0x1.fep127")       # beyond max bf16
    r = np.where(big, np.copysign(np.inf, a), r)
    return np.where(np.isfinite(a), r, a)


# --------------------------------------------------------------------------
# per-token operators
# --------------------------------------------------------------------------
def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis.

    The layer normalises its input before QKV and its residual stream before
    the FFN (Decode Token Parallelism §4.3: "output projection, residual and
    normalization, and MLP"); RMSNorm is the norm of the Llama/Qwen shapes.
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotary embedding, rotate-half form, on x[..., n, heads, d] at pos[n].

    For i < d/2 with angle a_i = pos * theta^(-2i/d):
      x'[i]       = x[i] cos a_i - x[i + d/2] sin a_i
      x'[i + d/2] = x[i] sin a_i + x[i + d/2] cos a_i
    (Decode Token Parallelism §4.3 applies rotary embeddings before the KV
    append, so the cache holds rotated keys.)
    """
    d = x.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / d)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]   # [n, d/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z)."""
    return z / (1.0 + np.exp(-z))


def swiglu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """silu(gate) * up — the gated FFN activation of the Llama/Qwen shapes."""
    return silu(gate) * up


# --------------------------------------------------------------------------
# paged KV
# --------------------------------------------------------------------------
def slot_of(pages: np.ndarray, pos, page_size: int) -> np.ndarray:
    """Pool slot of token position ``pos`` of a request with page table ``pages``.

    ConfluxServe §7 (PagedAttention blocks addressed through per-request
    block tables): slot = pages[pos // ps] * ps + pos % ps.
    """
    pos = np.asarray(pos, dtype=np.int64)
    return np.asarray(pages, dtype=np.int64)[pos // page_size] * page_size + pos % page_size


def gather_request_kv(pool, pages: np.ndarray, n: int, page_size: int) -> np.ndarray:
    """Positions 0..n-1 of one request from a pool [num_pages, Hkv, ps, d].

    Returns a contiguous float64 array [n, Hkv, d] (token-major)."""
    if n == 0:
        shape = tuple(pool.shape)
        return np.zeros((0, shape[1], shape[3]))
    npg = (n + page_size - 1) // page_size
    idx = np.asarray(pages[:npg], dtype=np.int64)
    if isinstance(pool, torch.Tensor):
        blk = to_f64(pool[torch.as_tensor(idx, device=pool.device)])
    else:
        blk = np.asarray(pool, dtype=np.float64)[idx]
    # [npg, Hkv, ps, d] -> [npg, ps, Hkv, d] -> [npg*ps, Hkv, d]
    tok = blk.transpose(0, 2, 1, 3).reshape(npg * page_size, blk.shape[1], blk.shape[3])
    return tok[:n]


def kv_append(k_pool: np.ndarray, v_pool: np.ndarray, k: np.ndarray, v: np.ndarray,
              slots: np.ndarray, page_size: int) -> None:
    """Scatter rows k[r], v[r] ([n, Hkv, d]) to pool slots ``slots[r]`` in place.

    ConfluxServe §4 (Fig. 8): a decode request extends its own KV with its new
    token; a prefill request appends its chunk's K/V.
    """
    slots = np.asarray(slots, dtype=np.int64)
    page, off = slots // page_size, slots % page_size
    for r in range(len(slots)):
        k_pool[page[r], :, off[r], :] = k[r]
        v_pool[page[r], :, off[r], :] = v[r]


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, qpos: np.ndarray,
              block: int = 256) -> np.ndarray:
    """Causal GQA attention for one request.

    q [nq, Hq, d] at positions qpos[nq]; K, V [n, Hkv, d] hold positions
    0..n-1.  Output [nq, Hq, d] with, for query r and head h,
      softmax_j(q[r,h] . K[j, h // G] / sqrt(d) + M[r, j]) V[j, h // G],
    M[r, j] = 0 if j <= qpos[r] else -inf (Adaptive Context Parallelism
    §2.1).  Softmax subtracts the row max, exponentiates and divides.
    """
    nq, Hq, d = q.shape
    n, Hkv, _ = K.shape
    G = Hq // Hkv
    out = np.zeros_like(q)
    keypos = np.arange(n)
    scale = 1.0 / math.sqrt(d)
    for h in range(Hq):
        kh, vh = K[:, h // G, :], V[:, h // G, :]
        for r0 in range(0, nq, block):
            r1 = min(nq, r0 + block)
            s = (q[r0:r1, h, :] @ kh.T) * scale                     # [b, n]
            s = np.where(keypos[None, :] <= qpos[r0:r1, None], s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=1, keepdims=True)
            out[r0:r1, h, :] = p @ vh
    return out


def decode_attention(q: np.ndarray, k_pool, v_pool, ctx_incl: np.ndarray,
                     pages: np.ndarray, page_size: int) -> np.ndarray:
    """Decode attention: request j's single query sees its ctx_incl[j] keys.

    ConfluxServe Table 7 ("each request attends to its own KV state"); the
    query sits at position ctx_incl[j] - 1, so every cached key is visible.
    """
    out = np.zeros_like(q)
    for j in range(q.shape[0]):
        n = int(ctx_incl[j])
        K = gather_request_kv(k_pool, pages[j], n, page_size)
        V = gather_request_kv(v_pool, pages[j], n, page_size)
        out[j:j + 1] = attention(q[j:j + 1], K, V, np.array([n - 1]))
    return out


def prefill_attention(q: np.ndarray, k_pool, v_pool, prefix: int, pages: np.ndarray,
                      page_size: int) -> np.ndarray:
    """Chunked causal prefill attention over the cached prefix plus the chunk.

    Chunk query i sits at position prefix + i and sees keys 0..prefix+i
    (ConfluxServe §4 "subsequent chunks reuse historical KV"; Adaptive
    Context Parallelism §2.2: uncached queries attend to the cached prefix
    and causally to the preceding uncached tokens).
    """
    l = q.shape[0]
    n = prefix + l
    K = gather_request_kv(k_pool, pages, n, page_size)
    V = gather_request_kv(v_pool, pages, n, page_size)
    return attention(q, K, V, prefix + np.arange(l))


def chunk_workload(R: int, P: int) -> int:
    """Unmasked (query, key) pairs of an R-token chunk on a P-token prefix.

    Adaptive Context Parallelism §2.2 Eq. 1: W(R, P) = RP + R(R+1)/2;
    ConfluxServe App. D Eq. 9 writes it l(c + (l+1)/2).
    """
    return R * P + R * (R + 1) // 2


# --------------------------------------------------------------------------
# the layer step
# --------------------------------------------------------------------------
@dataclass
class LayerWeights64:
    w_qkv: np.ndarray   # [(Hq+2Hkv)d, H]
    w_o: np.ndarray     # [H, Hq d]
    w_gate: np.ndarray  # [F, H]
    w_up: np.ndarray    # [F, H]
    w_down: np.ndarray  # [H, F]
    g_attn: np.ndarray
    g_ffn: np.ndarray
    g_q: Optional[np.ndarray] = None
    g_k: Optional[np.ndarray] = None

    @staticmethod
    def from_torch(w: Dict[str, torch.Tensor]) -> "LayerWeights64":
        return LayerWeights64(**{k: to_f64(v) for k, v in w.items()})


def layer_step(x: np.ndarray, W: LayerWeights64, shape, batch, k_pool, v_pool,
               round_bf16: bool = True, rows: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """One co-batched layer step.

    x [T, H] is the stacked token matrix, rows ordered [prefill chunks; decodes]
    (ConfluxServe §4, Fig. 7); the chunks of several requests (the batch P of
    ConfluxServe §6.2 Eq. 6) follow one another, chunk i's row r sitting at
    position c_i + r of its own request.  ``k_pool``/``v_pool`` hold the cache BEFORE the
    step (torch or numpy, [num_pages, Hkv, ps, d]); they are not modified.

    Steps (ConfluxServe Fig. 1 and §4; Decode Token Parallelism §4.3):
      1. xn = RMSNorm(x) g_attn
      2. qkv = xn W_qkv^T, split Q | K | V heads (Decode Token Parallelism §4.4)
      3. optional per-head RMSNorm of q and k over d (QK-norm)
      4. RoPE at each row's position (chunk row i: c_i + i; decode j: c_j)
      5. append k, v at slot(position) of the row's request
      6. attention: each chunk's rows causal over its own request's prefix +
         chunk, decode rows over their own c_j + 1 keys
      7. h = x + O W_o^T
      8. hn = RMSNorm(h) g_ffn
      9. out = h + (silu(hn W_gate^T) * (hn W_up^T)) W_down^T

    With ``round_bf16`` every tensor handed from one step to the next (xn;
    q, k, v after RoPE; the attention output; hn; the FFN activation; out) is
    rounded to bf16; h stays unrounded.  ``rows`` restricts the returned
    outputs to those stacked rows (all K/V rows a selected row depends on are
    still computed).
    """
    s = shape
    Hq, Hkv, d, ps = s.n_q_heads, s.n_kv_heads, s.head_dim, batch.page_size
    chunks = list(batch.chunks)            # (l_i, c_i, page ids), stacked in this order
    nd = batch.n_decode
    P = sum(c[0] for c in chunks)          # prefill rows
    T = P + nd
    R = bf16_round if round_bf16 else (lambda a: a)
    rows = np.arange(T) if rows is None else np.asarray(sorted(set(int(r) for r in rows)))
    pre_rows = rows[rows < P]
    dec_rows = rows[rows >= P]
    # rows whose q/k/v are needed: in each chunk every row up to its last
    # selected one (its keys are visible to later rows of the same chunk),
    # plus the selected decode rows.
    segs, need_parts, pos_parts = [], [], []
    r0 = 0
    for l_i, c_i, pages_i in chunks:
        sel = pre_rows[(pre_rows >= r0) & (pre_rows < r0 + l_i)]
        n_i = int(sel.max()) - r0 + 1 if len(sel) else 0
        segs.append((r0, l_i, c_i, pages_i, n_i, sel))
        need_parts.append(r0 + np.arange(n_i))
        pos_parts.append(c_i + np.arange(n_i))
        r0 += l_i
    need_pre = np.concatenate(need_parts) if need_parts else np.arange(0)
    need = np.concatenate([need_pre, dec_rows]).astype(np.int64)
    pos = np.concatenate(pos_parts + [batch.dec_ctx[dec_rows - P].astype(np.int64)]).astype(np.int64)

    xs = x[need]
    xn = R(rmsnorm(xs, W.g_attn, s.rms_eps))
    qkv = xn @ W.w_qkv.T
    q = qkv[:, :Hq * d].reshape(-1, Hq, d)
    k = qkv[:, Hq * d:(Hq + Hkv) * d].reshape(-1, Hkv, d)
    v = qkv[:, (Hq + Hkv) * d:].reshape(-1, Hkv, d)
    if s.qk_norm:
        q = rmsnorm(q, W.g_q, s.rms_eps)
        k = rmsnorm(k, W.g_k, s.rms_eps)
    q = R(rope(q, pos, s.rope_theta))
    k = R(rope(k, pos, s.rope_theta))
    v = R(v)

    attn = np.zeros((len(need), Hq, d))
    where_pre = []
    off = 0                                # index of the chunk's first row in ``need``
    for r0, l_i, c_i, pages_i, n_i, sel in segs:
        if n_i:
            # the request's cached prefix followed by the chunk's own (appended) keys
            Kc = gather_request_kv(k_pool, pages_i, c_i, ps)
            Vc = gather_request_kv(v_pool, pages_i, c_i, ps)
            K = np.concatenate([Kc, k[off:off + n_i]])
            V = np.concatenate([Vc, v[off:off + n_i]])
            loc = sel - r0                 # only the selected rows need attention
            attn[off + loc] = attention(q[off + loc], K, V, c_i + loc)
            where_pre.append(off + loc)
        off += n_i
    npre = off
    for t, r in enumerate(dec_rows):
        j = int(r) - P
        c = int(batch.dec_ctx[j])
        Kc = gather_request_kv(k_pool, batch.dec_pages[j], c, ps)
        Vc = gather_request_kv(v_pool, batch.dec_pages[j], c, ps)
        K = np.concatenate([Kc, k[npre + t:npre + t + 1]])
        V = np.concatenate([Vc, v[npre + t:npre + t + 1]])
        attn[npre + t] = attention(q[npre + t:npre + t + 1], K, V, np.array([c]))[0]
    attn = R(attn)

    # positions in ``need`` of the selected rows
    where = np.concatenate(where_pre + [npre + np.arange(len(dec_rows))]).astype(np.int64)
    a_sel = attn[where].reshape(len(rows), Hq * d)
    h = x[rows] + a_sel @ W.w_o.T
    hn = R(rmsnorm(h, W.g_ffn, s.rms_eps))
    act = R(swiglu(hn @ W.w_gate.T, hn @ W.w_up.T))
    out = R(h + act @ W.w_down.T)

    # slots written by the append, for the selected rows
    slots = []
    for r in rows:
        if r < P:
            for r0, l_i, c_i, pages_i, _, _ in segs:
                if r0 <= r < r0 + l_i:
                    slots.append(int(slot_of(pages_i, c_i + int(r) - r0, ps)))
                    break
        else:
            j = int(r) - P
            slots.append(int(slot_of(batch.dec_pages[j], int(batch.dec_ctx[j]), ps)))
    return {
        "rows": rows, "out": out, "h": h, "hn": hn, "act": act,
        "attn": attn[where], "q": q[where], "k": k[where], "v": v[where],
        "xn": xn[where], "slots": np.asarray(slots, dtype=np.int64),
        # every row whose q/k/v were computed (all chunk rows up to the last
        # selected one, then the selected decode rows), in stacked-row order
        "need_rows": need, "q_need": q, "k_need": k, "v_need": v, "xn_need": xn,
    }
