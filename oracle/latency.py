"""fp64 oracle of the ConfluxServe iteration-latency estimator.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm may use it.  It shares no code
with the native estimator in ``co_prefill_decode_gb300`` (which is C++ behind
the C ABI).

Source: ConfluxServe: Reconciling Resource Utilization and Parallelism
Efficiency across Prefill and Decode in LLM Serving — §6.2 "Latency Modeling
and Estimation" (Eq. 2-6), App. D "Latency Model Details" (Eq. 7-11) and
§8.4 "Latency-Estimator Accuracy" (MAPE over randomly sampled heterogeneous
batches).

The model, per iteration over L layers and N ranks:

* T_iter = L (T_GEMM + T_ATTN)                                    (Eq. 2)
* T_GEMM = f_GEMM(max_r (n_p^r + n_d^r))                          (Eq. 3)
* T_ATTN = max{beta T_P, alpha T_D}, alpha, beta >= 1             (Eq. 4)
* T_D = max_r f_D(sum_{i in D_r} c_i)                             (Eq. 5)
* T_P = f_comm(max_r n_p^r) + f_P((1/N) sum_{i in P} W_i)         (Eq. 6)
* W_i = l_i (c_i + (l_i + 1) / 2), the causal chunk workload      (Eq. 9)
* f_GEMM(n) = gamma n + gamma_0                                   (Eq. 7)
* f_D(W) = a_D W + a_D0                                           (Eq. 8)
* f_P(W) = a_P W + a_P0                                           (Eq. 10)
* f_comm(n) = a_comm n + a_comm0                                  (Eq. 11)

Readings where the pages are silent (listed in the design notes too):

* A path with no work takes no time: T_D = 0 when no rank holds a decode
  (the max of Eq. 5 runs over the ranks that hold one), T_P = 0 when no
  chunk is scheduled, T_GEMM = 0 when no rank has a token.  The fitted
  intercepts are the fixed cost of running a path, not of skipping it.
* f_comm is the Ulysses All-to-All of the prefill path; on one GPU it is
  zero (its coefficients are left at 0).
* "fit the corresponding coefficients from offline execution profiles"
  (App. D) is read as ordinary least squares of each line on its profile.
* "calibrate the contention factors alpha and beta" on heterogeneous
  profiles is read as: the pair on the grid {1, 1 + s, 1 + 2s, ...} <= f_max
  that minimises the MAPE (the accuracy measure of §8.4) of the model's
  prediction over the calibration batches; ties go to the smaller alpha,
  then the smaller beta.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np


@dataclass(frozen=True)
class LatencyModel:
    """Coefficients of the base latency functions (App. D Eq. 7, 8, 10, 11)
    and the contention factors of Eq. 4."""
    gamma: float = 0.0
    gamma0: float = 0.0
    a_d: float = 0.0
    a_d0: float = 0.0
    a_p: float = 0.0
    a_p0: float = 0.0
    a_comm: float = 0.0
    a_comm0: float = 0.0
    alpha: float = 1.0
    beta: float = 1.0


@dataclass(frozen=True)
class RankLoad:
    """One rank's share of an iteration: n_p^r prefill tokens, n_d^r decode
    tokens and the context lengths c_i of its resident decodes (§6.2)."""
    n_prefill: int = 0
    n_decode: int = 0
    contexts: Tuple[int, ...] = ()


# ---------------------------------------------------------------- Eq. 7-11
def f_gemm(m: LatencyModel, n: float) -> float:
    """App. D Eq. 7: shared linear operators over n rank-local tokens."""
    return m.gamma * float(n) + m.gamma0


def f_decode(m: LatencyModel, w: float) -> float:
    """App. D Eq. 8: decode attention with aggregate context W = sum c_i."""
    return m.a_d * float(w) + m.a_d0


def f_prefill(m: LatencyModel, w: float) -> float:
    """App. D Eq. 10: prefill attention with per-rank workload W."""
    return m.a_p * float(w) + m.a_p0


def f_comm(m: LatencyModel, n: float) -> float:
    """App. D Eq. 11: the two Ulysses All-to-Alls, largest prefill shard n."""
    return m.a_comm * float(n) + m.a_comm0


def chunk_workload(l: int, c: int) -> float:
    """App. D Eq. 9: causal attention work of a chunk of l tokens after c
    processed tokens, l (c + (l + 1) / 2)."""
    return float(l) * (float(c) + (float(l) + 1.0) / 2.0)


# ---------------------------------------------------------------- Eq. 2-6
def t_gemm(m: LatencyModel, ranks: Sequence[RankLoad]) -> float:
    """§6.2 Eq. 3: the largest combined token load across ranks."""
    n = max((r.n_prefill + r.n_decode for r in ranks), default=0)
    return f_gemm(m, n) if n > 0 else 0.0


def t_decode(m: LatencyModel, ranks: Sequence[RankLoad]) -> float:
    """§6.2 Eq. 5: the slowest rank's decode attention (ranks holding a
    decode only)."""
    vals = [f_decode(m, sum(float(c) for c in r.contexts)) for r in ranks if r.n_decode > 0]
    return max(vals) if vals else 0.0


def t_prefill(m: LatencyModel, ranks: Sequence[RankLoad],
              chunks: Sequence[Tuple[int, int]]) -> float:
    """§6.2 Eq. 6: All-to-All on the largest prefill shard plus the
    aggregate chunk workload spread evenly over the N ranks.  ``chunks`` are
    the scheduled (l_i, c_i)."""
    chunks = [(l, c) for l, c in chunks if l > 0]
    if not chunks:
        return 0.0
    n = len(ranks)
    w = sum(chunk_workload(l, c) for l, c in chunks) / n
    comm = f_comm(m, max(r.n_prefill for r in ranks)) if n > 1 else 0.0
    return comm + f_prefill(m, w)


def t_attn(m: LatencyModel, tp: float, td: float) -> float:
    """§6.2 Eq. 4: the two attention paths run concurrently, each slowed by
    its contention factor."""
    return max(m.beta * tp, m.alpha * td)


def t_iter(m: LatencyModel, ranks: Sequence[RankLoad], chunks: Sequence[Tuple[int, int]],
           n_layers: int = 1) -> dict:
    """§6.2 Eq. 2: T_iter = L (T_GEMM + T_ATTN), with the parts."""
    tg = t_gemm(m, ranks)
    td = t_decode(m, ranks)
    tp = t_prefill(m, ranks, chunks)
    ta = t_attn(m, tp, td)
    return {"t_iter": n_layers * (tg + ta), "t_gemm": tg, "t_attn": ta, "t_prefill": tp, "t_decode": td}


def one_gpu(l: int, c_p: int, contexts: Sequence[int]) -> Tuple[list, list]:
    """The single-rank batch of one co-batched layer step: a chunk of l
    tokens after c_p processed ones plus the decodes at ``contexts``."""
    ranks = [RankLoad(n_prefill=l, n_decode=len(contexts), contexts=tuple(int(c) for c in contexts))]
    return ranks, ([(l, c_p)] if l > 0 else [])


# ---------------------------------------------------------------- fitting
def fit_line(x: Sequence[float], y: Sequence[float]) -> Tuple[float, float]:
    """Ordinary least squares y ~ slope x + intercept (App. D: coefficients
    fitted from offline profiles).  Solved as a 2-column least-squares
    problem by numpy's lstsq."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    if x.size < 2 or np.ptp(x) == 0.0:
        raise ValueError("need at least two distinct x")
    a = np.stack([x, np.ones_like(x)], axis=1)
    sol, *_ = np.linalg.lstsq(a, y, rcond=None)
    return float(sol[0]), float(sol[1])


def mape(pred: Sequence[float], meas: Sequence[float]) -> float:
    """§8.4: mean absolute percentage error, in percent."""
    p = np.asarray(pred, dtype=np.float64)
    t = np.asarray(meas, dtype=np.float64)
    return float(100.0 * np.mean(np.abs(p - t) / np.abs(t)))


def factor_grid(f_max: float, step: float) -> np.ndarray:
    """{1, 1 + s, 1 + 2s, ...} up to f_max (inclusive within 1e-9)."""
    k = int(np.floor((f_max - 1.0) / step + 1e-9))
    return 1.0 + step * np.arange(k + 1, dtype=np.float64)


def calibrate(m: LatencyModel, t_g: Sequence[float], t_p: Sequence[float], t_d: Sequence[float],
              t_meas: Sequence[float], f_max: float = 3.0, step: float = 0.01) -> Tuple[LatencyModel, float]:
    """Contention factors of Eq. 4 from co-batched profiles: the grid pair
    minimising the MAPE of t_g + max(beta t_p, alpha t_d) against t_meas.
    Every (alpha, beta) is scored; the first minimum in (alpha, beta) order
    wins."""
    t_g = np.asarray(t_g, dtype=np.float64)
    t_p = np.asarray(t_p, dtype=np.float64)
    t_d = np.asarray(t_d, dtype=np.float64)
    t_m = np.asarray(t_meas, dtype=np.float64)
    grid = factor_grid(f_max, step)
    best = (np.inf, 1.0, 1.0)
    for a in grid:
        for b in grid:
            e = mape(t_g + np.maximum(b * t_p, a * t_d), t_m)
            if e < best[0]:
                best = (e, float(a), float(b))
    return replace(m, alpha=best[1], beta=best[2]), best[0]
