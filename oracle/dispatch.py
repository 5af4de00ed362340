"""Oracle of the ConfluxServe waterfill prefill dispatcher.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU arms may use it; it shares no code with the native
dispatcher in ``co_prefill_decode_gb300`` (C++ behind the C ABI).

Sources: ConfluxServe: Reconciling Resource Utilization and Parallelism
Efficiency across Prefill and Decode in LLM Serving — §6.3 "Prefill:
waterfill dispatch" and App. E "Waterfill Dispatch" (Algorithm 2); the
worked example in the paper-daily.com summary of the same paper (section
on per-iteration scheduling: decode loads 40 / 10 / 10 / 0, level 300,
capacities 260 / 290 / 290 / 300, budget 1140, a 2000-token prompt cut to
1140).

What the dispatcher computes (Algorithm 2):

1. n_target: the largest combined-load level, restricted to multiples of
   the alignment quantum q, whose iteration latency (the estimator of
   §6.2, ``oracle.latency``) stays within the TBT SLO tau;
2. B = sum_r max{0, n_target - n_d^r - n_p^r(A_p)};
3. without a request: return B;
4. with request i (remaining prefill m_i): l_i = min{m_i, B};
5. A_i = WaterfillAssign(D, A_p, l_i, n_target).

Readings where the pages are silent (listed in the design notes too):

* Feasibility of a level n: the iteration that level would run.  Rank r
  gets the prefill tokens it has (n_p^r) plus what the waterfill gives it;
  with a request those are A_i(n) for l_i(n) = min{m_i, B(n)}, and the
  request's chunk (l_i(n), c_i) joins the scheduled chunks P; without a
  request every rank is filled to the level (capacity tokens count toward
  Eq. 3 and the f_comm shard, but carry no attention workload: "omits the
  candidate-specific prefill workload").  Feasible iff T_iter <= tau.
* Search: level 0 first (infeasible: nothing fits, B = 0); with a request
  the search stops at the first level whose budget covers m_i (above it
  nothing changes); without one the upper end is found by doubling, up to
  2^40 tokens.  Then bisection between the last feasible and the first
  infeasible multiple of q.
* WaterfillAssign: water-filling in the literal sense.  Starting from the
  loads n_d^r + n_p^r, the l_i tokens raise the lowest ranks first to a
  common level w (never above n_target); tokens left over after the last
  whole level go one each to the ranks standing at w, lowest rank index
  first.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

from oracle import latency as L

LEVEL_CAP = 1 << 40


@dataclass(frozen=True)
class DecodeState:
    """Per-rank decode state D: n_d^r and the contexts of the resident decodes."""
    n_decode: Tuple[int, ...]
    contexts: Tuple[Tuple[int, ...], ...]


def waterfill_assign(loads: Sequence[int], tokens: int, n_target: int) -> List[int]:
    """Raise the lowest loads first; returns the tokens each rank receives."""
    n = len(loads)
    cap = [max(0, n_target - x) for x in loads]
    assert tokens <= sum(cap), "more tokens than the level admits"
    give = [0] * n
    left = tokens
    # pour one level at a time: every rank below the current water line
    # (and below n_target) takes one token per level
    w = min(loads) if loads else 0
    while left > 0:
        below = [r for r in range(n) if loads[r] + give[r] <= w and give[r] < cap[r]]
        if len(below) <= left:
            for r in below:
                give[r] += 1
            left -= len(below)
            w += 1
        else:
            for r in below[:left]:
                give[r] += 1
            left = 0
    return give


def _ranks(dec: DecodeState, n_prefill: Sequence[int]) -> List[L.RankLoad]:
    return [L.RankLoad(int(p), int(d), tuple(c)) for p, d, c in zip(n_prefill, dec.n_decode, dec.contexts)]


def _plan(m: L.LatencyModel, n_layers: int, dec: DecodeState, a_p: Sequence[int],
          chunks: Sequence[Tuple[int, int]], level: int, request: Optional[Tuple[int, int]]):
    """(T_iter, B, l_i, A_i) of the iteration level n would run."""
    loads = [d + p for d, p in zip(dec.n_decode, a_p)]
    budget = sum(max(0, level - x) for x in loads)
    if request is None:
        fill = [max(0, level - x) for x in loads]
        t = L.t_iter(m, _ranks(dec, [p + f for p, f in zip(a_p, fill)]), list(chunks), n_layers)["t_iter"]
        return t, budget, 0, fill
    m_i, c_i = request
    l_i = min(m_i, budget)
    give = waterfill_assign(loads, l_i, level)
    t = L.t_iter(m, _ranks(dec, [p + g for p, g in zip(a_p, give)]),
                 list(chunks) + ([(l_i, c_i)] if l_i > 0 else []), n_layers)["t_iter"]
    return t, budget, l_i, give


def waterfill(m: L.LatencyModel, n_layers: int, tau: float, quantum: int, dec: DecodeState,
              a_p: Sequence[int], chunks: Sequence[Tuple[int, int]],
              request: Optional[Tuple[int, int]] = None) -> dict:
    """Algorithm 2.  ``request`` = (m_i, c_i) or None.  Returns n_target, B,
    and with a request l_i and A_i."""
    assert quantum >= 1
    loads = [d + p for d, p in zip(dec.n_decode, a_p)]

    def feasible(k):
        return _plan(m, n_layers, dec, a_p, chunks, k * quantum, request)[0] <= tau

    if not feasible(0):
        k_best = None
    else:
        if request is not None:
            hi = -(-(max(loads) + request[0]) // quantum)
            if feasible(hi):
                k_best = hi
                hi = None
        else:
            k = 1
            hi = None
            k_best = None
            while True:
                if not feasible(k):
                    hi = k
                    break
                if k * quantum >= LEVEL_CAP:
                    k_best = k
                    break
                k *= 2
        if hi is not None:
            lo = 0 if request is not None else hi // 2
            while hi - lo > 1:
                mid = (lo + hi) // 2
                if feasible(mid):
                    lo = mid
                else:
                    hi = mid
            k_best = lo
    if k_best is None:
        return {"n_target": 0, "budget": 0, "chunk": 0, "assign": [0] * len(loads), "feasible": False}
    level = k_best * quantum
    t, budget, l_i, give = _plan(m, n_layers, dec, a_p, chunks, level, request)
    return {"n_target": level, "budget": budget, "chunk": l_i if request is not None else 0,
            "assign": give if request is not None else [0] * len(loads), "feasible": True, "t_iter": t}
