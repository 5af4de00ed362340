// Waterfill prefill dispatch of ConfluxServe (§6.3, App. E Algorithm 2):
// host code only, no CUDA call.  Binary search over the combined-load level
// with the iteration-latency estimator, then water-filling of the request's
// chunk toward that level.
#include <algorithm>
#include <vector>

#include "cf.h"

namespace {

constexpr long long kLevelCap = 1ll << 40;

// tokens rank r takes when the water stands at level w: min(cap_r, max(0, w - load_r))
long long filled(const long long* loads, const long long* cap, int n, long long w) {
  long long s = 0;
  for (int r = 0; r < n; ++r) {
    const long long f = w - loads[r];
    if (f > 0) s += f < cap[r] ? f : cap[r];
  }
  return s;
}

// Raises the lowest loads first to a common level (never above n_target);
// the tokens left after the last whole level go one each to the ranks
// standing at that level, lowest index first.
void assign(const long long* loads, int n, long long tokens, long long n_target, long long* give) {
  std::vector<long long> cap(n);
  long long lo = loads[0];
  for (int r = 0; r < n; ++r) {
    cap[r] = n_target - loads[r] > 0 ? n_target - loads[r] : 0;
    lo = std::min(lo, loads[r]);
  }
  // largest whole level w in [min load, n_target] with filled(w) <= tokens
  long long hi = std::max(lo, n_target);
  while (lo < hi) {
    const long long mid = lo + (hi - lo + 1) / 2;
    if (filled(loads, cap.data(), n, mid) <= tokens)
      lo = mid;
    else
      hi = mid - 1;
  }
  const long long w = lo;
  long long left = tokens;
  for (int r = 0; r < n; ++r) {
    const long long f = w - loads[r];
    give[r] = f > 0 ? (f < cap[r] ? f : cap[r]) : 0;
    left -= give[r];
  }
  for (int r = 0; r < n && left > 0; ++r)
    if (loads[r] + give[r] == w && give[r] < cap[r]) {
      give[r] += 1;
      --left;
    }
}

struct Planner {
  const cf_latency_model* m;
  int n_layers;
  const cf_dispatch_state* s;
  long long remaining, context;   // remaining < 0: no request
  std::vector<long long> loads, give, len, ctx;
  std::vector<cf_rank_load> ranks;

  // T_iter, B and l_i of the iteration level `level` would run; fills `give`
  cf_status plan(long long level, double* t, long long* budget, long long* chunk) {
    const int n = s->n_ranks;
    long long b = 0;
    for (int r = 0; r < n; ++r) b += level - loads[r] > 0 ? level - loads[r] : 0;
    long long l = 0;
    int nc = s->n_chunks;
    if (remaining < 0) {
      for (int r = 0; r < n; ++r) give[r] = level - loads[r] > 0 ? level - loads[r] : 0;
    } else {
      l = remaining < b ? remaining : b;
      assign(loads.data(), n, l, level, give.data());
      if (l > 0) {
        len[nc] = l;
        ctx[nc] = context;
        ++nc;
      }
    }
    for (int r = 0; r < n; ++r) {
      ranks[r].n_prefill = s->n_prefill[r] + give[r];
      ranks[r].n_decode = s->n_decode[r];
      ranks[r].ctx_sum = s->ctx_sum[r];
    }
    cf_latency_parts p;
    const cf_status st = cf_latency_predict(m, n, ranks.data(), nc, len.data(), ctx.data(), n_layers, &p);
    if (st != CF_OK) return st;
    *t = p.t_iter;
    *budget = b;
    *chunk = l;
    return CF_OK;
  }
};

}  // namespace

extern "C" {

cf_status cf_waterfill_assign(const long long* loads, int n_ranks, long long tokens, long long n_target,
                              long long* give) {
  if (!loads || !give || n_ranks < 1 || tokens < 0) return CF_ERR_INVALID_ARG;
  long long room = 0;
  for (int r = 0; r < n_ranks; ++r) {
    if (loads[r] < 0) return CF_ERR_INVALID_ARG;
    room += n_target - loads[r] > 0 ? n_target - loads[r] : 0;
  }
  if (tokens > room) return CF_ERR_INVALID_ARG;
  assign(loads, n_ranks, tokens, n_target, give);
  return CF_OK;
}

cf_status cf_waterfill_dispatch(const cf_latency_model* m, int n_layers, double tbt_slo, long long quantum,
                                const cf_dispatch_state* s, long long remaining, long long context,
                                cf_dispatch_result* out, long long* assign_out) {
  if (!m || !s || !out || n_layers < 0 || quantum < 1 || s->n_ranks < 1 || !s->n_decode || !s->ctx_sum ||
      !s->n_prefill || s->n_chunks < 0 || (s->n_chunks > 0 && (!s->chunk_len || !s->chunk_ctx)) ||
      (remaining >= 0 && context < 0) || !(tbt_slo == tbt_slo))
    return CF_ERR_INVALID_ARG;
  const int n = s->n_ranks;
  Planner P{m, n_layers, s, remaining, context};
  P.loads.resize(n);
  P.give.assign(n, 0);
  P.ranks.resize(n);
  P.len.assign(s->n_chunks + 1, 0);
  P.ctx.assign(s->n_chunks + 1, 0);
  long long max_load = 0;
  for (int r = 0; r < n; ++r) {
    if (s->n_decode[r] < 0 || s->n_prefill[r] < 0) return CF_ERR_INVALID_ARG;
    P.loads[r] = s->n_decode[r] + s->n_prefill[r];
    max_load = std::max(max_load, P.loads[r]);
  }
  for (int j = 0; j < s->n_chunks; ++j) {
    P.len[j] = s->chunk_len[j];
    P.ctx[j] = s->chunk_ctx[j];
  }
  cf_status st = CF_OK;
  auto feasible = [&](long long k, bool* ok) {
    double t;
    long long b, l;
    st = P.plan(k * quantum, &t, &b, &l);
    *ok = st == CF_OK && t <= tbt_slo;
    return st == CF_OK;
  };
  bool ok = false;
  if (!feasible(0, &ok)) return st;
  long long k_best = -1;
  if (ok) {
    long long lo = 0, hi = -1;
    if (remaining >= 0) {
      // above the first level whose budget covers the request nothing changes
      const long long top = (max_load + remaining + quantum - 1) / quantum;
      if (!feasible(top, &ok)) return st;
      if (ok)
        k_best = top;
      else
        hi = top;
    } else {
      long long k = 1;
      for (;;) {
        if (!feasible(k, &ok)) return st;
        if (!ok) {
          hi = k;
          lo = k / 2;
          break;
        }
        if (k * quantum >= kLevelCap) {
          k_best = k;
          break;
        }
        k *= 2;
      }
    }
    if (k_best < 0) {
      while (hi - lo > 1) {
        const long long mid = lo + (hi - lo) / 2;
        if (!feasible(mid, &ok)) return st;
        if (ok)
          lo = mid;
        else
          hi = mid;
      }
      k_best = lo;
    }
  }
  if (k_best < 0) {
    out->n_target = 0;
    out->budget = 0;
    out->chunk = 0;
    out->feasible = 0;
    out->t_iter = 0.0;
    if (assign_out)
      for (int r = 0; r < n; ++r) assign_out[r] = 0;
    return CF_OK;
  }
  double t;
  long long b, l;
  st = P.plan(k_best * quantum, &t, &b, &l);
  if (st != CF_OK) return st;
  out->n_target = k_best * quantum;
  out->budget = b;
  out->chunk = remaining >= 0 ? l : 0;
  out->feasible = 1;
  out->t_iter = t;
  if (assign_out)
    for (int r = 0; r < n; ++r) assign_out[r] = remaining >= 0 ? P.give[r] : 0;
  return CF_OK;
}

}  // extern "C"
