// Iteration-latency estimator of ConfluxServe (§6.2 Eq. 2-6, App. D
// Eq. 7-11): host code only, no CUDA call.  A scheduler queries it once per
// candidate batch, so prediction is O(ranks + chunks) with no allocation.
#include <cmath>
#include <cstddef>

#include "cf.h"

namespace {

inline double lin(double a, double a0, double x) { return a * x + a0; }

bool finite_model(const cf_latency_model& m) {
  const double v[] = {m.gamma, m.gamma0, m.a_d, m.a_d0, m.a_p, m.a_p0, m.a_comm, m.a_comm0, m.alpha, m.beta};
  for (double x : v)
    if (!std::isfinite(x)) return false;
  return true;
}

}  // namespace

extern "C" {

cf_status cf_latency_predict(const cf_latency_model* m, int n_ranks, const cf_rank_load* ranks, int n_chunks,
                             const long long* chunk_len, const long long* chunk_ctx, int n_layers,
                             cf_latency_parts* out) {
  if (!m || !out || n_ranks < 1 || !ranks || n_chunks < 0 || n_layers < 0) return CF_ERR_INVALID_ARG;
  if (n_chunks > 0 && (!chunk_len || !chunk_ctx)) return CF_ERR_INVALID_ARG;
  if (!finite_model(*m)) return CF_ERR_INVALID_ARG;
  // Eq. 3: the shared linear region waits for the largest combined load.
  // Eq. 5: decode waits for the rank with the largest f_D over the ranks
  // that hold decodes.  f_comm's shard is the largest n_p^r (Eq. 6).
  long long max_load = 0, max_np = 0;
  double t_d = 0.0;
  bool any_decode = false;
  for (int r = 0; r < n_ranks; ++r) {
    const cf_rank_load& q = ranks[r];
    if (q.n_prefill < 0 || q.n_decode < 0 || !(q.ctx_sum >= 0.0) || !std::isfinite(q.ctx_sum))
      return CF_ERR_INVALID_ARG;
    if (q.n_prefill + q.n_decode > max_load) max_load = q.n_prefill + q.n_decode;
    if (q.n_prefill > max_np) max_np = q.n_prefill;
    if (q.n_decode > 0) {
      const double f = lin(m->a_d, m->a_d0, q.ctx_sum);
      if (!any_decode || f > t_d) t_d = f;
      any_decode = true;
    }
  }
  // Eq. 6 + Eq. 9: the chunks' causal workload l (c + (l+1)/2), spread
  // evenly over the ranks by the sequence-parallel attention.
  double w = 0.0;
  bool any_chunk = false;
  for (int i = 0; i < n_chunks; ++i) {
    if (chunk_len[i] < 0 || chunk_ctx[i] < 0) return CF_ERR_INVALID_ARG;
    if (chunk_len[i] == 0) continue;
    const double l = (double)chunk_len[i], c = (double)chunk_ctx[i];
    w += l * (c + (l + 1.0) / 2.0);
    any_chunk = true;
  }
  double t_p = 0.0;
  if (any_chunk) {
    t_p = lin(m->a_p, m->a_p0, w / n_ranks);
    if (n_ranks > 1) t_p += lin(m->a_comm, m->a_comm0, (double)max_np);
  }
  const double t_g = max_load > 0 ? lin(m->gamma, m->gamma0, (double)max_load) : 0.0;
  // Eq. 4: the paths overlap; each is slowed by its contention factor.
  const double bp = m->beta * t_p, ad = m->alpha * t_d;
  const double t_a = bp > ad ? bp : ad;
  out->t_gemm = t_g;
  out->t_prefill = t_p;
  out->t_decode = t_d;
  out->t_attn = t_a;
  out->t_iter = (double)n_layers * (t_g + t_a);   // Eq. 2
  return CF_OK;
}

cf_status cf_latency_fit_line(const double* x, const double* y, int n, double* slope, double* intercept) {
  if (!x || !y || !slope || !intercept || n < 2) return CF_ERR_INVALID_ARG;
  double mx = 0.0, my = 0.0;
  for (int i = 0; i < n; ++i) {
    if (!std::isfinite(x[i]) || !std::isfinite(y[i])) return CF_ERR_INVALID_ARG;
    mx += x[i];
    my += y[i];
  }
  mx /= n;
  my /= n;
  double sxx = 0.0, sxy = 0.0;
  for (int i = 0; i < n; ++i) {
    const double dx = x[i] - mx;
    sxx += dx * dx;
    sxy += dx * (y[i] - my);
  }
  if (!(sxx > 0.0)) return CF_ERR_INVALID_ARG;   // all x equal
  *slope = sxy / sxx;
  *intercept = my - *slope * mx;
  return CF_OK;
}

cf_status cf_latency_calibrate(cf_latency_model* m, int n, const double* t_gemm, const double* t_prefill,
                               const double* t_decode, const double* t_meas, double f_max, double step,
                               double* mape) {
  if (!m || n < 1 || !t_gemm || !t_prefill || !t_decode || !t_meas) return CF_ERR_INVALID_ARG;
  if (!(step > 0.0) || !(f_max >= 1.0) || !std::isfinite(f_max)) return CF_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (!(t_meas[i] != 0.0) || !std::isfinite(t_meas[i]) || !std::isfinite(t_gemm[i]) ||
        !std::isfinite(t_prefill[i]) || !std::isfinite(t_decode[i]))
      return CF_ERR_INVALID_ARG;
  const long long k = (long long)std::floor((f_max - 1.0) / step + 1e-9);
  if (k > 100000) return CF_ERR_INVALID_ARG;
  double best = INFINITY, best_a = 1.0, best_b = 1.0;
  for (long long ia = 0; ia <= k; ++ia) {
    const double a = 1.0 + step * (double)ia;
    for (long long ib = 0; ib <= k; ++ib) {
      const double b = 1.0 + step * (double)ib;
      double s = 0.0;
      for (int i = 0; i < n; ++i) {
        const double bp = b * t_prefill[i], ad = a * t_decode[i];
        const double pred = t_gemm[i] + (bp > ad ? bp : ad);
        s += std::fabs(pred - t_meas[i]) / std::fabs(t_meas[i]);
      }
      const double e = 100.0 * s / n;
      if (e < best) {
        best = e;
        best_a = a;
        best_b = b;
      }
    }
  }
  m->alpha = best_a;
  m->beta = best_b;
  if (mape) *mape = best;
  return CF_OK;
}

}  // extern "C"
