// Split-K decode attention over paged KV (flash-decoding).
//
// Decode attention is bound by HBM: every cached K/V byte of a request is
// read once per KV head, never once per query head (ConfluxServe App. B,
// Table 7, "Decode Attention": traffic B L H / G).  A work item is
// (request j, KV head h, chunk of pages); one warp serves all G query heads
// of KV head h, so each 4 KB (page, head) tile is streamed once.
//
// Each lane loads 16-byte vectors straight from HBM into registers (the
// next page's loads are issued before the current page is processed), and
// the two small contractions per page, S = Q_g K^T (G x 16 keys) and
// O += P V (G x d), run on mma.sync m16n8k16 with the G query heads as the
// M rows: G = 4..8 rows would need 2-8x more CUDA-core FMAs than the HBM
// stream allows when decode owns only part of the SMs.  The register
// layouts are chosen so that K feeds the B fragment directly (a fixed
// permutation of d shared by Q and K leaves the dot products unchanged) and
// V feeds it after one byte-permute, with no shared-memory staging.
//
// Partial results (unnormalised O, running max m in log2 units, sum l) of
// the chunks of one (request, head) are merged with the log-sum-exp rule
// (Decode Token Parallelism §4.4, Eq. 4: partial outputs with fp32
// log-sum-exp statistics): o = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.
#include "common.cuh"
#include "internal.h"

namespace cf {

namespace {

constexpr int kThreads = kDecodeWarps * 32;
constexpr int kDecodeSmem = 64 * 1024;   // also keeps decode CTAs off prefill SMs
constexpr int kItemsPerWarp = 3;

CF_DEV void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
CF_DEV uint32_t word(const uint4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }
CF_DEV uint32_t pair_lo(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x5410); }
CF_DEV uint32_t pair_hi(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x7632); }

template <int D>
struct PageRegs {
  uint4 k[2][D / 32];   // n-tile (8 keys), 16-byte chunk (4jj + t)
  uint4 v[4][D / 64];   // keys 2t, 2t+1, 2t+8, 2t+9; d block 64*half + 8g
  int valid;            // keys of this page that exist (0..16)
};

template <int D>
CF_DEV void load_page(PageRegs<D>& r, const DecodeArgs& a, const int* table, int p, int keys, int h, int g, int t) {
  const int pid = table[p];
  int valid = keys - p * 16;
  valid = valid > 16 ? 16 : valid;
  if (pid < 0 || pid >= a.num_pages) {
    if ((threadIdx.x & 31) == 0) set_error(a.err, CF_DEVERR_PAGE);
    valid = 0;
  }
  r.valid = valid;
  if (valid <= 0) {
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int jj = 0; jj < D / 32; ++jj) r.k[n][jj] = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int hh = 0; hh < D / 64; ++hh) r.v[kk][hh] = make_uint4(0, 0, 0, 0);
    return;
  }
  const size_t base = ((size_t)pid * a.Hkv + h) * 16 * D;
  const __nv_bfloat16* kb = a.k_pool + base;
  const __nv_bfloat16* vb = a.v_pool + base;
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int jj = 0; jj < D / 32; ++jj) r.k[n][jj] = ldg_stream(kb + (n * 8 + g) * D + (4 * jj + t) * 8);
  const int keys4[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
#pragma unroll
    for (int hh = 0; hh < D / 64; ++hh) r.v[kk][hh] = ldg_stream(vb + keys4[kk] * D + hh * 64 + 8 * g);
}

template <int D, bool G16>
struct Acc {
  float o[D / 8][2];      // row g: d = 64*(m/8) + 16t + (m%8) [+8]
  float o8[D / 8][2];     // row g + 8: heads 8..15 (G > 8) or the low part of P (G <= 8)
  float m0, l0, m1, l1;
};

template <int D, bool G16>
CF_DEV void process_page(Acc<D, G16>& A, PageRegs<D>& r, const uint32_t (*qa)[2], const uint32_t (*qb)[2],
                         float scale_log2, int t) {
  // ---- S = Q K^T for two n-tiles of 8 keys
  float s[2][4];
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int st = 0; st < D / 16; ++st) {
      const uint4& kv = r.k[n][st >> 1];
      const uint32_t b0 = word(kv, (st & 1) * 2), b1 = word(kv, (st & 1) * 2 + 1);
      mma16816(s[n], qa[st][0], G16 ? qb[st][0] : 0u, qa[st][1], G16 ? qb[st][1] : 0u, b0, b1);
    }
  }
  // ---- mask, scale, online softmax (log2 domain)
  const int valid = r.valid;
  float x[2][2], y[2][2];
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const bool ok = n * 8 + 2 * t + e < valid;
      x[n][e] = ok ? s[n][e] * scale_log2 : -INFINITY;
      y[n][e] = ok ? s[n][2 + e] * scale_log2 : -INFINITY;
    }
  float mx = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const float mnew = fmaxf(A.m0, mx);
  const float muse = mnew == -INFINITY ? 0.f : mnew;
  const float alpha = fast_exp2(A.m0 - muse);
  float p[2][2];
  float ls = 0.f;
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      p[n][e] = fast_exp2(x[n][e] - muse);
      ls += p[n][e];
    }
  A.l0 = A.l0 * alpha + ls;
  A.m0 = mnew;
#pragma unroll
  for (int m = 0; m < D / 8; ++m) {
    A.o[m][0] *= alpha;
    A.o[m][1] *= alpha;
  }
  // P is split into bf16 high and low parts so that P V is accurate to
  // ~2^-16 relative: P ~= hi + lo, hi = bf16(P), lo = bf16(P - hi).
  const uint32_t pa0 = pack_bf16(p[0][0], p[0][1]), pa2 = pack_bf16(p[1][0], p[1][1]);
  const uint32_t pl0 = pack_bf16(p[0][0] - bf16lo(pa0), p[0][1] - bf16hi(pa0));
  const uint32_t pl2 = pack_bf16(p[1][0] - bf16lo(pa2), p[1][1] - bf16hi(pa2));
  uint32_t pa1 = pl0, pa3 = pl2;     // G <= 8: rows g+8 of the MMA carry the low part
  uint32_t qa1 = 0u, qa3 = 0u, ql1 = 0u, ql3 = 0u;
  if constexpr (G16) {
    float my = fmaxf(fmaxf(y[0][0], y[0][1]), fmaxf(y[1][0], y[1][1]));
    my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 1));
    my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 2));
    const float m1n = fmaxf(A.m1, my);
    const float m1u = m1n == -INFINITY ? 0.f : m1n;
    const float a1 = fast_exp2(A.m1 - m1u);
    float q[2][2], lq = 0.f;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        q[n][e] = fast_exp2(y[n][e] - m1u);
        lq += q[n][e];
      }
    A.l1 = A.l1 * a1 + lq;
    A.m1 = m1n;
#pragma unroll
    for (int m = 0; m < D / 8; ++m) {
      A.o8[m][0] *= a1;
      A.o8[m][1] *= a1;
    }
    qa1 = pack_bf16(q[0][0], q[0][1]);
    qa3 = pack_bf16(q[1][0], q[1][1]);
    ql1 = pack_bf16(q[0][0] - bf16lo(qa1), q[0][1] - bf16hi(qa1));
    ql3 = pack_bf16(q[1][0] - bf16lo(qa3), q[1][1] - bf16hi(qa3));
    pa1 = qa1;
    pa3 = qa3;
  } else {
#pragma unroll
    for (int m = 0; m < D / 8; ++m) {
      A.o8[m][0] *= alpha;
      A.o8[m][1] *= alpha;
    }
  }
  // ---- zero V of keys past the end (their slots may hold anything)
  if (valid < 16) {
    const int keys4[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      if (keys4[kk] >= valid)
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) r.v[kk][hh] = make_uint4(0, 0, 0, 0);
  }
  // ---- O += P V, n-tile m covers d = 64*(m/8) + 8*col + (m%8)
#pragma unroll
  for (int m = 0; m < D / 8; ++m) {
    const int hh = m >> 3, e = m & 7;
    const uint32_t w0 = word(r.v[0][hh], e >> 1), w1 = word(r.v[1][hh], e >> 1);
    const uint32_t w2 = word(r.v[2][hh], e >> 1), w3 = word(r.v[3][hh], e >> 1);
    const uint32_t b0 = (e & 1) ? pair_hi(w0, w1) : pair_lo(w0, w1);
    const uint32_t b1 = (e & 1) ? pair_hi(w2, w3) : pair_lo(w2, w3);
    float c[4] = {A.o[m][0], A.o[m][1], A.o8[m][0], A.o8[m][1]};
    mma16816(c, pa0, pa1, pa2, pa3, b0, b1);
    if constexpr (G16) mma16816(c, pl0, ql1, pl2, ql3, b0, b1);   // low parts of both row groups
    A.o[m][0] = c[0];
    A.o[m][1] = c[1];
    A.o8[m][0] = c[2];
    A.o8[m][1] = c[3];
  }
}

// Writes one query head's row: either the normalised bf16 output or the
// fp32 partial (unnormalised O plus m, l).
template <int D>
CF_DEV void write_row(const float (*o)[2], float m, float l, bool final_out, __nv_bfloat16* out_row,
                      float* part_row, float* ml, int t) {
  if (final_out) {
    const float inv = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll
    for (int hh = 0; hh < D / 64; ++hh) {
      uint4 lo, hi;
      lo.x = pack_bf16(o[8 * hh + 0][0] * inv, o[8 * hh + 1][0] * inv);
      lo.y = pack_bf16(o[8 * hh + 2][0] * inv, o[8 * hh + 3][0] * inv);
      lo.z = pack_bf16(o[8 * hh + 4][0] * inv, o[8 * hh + 5][0] * inv);
      lo.w = pack_bf16(o[8 * hh + 6][0] * inv, o[8 * hh + 7][0] * inv);
      hi.x = pack_bf16(o[8 * hh + 0][1] * inv, o[8 * hh + 1][1] * inv);
      hi.y = pack_bf16(o[8 * hh + 2][1] * inv, o[8 * hh + 3][1] * inv);
      hi.z = pack_bf16(o[8 * hh + 4][1] * inv, o[8 * hh + 5][1] * inv);
      hi.w = pack_bf16(o[8 * hh + 6][1] * inv, o[8 * hh + 7][1] * inv);
      uint4* dst = reinterpret_cast<uint4*>(out_row + 64 * hh + 16 * t);
      dst[0] = lo;
      dst[1] = hi;
    }
  } else {
#pragma unroll
    for (int hh = 0; hh < D / 64; ++hh) {
      float4* dst = reinterpret_cast<float4*>(part_row + 64 * hh + 16 * t);
      dst[0] = make_float4(o[8 * hh + 0][0], o[8 * hh + 1][0], o[8 * hh + 2][0], o[8 * hh + 3][0]);
      dst[1] = make_float4(o[8 * hh + 4][0], o[8 * hh + 5][0], o[8 * hh + 6][0], o[8 * hh + 7][0]);
      dst[2] = make_float4(o[8 * hh + 0][1], o[8 * hh + 1][1], o[8 * hh + 2][1], o[8 * hh + 3][1]);
      dst[3] = make_float4(o[8 * hh + 4][1], o[8 * hh + 5][1], o[8 * hh + 6][1], o[8 * hh + 7][1]);
    }
    if (t == 0) {
      ml[0] = m;
      ml[1] = l;
    }
  }
}

// Chunking plan, computed identically by every CTA from the key counts:
// pages_j = ceil(keys_j / 16); chunk = max(4, ceil(sum_j pages_j * Hkv /
// (3 * warps))); chunks_j = ceil(pages_j / chunk); S_j = prefix sums.
CF_DEV int build_plan(const DecodeArgs& a, int* s_pref, int* s_pages) {
  const int n = a.n;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    long long keys = (long long)a.n_keys[j] + a.key_offset;
    long long pg = keys > 0 ? (keys + 15) / 16 : 0;
    if (keys <= 0 || pg > a.page_stride) {
      if (blockIdx.x == 0) set_error(a.err, CF_DEVERR_CONTEXT);
      if (pg > a.page_stride) pg = a.page_stride;
      if (keys <= 0) pg = 0;
    }
    s_pages[j] = (int)pg;
  }
  __syncthreads();
  __shared__ int s_chunk;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    long long tot = 0;
    for (int j = lane; j < n; j += 32) tot += s_pages[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    const long long warps = (long long)gridDim.x * kDecodeWarps;
    long long chunk = (tot * a.Hkv + kItemsPerWarp * warps - 1) / (kItemsPerWarp * warps);
    if (chunk < 4) chunk = 4;
    // exclusive prefix sum of chunks_j: lane owns a contiguous block of j
    const int per = (n + 31) / 32;
    const int j0 = lane * per, j1 = min(n, j0 + per);
    int local = 0;
    for (int j = j0; j < j1; ++j) local += (int)((s_pages[j] + chunk - 1) / chunk);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - local;
    for (int j = j0; j < j1; ++j) {
      s_pref[j] = run;
      run += (int)((s_pages[j] + chunk - 1) / chunk);
    }
    if (lane == 31) s_pref[n] = incl;
    if (lane == 0) s_chunk = (int)chunk;
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int j = threadIdx.x; j <= n; j += blockDim.x) a.plan[2 + j] = s_pref[j];
    if (threadIdx.x == 0) {
      a.plan[0] = s_chunk;
      a.plan[1] = s_pref[n];
    }
  }
  return s_chunk;
}

template <int D, bool G16>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(DecodeArgs a) {
  extern __shared__ int dsm[];
  int* s_pref = dsm;              // [n + 1]
  int* s_pages = dsm + a.n + 1;   // [n]
  const int chunk = build_plan(a, s_pref, s_pages);
  const int G = a.Hq / a.Hkv;
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const long long total = (long long)s_pref[a.n] * a.Hkv;
  const int nwarps = gridDim.x * kDecodeWarps;
  const int gw = blockIdx.x * kDecodeWarps + (threadIdx.x >> 5);

  for (long long item = gw; item < total; item += nwarps) {
    const int cg = (int)(item / a.Hkv), h = (int)(item % a.Hkv);
    int lo = 0, hi = a.n;  // largest j with s_pref[j] <= cg
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pref[mid] <= cg) lo = mid; else hi = mid;
    }
    const int j = lo;
    const int c = cg - s_pref[j];
    const int nch = s_pref[j + 1] - s_pref[j];
    const int keys = a.n_keys[j] + a.key_offset;
    const int pages = s_pages[j];
    const int p0 = c * chunk, p1 = min(pages, p0 + chunk);
    const int* table = a.pages + (size_t)j * a.page_stride;

    // Q fragments of rows g (head h*G + g) and g + 8
    uint32_t qa[D / 16][2], qb[G16 ? D / 16 : 1][2];
    const __nv_bfloat16* qrow = a.q + (size_t)j * a.q_stride + (size_t)h * G * D;
#pragma unroll
    for (int jj = 0; jj < D / 32; ++jj) {
      const uint4 v = g < G ? *reinterpret_cast<const uint4*>(qrow + g * D + (4 * jj + t) * 8) : make_uint4(0, 0, 0, 0);
      qa[2 * jj][0] = v.x; qa[2 * jj][1] = v.y; qa[2 * jj + 1][0] = v.z; qa[2 * jj + 1][1] = v.w;
      if constexpr (G16) {
        const uint4 u = g + 8 < G ? *reinterpret_cast<const uint4*>(qrow + (g + 8) * D + (4 * jj + t) * 8)
                                  : make_uint4(0, 0, 0, 0);
        qb[2 * jj][0] = u.x; qb[2 * jj][1] = u.y; qb[2 * jj + 1][0] = u.z; qb[2 * jj + 1][1] = u.w;
      }
    }
    Acc<D, G16> A;
#pragma unroll
    for (int m = 0; m < D / 8; ++m) {
      A.o[m][0] = A.o[m][1] = 0.f;
      A.o8[m][0] = A.o8[m][1] = 0.f;
    }
    A.m0 = A.m1 = -INFINITY;
    A.l0 = A.l1 = 0.f;

    PageRegs<D> ra, rb;
    if (p0 < p1) load_page<D>(ra, a, table, p0, keys - 0, h, g, t);
    for (int p = p0; p < p1; p += 2) {
      if (p + 1 < p1) load_page<D>(rb, a, table, p + 1, keys, h, g, t);
      process_page<D, G16>(A, ra, qa, qb, a.scale_log2, t);
      if (p + 1 >= p1) break;
      if (p + 2 < p1) load_page<D>(ra, a, table, p + 2, keys, h, g, t);
      process_page<D, G16>(A, rb, qa, qb, a.scale_log2, t);
    }
    A.l0 += __shfl_xor_sync(0xffffffffu, A.l0, 1);
    A.l0 += __shfl_xor_sync(0xffffffffu, A.l0, 2);
    if constexpr (G16) {
      A.l1 += __shfl_xor_sync(0xffffffffu, A.l1, 1);
      A.l1 += __shfl_xor_sync(0xffffffffu, A.l1, 2);
    }
    if constexpr (!G16) {
#pragma unroll
      for (int m = 0; m < D / 8; ++m) {
        A.o[m][0] += A.o8[m][0];
        A.o[m][1] += A.o8[m][1];
      }
    }
    const bool final_out = nch == 1;
    const long long slot = item;  // partial index = (S_j + c) * Hkv + h
    if (g < G) {
      __nv_bfloat16* orow = a.out + (size_t)j * a.out_stride + (size_t)(h * G + g) * D;
      float* prow = a.part_o + ((size_t)slot * G + g) * D;
      float* ml = a.part_ml + ((size_t)slot * G + g) * 2;
      write_row<D>(A.o, A.m0, A.l0, final_out, orow, prow, ml, t);
    }
    if constexpr (G16) {
      if (g + 8 < G) {
        __nv_bfloat16* orow = a.out + (size_t)j * a.out_stride + (size_t)(h * G + g + 8) * D;
        float* prow = a.part_o + ((size_t)slot * G + g + 8) * D;
        float* ml = a.part_ml + ((size_t)slot * G + g + 8) * 2;
        write_row<D>(A.o8, A.m1, A.l1, final_out, orow, prow, ml, t);
      }
    }
  }
}

// One warp per (request, query head): merges the chunk partials.
template <int D>
__global__ void decode_merge_kernel(DecodeArgs a) {
  const int G = a.Hq / a.Hkv;
  const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= (long long)a.n * a.Hq) return;
  const int j = (int)(w / a.Hq), hq = (int)(w % a.Hq);
  const int h = hq / G, g = hq % G;
  const int s0 = a.plan[2 + j], nch = a.plan[2 + j + 1] - s0;
  __nv_bfloat16* orow = a.out + (size_t)j * a.out_stride + (size_t)hq * D;
  constexpr int PER = D / 32;
  if (nch == 1) return;  // written directly by the decode kernel
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  if (nch == 0) {  // no keys: defined as zeros (flagged in the error word)
#pragma unroll
    for (int i = 0; i < PER; ++i) orow[lane * PER + i] = __float2bfloat16(0.f);
    return;
  }
  float M = -INFINITY;
  for (int c = 0; c < nch; ++c) {
    const long long slot = (long long)(s0 + c) * a.Hkv + h;
    M = fmaxf(M, a.part_ml[(slot * G + g) * 2]);
  }
  const float Mu = M == -INFINITY ? 0.f : M;
  float L = 0.f;
  for (int c = 0; c < nch; ++c) {
    const long long slot = (long long)(s0 + c) * a.Hkv + h;
    const float* ml = a.part_ml + (slot * G + g) * 2;
    const float wgt = fast_exp2(ml[0] - Mu);
    L += wgt * ml[1];
    const float* po = a.part_o + (slot * G + g) * D + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] += wgt * po[i];
  }
  const float inv = L > 0.f ? 1.0f / L : 0.f;
#pragma unroll
  for (int i = 0; i < PER; i += 2)
    *reinterpret_cast<uint32_t*>(orow + lane * PER + i) = pack_bf16(acc[i] * inv, acc[i + 1] * inv);
}

template <int D, bool G16>
cudaError_t launch_t(const DecodeArgs& a, int ctas, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, G16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kDecodeSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  decode_kernel<D, G16><<<ctas, kThreads, kDecodeSmem, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long warps = (long long)a.n * a.Hq;
  const int blocks = (int)((warps * 32 + 255) / 256);
  decode_merge_kernel<D><<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

long long decode_max_items(int max_decode, int Hkv, int max_ctas) {
  return (long long)kItemsPerWarp * max_ctas * kDecodeWarps + (long long)max_decode * Hkv + 64;
}

cudaError_t launch_decode(const DecodeArgs& a, int num_ctas, cudaStream_t s) {
  if (a.n <= 0) return cudaSuccess;
  if ((a.n * 2 + 2) * 4 > kDecodeSmem) return cudaErrorInvalidValue;
  const bool g16 = a.Hq / a.Hkv > 8;
  if (a.head_dim == 128) return g16 ? launch_t<128, true>(a, num_ctas, s) : launch_t<128, false>(a, num_ctas, s);
  if (a.head_dim == 64) return g16 ? launch_t<64, true>(a, num_ctas, s) : launch_t<64, false>(a, num_ctas, s);
  return cudaErrorInvalidValue;
}

}  // namespace cf
