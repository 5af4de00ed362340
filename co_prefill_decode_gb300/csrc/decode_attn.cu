// Split-K decode attention over paged KV (flash-decoding).
//
// Decode attention is bound by HBM: every cached K/V byte of a request is
// read once per KV head, never once per query head (ConfluxServe App. B,
// Table 7, "Decode Attention": traffic B L H / G).  A work item is
// (request j, KV head h, chunk of pages); one warp serves all G query heads
// of KV head h, so each 4 KB (page, head) tile is streamed once.
//
// Loads: one lane of each warp issues TMA tensor copies of the page's K and
// V tiles (16 rows x 64 columns per box, 128-byte swizzle) into a per-warp
// ring of page slots, completed on one mbarrier per slot, so the bytes in
// flight are bounded by shared memory rather than by the SM's outstanding
// load slots.  Fragments are then read with ldmatrix (K) and ldmatrix.trans
// (V), which the swizzle makes bank-conflict free.
//
// The two small contractions per page, S = Q_g K^T (G x 16 keys) and
// O += P V (G x d), run on mma.sync m16n8k16: with only part of the SMs,
// G = 4..8 rows of CUDA-core FMAs per key would not keep up with the HBM
// stream.  For G <= 8 they are computed transposed (S^T = K Q^T, O^T += V^T
// P^T), with the page's 16 keys as the M rows and the heads as N = 8: half
// the MMAs of the heads-as-rows form, whose S products were half padding.
// For 8 < G <= 16 the heads are the M rows, and P is split into bf16 high
// and low parts (P = hi + lo) so that P V keeps ~2^-16 of P's precision.
//
// Partial results (unnormalised O, running max m in log2 units, sum l) of
// the chunks of one (request, head) are merged with the log-sum-exp rule
// (Decode Token Parallelism §4.4, Eq. 4: partial outputs with fp32
// log-sum-exp statistics): o = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace cf {

namespace {

constexpr int kThreads = kDecodeWarps * 32;
constexpr int kMaxDecodeReqs = 2048;                 // plan arrays in shared memory
// plan arrays, padded so that the page ring after them starts 1 KB aligned
// (the 128-byte swizzle repeats every 1024 bytes)
constexpr int kPlanBytes = (((2 * kMaxDecodeReqs + 2) * 4 + 1023) / 1024) * 1024;
constexpr int kRingBytes = 192 * 1024;               // per CTA, split over the warps
constexpr int kBarBytes = 1024;                      // per-slot mbarriers
// + 1 KB so the base can be aligned to 1 KB by hand; > half an SM, so a decode
// CTA never shares an SM with a prefill CTA
constexpr int kDecodeSmem = kPlanBytes + kRingBytes + kBarBytes + 1024;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: O is rescaled only when the max grows more

template <int D>
struct Ring {
  static constexpr int HALF = 16 * 128;                // one 16 x 64 box (2 KB)
  static constexpr int KV = HALF * (D / 64);           // K (or V) tile of one page
  static constexpr int PAGE = 2 * KV;                  // 8 KB for d = 128
  static constexpr int STAGES = kRingBytes / kDecodeWarps / PAGE;
  static_assert(STAGES >= 2 && STAGES * kDecodeWarps * 8 <= kBarBytes, "ring shape");
  static_assert(kPlanBytes % 1024 == 0 && PAGE % 1024 == 0, "swizzled boxes need 1 KB alignment");
};

// byte offset of 16-byte chunk c (of d) in row r of a swizzled K or V tile
CF_DEV uint32_t swz(int r, int c) { return (c >> 3) * (16 * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4); }

CF_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
CF_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

CF_DEV void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- 8 < G <= 16: the query heads are the MMA's M rows (heads 0..7 in
// rows g, heads 8..15 in rows g + 8).
template <int D>
struct Acc16 {
  float o[D / 8][2];      // head g: d = 8 m + 2 t, +1
  float o8[D / 8][2];     // head g + 8
  float m0, l0, m1, l1;   // running max (log2 units) and sum of heads g and g + 8
};

// One page (16 keys) of one item: S = Q K^T, online softmax, O += P V.
// kt, vt: shared-memory addresses of the page's K and V tiles.
template <int D>
CF_DEV void process_page16(Acc16<D>& A, uint32_t kt, uint32_t vt, int valid, const uint32_t (*qa)[2],
                           const uint32_t (*qb)[2], float scale_log2, int lane) {
  const int t = lane & 3;
  // ---- S = Q K^T: two n-tiles of 8 keys, two accumulator chains each
  float s[2][4];
  {
    float e0[2][4], e1[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) e0[n][i] = e1[n][i] = 0.f;
#pragma unroll
    for (int sp = 0; sp < D / 32; ++sp)
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        uint32_t b[4];
        ldsm_x4(kt + swz(8 * n + (lane & 7), 4 * sp + (lane >> 3)), b[0], b[1], b[2], b[3]);
        mma16816(e0[n], qa[2 * sp][0], qb[2 * sp][0], qa[2 * sp][1], qb[2 * sp][1], b[0], b[1]);
        mma16816(e1[n], qa[2 * sp + 1][0], qb[2 * sp + 1][0], qa[2 * sp + 1][1], qb[2 * sp + 1][1], b[2], b[3]);
      }
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) s[n][i] = e0[n][i] + e1[n][i];
  }
  // ---- mask, scale, online softmax (log2 domain)
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
  // lazy rescaling: keep the running max unless it grows by more than 2^8
  // (P then stays below 256, exact enough in fp32 and in the bf16 hi/lo split);
  // heads g first, then heads g + 8
  const bool first = A.m0 == -INFINITY;
  const bool grow = !first && mx > A.m0 + kRescaleThreshold;
  if (first) A.m0 = mx;
  if (__any_sync(0xffffffffu, grow)) {
    const float alpha = grow ? fast_exp2(A.m0 - mx) : 1.0f;
    if (grow) A.m0 = mx;
    A.l0 *= alpha;
#pragma unroll
    for (int m = 0; m < D / 8; ++m) {
      A.o[m][0] *= alpha;
      A.o[m][1] *= alpha;
    }
  }
  const float muse = A.m0 == -INFINITY ? 0.f : A.m0;
  float p[2][2];
  float ls = 0.f;
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      p[n][e] = fast_exp2(x[n][e] - muse);
      ls += p[n][e];
    }
  A.l0 += ls;
  // P is split into bf16 high and low parts: P ~= hi + lo, hi = bf16(P),
  // lo = bf16(P - hi); the low parts go through a second MMA.
  const uint32_t pa0 = pack_bf16(p[0][0], p[0][1]), pa2 = pack_bf16(p[1][0], p[1][1]);
  const uint32_t pl0 = pack_bf16(p[0][0] - bf16lo(pa0), p[0][1] - bf16hi(pa0));
  const uint32_t pl2 = pack_bf16(p[1][0] - bf16lo(pa2), p[1][1] - bf16hi(pa2));
  uint32_t pa1, pa3, ql1, ql3;
  {
    float my = fmaxf(fmaxf(y[0][0], y[0][1]), fmaxf(y[1][0], y[1][1]));
    my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 1));
    my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 2));
    const bool first1 = A.m1 == -INFINITY;
    const bool grow1 = !first1 && my > A.m1 + kRescaleThreshold;
    if (first1) A.m1 = my;
    if (__any_sync(0xffffffffu, grow1)) {
      const float a1 = grow1 ? fast_exp2(A.m1 - my) : 1.0f;
      if (grow1) A.m1 = my;
      A.l1 *= a1;
#pragma unroll
      for (int m = 0; m < D / 8; ++m) {
        A.o8[m][0] *= a1;
        A.o8[m][1] *= a1;
      }
    }
    const float m1u = A.m1 == -INFINITY ? 0.f : A.m1;
    float q[2][2], lq = 0.f;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        q[n][e] = fast_exp2(y[n][e] - m1u);
        lq += q[n][e];
      }
    A.l1 += lq;
    pa1 = pack_bf16(q[0][0], q[0][1]);
    pa3 = pack_bf16(q[1][0], q[1][1]);
    ql1 = pack_bf16(q[0][0] - bf16lo(pa1), q[0][1] - bf16hi(pa1));
    ql3 = pack_bf16(q[1][0] - bf16lo(pa3), q[1][1] - bf16hi(pa3));
  }
  // keys past the end of the request: their V (any bits, even NaN) must not
  // reach the product, so zero those halves of the B fragments
  uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
  if (valid < 16) {
    vm0 = (2 * t < valid ? 0x0000ffffu : 0u) | (2 * t + 1 < valid ? 0xffff0000u : 0u);
    vm1 = (2 * t + 8 < valid ? 0x0000ffffu : 0u) | (2 * t + 9 < valid ? 0xffff0000u : 0u);
  }
  // ---- O += P V, two n-tiles (16 d) per ldmatrix.x4.trans
#pragma unroll
  for (int m = 0; m < D / 8; m += 2) {
    uint32_t b[4];
    ldsm_x4_t(vt + swz((lane & 7) + 8 * ((lane >> 3) & 1), m + (lane >> 4)), b[0], b[1], b[2], b[3]);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t b0 = b[2 * u] & vm0, b1 = b[2 * u + 1] & vm1;
      float c[4] = {A.o[m + u][0], A.o[m + u][1], A.o8[m + u][0], A.o8[m + u][1]};
      mma16816(c, pa0, pa1, pa2, pa3, b0, b1);
      mma16816(c, pl0, ql1, pl2, ql3, b0, b1);   // low parts of both row groups
      A.o[m + u][0] = c[0];
      A.o[m + u][1] = c[1];
      A.o8[m + u][0] = c[2];
      A.o8[m + u][1] = c[3];
    }
  }
}

// ---- G <= 8: the products transposed, so the 16 keys of a page are the
// MMA's M rows and the query heads its N columns:
//   S^T = K Q^T   (m16n8k16: 16 keys x 8 heads, d in steps of 16),
//   O^T += V^T P^T (16 values of d x 8 heads per MMA, the page's 16 keys as K).
// A page then costs D/16 + D/16 MMAs instead of 2 D/8 with the heads as rows,
// where half of every S product was padding.  P is rounded to bf16 as the B
// operand; each head's running max moves only when one of its scores passes
// it by more than 2^8, which a warp vote detects without a reduction.
template <int D>
struct AccT {
  float o[D / 16][4];   // O^T: d = 16 m + g ([0], [1]) and 16 m + g + 8 ([2], [3]); heads 2t (+0), 2t+1 (+1)
  float m[2];           // running max (log2 units) of heads 2t and 2t + 1
  float l[2];           // their sums over the keys this lane holds
};

CF_DEV uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <int D>
CF_DEV void process_page_t(AccT<D>& A, uint32_t kt, uint32_t vt, int valid, const uint32_t (*qa)[2],
                           float scale_log2, int lane) {
  const int g = lane >> 2, t = lane & 3;
  // ---- S^T = K Q^T; K rows are the A operand, the Q fragments (head g,
  // d = 16 s + 2t (+8)) are exactly the B operand's; two accumulator chains
  float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int st = 0; st < D / 16; ++st) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(kt + swz((lane & 7) + 8 * ((lane >> 3) & 1), 2 * st + (lane >> 4)), a0, a1, a2, a3);
    mma16816(st & 1 ? c1 : c0, a0, a1, a2, a3, qa[st][0], qa[st][1]);
  }
  // x[k][e]: key g + 8 k, head 2t + e, in log2 units; keys past the end are -inf
  float x[2][2];
  x[0][0] = g < valid ? (c0[0] + c1[0]) * scale_log2 : -INFINITY;
  x[0][1] = g < valid ? (c0[1] + c1[1]) * scale_log2 : -INFINITY;
  x[1][0] = g + 8 < valid ? (c0[2] + c1[2]) * scale_log2 : -INFINITY;
  x[1][1] = g + 8 < valid ? (c0[3] + c1[3]) * scale_log2 : -INFINITY;
  bool need = false;
#pragma unroll
  for (int e = 0; e < 2; ++e) need |= fmaxf(x[0][e], x[1][e]) > A.m[e] + kRescaleThreshold;   // -inf + 8 = -inf
  if (__any_sync(0xffffffffu, need)) {
    // the page's max per head: keys g, g + 8 here, g over the lanes 4 g + t
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float mx = fmaxf(x[0][e], x[1][e]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      if (mx > A.m[e] + kRescaleThreshold) {   // the same for the 8 lanes of this head
        const float alpha = fast_exp2(A.m[e] - mx);   // 0 when the head had no keys yet
        A.l[e] *= alpha;
#pragma unroll
        for (int m = 0; m < D / 16; ++m) {
          A.o[m][e] *= alpha;
          A.o[m][2 + e] *= alpha;
        }
        A.m[e] = mx;
      }
    }
  }
  float p[2][2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const float mu = A.m[e] == -INFINITY ? 0.f : A.m[e];
    p[0][e] = fast_exp2(x[0][e] - mu);
    p[1][e] = fast_exp2(x[1][e] - mu);
    A.l[e] += p[0][e] + p[1][e];
  }
  // P^T as this lane holds it (key g or g + 8; heads 2t, 2t + 1) is one row
  // of an 8x8 block; the B operand wants keys 2t, 2t + 1 of head g: the
  // transpose of that block
  const uint32_t b0 = movmatrix_trans(pack_bf16(p[0][0], p[0][1]));
  const uint32_t b1 = movmatrix_trans(pack_bf16(p[1][0], p[1][1]));
  // keys past the end of the request: their V (any bits, even NaN) must not
  // reach the product, so zero those halves of the A fragments
  uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
  if (valid < 16) {
    vm0 = (2 * t < valid ? 0x0000ffffu : 0u) | (2 * t + 1 < valid ? 0xffff0000u : 0u);
    vm1 = (2 * t + 8 < valid ? 0x0000ffffu : 0u) | (2 * t + 9 < valid ? 0xffff0000u : 0u);
  }
  // ---- O^T += V^T P^T: V read transposed (rows of d, the page's keys as K)
#pragma unroll
  for (int m = 0; m < D / 16; ++m) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4_t(vt + swz((lane & 7) + 8 * (lane >> 4), 2 * m + ((lane >> 3) & 1)), a0, a1, a2, a3);
    mma16816(A.o[m], a0 & vm0, a1 & vm0, a2 & vm1, a3 & vm1, b0, b1);
  }
}

// Writes one query head's row: either the normalised bf16 output or the
// fp32 partial (unnormalised O plus m, l).  Lane (g, t) holds d = 8m + 2t, +1.
template <int D>
CF_DEV void write_row(const float (*o)[2], float m, float l, bool final_out, __nv_bfloat16* out_row,
                      float* part_row, float* ml, int t) {
  if (final_out) {
    const float inv = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll
    for (int k = 0; k < D / 8; ++k)
      *reinterpret_cast<uint32_t*>(out_row + 8 * k + 2 * t) = pack_bf16(o[k][0] * inv, o[k][1] * inv);
  } else {
#pragma unroll
    for (int k = 0; k < D / 8; ++k)
      *reinterpret_cast<float2*>(part_row + 8 * k + 2 * t) = make_float2(o[k][0], o[k][1]);
    if (t == 0) {
      ml[0] = m;
      ml[1] = l;
    }
  }
}


// Per item: zero the accumulator, and at the end write the item's rows.
template <int D>
CF_DEV void acc_init(Acc16<D>& A) {
#pragma unroll
  for (int m = 0; m < D / 8; ++m) {
    A.o[m][0] = A.o[m][1] = 0.f;
    A.o8[m][0] = A.o8[m][1] = 0.f;
  }
  A.m0 = A.m1 = -INFINITY;
  A.l0 = A.l1 = 0.f;
}
template <int D>
CF_DEV void acc_init(AccT<D>& A) {
#pragma unroll
  for (int m = 0; m < D / 16; ++m) A.o[m][0] = A.o[m][1] = A.o[m][2] = A.o[m][3] = 0.f;
  A.m[0] = A.m[1] = -INFINITY;
  A.l[0] = A.l[1] = 0.f;
}
template <int D>
CF_DEV void acc_page(Acc16<D>& A, uint32_t kt, uint32_t vt, int valid, const uint32_t (*qa)[2],
                     const uint32_t (*qb)[2], float scale_log2, int lane) {
  process_page16<D>(A, kt, vt, valid, qa, qb, scale_log2, lane);
}
template <int D>
CF_DEV void acc_page(AccT<D>& A, uint32_t kt, uint32_t vt, int valid, const uint32_t (*qa)[2],
                     const uint32_t (*)[2], float scale_log2, int lane) {
  process_page_t<D>(A, kt, vt, valid, qa, scale_log2, lane);
}
// rows of query heads h G + i, i < G, of request j: the output (final) or
// the item's partial at index `slot`
template <int D>
CF_DEV void acc_finish(Acc16<D>& A, const DecodeArgs& a, int j, int h, int G, long long slot, bool final_out,
                       int lane) {
  const int g = lane >> 2, t = lane & 3;
  A.l0 += __shfl_xor_sync(0xffffffffu, A.l0, 1);
  A.l0 += __shfl_xor_sync(0xffffffffu, A.l0, 2);
  A.l1 += __shfl_xor_sync(0xffffffffu, A.l1, 1);
  A.l1 += __shfl_xor_sync(0xffffffffu, A.l1, 2);
  if (g < G) {
    __nv_bfloat16* orow = a.out + (size_t)j * a.out_stride + (size_t)(h * G + g) * D;
    float* prow = a.part_o + ((size_t)slot * G + g) * D;
    float* ml = a.part_ml + ((size_t)slot * G + g) * 2;
    write_row<D>(A.o, A.m0, A.l0, final_out, orow, prow, ml, t);
  }
  if (g + 8 < G) {
    __nv_bfloat16* orow = a.out + (size_t)j * a.out_stride + (size_t)(h * G + g + 8) * D;
    float* prow = a.part_o + ((size_t)slot * G + g + 8) * D;
    float* ml = a.part_ml + ((size_t)slot * G + g + 8) * 2;
    write_row<D>(A.o8, A.m1, A.l1, final_out, orow, prow, ml, t);
  }
}
template <int D>
CF_DEV void acc_finish(AccT<D>& A, const DecodeArgs& a, int j, int h, int G, long long slot, bool final_out,
                       int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int e = 0; e < 2; ++e) {   // a head's keys are spread over the lanes 4 g + t
    A.l[e] += __shfl_xor_sync(0xffffffffu, A.l[e], 4);
    A.l[e] += __shfl_xor_sync(0xffffffffu, A.l[e], 8);
    A.l[e] += __shfl_xor_sync(0xffffffffu, A.l[e], 16);
  }
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int hh = 2 * t + e;
    if (hh >= G) continue;
    if (final_out) {
      const float inv = A.l[e] > 0.f ? 1.0f / A.l[e] : 0.f;
      __nv_bfloat16* orow = a.out + (size_t)j * a.out_stride + (size_t)(h * G + hh) * D;
#pragma unroll
      for (int m = 0; m < D / 16; ++m) {
        orow[16 * m + g] = __float2bfloat16(A.o[m][e] * inv);
        orow[16 * m + g + 8] = __float2bfloat16(A.o[m][2 + e] * inv);
      }
    } else {
      float* prow = a.part_o + ((size_t)slot * G + hh) * D;
#pragma unroll
      for (int m = 0; m < D / 16; ++m) {
        prow[16 * m + g] = A.o[m][e];
        prow[16 * m + g + 8] = A.o[m][2 + e];
      }
      if (g == 0) {
        float* ml = a.part_ml + ((size_t)slot * G + hh) * 2;
        ml[0] = A.m[e];
        ml[1] = A.l[e];
      }
    }
  }
}
// Chunking plan, computed identically by every CTA of every grid from the
// key counts: pages_j = ceil(keys_j / 16); chunk = max(4, ceil(sum_j pages_j
// * Hkv / (ipw * warps))) with warps = 8 * plan_ctas; chunks_j =
// ceil(pages_j / chunk); S_j = prefix sums.  ipw = 4 items per warp, or 2
// when every request has about the same length (longest <= 1.25 x mean):
// equal requests give equal items, so the queue stays balanced with fewer,
// longer items, which start up fewer times and leave fewer partials to merge.
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
    int pmax = 0;
    for (int j = lane; j < n; j += 32) {
      tot += s_pages[j];
      pmax = max(pmax, s_pages[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tot += __shfl_xor_sync(0xffffffffu, tot, o);
      pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
    }
    const long long chunk = decode_plan_chunk(tot, pmax, n, a.Hkv, a.plan_ctas);
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
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, DecodeArgs a) {
  using R = Ring<D>;
  extern __shared__ __align__(16) uint8_t dsm_raw[];
  int* dsm;
  {
    const uint32_t s0 = smem_u32(dsm_raw);
    dsm = reinterpret_cast<int*>(dsm_raw + (((s0 + 1023u) & ~1023u) - s0));
  }
  int* s_pref = dsm;                          // [n + 1]
  int* s_pages = dsm + kMaxDecodeReqs + 1;    // [n]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch();
  if (!a.pdl) griddep_wait();
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(dsm) + kPlanBytes + kRingBytes);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kDecodeWarps * R::STAGES; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  const int chunk = build_plan(a, s_pref, s_pages);   // ends with __syncthreads
  uint64_t* full = bars + warp * R::STAGES;
  const uint32_t ring = smem_u32(dsm) + kPlanBytes + warp * R::STAGES * R::PAGE;
  const int G = a.Hq / a.Hkv;
  const int g = lane >> 2, t = lane & 3;
  const long long total = (long long)s_pref[a.n] * a.Hkv;
  const int oob_row = a.num_pages * a.Hkv * 16;   // first row past the pool: zero-filled box
  volatile int no_abort = 0;
  const WaitCtl wc{&no_abort, a.err, a.wait_ns};

  if (total > a.max_items) {   // cannot happen with the plan bound; never write past the partials
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(a.err, CF_DEVERR_CONTEXT);
    return;
  }
  uint32_t issued = 0, consumed = 0;   // pages of this warp, over all its items
  bool ok_run = true;
  // items are taken from a global queue: (request, chunk, KV head), head fastest
  int item = 0;
  if (lane == 0) item = atomicAdd(a.counter, 1);
  item = __shfl_sync(0xffffffffu, item, 0);
  while (item < total && ok_run) {
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

    // Q fragments (natural d order): k-step s uses d = 16 s + 2 t (+8)
    uint32_t qa[D / 16][2], qb[G16 ? D / 16 : 1][2];
    const __nv_bfloat16* qrow = a.q + (size_t)j * a.q_stride + (size_t)h * G * D;
#pragma unroll
    for (int st = 0; st < D / 16; ++st) {
      qa[st][0] = g < G ? *reinterpret_cast<const uint32_t*>(qrow + g * D + 16 * st + 2 * t) : 0u;
      qa[st][1] = g < G ? *reinterpret_cast<const uint32_t*>(qrow + g * D + 16 * st + 8 + 2 * t) : 0u;
      if constexpr (G16) {
        qb[st][0] = g + 8 < G ? *reinterpret_cast<const uint32_t*>(qrow + (g + 8) * D + 16 * st + 2 * t) : 0u;
        qb[st][1] = g + 8 < G ? *reinterpret_cast<const uint32_t*>(qrow + (g + 8) * D + 16 * st + 8 + 2 * t) : 0u;
      }
    }
    // G <= 8: the transposed products; G > 8: the query heads as MMA rows
    typename std::conditional<G16, Acc16<D>, AccT<D>>::type A;
    acc_init(A);

    // ring pipeline: up to STAGES pages in flight; lane 0 issues the TMA
    // copies of page p0 + k into slot (issued % STAGES)
    const int np = p1 - p0;
    uint32_t okmask = 0;   // bit s: the page in ring slot s has a valid id
    int k_issue = 0;
    for (; k_issue < np && k_issue < R::STAGES; ++k_issue) {
      const int sl = issued % R::STAGES;
      const int pid = table[p0 + k_issue];
      const bool ok = pid >= 0 && pid < a.num_pages;
      okmask = ok ? (okmask | (1u << sl)) : (okmask & ~(1u << sl));
      if (lane == 0) {
        const int row = ok ? (pid * a.Hkv + h) * 16 : oob_row;
        const uint32_t kt = ring + sl * R::PAGE;
        mbar_expect_tx(&full[sl], R::PAGE);
#pragma unroll
        for (int hd = 0; hd < D / 64; ++hd) {
          tma_load_2d_u32(kt + hd * R::HALF, &tmK, &full[sl], hd * 64, row);
          tma_load_2d_u32(kt + R::KV + hd * R::HALF, &tmV, &full[sl], hd * 64, row);
        }
      }
      ++issued;
    }
    int pid_next = k_issue < np ? table[p0 + k_issue] : -1;
    for (int i = 0; i < np; ++i) {
      const int sl = consumed % R::STAGES;
      if (!mbar_wait(&full[sl], (consumed / R::STAGES) & 1, wc)) {
        ok_run = false;
        break;
      }
      const int p = p0 + i;
      int valid = keys - p * 16;
      valid = valid > 16 ? 16 : valid;
      if (!((okmask >> sl) & 1u)) {
        if (lane == 0) set_error(a.err, CF_DEVERR_PAGE);
        valid = 0;
      }
      const uint32_t kt = ring + sl * R::PAGE;
      acc_page(A, kt, kt + R::KV, valid, qa, qb, a.scale_log2, lane);
      ++consumed;
      __syncwarp();   // every lane has read the slot before it is refilled
      if (k_issue < np) {
        const int sl2 = issued % R::STAGES;
        const bool ok = pid_next >= 0 && pid_next < a.num_pages;
        okmask = ok ? (okmask | (1u << sl2)) : (okmask & ~(1u << sl2));
        if (lane == 0) {
          fence_proxy_async_smem();   // the slot's generic-proxy reads come before the TMA refill
          const int row = ok ? (pid_next * a.Hkv + h) * 16 : oob_row;
          const uint32_t kt2 = ring + sl2 * R::PAGE;
          mbar_expect_tx(&full[sl2], R::PAGE);
#pragma unroll
          for (int hd = 0; hd < D / 64; ++hd) {
            tma_load_2d_u32(kt2 + hd * R::HALF, &tmK, &full[sl2], hd * 64, row);
            tma_load_2d_u32(kt2 + R::KV + hd * R::HALF, &tmV, &full[sl2], hd * 64, row);
          }
        }
        ++issued;
        ++k_issue;
        pid_next = k_issue < np ? table[p0 + k_issue] : -1;
      }
    }
    if (!ok_run) break;
    acc_finish(A, a, j, h, G, item, nch == 1, lane);   // partial index = (S_j + c) * Hkv + h
    if (lane == 0) item = atomicAdd(a.counter, 1);
    item = __shfl_sync(0xffffffffu, item, 0);
  }
  if (!ok_run) {   // a wait gave up: let this warp's own copies land before exiting
    volatile int dummy = 0;
    const WaitCtl w2{&dummy, nullptr, a.wait_ns};
    while (consumed < issued) {
      mbar_wait(&full[consumed % R::STAGES], (consumed / R::STAGES) & 1, w2);
      ++consumed;
    }
  }
}
// One warp per (request, query head): merges the chunk partials.
template <int D>
__global__ void decode_merge_kernel(DecodeArgs a) {
  const int G = a.Hq / a.Hkv;
  const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.counter = 0;   // the decode kernel has finished with it
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
  // chunk c's partial of this (request, head) sits at ((s0 + c) Hkv + h) G + g
  const long long stride = (long long)a.Hkv * G;
  const long long base = ((long long)s0 * a.Hkv + h) * G + g;
  const float2* mlp = reinterpret_cast<const float2*>(a.part_ml);
  // (m, l) of chunks lane and lane + 32 stay in registers; later chunks
  // (more than 64, rare) are read again in the O pass
  const float2 ninf = make_float2(-INFINITY, 0.f);
  const float2 ml0 = lane < nch ? mlp[base + lane * stride] : ninf;
  const float2 ml1 = lane + 32 < nch ? mlp[base + (lane + 32) * stride] : ninf;
  float M = fmaxf(ml0.x, ml1.x);
  for (int c = lane + 64; c < nch; c += 32) M = fmaxf(M, mlp[base + c * stride].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float Mu = M == -INFINITY ? 0.f : M;
  const float w0 = fast_exp2(ml0.x - Mu), w1 = fast_exp2(ml1.x - Mu);   // exp2(-inf) = 0
  float L = fmaf(w0, ml0.y, w1 * ml1.y);
  for (int c = lane + 64; c < nch; c += 32) {
    const float2 ml = mlp[base + c * stride];
    L = fmaf(fast_exp2(ml.x - Mu), ml.y, L);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  // O: the chunks in order (the sum order does not depend on the lanes),
  // sixteen chunks' loads in flight; chunk c's weight comes from lane c % 32
  constexpr int B = 16;
  int c = 0;
  for (; c + B <= nch; c += B) {
    float po[B][PER];
#pragma unroll
    for (int u = 0; u < B; ++u) {
      const float* src = a.part_o + (base + (c + u) * stride) * D + lane * PER;
      if constexpr (PER == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        po[u][0] = v.x; po[u][1] = v.y; po[u][2] = v.z; po[u][3] = v.w;
      } else {
#pragma unroll
        for (int i = 0; i < PER; ++i) po[u][i] = src[i];
      }
    }
#pragma unroll
    for (int u = 0; u < B; ++u) {
      const int cu = c + u;
      const float wa = __shfl_sync(0xffffffffu, w0, cu & 31), wb = __shfl_sync(0xffffffffu, w1, cu & 31);
      const float w = cu < 32 ? wa : (cu < 64 ? wb : fast_exp2(mlp[base + cu * stride].x - Mu));
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] = fmaf(w, po[u][i], acc[i]);
    }
  }
  for (; c < nch; ++c) {
    const float wa = __shfl_sync(0xffffffffu, w0, c & 31), wb = __shfl_sync(0xffffffffu, w1, c & 31);
    const float w = c < 32 ? wa : (c < 64 ? wb : fast_exp2(mlp[base + c * stride].x - Mu));
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = fmaf(w, a.part_o[(base + c * stride) * D + lane * PER + i], acc[i]);
  }
  const float inv = L > 0.f ? 1.0f / L : 0.f;
#pragma unroll
  for (int i = 0; i < PER; i += 2)
    *reinterpret_cast<uint32_t*>(orow + lane * PER + i) = pack_bf16(acc[i] * inv, acc[i + 1] * inv);
}

template <int D, bool G16>
cudaError_t launch_t(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, int ctas, cudaStream_t s) {
  static std::atomic<unsigned long long> attr{0};
  const cudaError_t e = smem_limit_per_device(decode_kernel<D, G16>, kDecodeSmem, attr);
  if (e != cudaSuccess) return e;
  if (a.pdl) return launch_pdl(decode_kernel<D, G16>, dim3(ctas), dim3(kThreads), kDecodeSmem, s, tk, tv, a);
  decode_kernel<D, G16><<<ctas, kThreads, kDecodeSmem, s>>>(tk, tv, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t merge_t(const DecodeArgs& a, cudaStream_t s) {
  const long long warps = (long long)a.n * a.Hq;
  const int blocks = (int)((warps * 32 + 255) / 256);
  decode_merge_kernel<D><<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

long long decode_max_items(int max_decode, int Hkv, int max_ctas) {
  return (long long)kItemsPerWarp * max_ctas * kDecodeWarps + (long long)max_decode * Hkv + 64;
}

cudaError_t launch_decode_kernel(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, int num_ctas,
                                 cudaStream_t s) {
  if (a.n <= 0) return cudaSuccess;
  if (a.n > kMaxDecodeReqs || a.plan_ctas <= 0) return cudaErrorInvalidValue;
  const bool g16 = a.Hq / a.Hkv > 8;
  if (a.head_dim == 128)
    return g16 ? launch_t<128, true>(tk, tv, a, num_ctas, s) : launch_t<128, false>(tk, tv, a, num_ctas, s);
  if (a.head_dim == 64)
    return g16 ? launch_t<64, true>(tk, tv, a, num_ctas, s) : launch_t<64, false>(tk, tv, a, num_ctas, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_merge(const DecodeArgs& a, cudaStream_t s) {
  if (a.n <= 0) return cudaSuccess;
  if (a.head_dim == 128) return merge_t<128>(a, s);
  if (a.head_dim == 64) return merge_t<64>(a, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, int num_ctas,
                          cudaStream_t s) {
  cudaError_t e = launch_decode_kernel(tk, tv, a, num_ctas, s);
  return e == cudaSuccess ? launch_decode_merge(a, s) : e;
}

}  // namespace cf
