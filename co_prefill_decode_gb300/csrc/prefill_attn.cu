// Causal chunked-prefill attention over a paged, cached prefix on tcgen05.
//
// Chunk query i sits at position c_p + i and attends to keys 0..c_p+i of its
// request (Adaptive Context Parallelism §2.1, mask M_ij = 0 iff j <= i;
// ConfluxServe §4: later chunks reuse the historical KV in place).  The
// useful work is W(l, c_p) = l c_p + l(l+1)/2 query-key pairs (Adaptive
// Context Parallelism §2.2 Eq. 1, ConfluxServe App. D Eq. 9); key tiles that
// are entirely masked are never visited and only tiles that cross the
// diagonal are masked.
//
// A work item is (128-row query tile, query head).  Persistent CTAs draw
// items from a device-wide queue (an atomic counter zeroed earlier in the
// step), so several grids can share one chunk's items: the layer step runs
// one grid on the prefill SM partition and, once decode attention is done,
// a second one on the decode partition.  11 warps per CTA:
//   warp 0   TMA producer of the Q tile and, per 128-key tile, of the eight
//            (page, KV head) K boxes of 16 x 64 (x2 for d = 128; each page
//            is a contiguous 4 KB tile of the pool), one box per lane; lane
//            0 also takes the next item from the queue and publishes it to
//            the other roles through a small shared-memory ring;
//   warp 2   TMA producer of the V boxes, a 3-stage K/V ring in all;
//   warp 1   one thread issues tcgen05.mma: S = Q K^T into one of two TMEM
//            buffers, O += P V into a TMEM accumulator;
//   warps 3+ two threads per query row, each on 64 of a tile's keys and
//            half of the output columns: load S from TMEM, combine the row
//            maximum and sum through shared memory, online softmax in the
//            log2 domain with lazy rescaling (O is rescaled in TMEM only
//            when the running max grows by more than 2^8), write P back to
//            TMEM as bf16, and at the end normalise O and store it.
// S_{j+1} is computed while the softmax works on S_j, and PV_j runs while
// the softmax works on S_{j+1}.  P lives in TMEM (two buffers) and is the A
// operand of the PV MMA, which leaves shared memory for three K/V stages.
#include "common.cuh"
#include "internal.h"

namespace cf {

namespace {

// threads per query row in the softmax (8 softmax warps, two per SM
// sub-partition, so the MMA-issuing warp is not starved of issue slots);
// each thread handles 128/NSPLIT keys of a tile and D/NSPLIT output columns
template <int D>
struct Split {
  static constexpr int NSPLIT = 2;
  static constexpr int SOFTMAX_THREADS = 128 * NSPLIT;
  static constexpr int THREADS = 96 + SOFTMAX_THREADS;   // + 2 producer warps + MMA warp
};
constexpr int BQ = 128;     // query rows per tile
constexpr int BKV = 128;    // keys per tile (8 pages of 16)
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D>
struct PfCfg {
  static constexpr uint32_t HALF = BQ * 64 * 2;          // 16 KB: 128 rows x 64 bf16
  static constexpr uint32_t Q_BYTES = HALF * (D / 64);
  static constexpr uint32_t KV_BYTES = HALF * (D / 64);  // one K (or V) tile of 128 keys
  static constexpr int KV_STAGES = 3;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + KV_STAGES * KV_BYTES;
  static constexpr uint32_t OFF_X = OFF_V + KV_STAGES * KV_BYTES;   // row exchange [NSPLIT][128] fp32
  static constexpr uint32_t OFF_BAR = OFF_X + Split<D>::NSPLIT * 128 * 4;
  // no alignment slack: the kernel checks that the base is 1 KB aligned
  static constexpr size_t SMEM = OFF_BAR + 512;   // mbarriers, item ring, TMEM address
  static_assert(SMEM <= 232448, "shared memory per CTA");
  // TMEM columns: S0 [0,128), S1 [128,256), O [256, 256 + D), P0 [384, 448), P1 [448, 512)
  // (P holds 128 bf16 keys per row, two per 32-bit column)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_O = 256, T_P = 384;
};

struct Item {
  int qt, head;
};


CF_DEV Item item_of(int idx, int Hq, int n_qt) {
  Item it;
  it.qt = n_qt - 1 - idx / Hq;   // heaviest (last) query tiles first
  it.head = idx % Hq;
  return it;
}
CF_DEV int kv_tiles(const PrefillArgs& a, int qt) {
  const int end = min(a.prefix + qt * BQ + BQ, a.prefix + a.l);   // exclusive key end
  return (end + BKV - 1) / BKV;
}

template <int D>
__global__ void __launch_bounds__(Split<D>::THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, PrefillArgs a) {
  using C = PfCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (smem_u32(smem_raw) & 1023u) {   // the swizzled tiles need a 1 KB aligned base
    if (threadIdx.x == 0) set_error(a.err, CF_DEVERR_INTERNAL);
    return;
  }
  constexpr int NS = C::KV_STAGES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;             // [NS]
  uint64_t* k_empty = k_full + NS;         // [NS]
  uint64_t* v_full = k_empty + NS;         // [NS]
  uint64_t* v_empty = v_full + NS;         // [NS]
  uint64_t* s_full = v_empty + NS;         // [2] per S buffer
  uint64_t* s_free = s_full + 2;           // [2]
  uint64_t* p_full = s_free + 2;           // [2] per P buffer
  uint64_t* pv_done = p_full + 2;          // [2]
  uint64_t* o_free = pv_done + 2;
  uint64_t* drain = o_free + 1;
  uint64_t* item_ready = drain + 1;        // [8] per item-ring slot
  volatile int* ring = reinterpret_cast<volatile int*>(item_ready + 8);   // [8] item ids
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(const_cast<int*>(ring) + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch();
  if (!a.pdl) griddep_wait();
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], Split<D>::SOFTMAX_THREADS);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], Split<D>::SOFTMAX_THREADS);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(o_free, Split<D>::SOFTMAX_THREADS);
    for (int i = 0; i < 8; ++i) mbar_init(&item_ready[i], 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const WaitCtl wc{abort_flag, a.err, a.wait_ns};

  const int G = a.Hq / a.Hkv;
  const int n_qt = (a.l + BQ - 1) / BQ;
  const int n_items = n_qt * a.Hq;
  const int n_pages_req = (a.prefix + a.l + a.page_size - 1) / a.page_size;
  const int oob_row = a.num_pages * a.Hkv * a.page_size;   // first row past the pool

  if (warp == 0 || warp == 2) {  // ------------------------------------ producers
    // Warp 0 loads Q and the K tiles, warp 2 the V tiles, so the two streams
    // of small boxes are issued in parallel.  In each, lane 0 waits on the
    // ring and arms the barrier; lanes 0..8*(D/64)-1 then each issue one
    // (page, d-half) box.  Lanes 0..7 hold the page ids of the tile, loaded
    // one tile ahead.
    const bool is_v = warp == 2;
    constexpr int NBOX = 8 * (D / 64);
    int qc = 0, kc = 0;
    bool ok = true;
    uint32_t last_q = 0xffffffffu, last_k[NS], last_v[NS];
    for (int i = 0; i < NS; ++i) last_k[i] = last_v[i] = 0xffffffffu;
    for (int k = 0; ok; ++k) {
      // Work items come from a queue shared by every CTA of this launch and
      // of a second launch that picks up the SMs decode leaves behind.  Warp
      // 0 takes the next item once the Q buffer is free and publishes it to
      // the other warps through an 8-slot ring (no warp is more than 4 items
      // behind the fetcher, so a slot is always read before it is reused).
      int idx = -1;
      if (!is_v) {
        if (lane == 0) {
          ok = mbar_wait(q_empty, (qc & 1) ^ 1, wc);
          if (ok) {
            const unsigned got = atomicAdd(a.counter, 1u) - a.base;
            idx = got < (unsigned)n_items ? (int)got : -1;
            ring[k & 7] = idx;
            mbar_arrive(&item_ready[k & 7]);
            if (idx >= 0) {
              const Item it0 = item_of(idx, a.Hq, n_qt);
              mbar_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
              for (int hd = 0; hd < D / 64; ++hd)
                tma_load_3d(smem + C::OFF_Q + hd * C::HALF, &tmQ, q_full, hd * 64, it0.head, it0.qt * BQ);
              last_q = qc & 1;
            }
          }
        }
      } else if (lane == 0) {
        ok = mbar_wait(&item_ready[k & 7], (k >> 3) & 1, wc);
        idx = ok ? ring[k & 7] : -1;
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      if (!ok || idx < 0) break;
      const Item it = item_of(idx, a.Hq, n_qt);
      const int kvh = it.head / G;
      ++qc;
      const int nkv = kv_tiles(a, it.qt);
      int pid = (lane < 8 && lane < n_pages_req) ? a.pages[lane] : -1;
      for (int j = 0; j < nkv; ++j, ++kc) {
        const int st = kc % NS;
        const uint32_t ph = (kc / NS) & 1;
        const int pi = j * 8 + lane;
        int row = oob_row;   // a missing page reads as zeros
        if (lane < 8 && pi < n_pages_req) {
          if (pid >= 0 && pid < a.num_pages)
            row = (pid * a.Hkv + kvh) * a.page_size;
          else
            set_error(a.err, CF_DEVERR_PAGE);
        }
        // page ids of the next tile, so the next copies do not wait on them
        const int pin = (j + 1) * 8 + lane;
        const int pid_next = (lane < 8 && j + 1 < nkv && pin < n_pages_req) ? a.pages[pin] : -1;
        const int my_page = lane / (D / 64), my_hd = lane % (D / 64);
        const int my_row = __shfl_sync(0xffffffffu, row, my_page & 7);
        // K tile
        if (!is_v) {
          if (lane == 0) {
            ok = mbar_wait(&k_empty[st], ph ^ 1, wc);
            if (ok) mbar_expect_tx(&k_full[st], C::KV_BYTES);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          if (lane < NBOX)
            tma_load_2d(smem + C::OFF_K + st * C::KV_BYTES + my_hd * C::HALF + my_page * 2048, &tmK, &k_full[st],
                        my_hd * 64, my_row);
          if (lane == 0) last_k[st] = ph;
        }
        // V tile
        if (is_v) {
          if (lane == 0) {
            ok = mbar_wait(&v_empty[st], ph ^ 1, wc);
            if (ok) mbar_expect_tx(&v_full[st], C::KV_BYTES);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          if (lane < NBOX)
            tma_load_2d(smem + C::OFF_V + st * C::KV_BYTES + my_hd * C::HALF + my_page * 2048, &tmV, &v_full[st],
                        my_hd * 64, my_row);
          if (lane == 0) last_v[st] = ph;
        }
        pid = pid_next;
      }
    }
    // Let our own copies land before the CTA exits (normally consumed long
    // ago; after an expired wait anywhere in the CTA they may be in flight).
    if (lane == 0) {
      volatile int dummy = 0;
      const WaitCtl w2{&dummy, nullptr, a.wait_ns};
      if (last_q != 0xffffffffu) mbar_wait(q_full, last_q, w2);
      for (int i = 0; i < NS; ++i) {
        if (last_k[i] != 0xffffffffu) mbar_wait(&k_full[i], last_k[i], w2);
        if (last_v[i] != 0xffffffffu) mbar_wait(&v_full[i], last_v[i], w2);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------------ MMA issuer
      constexpr uint32_t IDESC_S = idesc_bf16(128, BKV, false);
      constexpr uint32_t IDESC_PV = idesc_bf16(128, D, true);
      const uint64_t qdesc = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
      int qc = 0, kc = 0, sc = 0, pc = 0, oc = 0;
      bool ok = true, issued = false;
      for (int k = 0; ok; ++k) {
        if (!mbar_wait(&item_ready[k & 7], (k >> 3) & 1, wc)) { ok = false; break; }
        const int idx = ring[k & 7];
        if (idx < 0) break;
        const Item it = item_of(idx, a.Hq, n_qt);
        const int nkv = kv_tiles(a, it.qt);
        if (!mbar_wait(q_full, qc & 1, wc)) { ok = false; break; }
        ++qc;
        int vc = kc;   // V tile counter trails the K tile counter
        for (int j = 0; j <= nkv && ok; ++j) {
          if (j < nkv) {  // S_j = Q K_j^T
            const int sb = sc & 1;
            const int st = kc % NS;
            if (!mbar_wait(&s_free[sb], ((sc >> 1) & 1) ^ 1, wc)) { ok = false; break; }
            if (!mbar_wait(&k_full[st], (kc / NS) & 1, wc)) { ok = false; break; }
            tc_fence_after();
            const uint64_t kdesc = sdesc_sw128(smem_u32(smem + C::OFF_K + st * C::KV_BYTES), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = ((kk >> 2) * C::HALF + (kk & 3) * 32) >> 4;   // in the start-address field
              umma_bf16(tmem + sb * BKV, qdesc + off, kdesc + off, IDESC_S, kk > 0);
            }
            issued = true;
            umma_commit(&k_empty[st]);
            umma_commit(&s_full[sb]);
            if (j == nkv - 1) umma_commit(q_empty);
            ++sc;
            ++kc;
          }
          if (j >= 1) {  // O += P_{j-1} V_{j-1}, P read from TMEM
            const int st = vc % NS;
            const int pb = pc & 1;   // P buffer of this PV
            if (!mbar_wait(&p_full[pb], (pc >> 1) & 1, wc)) { ok = false; break; }
            if (!mbar_wait(&v_full[st], (vc / NS) & 1, wc)) { ok = false; break; }
            if (j == 1 && !mbar_wait(o_free, (oc & 1) ^ 1, wc)) { ok = false; break; }
            tc_fence_after();
            const uint64_t vdesc = sdesc_sw128(smem_u32(smem + C::OFF_V + st * C::KV_BYTES), C::HALF, 1024);
#pragma unroll
            for (int kk = 0; kk < BKV / 16; ++kk)
              umma_bf16_ta(tmem + C::T_O, tmem + C::T_P + pb * 64 + kk * 8, vdesc + ((kk * 2048) >> 4), IDESC_PV,
                           (j > 1 || kk > 0));
            umma_commit(&v_empty[st]);
            umma_commit(&pv_done[pb]);
            ++pc;
            ++vc;
          }
        }
        ++oc;
      }
      if (!ok && issued) {
        volatile int dummy = 0;
        const WaitCtl w2{&dummy, nullptr, a.wait_ns};
        umma_commit(drain);
        mbar_wait(drain, 0, w2);
      }
    }
  } else {  // --------------------------------------------------- softmax warps
    constexpr int NSPLIT = Split<D>::NSPLIT;
    constexpr int HK = BKV / NSPLIT;          // keys of each thread per tile
    constexpr int HD = D / NSPLIT;            // output columns of each thread (32)
    static_assert(HD % 32 == 0, "32-column TMEM loads");
    const int quarter = warp & 3;             // the TMEM lane quarter this warp may access
    const int sub = (warp - 3) >> 2;          // which slice of the keys / output columns
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t bar_id = 1 + quarter;      // the NSPLIT warps of this quarter
    float* xbuf = reinterpret_cast<float*>(smem + C::OFF_X);
    int sc = 0, tc = 0, vc = 0;   // tc: KV tiles this thread has processed (P buffer tc & 1)
    bool ok = true;
    // Within an item the softmax threads never leave a loop early: a failed
    // wait only clears `ok`, so the threads of a row always meet at the same
    // exchanges.
    // Combine one value over the NSPLIT threads of this row (max or sum).
    auto row_sync = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(32 * NSPLIT) : "memory"); };
    auto row_max = [&](float v) {
      xbuf[sub * 128 + r] = v;
      row_sync();
      float m = v;
#pragma unroll
      for (int k = 0; k < NSPLIT; ++k) m = fmaxf(m, xbuf[k * 128 + r]);
      row_sync();   // every read is done before the buffer is written again
      return m;
    };
    auto row_sum = [&](float v) {
      xbuf[sub * 128 + r] = v;
      row_sync();
      float t = 0.f;
#pragma unroll
      for (int k = 0; k < NSPLIT; ++k) t += xbuf[k * 128 + r];
      row_sync();
      return t;
    };
    for (int k = 0; ok; ++k) {
      if (!mbar_wait(&item_ready[k & 7], (k >> 3) & 1, wc)) ok = false;
      const int idx = ok ? ring[k & 7] : -1;
      // every thread of a row reads the same slot: they leave together
      if (idx < 0) break;
      const Item it = item_of(idx, a.Hq, n_qt);
      const int nkv = kv_tiles(a, it.qt);
      const int qi = it.qt * BQ + r;
      const int qpos = a.prefix + qi;
      const int kend = a.prefix + a.l;          // first key that does not exist
      const int diag = a.prefix + it.qt * BQ;   // smallest query position of the tile
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nkv; ++j) {
        const int sb = sc & 1;
        if (!mbar_wait(&s_full[sb], (sc >> 1) & 1, wc)) ok = false;
        tc_fence_after();
        float s[HK];
        if constexpr (HK == 32) {
          tmem_ld32(tmem + lane_off + sb * BKV + sub * HK, s);
        } else {
#pragma unroll
          for (int c = 0; c < HK / 32; ++c) tmem_ld32(tmem + lane_off + sb * BKV + sub * HK + c * 32, s + c * 32);
        }
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&s_free[sb]);
        ++sc;
        const int kv0 = j * BKV + sub * HK;    // first key of this thread's slice
        if (j * BKV + BKV - 1 > diag) {         // tile crosses the diagonal or the end of the request
#pragma unroll
          for (int c = 0; c < HK; ++c) {
            const int kp = kv0 + c;
            if (!(kp <= qpos && kp < kend)) s[c] = -INFINITY;
          }
        }
        // row max: 8 independent partial maxima, then the other slices'
        float mp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mp[i] = s[i];
#pragma unroll
        for (int c = 8; c < HK; ++c) mp[c & 7] = fmaxf(mp[c & 7], s[c]);
        const float mh = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                               fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
        const float mx = row_max(mh) * a.scale_log2;
        // P buffer pb was last read by the PV of tile tc - 2: wait for it
        const int pb = tc & 1;
        if (tc >= 2 && !mbar_wait(&pv_done[pb], ((tc - 2) >> 1) & 1, wc)) ok = false;
        const bool grow = (m == -INFINITY) ? false : (mx > m + kRescaleThreshold);
        if (m == -INFINITY) m = mx;
        if (__any_sync(0xffffffffu, grow)) {
          // O is about to be rescaled: the PV of the previous tile must be done
          if (!mbar_wait(&pv_done[pb ^ 1], ((tc - 1) >> 1) & 1, wc)) ok = false;
          tc_fence_after();
          const float alpha = grow ? fast_exp2(m - mx) : 1.0f;
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            float o[32];
            tmem_ld32(tmem + lane_off + C::T_O + sub * HD + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(tmem + lane_off + C::T_O + sub * HD + c * 32, o);
          }
          tmem_st_wait();
          if (grow) {
            l *= alpha;
            m = mx;
          }
        }
        const float mu = m == -INFINITY ? 0.f : m;
        const float sc2 = a.scale_log2;
        float lp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) lp[i] = 0.f;
        uint32_t pk[HK / 2];   // P as bf16 pairs, low half = even key
#pragma unroll
        for (int c8 = 0; c8 < HK / 8; ++c8) {
          float p[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            p[i] = fast_exp2(fmaf(s[c8 * 8 + i], sc2, -mu));
            lp[i] += p[i];
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) pk[c8 * 4 + i] = pack_bf16(p[2 * i], p[2 * i + 1]);
        }
        // this thread's HK keys are HK/2 columns of P buffer pb in its TMEM lane
        if constexpr (HK == 32)
          tmem_st16(tmem + lane_off + C::T_P + pb * 64 + sub * 16, pk);
        else
          tmem_st32(tmem + lane_off + C::T_P + pb * 64 + sub * 32, reinterpret_cast<const float*>(pk));
        tmem_st_wait();
        l += ((lp[0] + lp[1]) + (lp[2] + lp[3])) + ((lp[4] + lp[5]) + (lp[6] + lp[7]));
        // keys past the end of the request: zero their V rows (slots may hold anything)
        const int vst = vc % NS;
        const int kt0 = j * BKV;
        if (kend - kt0 < BKV) {
          if (!mbar_wait(&v_full[vst], (vc / NS) & 1, wc)) ok = false;
          const int vk = max(0, kend - kt0);
          uint8_t* vt = smem + C::OFF_V + vst * C::KV_BYTES;
          const int nz = (BKV - vk) * (D / 64) * 8;   // 16-byte chunks
          for (int z = sub * 128 + r; z < nz; z += Split<D>::SOFTMAX_THREADS) {
            const int row = vk + z / ((D / 64) * 8);
            const int rem = z % ((D / 64) * 8);
            *reinterpret_cast<uint4*>(vt + (rem >> 3) * C::HALF + row * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();   // the zeros must be visible to the tensor core's V reads
        }
        ++vc;
        tc_fence_before();
        mbar_arrive(&p_full[pb]);
        ++tc;
      }
      // epilogue: O / l -> bf16, each thread its D/2 columns
      if (!mbar_wait(&pv_done[(tc - 1) & 1], ((tc - 1) >> 1) & 1, wc)) ok = false;   // the item's last PV
      tc_fence_after();
      const float lt = row_sum(l);
      const float inv = lt > 0.f ? 1.0f / lt : 0.f;
      __nv_bfloat16* orow = a.out + (size_t)qi * a.out_stride + (size_t)it.head * D + sub * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        float o[32];
        tmem_ld32(tmem + lane_off + C::T_O + sub * HD + c * 32, o);
        tmem_ld_wait();
        if (qi < a.l && ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 w;
            w.x = pack_bf16(o[8 * i + 0] * inv, o[8 * i + 1] * inv);
            w.y = pack_bf16(o[8 * i + 2] * inv, o[8 * i + 3] * inv);
            w.z = pack_bf16(o[8 * i + 4] * inv, o[8 * i + 5] * inv);
            w.w = pack_bf16(o[8 * i + 6] * inv, o[8 * i + 7] * inv);
            dst[i] = w;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(o_free);
      // both threads of a row leave together: after a failed (bounded) wait
      // every later wait of this CTA returns at once, so the pair only has to
      // agree here instead of at a barrier the other might never reach
      const bool row_ok = row_max(ok ? 0.f : 1.f) < 0.5f;
      if (!row_ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D>
cudaError_t launch_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const PrefillArgs& a,
                     int ctas, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e =
        cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PfCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  ctas = prefill_grid(a, ctas);
  if (a.pdl) return launch_pdl(prefill_kernel<D>, dim3(ctas), dim3(Split<D>::THREADS), PfCfg<D>::SMEM, s, q, k, v, a);
  prefill_kernel<D><<<ctas, Split<D>::THREADS, PfCfg<D>::SMEM, s>>>(q, k, v, a);
  return cudaGetLastError();
}

}  // namespace

int prefill_grid(const PrefillArgs& a, int ctas) {
  const int n_items = ((a.l + BQ - 1) / BQ) * a.Hq;
  if (ctas > n_items) ctas = n_items;
  return ctas < 1 ? 1 : ctas;
}

int prefill_items(const PrefillArgs& a) { return ((a.l + BQ - 1) / BQ) * a.Hq; }

cudaError_t launch_prefill(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const PrefillArgs& a, int num_ctas, cudaStream_t s) {
  if (a.l <= 0) return cudaSuccess;
  if (a.head_dim == 128) return launch_t<128>(tmQ, tmK, tmV, a, num_ctas, s);
  if (a.head_dim == 64) return launch_t<64>(tmQ, tmK, tmV, a, num_ctas, s);
  return cudaErrorInvalidValue;
}

}  // namespace cf
