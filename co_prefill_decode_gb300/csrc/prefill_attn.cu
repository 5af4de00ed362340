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
// Several chunks of different requests may share a launch (ConfluxServe §6.2
// Eq. 6, the scheduled prefill batch P): each has its own rows of Q and of
// the output, its own prefix c_i and its own page table.
// A work item is a pair of consecutive 128-row query tiles (A, B) of one
// query head of one chunk, and every 128-key K and V tile is loaded once for
// both; when the chunks have too few tile pairs to give every SM one, items
// are single tiles (A only) instead.
// Persistent CTAs draw items from a device-wide queue (an atomic counter
// zeroed earlier in the step), so several grids can share one chunk's items:
// the layer step runs one grid on the prefill SM partition and, once decode
// attention is done, a second one on the decode partition.  12 warps:
//   warp 0    TMA producer of the two Q tiles and, per key tile, of the eight
//             (page, KV head) K boxes of 16 x 64 (x2 for d = 128; each page
//             is a contiguous 4 KB tile of the pool), one box per lane; lane
//             0 also takes the next item from the queue and publishes it to
//             the other roles through a small shared-memory ring;
//   warp 2    TMA producer of the V boxes (2-stage K and V rings);
//   warp 1    one thread issues tcgen05.mma: S_A = Q_A K^T, S_B = Q_B K^T into
//             TMEM, O_A += P_A V and O_B += P_B V with P read from TMEM;
//   warps 4-7 softmax of tile A, warps 8-11 of tile B, one thread per query
//             row: load the row of S from TMEM, online softmax in the log2
//             domain with lazy rescaling (O is rescaled in TMEM only when the
//             running max grows by more than 2^8), write P back to TMEM as
//             bf16 over the first half of S, and at the end normalise O and
//             store it.
// The MMAs are issued in the order PV_A(j), S_A(j+1), PV_B(j), S_B(j+1): the
// tensor core computes tile B's products while tile A's softmax runs and the
// other way round, so the two softmax groups alternate on the exp units and
// the tensor pipe stays busy.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace cf {

namespace {

constexpr int BQ = 128;      // query rows per tile
constexpr int BKV = 128;     // keys per tile (8 pages of 16)
constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D>
struct PfCfg {
  static constexpr uint32_t HALF = BQ * 64 * 2;          // 16 KB: 128 rows x 64 bf16
  static constexpr uint32_t TILE = HALF * (D / 64);      // one Q, K or V tile
  // K ring one stage deeper than V: the next S needs the next K tile as soon
  // as the current PV is issued, while V(j) is needed a softmax later
  static constexpr int K_STAGES = 3, V_STAGES = 2;
  static constexpr uint32_t OFF_Q = 0;                   // Q_A, Q_B
  static constexpr uint32_t OFF_K = OFF_Q + 2 * TILE;
  static constexpr uint32_t OFF_V = OFF_K + K_STAGES * TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + V_STAGES * TILE;
  // no alignment slack: the kernel checks that the base is 1 KB aligned
  static constexpr size_t SMEM = OFF_BAR + 512;          // mbarriers, item ring, TMEM address
  static_assert(SMEM <= 232448, "shared memory per CTA");
  // TMEM columns: S of tile x at 128 x (P of tile x, 128 bf16 keys per row,
  // two per 32-bit column, over its first 64 columns); O of tile x at 256 + D x
  static constexpr uint32_t T_S = 0, T_O = 256;
  static constexpr uint32_t TMEM_COLS = 512;
};

// Registers per thread after the split: the loader / MMA warpgroup gives up
// registers it does not need and the two softmax warpgroups take them, so
// the 128 scores of a row stay in registers.  The kernel is launched with
// kLaunchRegs per thread (384 x 168 = 64512); the split uses all of them,
// 128 x 88 + 256 x 208 (each softmax thread keeps its row's 128 scores and
// 16 packed P words in registers without spilling).
constexpr int kLaunchRegs = 168, kLoaderRegs = 88, kSoftmaxRegs = 208;
static_assert(128 * kLoaderRegs + 256 * kSoftmaxRegs <= kThreads * kLaunchRegs, "register split");

CF_DEV float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <uint32_t N>
CF_DEV void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
CF_DEV void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

struct Item {
  int qa, ha, qb, hb;   // query tile and head of tiles A and B (qb = -1: no tile B)
  int k0, k1;           // the key tiles [k0, k1) this item visits
  int part;             // partial slot of tile A (B: part + 1) of a cut item; -1: not cut
  int row0, len, prefix;
  const int* pages;     // the chunk's page table
};

__host__ __device__ inline int units_of(int kind, int n_qt, int Hq) {
  return kind == kPfHeadPairs ? n_qt * (Hq / 2) : (kind == kPfTilePairs ? (n_qt + 1) / 2 : n_qt) * Hq;
}
// Unit u of a chunk with n_qt query tiles.  The query tiles are cut into
// bands of `band` tiles, the band with the most keys first; within a band
// the units are numbered KV head by KV head (query tiles with the most keys
// first, query heads fastest).  CTAs running at the same time then read the
// K/V of one or two KV heads (about 17 MB each for a 32K-token request at
// d = 128), which stay in L2, rather than every KV head of the request at
// scattered key positions.  The band is chosen per chunk so that its query
// tiles differ by at most about a quarter in key count (16 tiles on a long
// prefix, 1 without one), so the heaviest units still start first.
constexpr int kBandQ = 16;
constexpr int kTailSplits = 4, kTailMinTiles = 8;
// the KV-head-major position of unit u among n_g groups of c units per KV
// head (bands of b groups): *r = group index counted from the heaviest,
// *kvh, *j = index within the (group, KV head)
CF_DEV void band_order(int u, int n_g, int c, int Hkv, int b, int* r, int* kvh, int* j) {
  const int band = u / (b * c * Hkv);
  const int rem = u - band * b * c * Hkv;
  const int bt = min(b, n_g - band * b);    // groups in this band
  *kvh = rem / (bt * c);
  const int rem2 = rem % (bt * c);
  *r = band * b + rem2 / c;
  *j = rem2 % c;
}
CF_DEV void unit_tiles(int kind, int u, int n_qt, int Hq, int Hkv, int band, Item& it) {
  const int G = Hq / Hkv;
  int r, kvh, j;
  if (kind == kPfHeadPairs) {
    band_order(u, n_qt, G / 2, Hkv, band, &r, &kvh, &j);
    it.qa = it.qb = n_qt - 1 - r;
    it.ha = kvh * G + 2 * j;
    it.hb = it.ha + 1;
  } else {
    const bool tp = kind == kPfTilePairs;
    const int n_groups = tp ? (n_qt + 1) / 2 : n_qt;
    band_order(u, n_groups, G, Hkv, tp ? (band + 1) / 2 : band, &r, &kvh, &j);
    const int g = n_groups - 1 - r;
    it.ha = it.hb = kvh * G + j;
    it.qa = tp ? 2 * g : g;
    it.qb = (tp && 2 * g + 1 < n_qt) ? 2 * g + 1 : -1;
  }
}
CF_DEV int kv_tiles(const Item& it, int qt) {
  const int end = min(it.prefix + qt * BQ + BQ, it.prefix + it.len);   // exclusive key end
  return (end + BKV - 1) / BKV;
}
CF_DEV int slot_of(const PrefillArgs& a, int idx) {
  int sl = 0;
  while (sl + 1 < a.n_chunks && a.item_end[sl] <= idx) ++sl;
  return sl;
}
CF_DEV void chunk_of(const PrefillArgs& a, int sl, Item& it) {
  it.row0 = a.row0[sl];
  it.len = a.len[sl];
  it.prefix = a.prefix[sl];
  it.pages = a.pages + a.page_off[sl];
}

// Item idx: its chunk slot, its unit and its key range.  The slot's units
// before cut_from run whole, one item each; every later unit is cut into S
// items, split s covering key tiles [s r / S, (s+1) r / S) of the unit's
// reach r (the key tiles of its later query tile).
CF_DEV Item item_at(const PrefillArgs& a, int idx) {
  const int sl = slot_of(a, idx);
  const int local = idx - (sl ? a.item_end[sl - 1] : 0);
  Item it;
  chunk_of(a, sl, it);
  const int c0 = a.cut_from[sl];
  const int S = local < c0 ? 1 : a.splits[sl];
  const int rel = local - c0;   // index among the cut items
  const int u = local < c0 ? local : c0 + rel / S, sp = local < c0 ? 0 : rel % S;
  unit_tiles(a.pair, u, (it.len + BQ - 1) / BQ, a.Hq, a.Hkv, a.band[sl], it);
  const int reach = kv_tiles(it, it.qb > it.qa ? it.qb : it.qa);
  it.k0 = sp * reach / S;
  it.k1 = (sp + 1) * reach / S;
  it.part = S > 1 ? a.part_base[sl] + 2 * rel : -1;
  return it;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ PrefillArgs a) {
  using C = PfCfg<D>;
  constexpr int KS = C::K_STAGES, VS = C::V_STAGES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (smem_u32(smem_raw) & 1023u) {   // the swizzled tiles need a 1 KB aligned base
    if (threadIdx.x == 0) set_error(a.err, CF_DEVERR_INTERNAL);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;             // [KS]
  uint64_t* k_empty = k_full + KS;         // [KS]
  uint64_t* v_full = k_empty + KS;         // [VS]
  uint64_t* v_empty = v_full + VS;         // [VS]
  uint64_t* s_full = v_empty + VS;         // [2] per query tile: S ready
  uint64_t* p_full = s_full + 2;           // [2] P written
  uint64_t* o_done = p_full + 2;           // [2] the item's last PV is done
  uint64_t* o_free = o_done + 2;           // [2] O read by the epilogue
  uint64_t* drain = o_free + 2;
  uint64_t* item_ready = drain + 1;        // [8] per item-ring slot
  volatile int* ring = reinterpret_cast<volatile int*>(item_ready + 8);   // [8] item ids
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(const_cast<int*>(ring) + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch();
  if (!a.pdl) griddep_wait();
  if (a.pdl) {
    // A grid joining a running queue (the fork's second prefill grid): if
    // every item has been taken already, leave before any set-up.  The
    // counter only grows, so a stale read just means no early exit.
    __shared__ int s_drained;
    if (threadIdx.x == 0)
      s_drained = *reinterpret_cast<volatile unsigned*>(a.counter) - a.base >= (unsigned)a.item_end[a.n_chunks - 1];
    __syncthreads();
    if (s_drained) return;
  }
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < KS; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < VS; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], BQ);
      mbar_init(&o_done[x], 1);
      mbar_init(&o_free[x], BQ);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < 8; ++i) mbar_init(&item_ready[i], 1);
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
  const int n_items = a.item_end[a.n_chunks - 1];
  const int oob_row = a.num_pages * a.Hkv * a.page_size;   // first row past the pool

  // The register split is taken inside each warpgroup's own branch, so the
  // compiler allocates each branch for its own limit.
  if (warp >= 4) goto softmax_role;
  regs_dec<kLoaderRegs>();
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
    const int NS = is_v ? VS : KS;   // this warp's ring
    uint32_t last_q = 0xffffffffu, last_k[KS], last_v[VS];
#pragma unroll
    for (int i = 0; i < KS; ++i) last_k[i] = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < VS; ++i) last_v[i] = 0xffffffffu;
    for (int k = 0; ok; ++k) {
      // Warp 0 takes the next item once both Q buffers are free and
      // publishes it through an 8-slot ring (no role is more than two items
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
              const Item it0 = item_at(a, idx);
              const int nq = it0.qb >= 0 ? 2 : 1;
              mbar_expect_tx(q_full, nq * C::TILE);
              for (int t = 0; t < nq; ++t)
#pragma unroll
                for (int hd = 0; hd < D / 64; ++hd)
                  tma_load_3d(smem + C::OFF_Q + t * C::TILE + hd * C::HALF, &tmQ, q_full, hd * 64,
                              t ? it0.hb : it0.ha, it0.row0 + (t ? it0.qb : it0.qa) * BQ);
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
      const Item it = item_at(a, idx);
      const int kvh = it.ha / G;   // tile B's head reads the same KV head
      ++qc;
      const int n_pages_req = (it.prefix + it.len + a.page_size - 1) / a.page_size;
      int pid = (lane < 8 && it.k0 * 8 + lane < n_pages_req) ? it.pages[it.k0 * 8 + lane] : -1;
      for (int j = it.k0; j < it.k1; ++j, ++kc) {
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
        const int pid_next = (lane < 8 && j + 1 < it.k1 && pin < n_pages_req) ? it.pages[pin] : -1;
        const int my_page = lane / (D / 64), my_hd = lane % (D / 64);
        const int my_row = __shfl_sync(0xffffffffu, row, my_page & 7);
        uint64_t* full = is_v ? &v_full[st] : &k_full[st];
        uint64_t* empty = is_v ? &v_empty[st] : &k_empty[st];
        if (lane == 0) {
          ok = mbar_wait(empty, ph ^ 1, wc);
          if (ok) mbar_expect_tx(full, C::TILE);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane < NBOX)
          tma_load_2d(smem + (is_v ? C::OFF_V : C::OFF_K) + st * C::TILE + my_hd * C::HALF + my_page * 2048,
                      is_v ? &tmV : &tmK, full, my_hd * 64, my_row);
        if (lane == 0) {   // (unrolled so the arrays stay in registers)
          if (is_v) {
#pragma unroll
            for (int i = 0; i < VS; ++i)
              if (i == st) last_v[i] = ph;
          } else {
#pragma unroll
            for (int i = 0; i < KS; ++i)
              if (i == st) last_k[i] = ph;
          }
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
#pragma unroll
      for (int i = 0; i < KS; ++i)
        if (last_k[i] != 0xffffffffu) mbar_wait(&k_full[i], last_k[i], w2);
#pragma unroll
      for (int i = 0; i < VS; ++i)
        if (last_v[i] != 0xffffffffu) mbar_wait(&v_full[i], last_v[i], w2);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------------ MMA issuer
      constexpr uint32_t IDESC_S = idesc_bf16(128, BKV, false);
      constexpr uint32_t IDESC_PV = idesc_bf16(128, D, true);
      const uint64_t qdesc0 = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
      const uint64_t qdesc1 = sdesc_sw128(smem_u32(smem + C::OFF_Q + C::TILE), 16, 1024);
      int qc = 0, kc = 0, vc = 0;
      int pc[2] = {0, 0}, ofc[2] = {0, 0};
      bool ok = true, issued = false;
      // S_x = Q_x K^T from K stage st
      auto issue_s = [&](int x, int st) {
        const uint64_t kdesc = sdesc_sw128(smem_u32(smem + C::OFF_K + st * C::TILE), 16, 1024);
        const uint64_t qdesc = x ? qdesc1 : qdesc0;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::HALF + (kk & 3) * 32) >> 4;   // in the start-address field
          umma_bf16(tmem + C::T_S + 128 * x, qdesc + off, kdesc + off, IDESC_S, kk > 0);
        }
        issued = true;
        umma_commit(&s_full[x]);
      };
      // O_x (+)= P_x V from V stage st, P read from TMEM
      auto issue_pv = [&](int x, int st, bool first) {
        const uint64_t vdesc = sdesc_sw128(smem_u32(smem + C::OFF_V + st * C::TILE), C::HALF, 1024);
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk)
          umma_bf16_ta(tmem + C::T_O + D * x, tmem + C::T_S + 128 * x + kk * 8, vdesc + ((kk * 2048) >> 4),
                       IDESC_PV, (!first || kk > 0));
        issued = true;
      };
      for (int k = 0; ok; ++k) {
        if (!mbar_wait(&item_ready[k & 7], (k >> 3) & 1, wc)) { ok = false; break; }
        const int idx = ring[k & 7];
        if (idx < 0) break;
        const Item it = item_at(a, idx);
        // the key tiles of query tile x in this item end at e[x] (none if e[x] <= k0)
        int e[2];
        e[0] = min(it.k1, kv_tiles(it, it.qa));
        e[1] = it.qb >= 0 ? min(it.k1, kv_tiles(it, it.qb)) : 0;
        const int k0 = it.k0, n = it.k1;
        if (!mbar_wait(q_full, qc & 1, wc)) { ok = false; break; }
        ++qc;
        // S of key tile k0 for both query tiles
        if (!mbar_wait(&k_full[kc % KS], (kc / KS) & 1, wc)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if (e[x] > k0) issue_s(x, kc % KS);
        umma_commit(&k_empty[kc % KS]);
        ++kc;
        if (n - k0 == 1) umma_commit(q_empty);
        for (int j = k0; j < n && ok; ++j) {
          const int vst = vc % VS;
          if (!mbar_wait(&v_full[vst], (vc / VS) & 1, wc)) { ok = false; break; }
          const bool more = j + 1 < n;
          bool k_ready = false;
#pragma unroll
          for (int x = 0; x < 2 && ok; ++x) {
            if (j < e[x]) {   // O_x += P_x(j) V_j
              if (!mbar_wait(&p_full[x], pc[x] & 1, wc)) { ok = false; break; }
              ++pc[x];
              if (j == k0) {   // the previous item's epilogue has read O_x
                if (!mbar_wait(&o_free[x], (ofc[x] & 1) ^ 1, wc)) { ok = false; break; }
                ++ofc[x];
              }
              tc_fence_after();
              issue_pv(x, vst, j == k0);
              if (j == e[x] - 1) umma_commit(&o_done[x]);
            }
            if (more && j + 1 < e[x]) {   // S_x(j+1): overwrites P_x(j) after the PV above has read it
              if (!k_ready) {
                if (!mbar_wait(&k_full[kc % KS], (kc / KS) & 1, wc)) { ok = false; break; }
                tc_fence_after();
                k_ready = true;
              }
              issue_s(x, kc % KS);
            }
          }
          if (!ok) break;
          umma_commit(&v_empty[vst]);
          ++vc;
          if (more) {
            umma_commit(&k_empty[kc % KS]);
            ++kc;
            if (j + 2 == n) umma_commit(q_empty);   // the item's last S has been issued
          }
        }
      }
      if (!ok && issued) {
        volatile int dummy = 0;
        const WaitCtl w2{&dummy, nullptr, a.wait_ns};
        umma_commit(drain);
        mbar_wait(drain, 0, w2);
      }
    }
  }
  goto done;
softmax_role:
  {  // ------------------------------------------------------------------ softmax
    regs_inc<kSoftmaxRegs>();
    const int x = (warp - 4) >> 2;            // query tile A (0) or B (1) of the item
    const int quarter = warp & 3;             // the TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;        // row of the query tile
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t ts = tmem + lane_off + C::T_S + 128 * x;
    const uint32_t to = tmem + lane_off + C::T_O + D * x;
    int sc = 0, odc = 0, vbase = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!mbar_wait(&item_ready[k & 7], (k >> 3) & 1, wc)) break;
      const int idx = ring[k & 7];
      if (idx < 0) break;
      const Item it = item_at(a, idx);
      const int qt = x ? it.qb : it.qa;
      const int ea = min(it.k1, kv_tiles(it, it.qa));                  // tile A's key tiles end here
      const int ex = qt >= 0 ? min(it.k1, kv_tiles(it, qt)) : it.k0;   // this tile's
      const int qi = qt * BQ + r;               // query row within the chunk
      const int qpos = it.prefix + qi;
      const int kend = it.prefix + it.len;      // first key that does not exist
      float m = -INFINITY, l = 0.f;
      for (int j = it.k0; j < ex; ++j) {
        if (!mbar_wait(&s_full[x], sc & 1, wc)) { ok = false; break; }
        ++sc;
        tc_fence_after();
        const int kv0 = j * BKV;
        // this row's visible keys in the tile are a prefix [0, lim): causal
        // (key <= query position) and within the request
        const int lim = min(qpos + 1, kend) - kv0;
        const bool masked = lim < BKV;
        float s[BKV];
#pragma unroll
        for (int c = 0; c < BKV / 32; ++c) tmem_ld32(ts + c * 32, s + c * 32);
        tmem_ld_wait();
        if (masked) {
#pragma unroll
          for (int c = 0; c < BKV; ++c) s[c] = c < lim ? s[c] : -INFINITY;
        }
        float mp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mp[i] = max3f(s[i], s[i + 8], s[i + 16]);
#pragma unroll
        for (int c = 24; c < BKV; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) mp[i] = c + 8 + i < BKV ? max3f(mp[i], s[c + i], s[c + 8 + i]) : fmaxf(mp[i], s[c + i]);
        const float mx = max3f(max3f(mp[0], mp[1], mp[2]), max3f(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7])) *
                         a.scale_log2;
        const bool grow = (m == -INFINITY) ? false : (mx > m + kRescaleThreshold);
        if (m == -INFINITY) m = mx;
        if (__any_sync(0xffffffffu, grow)) {
          // S_x(j) is complete, so every earlier MMA (PV_x(j-1)) is too
          const float alpha = grow ? fast_exp2(m - mx) : 1.0f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(to + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(to + c * 32, o);
          }
          tmem_st_wait();
          if (grow) {
            l *= alpha;
            m = mx;
          }
        }
        const float mu = m == -INFINITY ? 0.f : m;
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
        const float2 nmu = make_float2(-mu, -mu);
        float2 lp[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        // P as bf16 pairs (low half = even key), from a second pass over S in
        // TMEM, 32 keys at a time in a loop that is not unrolled: a quarter
        // of the code of an unrolled pass, which keeps the hot loops of the
        // warps sharing each scheduler in its instruction cache.  P of chunk
        // h lands on columns [16 h, 16 h + 16), whose scores an earlier chunk
        // (or this one) has already read.  Scaling and row sums run as packed
        // fp32 pairs (one instruction per two keys).
#pragma unroll 1
        for (int h = 0; h < BKV / 32; ++h) {
          float sh[32];
          tmem_ld32(ts + 32 * h, sh);
          tmem_ld_wait();
          if (masked) {
#pragma unroll
            for (int c = 0; c < 32; ++c) sh[c] = 32 * h + c < lim ? sh[c] : -INFINITY;
          }
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 xs = __ffma2_rn(make_float2(sh[2 * i], sh[2 * i + 1]), sc2, nmu);
            const float2 p = make_float2(fast_exp2(xs.x), fast_exp2(xs.y));
            lp[i & 1] = __fadd2_rn(lp[i & 1], p);
            pk[i] = pack_bf16(p.x, p.y);
          }
          tmem_st16(ts + 16 * h, pk);
        }
        l += (lp[0].x + lp[1].x) + (lp[0].y + lp[1].y);
        // Keys past the end of the request: zero their V rows (the slots may
        // hold anything).  The tile whose PV reads V_j first does it: A while
        // it has key tile j, else B.
        const int vcnt = vbase + (j - it.k0);
        if (kend - kv0 < BKV && (x == 0 || j >= ea)) {
          const int vst = vcnt % VS;
          if (!mbar_wait(&v_full[vst], (vcnt / VS) & 1, wc)) ok = false;
          const int vk = max(0, kend - kv0);
          uint8_t* vt = smem + C::OFF_V + vst * C::TILE;
          const int nz = (BKV - vk) * (D / 64) * 8;   // 16-byte chunks
          for (int z = r; z < nz; z += BQ) {
            const int row = vk + z / ((D / 64) * 8);
            const int rem = z % ((D / 64) * 8);
            *reinterpret_cast<uint4*>(vt + (rem >> 3) * C::HALF + row * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();   // the zeros must be visible to the tensor core's V reads
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[x]);
        if (!ok) break;
      }
      vbase += it.k1 - it.k0;
      if (!ok) continue;
      if (ex <= it.k0) {   // no key tile of this query tile in the item
        if (qt >= 0 && it.part >= 0)
          reinterpret_cast<float2*>(a.part_ml)[(size_t)(it.part + x) * BQ + r] = make_float2(-INFINITY, 0.f);
        continue;
      }
      if (!mbar_wait(&o_done[x], odc & 1, wc)) {
        ok = false;
        break;
      }
      ++odc;
      tc_fence_after();
      if (it.part >= 0) {
        // a cut item: unnormalised O and (m, l) of this key range, merged later;
        // partial slot P holds O column-major [D][128] so a warp writes 128 B rows
        const size_t P = (size_t)(it.part + x);
        reinterpret_cast<float2*>(a.part_ml)[P * BQ + r] = make_float2(m, l);
        float* po = a.part_o + P * D * BQ + r;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(to + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) po[(size_t)(c * 32 + i) * BQ] = o[i];
        }
        tc_fence_before();
        mbar_arrive(&o_free[x]);
        continue;
      }
      // epilogue: O / l -> bf16
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      __nv_bfloat16* orow = a.out + (size_t)(it.row0 + qi) * a.out_stride + (size_t)(x ? it.hb : it.ha) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(to + c * 32, o);
        tmem_ld_wait();
        if (qi < it.len) {
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
      mbar_arrive(&o_free[x]);
    }
  }

done:
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// One CTA per (query tile of a cut unit, 8 output columns), one thread per
// query row: the partials of the unit's key ranges, each (O_s, m_s, l_s)
// with O_s = sum exp2(s - m_s) v, combine as
// O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, M = max m_s,
// in split order (deterministic).  Partials are column-major [D][128], so
// each warp load is 128 consecutive bytes; four ranges' loads are issued
// together.
constexpr int kMergeCols = 8;
template <int D>
__global__ void __launch_bounds__(BQ) prefill_merge_kernel(const __grid_constant__ PrefillArgs a) {
  constexpr int NG = D / kMergeCols;
  const int b = blockIdx.x / NG, cg = blockIdx.x % NG, r = threadIdx.x;
  int sl = 0;
  while (sl + 1 < a.n_chunks && a.merge_end[sl] <= b) ++sl;
  const int local = b - (sl ? a.merge_end[sl - 1] : 0);
  const int u = a.cut_from[sl] + (local >> 1), x = local & 1;
  Item it;
  chunk_of(a, sl, it);
  unit_tiles(a.pair, u, (it.len + BQ - 1) / BQ, a.Hq, a.Hkv, a.band[sl], it);
  const int qt = x ? it.qb : it.qa;
  if (qt < 0) return;
  const int qi = qt * BQ + r;
  if (qi >= it.len) return;
  const int S = a.splits[sl];
  const int P0 = a.part_base[sl] + 2 * (u - a.cut_from[sl]) * S + x;   // split s at P0 + 2 s
  const float2* mlp = reinterpret_cast<const float2*>(a.part_ml) + (size_t)P0 * BQ + r;
  float2 ml[kPfMaxSplits];
  float M = -INFINITY;
#pragma unroll
  for (int sp = 0; sp < kPfMaxSplits; ++sp) {
    ml[sp] = sp < S ? mlp[(size_t)2 * sp * BQ] : make_float2(-INFINITY, 0.f);
    if (ml[sp].y > 0.f) M = fmaxf(M, ml[sp].x);
  }
  float L = 0.f, o[kMergeCols];
#pragma unroll
  for (int i = 0; i < kMergeCols; ++i) o[i] = 0.f;
#pragma unroll
  for (int s4 = 0; s4 < kPfMaxSplits; s4 += 4) {
    if (s4 >= S) break;
    float v[4][kMergeCols], w[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int sp = s4 + t;
      // an empty range (l = 0) was never written: weight 0, nothing read
      const bool use = sp < S && ml[sp].y > 0.f;
      w[t] = use ? fast_exp2(ml[sp].x - M) : 0.f;
      const float* po = a.part_o + ((size_t)(P0 + 2 * sp) * D + cg * kMergeCols) * BQ + r;
#pragma unroll
      for (int i = 0; i < kMergeCols; ++i) v[t][i] = use ? po[(size_t)i * BQ] : 0.f;
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      L = fmaf(w[t], ml[s4 + t < kPfMaxSplits ? s4 + t : 0].y, L);
#pragma unroll
      for (int i = 0; i < kMergeCols; ++i) o[i] = fmaf(w[t], v[t][i], o[i]);
    }
  }
  const float inv = L > 0.f ? 1.0f / L : 0.f;
  __nv_bfloat16* orow =
      a.out + (size_t)(it.row0 + qi) * a.out_stride + (size_t)(x ? it.hb : it.ha) * D + cg * kMergeCols;
  *reinterpret_cast<uint4*>(orow) = make_uint4(pack_bf16(o[0] * inv, o[1] * inv), pack_bf16(o[2] * inv, o[3] * inv),
                                               pack_bf16(o[4] * inv, o[5] * inv), pack_bf16(o[6] * inv, o[7] * inv));
}

template <int D>
cudaError_t launch_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const PrefillArgs& a,
                     int ctas, cudaStream_t s) {
  static std::atomic<unsigned long long> attr{0};
  const cudaError_t e = smem_limit_per_device(prefill_kernel<D>, (int)PfCfg<D>::SMEM, attr);
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc waits until the registers it asks for are free in the
  // CTA's launch allocation: refuse to launch a build whose allocation per
  // thread is below what the split assumes (it would wait forever).
  static std::atomic<int> regs{0};
  if (regs.load(std::memory_order_acquire) == 0) {
    cudaFuncAttributes fa{};
    const cudaError_t r = cudaFuncGetAttributes(&fa, prefill_kernel<D>);
    if (r != cudaSuccess) return r;
    regs.store(fa.numRegs, std::memory_order_release);
  }
  if (regs.load(std::memory_order_acquire) < kLaunchRegs) return cudaErrorInvalidConfiguration;
  ctas = prefill_grid(a, ctas);
  if (a.pdl) return launch_pdl(prefill_kernel<D>, dim3(ctas), dim3(kThreads), PfCfg<D>::SMEM, s, q, k, v, a);
  prefill_kernel<D><<<ctas, kThreads, PfCfg<D>::SMEM, s>>>(q, k, v, a);
  return cudaGetLastError();
}

}  // namespace

int prefill_items(const PrefillArgs& a) { return a.n_chunks > 0 ? a.item_end[a.n_chunks - 1] : 0; }

int prefill_merge_blocks(const PrefillArgs& a) { return a.n_chunks > 0 ? a.merge_end[a.n_chunks - 1] : 0; }

namespace {
int kv_tiles_host(int prefix, int len, int qt) {
  const int end = std::min(prefix + qt * BQ + BQ, prefix + len);
  return (end + BKV - 1) / BKV;
}
}  // namespace

void prefill_set_chunks(PrefillArgs& a, int n, const int* len, const int* prefix, const int* row0,
                        const int* page_off, int sms, int split_mode) {
  // slot order: the chunk whose last query tile reaches furthest (most key
  // tiles per item) first, so the queue hands out the longest items first
  int order[kMaxChunks];
  for (int i = 0; i < n; ++i) order[i] = i;
  for (int i = 1; i < n; ++i)   // stable insertion sort, descending c_i + l_i
    for (int j = i; j > 0 && prefix[order[j]] + len[order[j]] > prefix[order[j - 1]] + len[order[j - 1]]; --j) {
      const int t = order[j];
      order[j] = order[j - 1];
      order[j - 1] = t;
    }
  // per unit the key tiles of its later query tile: the work of the launch
  // and the longest and shortest unit of each chunk
  long long total = 0;
  int reach_max[kMaxChunks], reach_min[kMaxChunks], units[kMaxChunks];
  for (int i = 0; i < n; ++i) {
    const int n_qt = (len[i] + BQ - 1) / BQ;
    units[i] = units_of(a.pair, n_qt, a.Hq);
    long long cost = 0;
    if (a.pair == kPfTilePairs) {
      for (int g = 0; g < (n_qt + 1) / 2; ++g) cost += kv_tiles_host(prefix[i], len[i], std::min(2 * g + 1, n_qt - 1));
      cost *= a.Hq;
      reach_min[i] = kv_tiles_host(prefix[i], len[i], std::min(1, n_qt - 1));
    } else {
      for (int qt = 0; qt < n_qt; ++qt) cost += kv_tiles_host(prefix[i], len[i], qt);
      cost *= a.pair == kPfHeadPairs ? a.Hq / 2 : a.Hq;
      reach_min[i] = kv_tiles_host(prefix[i], len[i], 0);
    }
    reach_max[i] = kv_tiles_host(prefix[i], len[i], n_qt - 1);
    total += cost;
  }
  const double avg = (double)total / (sms > 0 ? sms : 1);
  const double target = avg > 8.0 ? avg : 8.0;   // shortest range worth a split of its own
  // Few long units for the grid (fewer than 4 per SM) leave the last wave
  // part-empty: cut them so there are about 4 per SM, at most 4 ranges of at
  // least 16 key tiles each (a 2048-token chunk of 40 query heads: 320
  // tile-pair units on 152 SMs, cut in 2).
  int all_units = 0;
  for (int i = 0; i < n; ++i) all_units += units[i];
  const int quant = all_units > 0 && all_units < 4 * sms ? std::min(4, (4 * sms + all_units - 1) / all_units) : 1;
  a.n_chunks = n;
  int split[kMaxChunks], cut[kMaxChunks];
  bool any_cut = false;
  for (int s = 0; s < n; ++s) {
    const int i = order[s];
    int S = 1;
    if (split_mode >= 2)
      S = split_mode;
    else if (split_mode == 0) {
      if (reach_max[i] > 1.25 * target) S = (int)std::ceil(reach_max[i] / target);
      S = std::max(S, std::min(quant, reach_min[i] / 16));
    }
    S = std::min(S, std::min(reach_min[i], kPfMaxSplits));   // every split has a key tile
    split[s] = S < 2 ? 1 : S;
    cut[s] = 0;
    any_cut = any_cut || split[s] > 1;
  }
  // The tail of a long queue of whole units: when the queue runs dry, SMs
  // stop up to one unit's time apart (a unit of a Qwen3-32B-shaped chunk on
  // a 28K prefix runs ~400 us).  So when nothing else is cut and the units
  // make several waves, the last wave's worth of units (sms, counted from
  // the end of the queue) is cut into kTailSplits key ranges of at least
  // kTailMinTiles key tiles: the SMs that reach the tail first take more of
  // its short items, and the last ones finish close together.
  if (split_mode == 0 && !any_cut && all_units > 2 * sms) {
    int tail = sms;
    for (int s = n - 1; s >= 0 && tail > 0; --s) {
      const int i = order[s];
      const int S = std::min(kTailSplits, reach_min[i] / kTailMinTiles);
      if (S < 2) break;
      const int take = std::min(units[i], tail);
      split[s] = S;
      cut[s] = units[i] - take;
      tail -= take;
    }
  }
  int items = 0, parts = 0, merges = 0;
  for (int s = 0; s < n; ++s) {
    const int i = order[s];
    int S = split[s];
    const int n_cut = units[i] - cut[s];
    if (S > 1 && parts + 2 * n_cut * S > kPfPartTiles) S = (kPfPartTiles - parts) / (2 * n_cut);
    if (S < 2) S = 1;
    a.splits[s] = S;
    a.cut_from[s] = S > 1 ? cut[s] : units[i];
    a.part_base[s] = S > 1 ? parts : -1;
    if (S > 1) {
      parts += 2 * n_cut * S;
      merges += 2 * n_cut;
    }
    items += S > 1 ? cut[s] + n_cut * S : units[i];
    a.item_end[s] = items;
    a.merge_end[s] = merges;
    // query tiles per band of the unit order: tiles whose key counts differ
    // by at most about a quarter (all 16 on a long prefix, 1 without one)
    a.band[s] = std::max(1, std::min(kBandQ, (prefix[i] / BQ + 1) / 4));
    a.row0[s] = row0[i];
    a.len[s] = len[i];
    a.prefix[s] = prefix[i];
    a.page_off[s] = page_off[i];
  }
}

int prefill_grid(const PrefillArgs& a, int ctas) {
  const int n_items = prefill_items(a);
  if (ctas > n_items) ctas = n_items;
  return ctas < 1 ? 1 : ctas;
}

cudaError_t launch_prefill(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const PrefillArgs& a, int num_ctas, cudaStream_t s) {
  if (a.n_chunks <= 0 || prefill_items(a) <= 0) return cudaSuccess;
  if (a.head_dim == 128) return launch_t<128>(tmQ, tmK, tmV, a, num_ctas, s);
  if (a.head_dim == 64) return launch_t<64>(tmQ, tmK, tmV, a, num_ctas, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_merge(const PrefillArgs& a, cudaStream_t s) {
  const int blocks = prefill_merge_blocks(a);
  if (blocks <= 0) return cudaSuccess;
  if (a.head_dim == 128)
    prefill_merge_kernel<128><<<blocks * (128 / kMergeCols), BQ, 0, s>>>(a);
  else if (a.head_dim == 64)
    prefill_merge_kernel<64><<<blocks * (64 / kMergeCols), BQ, 0, s>>>(a);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace cf
