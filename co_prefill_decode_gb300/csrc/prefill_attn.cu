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
// A work item is (128-row query tile, query head).  Persistent CTAs, one per
// SM of the prefill partition, 6 warps:
//   warp 0   TMA producer: the Q tile once, then per 128-key tile eight
//            (page, KV head) boxes of 16 x 64 for K and for V (each page is a
//            contiguous 4 KB tile of the pool) into a 2-stage ring;
//   warp 1   one thread issues tcgen05.mma: S = Q K^T into one of two TMEM
//            buffers, O += P V into a TMEM accumulator;
//   warps 2-5 one query row per thread: load S from TMEM, online softmax in
//            the log2 domain with lazy rescaling (O is rescaled in TMEM only
//            when the running max grows by more than 2^8), write P as bf16
//            into a 128-byte-swizzled K-major tile, and at the end normalise
//            O and store it.
// S_{j+1} is computed while the softmax works on S_j, and PV_j runs while
// the softmax works on S_{j+1}.
#include "common.cuh"
#include "internal.h"

namespace cf {

namespace {

constexpr int kThreads = 192;
constexpr int BQ = 128;     // query rows per tile
constexpr int BKV = 128;    // keys per tile (8 pages of 16)
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D>
struct PfCfg {
  static constexpr uint32_t HALF = BQ * 64 * 2;          // 16 KB: 128 rows x 64 bf16
  static constexpr uint32_t Q_BYTES = HALF * (D / 64);
  static constexpr uint32_t KV_BYTES = HALF * (D / 64);  // one K (or V) tile
  static constexpr uint32_t P_BYTES = 2 * HALF;          // 128 rows x 128 keys
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + 2 * KV_BYTES;
  static constexpr uint32_t OFF_P = OFF_V + 2 * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_P + P_BYTES;
  static constexpr size_t SMEM = 1024 + OFF_BAR + 256 + 8192;   // spare tail
  static constexpr uint32_t TMEM_COLS = 512;   // S0 [0,128), S1 [128,256), O [256, 256+D)
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
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, PrefillArgs a) {
  using C = PfCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem;
  {
    const uint32_t s0 = smem_u32(smem_raw);
    smem = smem_raw + (((s0 + 1023u) & ~1023u) - s0);
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;    // [2]
  uint64_t* k_empty = bars + 4;   // [2]
  uint64_t* v_full = bars + 6;    // [2]
  uint64_t* v_empty = bars + 8;   // [2]
  uint64_t* s_full = bars + 10;   // [2]
  uint64_t* s_free = bars + 12;   // [2]
  uint64_t* p_full = bars + 14;
  uint64_t* pv_done = bars + 15;
  uint64_t* o_free = bars + 16;
  uint64_t* drain = bars + 17;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 18);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(o_free, 128);
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

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------------------ producer
      int qc = 0, kc = 0;   // Q tiles and K/V tiles issued
      bool ok = true;
      uint32_t last_q = 0xffffffffu, last_k[2] = {0xffffffffu, 0xffffffffu}, last_v[2] = {0xffffffffu, 0xffffffffu};
      for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x) {
        const Item it = item_of(idx, a.Hq, n_qt);
        const int kvh = it.head / G;
        if (!mbar_wait(q_empty, (qc & 1) ^ 1, wc)) { ok = false; break; }
        mbar_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
        for (int hd = 0; hd < D / 64; ++hd)
          tma_load_3d(smem + C::OFF_Q + hd * C::HALF, &tmQ, q_full, hd * 64, it.head, it.qt * BQ);
        last_q = qc & 1;
        ++qc;
        const int nkv = kv_tiles(a, it.qt);
        for (int j = 0; j < nkv; ++j, ++kc) {
          const int st = kc & 1;
          const uint32_t ph = (kc >> 1) & 1;
          int rows[8];
#pragma unroll
          for (int pg = 0; pg < 8; ++pg) {
            const int pi = j * 8 + pg;
            int r = oob_row;
            if (pi < n_pages_req) {
              const int pid = a.pages[pi];
              if (pid >= 0 && pid < a.num_pages)
                r = (pid * a.Hkv + kvh) * a.page_size;
              else
                set_error(a.err, CF_DEVERR_PAGE);
            }
            rows[pg] = r;
          }
          if (!mbar_wait(&k_empty[st], ph ^ 1, wc)) { ok = false; break; }
          mbar_expect_tx(&k_full[st], C::KV_BYTES);
          uint8_t* kt = smem + C::OFF_K + st * C::KV_BYTES;
#pragma unroll
          for (int pg = 0; pg < 8; ++pg)
#pragma unroll
            for (int hd = 0; hd < D / 64; ++hd)
              tma_load_2d(kt + hd * C::HALF + pg * 2048, &tmK, &k_full[st], hd * 64, rows[pg]);
          last_k[st] = ph;
          if (!mbar_wait(&v_empty[st], ph ^ 1, wc)) { ok = false; break; }
          mbar_expect_tx(&v_full[st], C::KV_BYTES);
          uint8_t* vt = smem + C::OFF_V + st * C::KV_BYTES;
#pragma unroll
          for (int pg = 0; pg < 8; ++pg)
#pragma unroll
            for (int hd = 0; hd < D / 64; ++hd)
              tma_load_2d(vt + hd * C::HALF + pg * 2048, &tmV, &v_full[st], hd * 64, rows[pg]);
          last_v[st] = ph;
        }
      }
      if (!ok) {  // let our own copies land before the CTA exits
        volatile int dummy = 0;
        const WaitCtl w2{&dummy, nullptr, a.wait_ns};
        if (last_q != 0xffffffffu) mbar_wait(q_full, last_q, w2);
        for (int s = 0; s < 2; ++s) {
          if (last_k[s] != 0xffffffffu) mbar_wait(&k_full[s], last_k[s], w2);
          if (last_v[s] != 0xffffffffu) mbar_wait(&v_full[s], last_v[s], w2);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------------ MMA issuer
      constexpr uint32_t IDESC_S = idesc_bf16(128, BKV, false);
      constexpr uint32_t IDESC_PV = idesc_bf16(128, D, true);
      const uint32_t q_s = smem_u32(smem + C::OFF_Q);
      const uint32_t p_s = smem_u32(smem + C::OFF_P);
      int qc = 0, kc = 0, sc = 0, pc = 0, oc = 0;
      bool ok = true, issued = false;
      for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x) {
        const Item it = item_of(idx, a.Hq, n_qt);
        const int nkv = kv_tiles(a, it.qt);
        if (!mbar_wait(q_full, qc & 1, wc)) { ok = false; break; }
        ++qc;
        int vc = kc;   // V tile counter trails the K tile counter
        for (int j = 0; j <= nkv && ok; ++j) {
          if (j < nkv) {  // S_j = Q K_j^T
            const int sb = sc & 1;
            const int st = kc & 1;
            if (!mbar_wait(&s_free[sb], ((sc >> 1) & 1) ^ 1, wc)) { ok = false; break; }
            if (!mbar_wait(&k_full[st], (kc >> 1) & 1, wc)) { ok = false; break; }
            tc_fence_after();
            const uint32_t k_s = smem_u32(smem + C::OFF_K + st * C::KV_BYTES);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * C::HALF + (kk & 3) * 32;
              umma_bf16(tmem + sb * BKV, sdesc_sw128(q_s + off, 16, 1024), sdesc_sw128(k_s + off, 16, 1024),
                        IDESC_S, kk > 0);
            }
            issued = true;
            umma_commit(&k_empty[st]);
            umma_commit(&s_full[sb]);
            if (j == nkv - 1) umma_commit(q_empty);
            ++sc;
            ++kc;
          }
          if (j >= 1) {  // O += P_{j-1} V_{j-1}
            const int st = vc & 1;
            if (!mbar_wait(p_full, pc & 1, wc)) { ok = false; break; }
            if (!mbar_wait(&v_full[st], (vc >> 1) & 1, wc)) { ok = false; break; }
            if (j == 1 && !mbar_wait(o_free, (oc & 1) ^ 1, wc)) { ok = false; break; }
            tc_fence_after();
            const uint32_t v_s = smem_u32(smem + C::OFF_V + st * C::KV_BYTES);
#pragma unroll
            for (int kk = 0; kk < BKV / 16; ++kk) {
              const uint32_t poff = (kk >> 2) * C::HALF + (kk & 3) * 32;
              umma_bf16(tmem + 256, sdesc_sw128(p_s + poff, 16, 1024),
                        sdesc_sw128(v_s + kk * 2048, C::HALF, 1024), IDESC_PV, (j > 1 || kk > 0));
            }
            umma_commit(&v_empty[st]);
            umma_commit(pv_done);
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
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint8_t* p_tile = smem + C::OFF_P;
    int sc = 0, pc = 0, vc = 0;
    bool ok = true;
    for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x) {
      const Item it = item_of(idx, a.Hq, n_qt);
      const int nkv = kv_tiles(a, it.qt);
      const int qi = it.qt * BQ + r;
      const int qpos = a.prefix + qi;
      const int kend = a.prefix + a.l;   // first key that does not exist
      const int diag = a.prefix + it.qt * BQ;   // smallest query position of the tile
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nkv; ++j) {
        const int sb = sc & 1;
        if (!mbar_wait(&s_full[sb], (sc >> 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        float s[BKV];
#pragma unroll
        for (int c = 0; c < BKV / 32; ++c) tmem_ld32(tmem + lane_off + sb * BKV + c * 32, s + c * 32);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&s_free[sb]);
        ++sc;
        const int kv0 = j * BKV;
        if (kv0 + BKV - 1 > diag) {   // tile crosses the diagonal or the end of the request
#pragma unroll
          for (int c = 0; c < BKV; ++c) {
            const int kp = kv0 + c;
            if (!(kp <= qpos && kp < kend)) s[c] = -INFINITY;
          }
        }
        // row max with 8 independent partial maxima (short dependency chains)
        float mp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mp[i] = s[i];
#pragma unroll
        for (int c = 8; c < BKV; ++c) mp[c & 7] = fmaxf(mp[c & 7], s[c]);
        const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                               fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7]))) * a.scale_log2;
        // wait until PV_{j-1} is done: O may be rescaled and P rewritten
        if (j > 0) {
          if (!mbar_wait(pv_done, (pc & 1), wc)) { ok = false; break; }
          ++pc;
          tc_fence_after();
        }
        const bool grow = (m == -INFINITY) ? false : (mx > m + kRescaleThreshold);
        if (m == -INFINITY) m = mx;
        if (__any_sync(0xffffffffu, grow)) {
          const float alpha = grow ? fast_exp2(m - mx) : 1.0f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(tmem + lane_off + 256 + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(tmem + lane_off + 256 + c * 32, o);
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
#pragma unroll
        for (int c8 = 0; c8 < BKV / 8; ++c8) {
          float p[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            p[i] = fast_exp2(fmaf(s[c8 * 8 + i], sc2, -mu));
            lp[i] += p[i];
          }
          uint4 w;
          w.x = pack_bf16(p[0], p[1]);
          w.y = pack_bf16(p[2], p[3]);
          w.z = pack_bf16(p[4], p[5]);
          w.w = pack_bf16(p[6], p[7]);
          const int half = c8 >> 3, ch = c8 & 7;
          *reinterpret_cast<uint4*>(p_tile + half * C::HALF + r * 128 + ((ch ^ (r & 7)) << 4)) = w;
        }
        const float ls = ((lp[0] + lp[1]) + (lp[2] + lp[3])) + ((lp[4] + lp[5]) + (lp[6] + lp[7]));
        l += ls;
        // keys past the end of the request: zero their V rows (slots may hold anything)
        const int vst = vc & 1;
        if (kend - kv0 < BKV) {
          if (!mbar_wait(&v_full[vst], (vc >> 1) & 1, wc)) { ok = false; break; }
          const int vk = max(0, kend - kv0);
          uint8_t* vt = smem + C::OFF_V + vst * C::KV_BYTES;
          const int nz = (BKV - vk) * (D / 64) * 8;   // 16-byte chunks
          for (int z = r; z < nz; z += 128) {
            const int row = vk + z / ((D / 64) * 8);
            const int rem = z % ((D / 64) * 8);
            *reinterpret_cast<uint4*>(vt + (rem >> 3) * C::HALF + row * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
        }
        ++vc;
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(p_full);
      }
      if (!ok) break;
      // epilogue: O / l -> bf16
      if (!mbar_wait(pv_done, (pc & 1), wc)) { ok = false; break; }
      ++pc;
      tc_fence_after();
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      __nv_bfloat16* orow = a.out + (size_t)qi * a.out_stride + (size_t)it.head * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(tmem + lane_off + 256 + c * 32, o);
        tmem_ld_wait();
        if (qi < a.l) {
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
  const int n_items = ((a.l + BQ - 1) / BQ) * a.Hq;
  if (ctas > n_items) ctas = n_items;
  if (ctas < 1) ctas = 1;
  prefill_kernel<D><<<ctas, kThreads, PfCfg<D>::SMEM, s>>>(q, k, v, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const PrefillArgs& a, int num_ctas, cudaStream_t s) {
  if (a.l <= 0) return cudaSuccess;
  if (a.head_dim == 128) return launch_t<128>(tmQ, tmK, tmV, a, num_ctas, s);
  if (a.head_dim == 64) return launch_t<64>(tmQ, tmK, tmV, a, num_ctas, s);
  return cudaErrorInvalidValue;
}

}  // namespace cf
