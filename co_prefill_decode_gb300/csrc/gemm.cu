// Dense GEMMs of the co-batched layer on the 5th-generation tensor cores.
//
// One persistent, warp-specialised kernel: warp 0 streams 128x64 A tiles and
// BNx64 B tiles with TMA (128-byte swizzle) through an mbarrier ring; one
// thread of warp 1 issues tcgen05.mma (M=128, N=BN, K=16, bf16 -> fp32 in
// TMEM) and commits each stage back to the producer; warps 2-5 read the
// accumulator from TMEM (double buffered, so the epilogue of tile i overlaps
// the MMAs of tile i+1) and apply the fused epilogue, storing whole row
// segments through a per-warp shared-memory transpose.  The stacked
// [prefill; decode] token matrix is the A operand, so every weight tile is
// fetched once for both phases (ConfluxServe §4 "Cross-SP co-batch", App. B
// Table 7: weight traffic amortised over all co-batched tokens).
//
// Work is dealt by a fixed schedule (gemm_schedule): every CTA takes whole
// tiles, one per wave, for all full waves.  When the tiles of the last wave
// would leave many SMs idle, each of them is cut into S equal k-chunks and
// the chunks are dealt chunk-major, one per CTA, so CTAs running at the same
// time read the same k range of the shared weight tiles.  A cut tile is
// finished by the CTA running its last chunk: the others store their fp32
// partial accumulators to a workspace; since the chunk is that CTA's final
// unit its TMA ring is idle by then, so it pulls the partials into the ring
// with bulk copies, adds them in k order followed by its own (a fixed order,
// so results are deterministic), puts the sum back into TMEM and applies the
// epilogue as for a whole tile.
#include <stdio.h>

#include "common.cuh"
#include "internal.h"

namespace cf {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 192;

template <int BN, int EPI>
struct GemmCfg {
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = BN * BK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 256 ? 4 : 6;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  // per epilogue warp: one 32 x 32 fp32 block being transposed (the SwiGLU
  // epilogue stores directly and needs none)
  static constexpr uint32_t XPOSE_BYTES = EPI == EPI_SWIGLU ? 0 : 4 * 32 * 32 * 4;
  static constexpr size_t SMEM = 1024 + STAGES * STAGE_BYTES + XPOSE_BYTES + 256;
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

CF_DEV uint8_t* align1024(uint8_t* p) {
  uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

// SiLU with the fast reciprocal-based division: its ~2-ulp error is far
// below the bf16 rounding of the product it feeds
CF_DEV float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// One unit of work: k-blocks [kb0, kb1) of tile `tile` (m-fastest numbering).
struct Unit {
  int tile, kb0, kb1;
};

// The units of CTA `c` in order: whole tiles c, c + G, ... below dp_tiles,
// then (if c < (tiles - dp_tiles) * split) chunk c / R of tail tile
// dp_tiles + c % R, R = tiles - dp_tiles; chunk s covers k-blocks
// [s * num_kb / split, (s + 1) * num_kb / split).
struct UnitIter {
  int c, G, num_kb, dp_tiles, tail, split;
  int j;
  bool tail_done;
  CF_DEV UnitIter(int c_, int G_, int num_kb_, int tiles, int dp_tiles_, int split_)
      : c(c_), G(G_), num_kb(num_kb_), dp_tiles(dp_tiles_), tail(tiles - dp_tiles_), split(split_), j(0),
        tail_done(false) {}
  CF_DEV bool next(Unit& u) {
    const int tile = c + j * G;
    if (tile < dp_tiles) {
      u = Unit{tile, 0, num_kb};
      ++j;
      return true;
    }
    if (tail_done || c >= tail * split) return false;
    tail_done = true;
    const int s = c / tail;
    u = Unit{dp_tiles + c % tail, s * num_kb / split, (s + 1) * num_kb / split};
    return true;
  }
};

CF_DEV void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// barrier of the 128 epilogue threads that also ANDs a flag over them, so a
// wait that ran out in one warp makes all four leave together (the fix-up's
// barriers then never wait for a warp that has left)
CF_DEV bool epi_bar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, 1, 128, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Split-K fix-up of a tail unit (a k-chunk of a cut tile).  Returns 1 when
// this CTA holds the tile's full sum in TMEM and must run the epilogue, 0
// when it handed its partial over, -1 when the wait for the other chunks
// gave up (error word set).  `ring` is the CTA's TMA stage memory, idle once
// the last unit's accumulator is full.
template <int BN>
CF_DEV int sk_fixup(uint32_t taddr, int r_in_tile, int ep_tid, const Unit& u, const GemmArgs& p, uint8_t* ring,
                    uint32_t ring_bytes, uint64_t* fix_bar, volatile int* sh_flag, const WaitCtl& wc) {
  const int tail = p.tiles - p.dp_tiles;
  const int it = u.tile - p.dp_tiles;   // tail tile index; its chunk s is run by CTA s * tail + it
  const int S = p.split;
  const int s_me = blockIdx.x / tail;
  int* flag = p.sk_flags + it;          // partials stored so far
  // Partial layout: float4 j (columns 4j..4j+3) of tile row r at
  // slot + j * BM + r, so the rows of a warp fill 512 contiguous bytes per
  // access, and the 32 columns c..c+31 form one contiguous 16 KB piece.
  constexpr uint32_t kPiece = BM * 32 * 4;
  constexpr size_t kSlot4 = (size_t)BM * BN / 4;
  float4* ws4 = reinterpret_cast<float4*>(p.sk_ws);
  float v[32];
  if (s_me < S - 1) {  // store the partial, then count it
    float4* dst = ws4 + (size_t)blockIdx.x * kSlot4 + r_in_tile;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      tmem_ld32(taddr + c, v);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 8; ++i)
        __stcg(dst + (size_t)(c / 4 + i) * BM, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
    }
    __threadfence();
    epi_bar();
    if (ep_tid == 0) atomicAdd(flag, 1);
    return 0;
  }
  // the last chunk: wait until the other S - 1 partials are stored
  if (ep_tid == 0) {
    const uint64_t t_start = globaltimer();
    int ok = 1;
    while (*reinterpret_cast<volatile int*>(flag) < S - 1) {
      if (*wc.abort) {
        ok = 0;
        break;
      }
      if (globaltimer() - t_start > wc.limit_ns) {
        *wc.abort = 1;
        set_error(wc.err, CF_DEVERR_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    *sh_flag = ok;
    __threadfence();
    fence_proxy_async_global();
  }
  epi_bar();
  if (!*sh_flag) return -1;
  // rounds of whole 32-column chunks: all S - 1 pieces of a chunk per round
  const int per_round = (int)(ring_bytes / kPiece) / (S - 1);
  const float4* ring4 = reinterpret_cast<const float4*>(ring);
  int round = 0;
  bool ok = true;
#pragma unroll 1
  for (int c0 = 0; c0 < BN / 32 && ok; c0 += per_round, ++round) {
    const int nc = BN / 32 - c0 < per_round ? BN / 32 - c0 : per_round;
    if (ep_tid == 0) {
      mbar_expect_tx(fix_bar, (uint32_t)(nc * (S - 1)) * kPiece);
      for (int c = 0; c < nc; ++c)
        for (int j = 0; j < S - 1; ++j)
          bulk_load(ring + (size_t)(c * (S - 1) + j) * kPiece,
                    ws4 + (size_t)(j * tail + it) * kSlot4 + (size_t)(c0 + c) * (kPiece / 16), kPiece, fix_bar);
    }
    ok = mbar_wait(fix_bar, round & 1, wc);
    if (!ok) {   // the bulk copies may still be landing in the ring: wait for them before leaving
      volatile int dummy = 0;
      const WaitCtl w2{&dummy, nullptr, p.wait_ns};
      mbar_wait(fix_bar, round & 1, w2);
    }
    if (ok) {
#pragma unroll 1
      for (int c = 0; c < nc; ++c) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
        for (int j = 0; j < S - 1; ++j) {   // chunks in k order ...
          const float4* src = ring4 + (size_t)(c * (S - 1) + j) * (kPiece / 16) + r_in_tile;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 q = src[i * BM];
            v[4 * i] += q.x;
            v[4 * i + 1] += q.y;
            v[4 * i + 2] += q.z;
            v[4 * i + 3] += q.w;
          }
        }
        float own[32];   // ... then this CTA's own, the last in k
        tmem_ld32(taddr + (c0 + c) * 32, own);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += own[i];
        tmem_st32(taddr + (c0 + c) * 32, v);
      }
    }
    ok = epi_bar_and(ok);   // the ring is read before the next round overwrites it
  }
  tmem_st_wait();
  if (ep_tid == 0) *flag = 0;   // free for the next launch
  return ok ? 1 : -1;
}

CF_DEV void store_bf16x32(__nv_bfloat16* dst, const float* v) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 w;
    w.x = pack_bf16(v[8 * i + 0], v[8 * i + 1]);
    w.y = pack_bf16(v[8 * i + 2], v[8 * i + 3]);
    w.z = pack_bf16(v[8 * i + 4], v[8 * i + 5]);
    w.w = pack_bf16(v[8 * i + 6], v[8 * i + 7]);
    d[i] = w;
  }
}

// The epilogue reads TMEM one row per thread, so a warp holds a 32-row x
// 32-column block with each row in one thread.  Stored as it is, every
// 16-byte store of the warp would touch 32 rows; the block is therefore
// turned around in shared memory so that each store instruction writes whole
// 64- or 128-byte row segments.  16-byte chunks are placed XOR-swizzled by
// the row, which keeps both directions free of bank conflicts.
//
// fp32 block (32 words per row): lane l puts row l; afterwards lane l takes
// row 4i + l/8, columns 4(l%8)..+3, for i = 0..7.
CF_DEV void xpose_f32_put(float4* sb, const float* v, int lane) {
#pragma unroll
  for (int k = 0; k < 8; ++k)
    sb[lane * 8 + (k ^ (lane & 7))] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
}
CF_DEV float4 xpose_f32_get(const float4* sb, int i, int lane) {
  const int row = 4 * i + (lane >> 3), k = lane & 7;
  return sb[row * 8 + (k ^ (row & 7))];
}
// bf16 block (16 words per row): lane l puts row l; afterwards lane l takes
// row 8i + l/4, columns 8(l%4)..+7, for i = 0..3.
CF_DEV void xpose_b16_put(uint4* sb, const uint32_t* w, int lane) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    sb[lane * 4 + (k ^ ((lane >> 1) & 3))] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
}
CF_DEV uint4 xpose_b16_get(const uint4* sb, int i, int lane) {
  const int row = 8 * i + (lane >> 2), k = lane & 3;
  return sb[row * 4 + (k ^ ((row >> 1) & 3))];
}
// 32 fp32 values as 16 words of bf16 pairs (low half = even column)
CF_DEV void pack32(const float* v, uint32_t* w) {
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
}
// stores the warp's bf16 block: row r of the block goes to dst0 + r * ld
CF_DEV void store_block_b16(const uint4* sb, __nv_bfloat16* dst0, size_t ld, int rows_left, int lane) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = 8 * i + (lane >> 2);
    const uint4 q = xpose_b16_get(sb, i, lane);
    if (row < rows_left) *reinterpret_cast<uint4*>(dst0 + (size_t)row * ld + 8 * (lane & 3)) = q;
  }
}

// Stores a warp's 32 rows x 32 columns as bf16 through the transpose: the
// row held by lane r goes to lane r's `dst` (nothing where it is null).
CF_DEV void store_rows_b16(uint4* sb, __nv_bfloat16* dst, const float* v, int lane) {
  uint32_t pk[16];
  pack32(v, pk);
  __syncwarp();
  xpose_b16_put(sb, pk, lane);
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = 8 * i + (lane >> 2);
    __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(dst), row));
    const uint4 q = xpose_b16_get(sb, i, lane);
    if (d) *reinterpret_cast<uint4*>(d + 8 * (lane & 3)) = q;
  }
}

// QKV epilogue for one head of one row: columns [hcol, hcol + D) of this
// thread's TMEM lane hold q, k or v of head `head` for stacked row `row`.
template <int D>
CF_DEV void qkv_head(uint32_t taddr, int row, bool valid, int head, const QkvEpilogue& e, uint4* sb, int lane) {
  const int Hq = e.Hq, Hkv = e.Hkv;
  const int kind = head < Hq ? 0 : (head < Hq + Hkv ? 1 : 2);
  __nv_bfloat16* dst = nullptr;
  if (valid) {
    if (kind == 0) {
      dst = e.q_out + ((size_t)row * Hq + head) * D;
    } else {
      const int s = e.slot[row];
      if (s >= 0) {
        const int page = s / e.page_size, off = s % e.page_size;
        const int kvh = kind == 1 ? head - Hq : head - Hq - Hkv;
        __nv_bfloat16* pool = kind == 1 ? e.k_pool : e.v_pool;
        dst = pool + (((size_t)page * Hkv + kvh) * e.page_size + off) * D;
      }
    }
  }
  float v[32], w[32];
  if (kind == 2) {  // V: plain copy to the pool
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      tmem_ld32(taddr + c * 32, v);
      tmem_ld_wait();
      store_rows_b16(sb, dst ? dst + c * 32 : nullptr, v, lane);
    }
    return;
  }
  float nrm = 1.0f;
  const __nv_bfloat16* g = kind == 0 ? e.g_q : e.g_k;
  if (e.qk_norm) {  // per-head RMSNorm over d (before RoPE)
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      tmem_ld32(taddr + c * 32, v);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) ss = fmaf(v[i], v[i], ss);
    }
    nrm = rsqrtf(ss / D + e.eps);
  }
  // pair-major table: for pair i the warp's 32 rows are 256 contiguous bytes
  const float2* cs = e.rope_cs + (valid ? row : 0);
  // rotate-half: element i pairs with i + D/2
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    tmem_ld32(taddr + c * 32, v);
    tmem_ld32(taddr + D / 2 + c * 32, w);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int i0 = c * 32 + i;
      float x1 = v[i] * nrm, x2 = w[i] * nrm;
      if (e.qk_norm) {
        x1 *= bf16f(g[i0]);
        x2 *= bf16f(g[i0 + D / 2]);
      }
      const float2 r = cs[(size_t)i0 * e.cs_ld];
      v[i] = x1 * r.x - x2 * r.y;
      w[i] = x1 * r.y + x2 * r.x;
    }
    store_rows_b16(sb, dst ? dst + c * 32 : nullptr, v, lane);
    store_rows_b16(sb, dst ? dst + D / 2 + c * 32 : nullptr, w, lane);
  }
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                const __grid_constant__ CUtensorMap tmB1, GemmArgs p) {
  using C = GemmCfg<BN, EPI>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* xpose = smem + STAGES * C::STAGE_BYTES;   // 4 KB per epilogue warp
  uint64_t* full = reinterpret_cast<uint64_t*>(xpose + C::XPOSE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* fix_bar = drain + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(fix_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* sh_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(drain, 1);
    mbar_init(fix_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    prefetch_tmap(&tmB1);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch();
  const uint32_t tmem_base = *tmem_holder;
  const WaitCtl wc{abort_flag, p.err, p.wait_ns};

  const int num_m = (p.M + BM - 1) / BM;
  const int num_kb = p.K / BK;

  if (warp == 0) {
    if (lane == 0) {  // ---------------- TMA producer
      uint32_t stage = 0, phase = 0;
      int issued_any = 0;
      uint32_t last_phase[8];
      for (int s = 0; s < 8; ++s) last_phase[s] = 0xffffffffu;
      bool ok = true;
      UnitIter ui(blockIdx.x, gridDim.x, num_kb, p.tiles, p.dp_tiles, p.split);
      Unit u;
      // Weight tiles of the first stages do not depend on the previous
      // kernel: load them before waiting for it (the ring starts empty).
      int pre = 0;
      {
        UnitIter first = ui;
        Unit u0;
        if (p.b_static && first.next(u0)) {
          const int n0 = u0.tile / num_m;
          const int brow0 = EPI == EPI_SWIGLU ? n0 * (BN / 2) : n0 * BN;
          const int brow1 = EPI == EPI_SWIGLU ? brow0 : brow0 + BN / 2;
          pre = u0.kb1 - u0.kb0 < STAGES ? u0.kb1 - u0.kb0 : STAGES;
          for (int i = 0; i < pre; ++i) {
            uint8_t* sb = smem + i * C::STAGE_BYTES + C::A_BYTES;
            mbar_expect_tx(&full[i], C::STAGE_BYTES);
            tma_load_2d(sb, &tmB0, &full[i], (u0.kb0 + i) * BK, brow0);
            tma_load_2d(sb + C::B_BYTES / 2, &tmB1, &full[i], (u0.kb0 + i) * BK, brow1);
          }
        }
      }
      griddep_wait();
      int n_issue = 0;
      while (ok && ui.next(u)) {
        const int mt = u.tile % num_m, nt = u.tile / num_m;
        const int brow0 = EPI == EPI_SWIGLU ? nt * (BN / 2) : nt * BN;
        const int brow1 = EPI == EPI_SWIGLU ? brow0 : brow0 + BN / 2;
        for (int kb = u.kb0; kb < u.kb1; ++kb, ++n_issue) {
          uint8_t* sa = smem + stage * C::STAGE_BYTES;
          uint8_t* sb = sa + C::A_BYTES;
          if (n_issue < pre) {   // B already in flight: add A to the same stage
            tma_load_2d(sa, &tmA, &full[stage], kb * BK, mt * BM);
          } else {
            if (!mbar_wait(&empty[stage], phase ^ 1, wc)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&full[stage], C::STAGE_BYTES);
            tma_load_2d(sa, &tmA, &full[stage], kb * BK, mt * BM);
            tma_load_2d(sb, &tmB0, &full[stage], kb * BK, brow0);
            tma_load_2d(sb + C::B_BYTES / 2, &tmB1, &full[stage], kb * BK, brow1);
          }
          last_phase[stage] = phase;
          issued_any = 1;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Let our own copies land before the CTA exits.  Normally the MMAs
      // have consumed them and these phases are long complete; after an
      // expired wait anywhere in the CTA they may still be in flight.
      if (issued_any) {
        volatile int dummy = 0;
        const WaitCtl w2{&dummy, nullptr, p.wait_ns};
        for (int s = 0; s < STAGES; ++s)
          if (last_phase[s] != 0xffffffffu) mbar_wait(&full[s], last_phase[s], w2);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------- MMA issuer
      constexpr uint32_t IDESC = idesc_bf16(BM, BN, false);
      uint32_t stage = 0, phase = 0;
      int it = 0;
      bool ok = true, issued = false;
      UnitIter ui(blockIdx.x, gridDim.x, num_kb, p.tiles, p.dp_tiles, p.split);
      Unit u;
      // self-test: nothing arrives on `drain` before an MMA is issued, so this
      // wait runs out, raises the abort flag and the timeout bit, and every
      // role then winds down as after any expired wait
      if (p.stall_test && !mbar_wait(drain, 0, wc)) ok = false;
      for (; ok && ui.next(u); ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, wc)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b0 = a0 + C::A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = sdesc_sw128(a0 + k * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b0 + k * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, IDESC, (kb != u.kb0) | (k != 0));
          }
          issued = true;
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) umma_commit(&tfull[acc]);
      }
      if (!ok && issued) {  // wait for our MMAs before TMEM is released
        volatile int dummy = 0;
        const WaitCtl w2{&dummy, nullptr, p.wait_ns};
        umma_commit(drain);
        mbar_wait(drain, 0, w2);
      }
    }
  } else {  // ---------------- epilogue warps 2..5
    const int quarter = warp & 3;
    const int r_in_tile = quarter * 32 + lane;
    const int ep_tid = threadIdx.x - 64;
    float4* xf32 = reinterpret_cast<float4*>(xpose + quarter * 4096);
    uint4* xb16 = reinterpret_cast<uint4*>(xpose + quarter * 4096);
    griddep_wait();   // the epilogue reads the residual / RoPE table and writes
    int it = 0;
    UnitIter ui(blockIdx.x, gridDim.x, num_kb, p.tiles, p.dp_tiles, p.split);
    Unit u;
    for (; ui.next(u); ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!epi_bar_and(mbar_wait(&tfull[acc], acc_phase, wc))) break;
      tc_fence_after();
      const int mt = u.tile % num_m, nt = u.tile / num_m;
      const int row = mt * BM + r_in_tile;
      const bool valid = row < p.M;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if (u.kb0 != 0 || u.kb1 != num_kb) {
        const int own = sk_fixup<BN>(taddr, r_in_tile, ep_tid, u, p, smem, STAGES * C::STAGE_BYTES, fix_bar,
                                     sh_flag, wc);
        if (own <= 0) {
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
          if (own < 0) break;
          continue;
        }
      }
      float v[32], w[32];
      uint32_t pk[16];
      // this warp's 32 rows of the tile start at tile row quarter * 32
      const int wrow0 = mt * BM + quarter * 32;
      const int rows_left = p.M - wrow0;
      if constexpr (EPI == EPI_BF16) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)wrow0 * p.ldo + nt * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          tmem_ld32(taddr + c, v);
          tmem_ld_wait();
          pack32(v, pk);
          __syncwarp();
          xpose_b16_put(xb16, pk, lane);
          __syncwarp();
          store_block_b16(xb16, out + c, p.ldo, rows_left, lane);
        }
      } else if constexpr (EPI == EPI_RESID_F32) {
        // out (fp32) = acc + residual (bf16); lane l handles rows 4i + l/8,
        // columns 4(l%8)..+3 of each 32-column block, and the residual of the
        // next block is loaded while this one is turned around and stored
        float* out = reinterpret_cast<float*>(p.out) + (size_t)wrow0 * p.ldo + nt * BN + 4 * (lane & 7);
        const __nv_bfloat16* res = reinterpret_cast<const __nv_bfloat16*>(p.aux) + (size_t)wrow0 * p.ld_aux +
                                   nt * BN + 4 * (lane & 7);
        uint2 rn[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int row = 4 * i + (lane >> 3);
          rn[i] = row < rows_left ? *reinterpret_cast<const uint2*>(res + (size_t)row * p.ld_aux) : make_uint2(0, 0);
        }
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint2 rc[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) rc[i] = rn[i];
          if (c + 32 < BN) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int row = 4 * i + (lane >> 3);
              if (row < rows_left) rn[i] = *reinterpret_cast<const uint2*>(res + (size_t)row * p.ld_aux + c + 32);
            }
          }
          tmem_ld32(taddr + c, v);
          tmem_ld_wait();
          __syncwarp();
          xpose_f32_put(xf32, v, lane);
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int row = 4 * i + (lane >> 3);
            const float4 a = xpose_f32_get(xf32, i, lane);
            if (row < rows_left)
              *reinterpret_cast<float4*>(out + (size_t)row * p.ldo + c) =
                  make_float4(a.x + bf16lo(rc[i].x), a.y + bf16hi(rc[i].x), a.z + bf16lo(rc[i].y), a.w + bf16hi(rc[i].y));
          }
        }
      } else if constexpr (EPI == EPI_RESID_BF16) {
        // out (bf16) = bf16(acc + residual (fp32)), same lane layout as above
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)wrow0 * p.ldo + nt * BN + 4 * (lane & 7);
        const float* res = reinterpret_cast<const float*>(p.aux) + (size_t)wrow0 * p.ld_aux + nt * BN + 4 * (lane & 7);
        float4 rn[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int row = 4 * i + (lane >> 3);
          rn[i] = row < rows_left ? *reinterpret_cast<const float4*>(res + (size_t)row * p.ld_aux) : make_float4(0, 0, 0, 0);
        }
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          float4 rc[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) rc[i] = rn[i];
          if (c + 32 < BN) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int row = 4 * i + (lane >> 3);
              if (row < rows_left) rn[i] = *reinterpret_cast<const float4*>(res + (size_t)row * p.ld_aux + c + 32);
            }
          }
          tmem_ld32(taddr + c, v);
          tmem_ld_wait();
          __syncwarp();
          xpose_f32_put(xf32, v, lane);
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int row = 4 * i + (lane >> 3);
            const float4 a = xpose_f32_get(xf32, i, lane);
            if (row < rows_left)
              *reinterpret_cast<uint2*>(out + (size_t)row * p.ldo + c) =
                  make_uint2(pack_bf16(a.x + rc[i].x, a.y + rc[i].y), pack_bf16(a.z + rc[i].z, a.w + rc[i].w));
          }
        }
      } else if constexpr (EPI == EPI_SWIGLU) {
        // stored directly, one row per thread: measured faster here than
        // through the transpose (the SiLU work already spaces the stores)
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)row * p.ldo + nt * (BN / 2);
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          tmem_ld32(taddr + c, v);
          tmem_ld32(taddr + BN / 2 + c, w);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = silu(v[i]) * w[i];
            store_bf16x32(out + c, v);
          }
        }
      } else if constexpr (EPI == EPI_QKV) {
        const int D = p.qkv.head_dim;
        const int col0 = nt * BN;
        if (D == 128) {
#pragma unroll 1
          for (int hh = 0; hh < BN / 128; ++hh)
            qkv_head<128>(taddr + hh * 128, row, valid, (col0 + hh * 128) / 128, p.qkv, xb16, lane);
        } else {
#pragma unroll 1
          for (int hh = 0; hh < BN / 64; ++hh)
            qkv_head<64>(taddr + hh * 64, row, valid, (col0 + hh * 64) / 64, p.qkv, xb16, lane);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

template <int BN, int EPI>
cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const GemmArgs& p,
                       int num_sms, cudaStream_t s) {
  using C = GemmCfg<BN, EPI>;
  auto k = gemm_kernel<BN, EPI>;
  static std::atomic<unsigned long long> attr{0};
  const cudaError_t e = smem_limit_per_device(k, (int)C::SMEM, attr);
  if (e != cudaSuccess) return e;
  const int cap = p.max_ctas > 0 && p.max_ctas < num_sms ? p.max_ctas : num_sms;
  GemmArgs q = p;
  const GemmSchedule sc = gemm_schedule(p.M, p.N, p.K, EPI, cap, (q.sk_ws && q.sk_flags) ? p.split_mode : 1);
  q.tiles = sc.tiles;
  q.dp_tiles = sc.dp_tiles;
  q.split = sc.split;
  return launch_pdl(k, dim3(sc.grid), dim3(kThreads), C::SMEM, s, a, b0, b1, q);
}

// Critical-path cost of the split-K fix-up, in k-blocks (one k-block of a
// 128x256 tile is ~0.3 us on an SM): storing a partial and signalling it,
// then per extra chunk a 128 KB bulk read back, measured as ~9 us in all.
constexpr int kFixupBaseKb = 30;
constexpr int kFixupPerChunkKb = 4;
// at most 12 partial pieces of a 32-column chunk fit the fix-up's ring rounds
constexpr int kMaxSplit = 13;

}  // namespace

// split_mode: 0 automatic, 1 whole tiles only, >= 2 that many k-chunks per
// tail tile (at most what fits in one wave).
GemmSchedule gemm_schedule(int M, int N, int K, int epi, int ctas, int split_mode) {
  if (ctas < 1) ctas = 1;
  GemmSchedule sc{};
  const int num_m = (M + BM - 1) / BM;
  const int num_n = epi == EPI_SWIGLU ? N / (kGemmBN / 2) : N / kGemmBN;
  sc.tiles = num_m * num_n;
  sc.num_kb = K / BK;
  sc.dp_tiles = sc.tiles;
  sc.split = 1;
  sc.grid = sc.tiles < ctas ? sc.tiles : ctas;
  if (sc.grid < 1) sc.grid = 1;
  const int rest = sc.tiles % ctas;
  if (split_mode == 1 || rest == 0 || sc.tiles <= 0) return sc;
  int max_split = ctas / rest < sc.num_kb ? ctas / rest : sc.num_kb;
  if (max_split > kMaxSplit) max_split = kMaxSplit;
  if (max_split < 2) return sc;
  int best = 1;
  if (split_mode >= 2) {
    best = split_mode < max_split ? split_mode : max_split;
  } else {
    long long best_t = sc.num_kb;   // the tail as one more wave of whole tiles
    for (int s = 2; s <= max_split; ++s) {
      const long long t = (sc.num_kb + s - 1) / s + kFixupBaseKb + (long long)kFixupPerChunkKb * (s - 1);
      if (t < best_t) {
        best_t = t;
        best = s;
      }
    }
  }
  if (best < 2) return sc;
  sc.dp_tiles = sc.tiles - rest;
  sc.split = best;
  sc.grid = sc.dp_tiles > 0 ? ctas : rest * best;
  return sc;
}

size_t gemm_sk_ws_bytes(int ctas) { return (size_t)ctas * BM * kGemmBN * sizeof(float); }
size_t gemm_sk_flag_bytes(int ctas) { return (size_t)ctas * sizeof(int); }

cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB0, const CUtensorMap& tmB1,
                        const GemmArgs& a, int num_sms, cudaStream_t s) {
  switch (a.epi) {
    case EPI_BF16: return launch_one<256, EPI_BF16>(tmA, tmB0, tmB1, a, num_sms, s);
    case EPI_RESID_F32: return launch_one<256, EPI_RESID_F32>(tmA, tmB0, tmB1, a, num_sms, s);
    case EPI_RESID_BF16: return launch_one<256, EPI_RESID_BF16>(tmA, tmB0, tmB1, a, num_sms, s);
    case EPI_SWIGLU: return launch_one<256, EPI_SWIGLU>(tmA, tmB0, tmB1, a, num_sms, s);
    case EPI_QKV: return launch_one<256, EPI_QKV>(tmA, tmB0, tmB1, a, num_sms, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace cf
