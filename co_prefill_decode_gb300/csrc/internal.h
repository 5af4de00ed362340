// Internal launch interfaces of libcf (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace cf {

constexpr int kPageSize = 16;

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device: the attribute belongs to the device that is
// current when it is set, so a process that launches on several GPUs needs
// it on each.  `done` holds one bit per device index below 64 (devices
// above that set it on every launch).
template <typename Kernel>
cudaError_t smem_limit_per_device(Kernel kernel, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Launches `kernel` with programmatic stream serialisation: it may be
// scheduled while the previous kernel of the stream finishes; the kernel
// itself waits (griddep_wait) before touching data that kernel may write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ------------------------------------------------------------------ GEMM
enum GemmEpi {
  EPI_BF16 = 0,        // C bf16 = acc
  EPI_RESID_F32 = 1,   // C fp32 = bf16 aux + acc
  EPI_RESID_BF16 = 2,  // C bf16 = fp32 aux + acc
  EPI_SWIGLU = 3,      // C bf16 = silu(acc[:, :BN/2]) * acc[:, BN/2:]
  EPI_QKV = 4,         // QK-norm, RoPE, Q write, paged K/V append
};

struct QkvEpilogue {
  int Hq, Hkv, head_dim, page_size, qk_norm, num_pages;
  float eps;
  const float2* rope_cs;          // [d/2][cs_ld] (cos, sin) at each row's position, pair-major
  int cs_ld;                      // row stride of rope_cs (>= T)
  const int* slot;                // [T] pool slot of each row (-1: skip)
  const __nv_bfloat16* g_q;       // [d]
  const __nv_bfloat16* g_k;       // [d]
  __nv_bfloat16* q_out;           // [T][Hq][d]
  __nv_bfloat16* k_pool;          // [pages][Hkv][ps][d]
  __nv_bfloat16* v_pool;
};

struct GemmArgs {
  int M, N, K;                    // N: output columns (SwiGLU: F)
  int epi;
  void* out;
  long long ldo;                  // elements
  const void* aux;                // residual
  long long ld_aux;
  QkvEpilogue qkv;
  int* err;
  unsigned long long wait_ns;
  int max_ctas;                   // persistent grid cap (0 = all SMs)
  // split-K tail of the last wave (tiles .. split set by launch_gemm from gemm_schedule)
  int split_mode;                 // 0 automatic, 1 whole tiles only, >= 2 forced chunk count
  float* sk_ws;                   // [grid][BM * BN] fp32 partial tiles, one slot per CTA
  int* sk_flags;                  // [tail tiles]: partials stored; 0 between launches
  int tiles, dp_tiles, split;     // tiles [dp_tiles, tiles) are cut into `split` k-chunks
  int b_static;                   // B is never written by other kernels: its first stages may be
                                  // loaded before the previous kernel of the stream has finished
  int stall_test;                 // failure-detection self-test: the MMA issuer first waits on a barrier
                                  // nothing arrives at, so the bounded wait runs out
};

// Persistent schedule of one GEMM on `ctas` CTAs: whole BMxBN tiles for the
// full waves; the tiles of a partial last wave are cut into `split` k-chunks
// when that shortens the critical path.
struct GemmSchedule {
  int grid, tiles, num_kb, dp_tiles, split;
};
GemmSchedule gemm_schedule(int M, int N, int K, int epi, int ctas, int split_mode);
constexpr int kGemmBN = 256;
// bytes of sk_ws / sk_flags a GEMM needs on up to `ctas` CTAs
size_t gemm_sk_ws_bytes(int ctas);
size_t gemm_sk_flag_bytes(int ctas);

// Builds a 2-D bf16 TMA descriptor with 128-byte swizzle: rows x cols
// (cols contiguous, row stride `ld` elements), box = box_rows x 64.
bool make_tmap_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                  uint32_t box_rows, uint32_t box_cols);
// 3-D: dims {d0 (contiguous), d1, d2}, strides in elements for d1, d2.
bool make_tmap_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                  uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2);

// A [M][K] (lda), B0/B1 halves of the weight tile: for plain GEMMs both
// describe B [N][K]; for SwiGLU B0 = gate and B1 = up.
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB0, const CUtensorMap& tmB1,
                        const GemmArgs& a, int num_sms, cudaStream_t s);

// ------------------------------------------------------------------ row kernels
// ------------------------------------------------------------------ prefill chunks
// The prefill chunks of one step (ConfluxServe §6.2 Eq. 6: the scheduled
// batch P), stacked one after another before the decode rows.
constexpr int kMaxChunks = 32;
struct ChunkRows {
  int n;                          // chunks
  int row0[kMaxChunks + 1];       // first stacked row of chunk i; row0[n] = prefill rows
  int prefix[kMaxChunks];         // c_i: chunk row r sits at position c_i + r - row0[i]
};

struct PrepArgs {
  // RMSNorm
  const void* x;                  // [T][H] bf16 (in_f32 = 0) or fp32
  int in_f32;
  const __nv_bfloat16* gain;
  float eps;
  int T, H;
  __nv_bfloat16* xn;              // [T][H]
  // rope table + slots (skipped when rope_cs == nullptr)
  float2* rope_cs;                // [d/2][cs_ld]: pair-major, so a warp's rows read 256 contiguous bytes
  int cs_ld;
  const double* inv_freq;         // [d/2]
  int half_dim;
  int* slot;                      // [T]
  ChunkRows cr;                   // the step's chunks (read from bdev instead when bdev is set)
  int n_decode;
  const int* dec_ctx;
  const int* dec_pages;
  int dec_stride;
  const int* pre_pages;           // chunk i's page table at pre_pages + i * pre_stride
  int pre_stride;
  int num_pages, page_size;
  int* err;
  unsigned* zero;                 // if set, block 0 stores 0 here (resets a work queue)
  const ChunkRows* bdev;          // if set, the chunks are read from device memory (graph replay)
};
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s);

cudaError_t launch_kv_append(const void* k, const void* v, int n, const int* slots, void* k_pool,
                             void* v_pool, int num_pages, int Hkv, int d, int ps, int* err,
                             cudaStream_t s);

// ------------------------------------------------------------------ decode attention
struct DecodeArgs {
  const __nv_bfloat16* q;         // row j at q + j * q_stride, [Hq][d]
  long long q_stride;
  const __nv_bfloat16* k_pool;
  const __nv_bfloat16* v_pool;
  int num_pages;
  int n;                          // requests
  const int* n_keys;              // [n]; keys of request j = n_keys[j] + key_offset
  int key_offset;
  const int* pages;               // [n][page_stride]
  int page_stride;
  __nv_bfloat16* out;             // row j at out + j * out_stride, [Hq][d]
  long long out_stride;
  int Hq, Hkv, head_dim, page_size;
  float scale_log2;               // log2(e) / sqrt(d)
  float* part_o;                  // [max_items][G][d] fp32 (unnormalised)
  float* part_ml;                 // [max_items][G][2] (max in log2 units, sum)
  int* plan;                      // [n + 2]: chunk prefix sums, chunk pages
  long long max_items;
  int* counter;                   // work-queue counter; 0 at launch, reset to 0 by the merge kernel
  int plan_ctas;                  // CTA count the chunk plan is sized for (the device's SMs): the items,
                                  // and so the results, depend on it, never on a launch's grid
  int pdl;                        // launch with programmatic serialisation: the grid reads nothing the
                                  // previous kernel of its stream writes, so it may start on SMs that
                                  // kernel frees before it has finished
  int* err;
  unsigned long long wait_ns;     // cap of one mbarrier wait
};
constexpr int kDecodeWarps = 8;
constexpr int kItemsPerWarp = 4;   // decode items per warp the plan aims at (unequal lengths)
// Pages per decode item (the chunk), from the total and the longest page
// count of the n requests and the CTAs the plan is sized for: about
// kItemsPerWarp items per warp, or half as many when every request has about
// the same length (longest <= 1.25 x mean), at least 4 pages.
__host__ __device__ inline long long decode_plan_chunk(long long tot_pages, long long max_pages, int n, int Hkv,
                                                       int plan_ctas) {
  const long long warps = (long long)plan_ctas * kDecodeWarps;
  const long long ipw = 4LL * max_pages * n <= 5LL * tot_pages ? kItemsPerWarp / 2 : kItemsPerWarp;
  const long long chunk = (tot_pages * Hkv + ipw * warps - 1) / (ipw * warps);
  return chunk < 4 ? 4 : chunk;
}
long long decode_max_items(int max_decode, int Hkv, int max_ctas);
// tmK/tmV: 2-D {d, pages*Hkv*ps} maps over the pools, box {64, 16}, 128-byte swizzle.
// launch_decode = launch_decode_kernel + launch_decode_merge.  Several
// decode kernel grids may drain one work queue (same args); the merge must
// follow all of them.
cudaError_t launch_decode(const CUtensorMap& tmK, const CUtensorMap& tmV, const DecodeArgs& a, int num_ctas,
                          cudaStream_t s);
cudaError_t launch_decode_kernel(const CUtensorMap& tmK, const CUtensorMap& tmV, const DecodeArgs& a,
                                 int num_ctas, cudaStream_t s);
cudaError_t launch_decode_merge(const DecodeArgs& a, cudaStream_t s);

// ------------------------------------------------------------------ prefill attention
// Query tiles of a prefill work item (pair kinds): one (query tile, head);
// two consecutive query tiles of one head; or one query tile of two heads
// that read the same KV head (GQA groups of even size).
constexpr int kPfSingle = 0, kPfTilePairs = 1, kPfHeadPairs = 2;
constexpr int kPfMaxSplits = 16;
constexpr int kPfPartTiles = 2048;  // fp32 partial (query tile) slots of split items per engine (128 MB at d = 128)

struct PrefillArgs {
  // Work items are numbered chunk slot by chunk slot (slots sorted so that the
  // chunk reaching furthest into its request comes first); slot s owns items
  // [item_end[s-1], item_end[s]).  A slot's units (tile or tile pair) before
  // cut_from[s] are one item each; the later ones are cut into splits[s] key
  // ranges each, item = cut_from + (unit - cut_from) * splits + split.
  int n_chunks;
  int item_end[kMaxChunks];
  int row0[kMaxChunks];           // the chunk's first row of Q and of out
  int len[kMaxChunks];            // l_i
  int prefix[kMaxChunks];         // c_i
  int page_off[kMaxChunks];       // its page table: pages + page_off, ceil((c_i + l_i) / ps) ids
  int splits[kMaxChunks];
  int cut_from[kMaxChunks];       // the slot's units before this one run whole; later ones are cut into splits
  int band[kMaxChunks];           // query tiles per band of the slot's unit order (see unit_tiles)
  int part_base[kMaxChunks];      // first partial slot of the slot's split items (2 per item: A, B)
  int merge_end[kMaxChunks];      // merge blocks of slots 0..s (2 per unit of a cut slot)
  float* part_o;                  // [kPfPartTiles][D][128] unnormalised O of a split's query tile
  float* part_ml;                 // [kPfPartTiles][128][2] its running max (log2 units) and sum
  int Hq, Hkv, head_dim, page_size, num_pages;
  const int* pages;
  __nv_bfloat16* out;             // row i at out + i * out_stride, [Hq][d]
  long long out_stride;
  float scale_log2;
  unsigned* counter;              // work queue shared by the launches of one step
  unsigned base;                  // counter value at the start of this launch's queue (0)
  int pdl;                        // as DecodeArgs::pdl
  int pair;                       // kPfSingle / kPfTilePairs / kPfHeadPairs; every grid draining one
                                  // queue must agree
  int* err;
  unsigned long long wait_ns;
};
// The pair kind of a launch: two heads of one KV head when the GQA group
// size is even; otherwise pairs of query tiles when that still leaves one
// item per SM of the device, else single tiles.
inline int prefill_pairing(const int* len, int n, int Hq, int Hkv, int sms) {
  if ((Hq / Hkv) % 2 == 0) return kPfHeadPairs;
  long long groups = 0;
  for (int i = 0; i < n; ++i) groups += ((len[i] + 127) / 128 + 1) / 2;
  return groups * Hq >= sms ? kPfTilePairs : kPfSingle;
}
// Fills the chunk slots, splits and item counts of `a` (a.Hq, a.Hkv and
// a.pair set) from chunks given in stacked-row order: lengths, prefixes,
// first rows and page table offsets.  split_mode 0 cuts the key range of a
// chunk's items when they would otherwise be the launch's critical path
// (longer than the average work per SM of `sms` CTAs); 1 never cuts; n >= 2
// cuts every chunk into n ranges where it can (at most its shortest item's
// key tiles, kPfMaxSplits, and the partial slots).
void prefill_set_chunks(PrefillArgs& a, int n, const int* len, const int* prefix, const int* row0,
                        const int* page_off, int sms, int split_mode);
// Merge blocks of a launch (0: no cut items).
int prefill_merge_blocks(const PrefillArgs& a);

// CTAs a launch really uses (<= items), and the items of a launch.
int prefill_grid(const PrefillArgs& a, int num_ctas);
int prefill_items(const PrefillArgs& a);
// tmQ: 3-D {d, Hq, rows} over q with box {64, 1, 128};
// tmK/tmV: 2-D {d, pages*Hkv*ps} over the pools with box {64, 16}.
cudaError_t launch_prefill(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const PrefillArgs& a, int num_ctas, cudaStream_t s);
// Combines the partials of cut items into the output (after every grid of
// the launch is done); does nothing when no item was cut.
cudaError_t launch_prefill_merge(const PrefillArgs& a, cudaStream_t s);

int device_sm_count();

}  // namespace cf
