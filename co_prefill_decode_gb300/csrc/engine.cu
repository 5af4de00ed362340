// libcf host runtime: the C ABI of include/cf.h.
//
// cf_layer_step queues one co-batched layer (ConfluxServe Fig. 1, Fig. 7):
//   main stream : RMSNorm (+RoPE table, slots) -> fused QKV GEMM (QK-norm,
//                 RoPE, Q write, paged K/V append) -> event `fork`
//   D stream    : waits `fork` -> split-K decode attention + merge on the
//                 decode SM partition -> event `join`
//   main stream : causal prefill attention on the remaining SMs -> waits
//                 `join` -> O-proj (+x, fp32 h) -> RMSNorm -> gate/up GEMM
//                 with SwiGLU -> down GEMM (+h) -> x_out
// The two attention kernels are persistent grids sized to disjoint SM
// counts; each CTA needs more than half of an SM's shared memory (or
// registers), so no SM runs CTAs of both (ConfluxServe §6.1: decode gets the
// SMs it needs for ~90% of its standalone HBM bandwidth, prefill the rest).
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace cf {

// ---------------------------------------------------------------- TMA descriptors
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}
}  // namespace

bool make_tmap_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows,
                  uint32_t box_cols) {
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                  uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1 * 2, s2 * 2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace cf

using namespace cf;

namespace {

constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s cap on any one device wait
// Decode batches are bucketed by ceil(log2 n_decode) (n_decode <= 2048) for
// the automatic SM share: each bucket is calibrated on its first step.
constexpr int kBuckets = 12;
int bucket_of(int n_decode) {
  int b = 0;
  while ((1 << b) < n_decode && b < kBuckets - 1) ++b;
  return b;
}
constexpr int kPhases = 12;
constexpr int kRing = 64;
enum { PH_PREP = 0, PH_QKV, PH_DEC, PH_PRE, PH_FORK, PH_OPROJ, PH_PREP2, PH_GU, PH_DOWN, PH_STEP, PH_FORK_IN,
       PH_FORK_OUT };
enum { EV_START = 0, EV_PREP, EV_QKV, EV_DEC0, EV_DEC1, EV_PRE0, EV_PRE1, EV_JOIN, EV_OPROJ, EV_PREP2, EV_GU, EV_END,
       EV_COUNT };

struct Tmaps {
  CUtensorMap xn, attn, hn, act;       // A operands (rows max_tokens)
  CUtensorMap wqkv, wo, wg, wu, wd;    // B operands
  CUtensorMap q3;                      // Q buffer, 3-D {d, Hq, rows}
};

struct PoolMaps {
  const void* k = nullptr;
  const void* v = nullptr;
  int pages = 0;
  CUtensorMap tk, tv;
};

}  // namespace

struct cf_engine {
  cf_config cfg;
  cf_weights w;
  int dev = 0, sms = 0;
  int decode_sms = 0;            // explicit share (cf_set_decode_sms); 0: the config's, else auto
  int fork_mode = 0;             // 0: concurrent work-conserving fork; 1: serial (decode, then prefill)
  int auto_sms[kBuckets] = {0};  // the 90%-rule share per decode-batch bucket; 0: not measured yet
  int last_bucket = -1;          // bucket of the last step with decodes
  cudaStream_t dstream = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_dec = nullptr;
  // workspace
  void* ws = nullptr;
  size_t ws_bytes = 0;
  __nv_bfloat16 *xn, *q, *attn, *hn, *act;
  float* h;
  float2* rope_cs;
  int* slot;
  double* inv_freq;
  float *part_o, *part_ml;
  int* plan;
  unsigned* counter;             // prefill work queue (set to 0 before each use)
  int* dec_counter;
  int split_mode = 0;            // GEMM split-K tail: 0 automatic, 1 off, >= 2 forced chunk count
  int prefill_pair = 0;          // prefill items: 0 automatic, 1 single query tiles, 2 tile pairs, 3 head pairs
  int prefill_split = 0;         // prefill key-range cuts: 0 automatic, 1 never, n >= 2 n ranges
  float* pf_part_o = nullptr;    // partials of cut prefill items
  float* pf_part_ml = nullptr;
  float* sk_ws;                  // split-K partial tiles of the GEMMs
  int* sk_flags;                 // their per-tile flags (0 between launches)
  int* err;
  long long max_items;
  Tmaps tm;
  PoolMaps pm;
  long long launches = 0;
  std::string last_error;
  // profiling
  int profiling = 0;
  std::vector<cudaEvent_t> ring;     // kRing * EV_COUNT
  std::vector<int> ring_used;        // 1 if slot holds an unresolved step
  std::vector<int> ring_has_dec, ring_has_pre;
  long long ring_next = 0;
  double phase_ms[kPhases] = {0};
  int phase_steps = 0;
  std::vector<std::pair<int, float>> calib;   // (decode CTAs, ms) of the last calibration
  // piecewise CUDA graphs of the shared linear segments (ConfluxServe §6.1, Fig. 10)
  int use_graphs = 0;
  cudaStream_t cstream = nullptr;    // capture stream
  ChunkRows* bdev = nullptr;         // device copy of the step's chunk table (graph replay)
  struct Graphs {
    long long T;
    const void *x_in, *x_out, *pk, *pv;
    int num_pages;
    const int *dec_ctx, *dec_pages, *pre_pages;
    int dec_stride, pre_stride, split_mode;
    cudaGraphExec_t a, b;            // RMSNorm + QKV; O-proj + RMSNorm + gate/up + down
  };
  std::vector<Graphs> graphs;
  long long graph_captures = 0;
};

namespace {

cf_status fail(cf_engine* e, cf_status s, const char* msg) {
  if (e) e->last_error = msg;
  return s;
}
cf_status cuda_fail(cf_engine* e, cudaError_t err, const char* what) {
  if (e) e->last_error = std::string(what) + ": " + cudaGetErrorString(err);
  return CF_ERR_CUDA;
}
#define CF_CUDA(e, call)                                  \
  do {                                                    \
    cudaError_t _r = (call);                              \
    if (_r != cudaSuccess) return cuda_fail((e), _r, #call); \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int qkv_dim(const cf_config& c) { return (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim; }

cf_status check_config(const cf_config* c) {
  if (!c) return CF_ERR_INVALID_ARG;
  if (c->hidden <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->ffn_dim <= 0 || c->max_tokens <= 0 ||
      c->max_decode < 0 || c->page_size <= 0)
    return CF_ERR_INVALID_ARG;
  if (c->n_q_heads % c->n_kv_heads) return CF_ERR_INVALID_ARG;
  if (c->n_q_heads / c->n_kv_heads > 16) return CF_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return CF_ERR_UNSUPPORTED;
  if (c->page_size != kPageSize) return CF_ERR_UNSUPPORTED;
  if (c->hidden % 256 || qkv_dim(*c) % 256 || c->ffn_dim % 128 || (c->n_q_heads * c->head_dim) % 64)
    return CF_ERR_UNSUPPORTED;
  if (c->max_decode > 2048) return CF_ERR_UNSUPPORTED;
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return CF_ERR_INVALID_ARG;
  return CF_OK;
}

// The share is, in order: the explicit one (cf_set_decode_sms), the
// configuration's, the measured 90%-rule share of the batch's bucket, and
// before any measurement a third of the SMs.
int pick_decode_sms(cf_engine* e, bool have_prefill, bool have_decode, int bucket) {
  if (!have_prefill) return e->sms;
  if (!have_decode) return 0;
  int n = e->decode_sms > 0 ? e->decode_sms : e->cfg.decode_sms;
  if (n <= 0 && bucket >= 0 && bucket < kBuckets) n = e->auto_sms[bucket];
  if (n <= 0) n = e->sms / 3;
  if (n < 1) n = 1;
  if (n > e->sms - 1) n = e->sms - 1;
  return n;
}

cf_status pool_maps(cf_engine* e, const cf_kv_pool* pool) {
  if (e->pm.k == pool->k && e->pm.v == pool->v && e->pm.pages == pool->num_pages) return CF_OK;
  const uint64_t rows = (uint64_t)pool->num_pages * e->cfg.n_kv_heads * e->cfg.page_size;
  const uint64_t d = e->cfg.head_dim;
  if (!make_tmap_2d(&e->pm.tk, pool->k, rows, d, d, 16, 64) || !make_tmap_2d(&e->pm.tv, pool->v, rows, d, d, 16, 64))
    return fail(e, CF_ERR_CUDA, "cuTensorMapEncodeTiled failed for the KV pool");
  e->pm.k = pool->k;
  e->pm.v = pool->v;
  e->pm.pages = pool->num_pages;
  return CF_OK;
}

cf_status check_pool(cf_engine* e, const cf_kv_pool* pool) {
  if (!pool || !pool->k || !pool->v || pool->num_pages <= 0) return fail(e, CF_ERR_INVALID_ARG, "bad KV pool");
  if (!aligned16(pool->k) || !aligned16(pool->v)) return fail(e, CF_ERR_INVALID_ARG, "KV pool not 16-byte aligned");
  const long long rows = (long long)pool->num_pages * e->cfg.n_kv_heads * e->cfg.page_size;
  if (rows >= (1ll << 31)) return fail(e, CF_ERR_UNSUPPORTED, "KV pool too large for 32-bit TMA coordinates");
  return CF_OK;
}

// The prefill chunks of a batch: the chunk list when n_chunks > 0, else the
// single chunk of prefill_len / prefill_prefix / pre_pages (or none).
struct StepChunks {
  int n = 0;
  int len[kMaxChunks], prefix[kMaxChunks];
  const int* pages = nullptr;   // chunk i's table at pages + i * stride
  int stride = 0;
  int rows = 0;                 // prefill rows, sum of len
};

cf_status chunks_of(cf_engine* e, const cf_batch* bt, StepChunks* ch) {
  ch->n = 0;
  ch->rows = 0;
  if (bt->n_chunks < 0) return fail(e, CF_ERR_INVALID_ARG, "negative n_chunks");
  if (bt->n_chunks > 0) {
    if (bt->prefill_len != 0) return fail(e, CF_ERR_INVALID_ARG, "prefill_len must be 0 when n_chunks > 0");
    if (bt->n_chunks > kMaxChunks) return fail(e, CF_ERR_UNSUPPORTED, "more than 32 prefill chunks");
    if (!bt->chunk_len || !bt->chunk_prefix || !bt->chunk_pages || bt->chunk_stride <= 0)
      return fail(e, CF_ERR_INVALID_ARG, "prefill chunks without lengths, prefixes or page tables");
    long long rows = 0;
    for (int i = 0; i < bt->n_chunks; ++i) {
      const int l = bt->chunk_len[i], c = bt->chunk_prefix[i];
      if (l <= 0 || c < 0) return fail(e, CF_ERR_INVALID_ARG, "chunk length < 1 or negative prefix");
      if (((long long)c + l + e->cfg.page_size - 1) / e->cfg.page_size > bt->chunk_stride)
        return fail(e, CF_ERR_INVALID_ARG, "chunk needs more pages than chunk_stride");
      ch->len[i] = l;
      ch->prefix[i] = c;
      rows += l;
      if (rows > e->cfg.max_tokens) return fail(e, CF_ERR_INVALID_ARG, "batch exceeds engine limits");
    }
    ch->n = bt->n_chunks;
    ch->rows = (int)rows;
    ch->pages = bt->chunk_pages;
    ch->stride = bt->chunk_stride;
    return CF_OK;
  }
  if (bt->prefill_len < 0 || bt->prefill_prefix < 0) return fail(e, CF_ERR_INVALID_ARG, "negative batch sizes");
  if (bt->prefill_len > 0) {
    if (!bt->pre_pages) return fail(e, CF_ERR_INVALID_ARG, "prefill chunk without a page table");
    ch->n = 1;
    ch->len[0] = bt->prefill_len;
    ch->prefix[0] = bt->prefill_prefix;
    ch->rows = bt->prefill_len;
    ch->pages = bt->pre_pages;
  }
  return CF_OK;
}

cf_status check_batch(cf_engine* e, const cf_batch* bt, StepChunks* ch) {
  const cf_config& c = e->cfg;
  cf_status st = chunks_of(e, bt, ch);
  if (st != CF_OK) return st;
  const int nd = bt->n_decode;
  if (nd < 0) return fail(e, CF_ERR_INVALID_ARG, "negative batch sizes");
  if ((long long)ch->rows + nd > c.max_tokens || nd > c.max_decode)
    return fail(e, CF_ERR_INVALID_ARG, "batch exceeds engine limits");
  if (nd > 0 && (!bt->dec_ctx || !bt->dec_pages || bt->dec_stride <= 0))
    return fail(e, CF_ERR_INVALID_ARG, "decode batch without context/page arrays");
  return CF_OK;
}

ChunkRows chunk_rows(const StepChunks& ch) {
  ChunkRows cr{};
  cr.n = ch.n;
  int r = 0;
  for (int i = 0; i < ch.n; ++i) {
    cr.row0[i] = r;
    cr.prefix[i] = ch.prefix[i];
    r += ch.len[i];
  }
  cr.row0[ch.n] = r;
  return cr;
}

// The chunk slots of a prefill launch: chunk i's rows of q and of out start
// at the sum of the earlier chunks' lengths.
void prefill_chunks_args(cf_engine* e, const StepChunks& ch, PrefillArgs& pf) {
  int row0[kMaxChunks], off[kMaxChunks];
  int r = 0;
  for (int i = 0; i < ch.n; ++i) {
    row0[i] = r;
    off[i] = i * ch.stride;
    r += ch.len[i];
  }
  pf.pages = ch.pages;
  pf.pair = e->prefill_pair ? e->prefill_pair - 1 : prefill_pairing(ch.len, ch.n, pf.Hq, pf.Hkv, e->sms);
  pf.part_o = e->pf_part_o;
  pf.part_ml = e->pf_part_ml;
  prefill_set_chunks(pf, ch.n, ch.len, ch.prefix, row0, off, e->sms, e->prefill_split);
}

// RoPE table + slots (and optionally the RMSNorm of x), then the fused QKV
// GEMM whose epilogue writes q and appends k, v.
cf_status qkv_stage(cf_engine* e, const cf_batch* bt, const StepChunks& ch, const void* x, const CUtensorMap& tm_xn,
                    void* q_out, const cf_kv_pool* pool, cudaStream_t s, cudaEvent_t ev_mid,
                    const ChunkRows* bdev = nullptr) {
  const cf_config& c = e->cfg;
  const int T = ch.rows + bt->n_decode;
  PrepArgs pa{};
  pa.x = x;
  pa.in_f32 = 0;
  pa.gain = static_cast<const __nv_bfloat16*>(e->w.g_attn);
  pa.eps = c.rms_eps;
  pa.T = T;
  pa.H = c.hidden;
  pa.xn = x ? e->xn : nullptr;
  pa.rope_cs = e->rope_cs;
  pa.cs_ld = c.max_tokens;
  pa.inv_freq = e->inv_freq;
  pa.half_dim = c.head_dim / 2;
  pa.slot = e->slot;
  pa.cr = chunk_rows(ch);
  pa.n_decode = bt->n_decode;
  pa.dec_ctx = bt->dec_ctx;
  pa.dec_pages = bt->dec_pages;
  pa.dec_stride = bt->dec_stride;
  pa.pre_pages = ch.pages;
  pa.pre_stride = ch.stride;
  pa.num_pages = pool->num_pages;
  pa.page_size = c.page_size;
  pa.err = e->err;
  pa.zero = e->counter;   // the prefill work queue of this step starts at 0
  pa.bdev = bdev;
  CF_CUDA(e, launch_prep(pa, s));
  e->launches++;
  if (ev_mid) CF_CUDA(e, cudaEventRecord(ev_mid, s));
  GemmArgs g{};
  g.M = T;
  g.N = qkv_dim(c);
  g.K = c.hidden;
  g.epi = EPI_QKV;
  g.err = e->err;
  g.wait_ns = kWaitNs;
  g.qkv.Hq = c.n_q_heads;
  g.qkv.Hkv = c.n_kv_heads;
  g.qkv.head_dim = c.head_dim;
  g.qkv.page_size = c.page_size;
  g.qkv.qk_norm = c.qk_norm;
  g.qkv.num_pages = pool->num_pages;
  g.qkv.eps = c.rms_eps;
  g.qkv.rope_cs = e->rope_cs;
  g.qkv.cs_ld = c.max_tokens;
  g.qkv.slot = e->slot;
  g.qkv.g_q = static_cast<const __nv_bfloat16*>(e->w.g_q);
  g.qkv.g_k = static_cast<const __nv_bfloat16*>(e->w.g_k);
  g.qkv.q_out = static_cast<__nv_bfloat16*>(q_out);
  g.qkv.k_pool = static_cast<__nv_bfloat16*>(pool->k);
  g.qkv.v_pool = static_cast<__nv_bfloat16*>(pool->v);
  g.split_mode = e->split_mode;
  g.sk_ws = e->sk_ws;
  g.sk_flags = e->sk_flags;
  g.b_static = 1;
  CF_CUDA(e, launch_gemm(tm_xn, e->tm.wqkv, e->tm.wqkv, g, e->sms, s));
  e->launches++;
  return CF_OK;
}

cf_status rmsnorm_stage(cf_engine* e, const void* x, int in_f32, const void* gain, void* out, int T,
                        cudaStream_t s) {
  PrepArgs pb{};
  pb.x = x;
  pb.in_f32 = in_f32;
  pb.gain = static_cast<const __nv_bfloat16*>(gain);
  pb.eps = e->cfg.rms_eps;
  pb.T = T;
  pb.H = e->cfg.hidden;
  pb.xn = static_cast<__nv_bfloat16*>(out);
  CF_CUDA(e, launch_prep(pb, s));
  e->launches++;
  return CF_OK;
}

void prof_resolve(cf_engine* e, int slot) {
  cudaEvent_t* ev = &e->ring[(size_t)slot * EV_COUNT];
  cudaEventSynchronize(ev[EV_END]);
  auto el = [&](int a, int b) {
    float ms = 0.f;
    cudaEventElapsedTime(&ms, ev[a], ev[b]);
    return (double)ms;
  };
  e->phase_ms[PH_PREP] += el(EV_START, EV_PREP);
  e->phase_ms[PH_QKV] += el(EV_PREP, EV_QKV);
  if (e->ring_has_dec[slot]) {
    e->phase_ms[PH_DEC] += el(EV_DEC0, EV_DEC1);
    e->phase_ms[PH_FORK_IN] += el(EV_QKV, EV_DEC0);
    e->phase_ms[PH_FORK_OUT] += el(EV_DEC1, EV_JOIN);
  }
  if (e->ring_has_pre[slot]) e->phase_ms[PH_PRE] += el(EV_PRE0, EV_PRE1);
  e->phase_ms[PH_FORK] += el(EV_QKV, EV_JOIN);
  e->phase_ms[PH_OPROJ] += el(EV_JOIN, EV_OPROJ);
  e->phase_ms[PH_PREP2] += el(EV_OPROJ, EV_PREP2);
  e->phase_ms[PH_GU] += el(EV_PREP2, EV_GU);
  e->phase_ms[PH_DOWN] += el(EV_GU, EV_END);
  e->phase_ms[PH_STEP] += el(EV_START, EV_END);
  e->phase_steps += 1;
  e->ring_used[slot] = 0;
}

// The decode attention of a step's batch: its Q rows (after the chunk rows
// of the engine's Q buffer), its output rows of the attention buffer.
DecodeArgs step_decode_args(cf_engine* e, const cf_batch* bt, int chunk_rows, const cf_kv_pool* pool) {
  const cf_config& c = e->cfg;
  const size_t row = (size_t)c.n_q_heads * c.head_dim;
  DecodeArgs da{};
  da.q = e->q + (size_t)chunk_rows * row;
  da.q_stride = (long long)row;
  da.k_pool = static_cast<const __nv_bfloat16*>(pool->k);
  da.v_pool = static_cast<const __nv_bfloat16*>(pool->v);
  da.num_pages = pool->num_pages;
  da.n = bt->n_decode;
  da.n_keys = bt->dec_ctx;
  da.key_offset = 1;
  da.pages = bt->dec_pages;
  da.page_stride = bt->dec_stride;
  da.out = e->attn + (size_t)chunk_rows * row;
  da.out_stride = (long long)row;
  da.Hq = c.n_q_heads;
  da.Hkv = c.n_kv_heads;
  da.head_dim = c.head_dim;
  da.page_size = c.page_size;
  da.scale_log2 = (float)(1.4426950408889634 / sqrt((double)c.head_dim));
  da.part_o = e->part_o;
  da.part_ml = e->part_ml;
  da.plan = e->plan;
  da.max_items = e->max_items;
  da.counter = e->dec_counter;
  da.plan_ctas = e->sms;
  da.wait_ns = kWaitNs;
  da.err = e->err;
  return da;
}

// ConfluxServe §6.1: decode gets "the minimum number of SMs needed to
// sustain 90% of its standalone peak HBM bandwidth".  Times the decode
// attention `da` alone (kernel + merge, on `s`) on 8, 12, 16, ..., all SMs,
// each point the median of three timed launches after a warm-up one, and
// picks the smallest CTA count whose time is within 1/frac of the fastest.
// Synchronous (waits for the work already queued on `s`); overwrites the
// decode rows of `da.out` and the partials, which the caller recomputes.
cf_status measure_decode_share(cf_engine* e, const DecodeArgs& da, cudaStream_t s, float frac, int* chosen) {
  cudaEvent_t ev[4];
  for (auto& x : ev) CF_CUDA(e, cudaEventCreate(&x));
  std::vector<std::pair<int, float>> res;
  cf_status st = CF_OK;
  for (int n = 8;; n += 4) {   // 4-SM steps: the pick sits close to where the curve crosses the rule
    const int ctas = n < e->sms ? n : e->sms;
    cudaError_t r = launch_decode(e->pm.tk, e->pm.tv, da, ctas, s);
    for (int k = 0; k < 3 && r == cudaSuccess; ++k) {
      r = cudaEventRecord(ev[k], s);
      if (r == cudaSuccess) r = launch_decode(e->pm.tk, e->pm.tv, da, ctas, s);
    }
    if (r == cudaSuccess) r = cudaEventRecord(ev[3], s);
    if (r == cudaSuccess) r = cudaEventSynchronize(ev[3]);
    if (r != cudaSuccess) {
      st = cuda_fail(e, r, "decode share calibration");
      break;
    }
    float t[3];
    for (int k = 0; k < 3; ++k) cudaEventElapsedTime(&t[k], ev[k], ev[k + 1]);
    const float lo = fminf(t[0], fminf(t[1], t[2])), hi = fmaxf(t[0], fmaxf(t[1], t[2]));
    res.push_back({ctas, t[0] + t[1] + t[2] - lo - hi});
    e->launches += 8;
    if (ctas == e->sms) break;
  }
  for (auto& x : ev) cudaEventDestroy(x);
  if (st != CF_OK) return st;
  float best = 1e30f;
  for (auto& r : res) best = r.second < best ? r.second : best;
  int pick = e->sms - 1;
  for (auto& r : res)
    if (best / r.second >= frac) {
      pick = r.first;
      break;
    }
  if (pick >= e->sms) pick = e->sms - 1;
  e->calib.assign(res.begin(), res.end());
  *chosen = pick;
  return CF_OK;
}

}  // namespace

extern "C" {

int cf_device_sm_count(void) { return device_sm_count(); }

cf_status cf_create(const cf_config* cfg, const cf_weights* w, cf_engine** out) {
  if (!out) return CF_ERR_INVALID_ARG;
  *out = nullptr;
  cf_status st = check_config(cfg);
  if (st != CF_OK) return st;
  if (!w || !w->w_qkv || !w->w_o || !w->w_gate || !w->w_up || !w->w_down || !w->g_attn || !w->g_ffn)
    return CF_ERR_INVALID_ARG;
  if (cfg->qk_norm && (!w->g_q || !w->g_k)) return CF_ERR_INVALID_ARG;
  const void* ptrs[] = {w->w_qkv, w->w_o, w->w_gate, w->w_up, w->w_down, w->g_attn, w->g_ffn};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CF_ERR_INVALID_ARG;
  if (!encoder()) return CF_ERR_CUDA;

  cf_engine* e = new cf_engine();
  e->cfg = *cfg;
  e->w = *w;
  cudaGetDevice(&e->dev);
  e->sms = device_sm_count();
  if (e->sms <= 0) {
    delete e;
    return CF_ERR_CUDA;
  }
  const cf_config& c = *cfg;
  const size_t T = c.max_tokens, H = c.hidden, d = c.head_dim, Hq = c.n_q_heads, F = c.ffn_dim;
  const int G = c.n_q_heads / c.n_kv_heads;
  e->max_items = decode_max_items(c.max_decode, c.n_kv_heads, e->sms);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += (bytes + 255) & ~(size_t)255;
    return o;
  };
  const size_t o_xn = take(T * H * 2), o_q = take(T * Hq * d * 2), o_attn = take(T * Hq * d * 2);
  const size_t o_h = take(T * H * 4), o_hn = take(T * H * 2), o_act = take(T * F * 2);
  const size_t o_cs = take(T * (d / 2) * 8), o_slot = take(T * 4), o_inv = take(d / 2 * 8);
  const size_t o_po = take((size_t)e->max_items * G * d * 4), o_pml = take((size_t)e->max_items * G * 2 * 4);
  const size_t o_plan = take((size_t)(c.max_decode + 4) * 4), o_cnt = take(4), o_err = take(4);
  const size_t o_dcnt = take(4), o_bdev = take(sizeof(ChunkRows));
  const size_t o_skw = take(gemm_sk_ws_bytes(e->sms)), o_skf = take(gemm_sk_flag_bytes(e->sms));
  const size_t o_ppo = take((size_t)kPfPartTiles * d * 128 * 4), o_ppml = take((size_t)kPfPartTiles * 128 * 2 * 4);
  e->ws_bytes = off;
  if (cudaMalloc(&e->ws, off) != cudaSuccess) {
    cudaGetLastError();
    delete e;
    return CF_ERR_OOM;
  }
  uint8_t* b = static_cast<uint8_t*>(e->ws);
  e->xn = reinterpret_cast<__nv_bfloat16*>(b + o_xn);
  e->q = reinterpret_cast<__nv_bfloat16*>(b + o_q);
  e->attn = reinterpret_cast<__nv_bfloat16*>(b + o_attn);
  e->h = reinterpret_cast<float*>(b + o_h);
  e->hn = reinterpret_cast<__nv_bfloat16*>(b + o_hn);
  e->act = reinterpret_cast<__nv_bfloat16*>(b + o_act);
  e->rope_cs = reinterpret_cast<float2*>(b + o_cs);
  e->slot = reinterpret_cast<int*>(b + o_slot);
  e->inv_freq = reinterpret_cast<double*>(b + o_inv);
  e->part_o = reinterpret_cast<float*>(b + o_po);
  e->part_ml = reinterpret_cast<float*>(b + o_pml);
  e->plan = reinterpret_cast<int*>(b + o_plan);
  e->counter = reinterpret_cast<unsigned*>(b + o_cnt);
  e->err = reinterpret_cast<int*>(b + o_err);
  e->dec_counter = reinterpret_cast<int*>(b + o_dcnt);
  e->bdev = reinterpret_cast<ChunkRows*>(b + o_bdev);
  e->sk_ws = reinterpret_cast<float*>(b + o_skw);
  e->sk_flags = reinterpret_cast<int*>(b + o_skf);
  e->pf_part_o = reinterpret_cast<float*>(b + o_ppo);
  e->pf_part_ml = reinterpret_cast<float*>(b + o_ppml);
  bool ok = cudaMemset(e->ws, 0, off) == cudaSuccess;
  // RoPE inverse frequencies theta^(-2i/d), in double
  std::vector<double> inv(d / 2);
  for (size_t i = 0; i < d / 2; ++i) inv[i] = pow((double)c.rope_theta, -2.0 * (double)i / (double)d);
  ok = ok && cudaMemcpy(e->inv_freq, inv.data(), inv.size() * 8, cudaMemcpyHostToDevice) == cudaSuccess;
  ok = ok && cudaStreamCreateWithFlags(&e->dstream, cudaStreamNonBlocking) == cudaSuccess;
  ok = ok && cudaStreamCreateWithFlags(&e->cstream, cudaStreamNonBlocking) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&e->ev_fork, cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&e->ev_join, cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&e->ev_dec, cudaEventDisableTiming) == cudaSuccess;
  const size_t QKV = qkv_dim(c);
  ok = ok && make_tmap_2d(&e->tm.xn, e->xn, T, H, H, 128, 64);
  ok = ok && make_tmap_2d(&e->tm.attn, e->attn, T, Hq * d, Hq * d, 128, 64);
  ok = ok && make_tmap_2d(&e->tm.hn, e->hn, T, H, H, 128, 64);
  ok = ok && make_tmap_2d(&e->tm.act, e->act, T, F, F, 128, 64);
  ok = ok && make_tmap_2d(&e->tm.wqkv, w->w_qkv, QKV, H, H, 128, 64);
  ok = ok && make_tmap_2d(&e->tm.wo, w->w_o, H, Hq * d, Hq * d, 128, 64);
  ok = ok && make_tmap_2d(&e->tm.wg, w->w_gate, F, H, H, 128, 64);
  ok = ok && make_tmap_2d(&e->tm.wu, w->w_up, F, H, H, 128, 64);
  ok = ok && make_tmap_2d(&e->tm.wd, w->w_down, H, F, F, 128, 64);
  ok = ok && make_tmap_3d(&e->tm.q3, e->q, d, Hq, T, d, Hq * d, 64, 1, 128);
  if (!ok) {
    cudaGetLastError();
    cf_destroy(e);
    return CF_ERR_CUDA;
  }
  *out = e;
  return CF_OK;
}

void cf_destroy(cf_engine* e) {
  if (!e) return;
  if (e->dstream) cudaStreamSynchronize(e->dstream);
  cudaDeviceSynchronize();
  for (cudaEvent_t ev : e->ring) cudaEventDestroy(ev);
  if (e->ev_fork) cudaEventDestroy(e->ev_fork);
  if (e->ev_join) cudaEventDestroy(e->ev_join);
  if (e->ev_dec) cudaEventDestroy(e->ev_dec);
  if (e->dstream) cudaStreamDestroy(e->dstream);
  for (auto& g : e->graphs) {
    if (g.a) cudaGraphExecDestroy(g.a);
    if (g.b) cudaGraphExecDestroy(g.b);
  }
  if (e->cstream) cudaStreamDestroy(e->cstream);
  if (e->ws) cudaFree(e->ws);
  delete e;
}

// a6 - a9: O-proj + residual -> h (fp32), RMSNorm, gate/up + SwiGLU, down +
// residual -> x_out.  Depends on the batch only through T.
cf_status ffn_stage(cf_engine* e, long long T, const void* x_in, void* x_out, cudaStream_t s, cudaEvent_t* ev) {
  const cf_config& c = e->cfg;
  const int H = c.hidden, d = c.head_dim, Hq = c.n_q_heads, F = c.ffn_dim;
  cf_status st = CF_OK;
  // a6: O-proj + residual -> h (fp32)
  GemmArgs g{};
  g.M = (int)T;
  g.N = H;
  g.K = Hq * d;
  g.epi = EPI_RESID_F32;
  g.out = e->h;
  g.ldo = H;
  g.aux = x_in;
  g.ld_aux = H;
  g.err = e->err;
  g.wait_ns = kWaitNs;
  g.split_mode = e->split_mode;
  g.sk_ws = e->sk_ws;
  g.sk_flags = e->sk_flags;
  g.b_static = 1;
  CF_CUDA(e, launch_gemm(e->tm.attn, e->tm.wo, e->tm.wo, g, e->sms, s));
  e->launches++;
  if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_OPROJ], s));

  // a7: RMSNorm of h
  st = rmsnorm_stage(e, e->h, 1, e->w.g_ffn, e->hn, (int)T, s);
  if (st != CF_OK) return st;
  if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_PREP2], s));

  // a8: gate/up GEMM + SwiGLU
  g = GemmArgs{};
  g.M = (int)T;
  g.N = F;
  g.K = H;
  g.epi = EPI_SWIGLU;
  g.out = e->act;
  g.ldo = F;
  g.err = e->err;
  g.wait_ns = kWaitNs;
  g.split_mode = e->split_mode;
  g.sk_ws = e->sk_ws;
  g.sk_flags = e->sk_flags;
  g.b_static = 1;
  CF_CUDA(e, launch_gemm(e->tm.hn, e->tm.wg, e->tm.wu, g, e->sms, s));
  e->launches++;
  if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_GU], s));

  // a9: down GEMM + residual -> x_out
  g = GemmArgs{};
  g.M = (int)T;
  g.N = H;
  g.K = F;
  g.epi = EPI_RESID_BF16;
  g.out = x_out;
  g.ldo = H;
  g.aux = e->h;
  g.ld_aux = H;
  g.err = e->err;
  g.wait_ns = kWaitNs;
  g.split_mode = e->split_mode;
  g.sk_ws = e->sk_ws;
  g.sk_flags = e->sk_flags;
  g.b_static = 1;
  CF_CUDA(e, launch_gemm(e->tm.act, e->tm.wd, e->tm.wd, g, e->sms, s));
  e->launches++;
  if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_END], s));
  return CF_OK;
}

// The graphs of one (T, buffers) key, captured on first use.
cf_engine::Graphs* graphs_for(cf_engine* e, const cf_batch* bt, const StepChunks& ch, long long T, const void* x_in,
                              void* x_out, const cf_kv_pool* pool, cf_status* st) {
  *st = CF_OK;
  for (auto& g : e->graphs)
    if (g.T == T && g.x_in == x_in && g.x_out == x_out && g.pk == pool->k && g.pv == pool->v &&
        g.num_pages == pool->num_pages && g.dec_ctx == bt->dec_ctx && g.dec_pages == bt->dec_pages &&
        g.pre_pages == ch.pages && g.dec_stride == bt->dec_stride && g.pre_stride == ch.stride &&
        g.split_mode == e->split_mode)
      return &g;
  if (e->graphs.size() >= 16) {   // keep the cache small: drop the oldest
    cudaGraphExecDestroy(e->graphs.front().a);
    cudaGraphExecDestroy(e->graphs.front().b);
    e->graphs.erase(e->graphs.begin());
  }
  cf_engine::Graphs g{T, x_in, x_out, pool->k, pool->v, pool->num_pages, bt->dec_ctx, bt->dec_pages,
                      ch.pages, bt->dec_stride, ch.stride, e->split_mode, nullptr, nullptr};
  const long long launches = e->launches;   // captured launches do not run now
  cudaGraph_t ga = nullptr, gb = nullptr;
  cudaError_t r = cudaStreamBeginCapture(e->cstream, cudaStreamCaptureModeThreadLocal);
  if (r == cudaSuccess) {
    *st = qkv_stage(e, bt, ch, x_in, e->tm.xn, e->q, pool, e->cstream, nullptr, e->bdev);
    r = cudaStreamEndCapture(e->cstream, &ga);
  }
  if (r == cudaSuccess && *st == CF_OK) {
    r = cudaStreamBeginCapture(e->cstream, cudaStreamCaptureModeThreadLocal);
    if (r == cudaSuccess) {
      *st = ffn_stage(e, T, x_in, x_out, e->cstream, nullptr);
      r = cudaStreamEndCapture(e->cstream, &gb);
    }
  }
  if (r == cudaSuccess && *st == CF_OK) r = cudaGraphInstantiate(&g.a, ga, 0);
  if (r == cudaSuccess && *st == CF_OK) r = cudaGraphInstantiate(&g.b, gb, 0);
  if (ga) cudaGraphDestroy(ga);
  if (gb) cudaGraphDestroy(gb);
  e->launches = launches;
  if (r != cudaSuccess || *st != CF_OK) {
    if (g.a) cudaGraphExecDestroy(g.a);
    if (g.b) cudaGraphExecDestroy(g.b);
    cudaGetLastError();
    if (*st == CF_OK) *st = cuda_fail(e, r, "graph capture");
    return nullptr;
  }
  e->graph_captures++;
  e->graphs.push_back(g);
  return &e->graphs.back();
}

cf_status cf_layer_step(cf_engine* e, const cf_batch* bt, const void* x_in, void* x_out, const cf_kv_pool* pool,
                        void* stream) {
  if (!e || !bt || !x_in || !x_out) return fail(e, CF_ERR_INVALID_ARG, "null argument");
  const cf_config& c = e->cfg;
  StepChunks ch;
  cf_status st = check_batch(e, bt, &ch);
  if (st != CF_OK) return st;
  const int l = ch.rows, nd = bt->n_decode;   // l: prefill rows of all chunks
  const long long T = (long long)l + nd;
  if (T == 0) return CF_OK;
  if (!aligned16(x_in) || !aligned16(x_out)) return fail(e, CF_ERR_INVALID_ARG, "x not 16-byte aligned");
  const size_t xbytes = (size_t)T * c.hidden * 2;
  const uint8_t *xi = static_cast<const uint8_t*>(x_in), *xo = static_cast<const uint8_t*>(x_out);
  if (xi < xo + xbytes && xo < xi + xbytes) return fail(e, CF_ERR_INVALID_ARG, "x_in and x_out overlap");
  st = check_pool(e, pool);
  if (st != CF_OK) return st;
  st = pool_maps(e, pool);
  if (st != CF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int d = c.head_dim, Hq = c.n_q_heads;

  cudaEvent_t* ev = nullptr;
  int slot = -1;
  if (e->profiling) {
    slot = (int)(e->ring_next % kRing);
    if (e->ring_used[slot]) prof_resolve(e, slot);
    ev = &e->ring[(size_t)slot * EV_COUNT];
    e->ring_used[slot] = 1;
    e->ring_has_dec[slot] = nd > 0;
    e->ring_has_pre[slot] = l > 0;
    e->ring_next++;
    CF_CUDA(e, cudaEventRecord(ev[EV_START], s));
  }

  // a1 + a2: RMSNorm (+ RoPE table, slots), fused QKV GEMM with append.
  // With graphs on, this segment and a6 - a9 replay captured graphs; the
  // batch's chunk lengths and prefixes reach the captured RMSNorm kernel
  // through a small device copy of the chunk table written just before.
  cf_engine::Graphs* ge = nullptr;
  if (e->use_graphs && !ev) {
    ge = graphs_for(e, bt, ch, T, x_in, x_out, pool, &st);
    if (st != CF_OK) return st;
  }
  if (ge) {
    const ChunkRows hb = chunk_rows(ch);
    CF_CUDA(e, cudaMemcpyAsync(e->bdev, &hb, sizeof(hb), cudaMemcpyHostToDevice, s));
    CF_CUDA(e, cudaGraphLaunch(ge->a, s));
    e->launches += 2;
  } else {
    st = qkv_stage(e, bt, ch, x_in, e->tm.xn, e->q, pool, s, ev ? ev[EV_PREP] : nullptr);
    if (st != CF_OK) return st;
  }
  if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_QKV], s));

  // a3 || a4: the attention fork.  Decode runs on a second stream with
  // n_dec_sms CTAs, prefill on `stream` with the rest.  Each kernel drains a
  // device-wide work queue, so it is work-conserving in both directions:
  // whichever path finishes first launches a second grid of the other
  // kernel on its SMs, which takes the remaining items (or none).  Decode's
  // merge runs once both decode grids are done.
  const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)d));
  DecodeArgs da{};
  PrefillArgs pf{};
  const int bucket = nd > 0 ? bucket_of(nd) : -1;
  if (nd > 0) {
    da = step_decode_args(e, bt, l, pool);
    e->last_bucket = bucket;
  }
  if (l > 0) {
    pf.Hq = Hq;
    pf.Hkv = c.n_kv_heads;
    pf.head_dim = d;
    pf.page_size = c.page_size;
    pf.num_pages = pool->num_pages;
    pf.out = e->attn;
    pf.out_stride = (long long)Hq * d;
    pf.scale_log2 = scale_log2;
    prefill_chunks_args(e, ch, pf);
    pf.counter = e->counter;   // zeroed by this step's prep kernel
    pf.base = 0;
    pf.err = e->err;
    pf.wait_ns = kWaitNs;
  }
  // The automatic decode share: the first concurrent step of a decode-batch
  // bucket measures the 90% rule on its own batch (synchronously, on
  // `stream`, after its QKV stage) unless `stream` is being captured.
  if (nd > 0 && l > 0 && e->fork_mode == 0 && e->decode_sms <= 0 && c.decode_sms <= 0 && !e->auto_sms[bucket]) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    CF_CUDA(e, cudaStreamIsCapturing(s, &cs));
    if (cs == cudaStreamCaptureStatusNone) {
      int pick = 0;
      st = measure_decode_share(e, da, s, 0.9f, &pick);
      if (st != CF_OK) return st;
      e->auto_sms[bucket] = pick;
    }
  }
  const int n_dec_sms = pick_decode_sms(e, l > 0, nd > 0, bucket);
  const int n_pre_sms = e->sms - n_dec_sms;
  if (e->fork_mode == 1) {
    // Serial execution (the baseline the fork is measured against,
    // ConfluxServe §8.3): decode alone on all SMs, then prefill alone on
    // all SMs, on `stream`, with the same kernels and work items.
    if (nd > 0) {
      if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_DEC0], s));
      CF_CUDA(e, launch_decode(e->pm.tk, e->pm.tv, da, e->sms, s));
      e->launches += 2;
      if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_DEC1], s));
    }
    if (l > 0) {
      if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_PRE0], s));
      CF_CUDA(e, launch_prefill(e->tm.q3, e->pm.tk, e->pm.tv, pf, e->sms, s));
      e->launches++;
      if (prefill_merge_blocks(pf) > 0) {
        CF_CUDA(e, launch_prefill_merge(pf, s));
        e->launches++;
      }
      if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_PRE1], s));
    }
    if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_JOIN], s));
  } else {
    if (nd > 0) {
      CF_CUDA(e, cudaEventRecord(e->ev_fork, s));
      CF_CUDA(e, cudaStreamWaitEvent(e->dstream, e->ev_fork, 0));
      if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_DEC0], e->dstream));
      CF_CUDA(e, launch_decode_kernel(e->pm.tk, e->pm.tv, da, n_dec_sms, e->dstream));
      e->launches++;
      // every decode item has been taken when this grid ends (a second grid
      // started later only takes items this one has not reached; it may still
      // be finishing its last ones), so this is decode's time in the fork
      if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_DEC1], e->dstream));
      CF_CUDA(e, cudaEventRecord(e->ev_dec, e->dstream));
      if (l > 0) {   // decode's SMs join prefill once decode is done
        PrefillArgs helper = pf;
        helper.pdl = 1;   // starts on each SM decode frees
        CF_CUDA(e, launch_prefill(e->tm.q3, e->pm.tk, e->pm.tv, helper, n_dec_sms, e->dstream));
        e->launches++;
      }
      CF_CUDA(e, cudaEventRecord(e->ev_join, e->dstream));
    }
    if (l > 0) {
      if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_PRE0], s));
      CF_CUDA(e, launch_prefill(e->tm.q3, e->pm.tk, e->pm.tv, pf, n_pre_sms, s));
      e->launches++;
      if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_PRE1], s));
      if (nd > 0) {   // prefill's SMs join decode once prefill is done
        DecodeArgs helper = da;
        helper.pdl = 1;   // starts on each SM prefill frees
        CF_CUDA(e, launch_decode_kernel(e->pm.tk, e->pm.tv, helper, n_pre_sms, s));
        e->launches++;
      }
    }
    if (nd > 0) {
      CF_CUDA(e, cudaStreamWaitEvent(s, e->ev_dec, 0));
      CF_CUDA(e, launch_decode_merge(da, s));
      e->launches++;
      CF_CUDA(e, cudaStreamWaitEvent(s, e->ev_join, 0));
    }
    if (l > 0 && prefill_merge_blocks(pf) > 0) {   // both prefill grids are done: merge the cut items
      CF_CUDA(e, launch_prefill_merge(pf, s));
      e->launches++;
    }
    if (ev) CF_CUDA(e, cudaEventRecord(ev[EV_JOIN], s));
  }

  // a6 - a9
  if (ge) {
    CF_CUDA(e, cudaGraphLaunch(ge->b, s));
    e->launches += 4;
    return CF_OK;
  }
  return ffn_stage(e, T, x_in, x_out, s, ev);
}

cf_status cf_rmsnorm(cf_engine* e, const void* x, int x_is_f32, const void* gain, void* out, int T, void* stream) {
  if (!e) return CF_ERR_INVALID_ARG;
  if (T < 0) return fail(e, CF_ERR_INVALID_ARG, "negative T");
  if (T == 0) return CF_OK;
  if (!x || !gain || !out) return fail(e, CF_ERR_INVALID_ARG, "null argument");
  if (!aligned16(x) || !aligned16(gain) || !aligned16(out)) return fail(e, CF_ERR_INVALID_ARG, "not 16-byte aligned");
  return rmsnorm_stage(e, x, x_is_f32 ? 1 : 0, gain, out, T, static_cast<cudaStream_t>(stream));
}

cf_status cf_qkv(cf_engine* e, const cf_batch* bt, const void* xn, const cf_kv_pool* pool, void* q_out,
                 void* stream) {
  if (!e || !bt || !xn || !q_out) return fail(e, CF_ERR_INVALID_ARG, "null argument");
  StepChunks ch;
  cf_status st = check_batch(e, bt, &ch);
  if (st != CF_OK) return st;
  const int T = ch.rows + bt->n_decode;
  if (T == 0) return CF_OK;
  if (!aligned16(xn) || !aligned16(q_out)) return fail(e, CF_ERR_INVALID_ARG, "not 16-byte aligned");
  st = check_pool(e, pool);
  if (st != CF_OK) return st;
  CUtensorMap tm;
  if (!make_tmap_2d(&tm, xn, T, e->cfg.hidden, e->cfg.hidden, 128, 64))
    return fail(e, CF_ERR_CUDA, "cuTensorMapEncodeTiled failed for xn");
  return qkv_stage(e, bt, ch, nullptr, tm, q_out, pool, static_cast<cudaStream_t>(stream), nullptr);
}

cf_status cf_decode_attn(cf_engine* e, const void* q, long long q_row_stride, const cf_kv_pool* pool, int n,
                         const int* n_keys, const int* pages, int page_stride, void* out, long long out_row_stride,
                         int num_sms, void* stream) {
  if (!e) return CF_ERR_INVALID_ARG;
  if (n < 0 || n > e->cfg.max_decode) return fail(e, CF_ERR_INVALID_ARG, "n outside [0, max_decode]");
  if (n == 0) return CF_OK;
  const cf_config& c = e->cfg;
  if (!q || !n_keys || !pages || !out || page_stride <= 0) return fail(e, CF_ERR_INVALID_ARG, "null argument");
  if (!aligned16(q) || !aligned16(out) || (q_row_stride * 2) % 16 || (out_row_stride * 2) % 16)
    return fail(e, CF_ERR_INVALID_ARG, "q/out must be 16-byte aligned with 16-byte row strides");
  if (q_row_stride < (long long)c.n_q_heads * c.head_dim || out_row_stride < (long long)c.n_q_heads * c.head_dim)
    return fail(e, CF_ERR_INVALID_ARG, "row stride shorter than Hq * d");
  cf_status st = check_pool(e, pool);
  if (st != CF_OK) return st;
  st = pool_maps(e, pool);
  if (st != CF_OK) return st;
  int ctas = num_sms > 0 ? num_sms : e->sms;
  if (ctas > e->sms) ctas = e->sms;
  DecodeArgs da{};
  da.q = static_cast<const __nv_bfloat16*>(q);
  da.q_stride = q_row_stride;
  da.k_pool = static_cast<const __nv_bfloat16*>(pool->k);
  da.v_pool = static_cast<const __nv_bfloat16*>(pool->v);
  da.num_pages = pool->num_pages;
  da.n = n;
  da.n_keys = n_keys;
  da.key_offset = 0;
  da.pages = pages;
  da.page_stride = page_stride;
  da.out = static_cast<__nv_bfloat16*>(out);
  da.out_stride = out_row_stride;
  da.Hq = c.n_q_heads;
  da.Hkv = c.n_kv_heads;
  da.head_dim = c.head_dim;
  da.page_size = c.page_size;
  da.scale_log2 = (float)(1.4426950408889634 / sqrt((double)c.head_dim));
  da.part_o = e->part_o;
  da.part_ml = e->part_ml;
  da.plan = e->plan;
  da.max_items = e->max_items;
  da.counter = e->dec_counter;
  da.plan_ctas = e->sms;
  da.wait_ns = kWaitNs;
  da.err = e->err;
  CF_CUDA(e, launch_decode(e->pm.tk, e->pm.tv, da, ctas, static_cast<cudaStream_t>(stream)));
  e->launches += 2;
  return CF_OK;
}

namespace {

cf_status prefill_attn_impl(cf_engine* e, const void* q, const cf_kv_pool* pool, const StepChunks& ch, void* out,
                            int num_sms, cudaStream_t s) {
  if (ch.rows == 0) return CF_OK;
  if (!q || !out) return fail(e, CF_ERR_INVALID_ARG, "null argument");
  if (!aligned16(q) || !aligned16(out)) return fail(e, CF_ERR_INVALID_ARG, "q/out not 16-byte aligned");
  const cf_config& c = e->cfg;
  cf_status st = check_pool(e, pool);
  if (st != CF_OK) return st;
  st = pool_maps(e, pool);
  if (st != CF_OK) return st;
  CUtensorMap tq;
  if (!make_tmap_3d(&tq, q, c.head_dim, c.n_q_heads, ch.rows, c.head_dim, (uint64_t)c.n_q_heads * c.head_dim, 64,
                    1, 128))
    return fail(e, CF_ERR_CUDA, "cuTensorMapEncodeTiled failed for q");
  int ctas = num_sms > 0 ? num_sms : e->sms;
  if (ctas > e->sms) ctas = e->sms;
  PrefillArgs pf{};
  pf.Hq = c.n_q_heads;
  pf.Hkv = c.n_kv_heads;
  pf.head_dim = c.head_dim;
  pf.page_size = c.page_size;
  pf.num_pages = pool->num_pages;
  pf.out = static_cast<__nv_bfloat16*>(out);
  pf.out_stride = (long long)c.n_q_heads * c.head_dim;
  pf.scale_log2 = (float)(1.4426950408889634 / sqrt((double)c.head_dim));
  prefill_chunks_args(e, ch, pf);
  pf.counter = e->counter;
  pf.base = 0;
  CF_CUDA(e, cudaMemsetAsync(e->counter, 0, sizeof(unsigned), s));
  pf.err = e->err;
  pf.wait_ns = kWaitNs;
  CF_CUDA(e, launch_prefill(tq, e->pm.tk, e->pm.tv, pf, ctas, s));
  e->launches++;
  if (prefill_merge_blocks(pf) > 0) {
    CF_CUDA(e, launch_prefill_merge(pf, s));
    e->launches++;
  }
  return CF_OK;
}

}  // namespace

cf_status cf_prefill_attn(cf_engine* e, const void* q, const cf_kv_pool* pool, int l, int prefix, const int* pages,
                          void* out, int num_sms, void* stream) {
  if (!e) return CF_ERR_INVALID_ARG;
  if (l < 0 || prefix < 0) return fail(e, CF_ERR_INVALID_ARG, "negative sizes");
  if (l == 0) return CF_OK;
  if (!pages) return fail(e, CF_ERR_INVALID_ARG, "null argument");
  StepChunks ch;
  ch.n = 1;
  ch.len[0] = l;
  ch.prefix[0] = prefix;
  ch.rows = l;
  ch.pages = pages;
  return prefill_attn_impl(e, q, pool, ch, out, num_sms, static_cast<cudaStream_t>(stream));
}

cf_status cf_prefill_attn_varlen(cf_engine* e, const void* q, const cf_kv_pool* pool, int n_chunks,
                                 const int* chunk_len, const int* chunk_prefix, const int* chunk_pages,
                                 int chunk_stride, void* out, int num_sms, void* stream) {
  if (!e) return CF_ERR_INVALID_ARG;
  if (n_chunks < 0) return fail(e, CF_ERR_INVALID_ARG, "negative n_chunks");
  if (n_chunks == 0) return CF_OK;
  cf_batch b{};
  b.n_chunks = n_chunks;
  b.chunk_len = chunk_len;
  b.chunk_prefix = chunk_prefix;
  b.chunk_pages = chunk_pages;
  b.chunk_stride = chunk_stride;
  StepChunks ch;
  const cf_status st = chunks_of(e, &b, &ch);
  if (st != CF_OK) return st;
  return prefill_attn_impl(e, q, pool, ch, out, num_sms, static_cast<cudaStream_t>(stream));
}

cf_status cf_gemm(cf_engine* e, const void* A, int lda, const void* B, int ldb, void* C, int ldc, int M, int N, int K,
                  int epilogue, const void* aux, void* stream) {
  if (!e) return CF_ERR_INVALID_ARG;
  if (M < 0 || N <= 0 || K <= 0) return fail(e, CF_ERR_INVALID_ARG, "bad GEMM sizes");
  if (M == 0) return CF_OK;
  if (!A || !B || !C) return fail(e, CF_ERR_INVALID_ARG, "null operand");
  if (epilogue < CF_EPI_NONE || epilogue > CF_EPI_SWIGLU) return fail(e, CF_ERR_INVALID_ARG, "unknown epilogue");
  if (epilogue != CF_EPI_NONE && !aux) return fail(e, CF_ERR_INVALID_ARG, "epilogue needs aux");
  if (K % 64) return fail(e, CF_ERR_UNSUPPORTED, "K must be a multiple of 64");
  if (epilogue == CF_EPI_SWIGLU ? (N % 128) : (N % 256))
    return fail(e, CF_ERR_UNSUPPORTED, "N must be a multiple of 256 (128 for SwiGLU)");
  if (lda < K || ldb < K || ldc < N || lda % 8 || ldb % 8 || ldc % 8)
    return fail(e, CF_ERR_INVALID_ARG, "leading dimensions must be >= the row length and multiples of 8");
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || (aux && !aligned16(aux)))
    return fail(e, CF_ERR_INVALID_ARG, "operands must be 16-byte aligned");
  CUtensorMap ta, tb0, tb1;
  bool ok = make_tmap_2d(&ta, A, M, K, lda, 128, 64) && make_tmap_2d(&tb0, B, N, K, ldb, 128, 64);
  if (epilogue == CF_EPI_SWIGLU)
    ok = ok && make_tmap_2d(&tb1, aux, N, K, ldb, 128, 64);
  else
    tb1 = tb0;
  if (!ok) return fail(e, CF_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  GemmArgs g{};
  g.M = M;
  g.N = N;
  g.K = K;
  g.out = C;
  g.ldo = ldc;
  g.err = e->err;
  g.wait_ns = kWaitNs;
  switch (epilogue) {
    case CF_EPI_NONE: g.epi = EPI_BF16; break;
    case CF_EPI_RESID_F32: g.epi = EPI_RESID_F32; g.aux = aux; g.ld_aux = ldc; break;
    case CF_EPI_RESID_BF16: g.epi = EPI_RESID_BF16; g.aux = aux; g.ld_aux = ldc; break;
    case CF_EPI_SWIGLU: g.epi = EPI_SWIGLU; break;
  }
  g.split_mode = e->split_mode;
  g.sk_ws = e->sk_ws;
  g.sk_flags = e->sk_flags;
  CF_CUDA(e, launch_gemm(ta, tb0, tb1, g, e->sms, static_cast<cudaStream_t>(stream)));
  e->launches++;
  return CF_OK;
}

cf_status cf_gemm_schedule(int M, int N, int K, int epilogue, int ctas, int split_mode, int* grid, int* tiles,
                           int* dp_tiles, int* split) {
  if (M <= 0 || N <= 0 || K <= 0 || ctas <= 0 || split_mode < 0) return CF_ERR_INVALID_ARG;
  if (epilogue < CF_EPI_NONE || epilogue > CF_EPI_SWIGLU) return CF_ERR_INVALID_ARG;
  const GemmSchedule sc =
      gemm_schedule(M, N, K, epilogue == CF_EPI_SWIGLU ? EPI_SWIGLU : EPI_BF16, ctas, split_mode);
  if (grid) *grid = sc.grid;
  if (tiles) *tiles = sc.tiles;
  if (dp_tiles) *dp_tiles = sc.dp_tiles;
  if (split) *split = sc.split;
  return CF_OK;
}

cf_status cf_decode_plan(int n, const int* n_keys, int page_stride, int n_kv_heads, int plan_ctas, int* chunk,
                         int* items, long long* max_items) {
  if (n <= 0 || !n_keys || page_stride <= 0 || n_kv_heads <= 0 || plan_ctas <= 0) return CF_ERR_INVALID_ARG;
  long long tot = 0, pmax = 0;
  std::vector<long long> pages(n);
  for (int j = 0; j < n; ++j) {   // as the kernel: no keys -> no pages, at most the page table's width
    const long long keys = n_keys[j];
    long long pg = keys > 0 ? (keys + 15) / 16 : 0;
    if (pg > page_stride) pg = page_stride;
    pages[j] = pg;
    tot += pg;
    pmax = pg > pmax ? pg : pmax;
  }
  const long long c = decode_plan_chunk(tot, pmax, n, n_kv_heads, plan_ctas);
  long long it = 0;
  for (int j = 0; j < n; ++j) it += (pages[j] + c - 1) / c;
  if (chunk) *chunk = (int)c;
  if (items) *items = (int)(it * n_kv_heads);
  if (max_items) *max_items = decode_max_items(n, n_kv_heads, plan_ctas);
  return CF_OK;
}

cf_status cf_prefill_plan(int n, const int* len, const int* prefix, int n_q_heads, int n_kv_heads, int sms,
                          int split_mode, int pairing_mode, int* kind, int* splits, int* cut_from, int* items) {
  if (n <= 0 || n > kMaxChunks || !len || !prefix || n_q_heads <= 0 || n_kv_heads <= 0 || sms <= 0 ||
      n_q_heads % n_kv_heads || split_mode < 0 || split_mode > kPfMaxSplits || pairing_mode < 0 || pairing_mode > 3)
    return CF_ERR_INVALID_ARG;
  if (pairing_mode == 3 && (n_q_heads / n_kv_heads) % 2) return CF_ERR_UNSUPPORTED;
  int row0[kMaxChunks], off[kMaxChunks];
  int r = 0;
  for (int i = 0; i < n; ++i) {
    if (len[i] <= 0 || prefix[i] < 0) return CF_ERR_INVALID_ARG;
    row0[i] = r;
    off[i] = 0;
    r += len[i];
  }
  PrefillArgs pf{};
  pf.Hq = n_q_heads;
  pf.Hkv = n_kv_heads;
  pf.pair = pairing_mode ? pairing_mode - 1 : prefill_pairing(len, n, n_q_heads, n_kv_heads, sms);
  prefill_set_chunks(pf, n, len, prefix, row0, off, sms, split_mode);
  for (int s = 0; s < n; ++s)   // slots are sorted by reach: map them back to the given order
    for (int i = 0; i < n; ++i)
      if (row0[i] == pf.row0[s]) {
        if (splits) splits[i] = pf.splits[s];
        if (cut_from) cut_from[i] = pf.cut_from[s];
      }
  if (kind) *kind = pf.pair;
  if (items) *items = prefill_items(pf);
  return CF_OK;
}

cf_status cf_set_prefill_pairing(cf_engine* e, int mode) {
  if (!e || mode < 0 || mode > 3) return CF_ERR_INVALID_ARG;
  if (mode == 3 && (e->cfg.n_q_heads / e->cfg.n_kv_heads) % 2) return fail(e, CF_ERR_UNSUPPORTED, "odd GQA group");
  e->prefill_pair = mode;
  return CF_OK;
}

cf_status cf_set_prefill_split(cf_engine* e, int mode) {
  if (!e || mode < 0 || mode > kPfMaxSplits) return CF_ERR_INVALID_ARG;
  e->prefill_split = mode;
  return CF_OK;
}

cf_status cf_set_graphs(cf_engine* e, int enable) {
  if (!e) return CF_ERR_INVALID_ARG;
  e->use_graphs = enable ? 1 : 0;
  return CF_OK;
}

long long cf_graph_captures(cf_engine* e) { return e ? e->graph_captures : 0; }

cf_status cf_set_split_k(cf_engine* e, int split_mode) {
  if (!e || split_mode < 0) return CF_ERR_INVALID_ARG;
  e->split_mode = split_mode;
  return CF_OK;
}

cf_status cf_selftest_timeout(cf_engine* e, unsigned long long wait_ns, void* stream) {
  if (!e || wait_ns == 0 || wait_ns > kWaitNs) return CF_ERR_INVALID_ARG;
  const cf_config& c = e->cfg;
  // one 128 x 256 tile: A = the engine's xn rows, B = the first W_qkv rows, C = its Q buffer
  GemmArgs g{};
  g.M = 128 < c.max_tokens ? 128 : c.max_tokens;
  g.N = 256;
  g.K = 64;
  g.epi = EPI_BF16;
  g.out = e->q;
  g.ldo = 256;
  g.err = e->err;
  g.wait_ns = wait_ns;
  g.split_mode = 1;
  g.stall_test = 1;
  CF_CUDA(e, launch_gemm(e->tm.xn, e->tm.wqkv, e->tm.wqkv, g, 1, static_cast<cudaStream_t>(stream)));
  e->launches++;
  return CF_OK;
}

cf_status cf_kv_append(cf_engine* e, const void* k, const void* v, int n, const int* slots, const cf_kv_pool* pool,
                       int n_kv_heads, int head_dim, int page_size, void* stream) {
  if (n < 0 || n_kv_heads <= 0 || page_size <= 0 || head_dim <= 0 || head_dim % 8)
    return fail(e, CF_ERR_INVALID_ARG, "bad append sizes");
  if (n == 0) return CF_OK;
  if (!k || !v || !slots || !pool || !pool->k || !pool->v || pool->num_pages <= 0)
    return fail(e, CF_ERR_INVALID_ARG, "null argument");
  if (!aligned16(k) || !aligned16(v) || !aligned16(pool->k) || !aligned16(pool->v))
    return fail(e, CF_ERR_INVALID_ARG, "append operands must be 16-byte aligned");
  cudaError_t r = launch_kv_append(k, v, n, slots, pool->k, pool->v, pool->num_pages, n_kv_heads, head_dim, page_size,
                                   e ? e->err : nullptr, static_cast<cudaStream_t>(stream));
  if (r != cudaSuccess) return cuda_fail(e, r, "kv_append launch");
  if (e) e->launches++;
  return CF_OK;
}

cf_status cf_get_error(cf_engine* e, char* buf, int len) {
  if (!e) return CF_ERR_INVALID_ARG;
  cudaError_t r = cudaStreamSynchronize(e->dstream);
  if (r == cudaSuccess) r = cudaDeviceSynchronize();
  int word = 0;
  if (r == cudaSuccess) r = cudaMemcpy(&word, e->err, 4, cudaMemcpyDeviceToHost);
  if (r == cudaSuccess && word) r = cudaMemset(e->err, 0, 4);
  // a launch that gave up may leave split-K tile flags set: clear them
  if (r == cudaSuccess && word) r = cudaMemset(e->sk_flags, 0, gemm_sk_flag_bytes(e->sms));
  std::string msg;
  cf_status st = CF_OK;
  if (r != cudaSuccess) {
    msg = std::string("CUDA error: ") + cudaGetErrorString(r);
    st = CF_ERR_CUDA;
  } else if (word) {
    msg = "device error:";
    if (word & CF_DEVERR_PAGE) msg += " page id outside the pool;";
    if (word & CF_DEVERR_CONTEXT) msg += " context longer than its page table;";
    if (word & CF_DEVERR_TIMEOUT) msg += " bounded wait expired;";
    if (word & CF_DEVERR_INTERNAL) msg += " kernel refused to run (internal check);";
    st = (word & CF_DEVERR_TIMEOUT) ? CF_ERR_TIMEOUT : CF_ERR_DEVICE;
  } else if (!e->last_error.empty()) {
    msg = e->last_error;
  }
  if (buf && len > 0) {
    strncpy(buf, msg.c_str(), (size_t)len - 1);
    buf[len - 1] = 0;
  }
  e->last_error.clear();
  return st;
}

void* cf_engine_buffer(cf_engine* e, const char* name) {
  if (!e || !name) return nullptr;
  if (!strcmp(name, "xn")) return e->xn;
  if (!strcmp(name, "q")) return e->q;
  if (!strcmp(name, "attn")) return e->attn;
  if (!strcmp(name, "h")) return e->h;
  if (!strcmp(name, "hn")) return e->hn;
  if (!strcmp(name, "act")) return e->act;
  return nullptr;
}

int cf_engine_decode_sms(cf_engine* e) { return e ? pick_decode_sms(e, true, true, e->last_bucket) : 0; }

cf_status cf_set_fork_mode(cf_engine* e, int mode) {
  if (!e || mode < 0 || mode > 1) return CF_ERR_INVALID_ARG;
  e->fork_mode = mode;
  return CF_OK;
}

cf_status cf_set_decode_sms(cf_engine* e, int n) {
  if (!e || n < 0 || n >= e->sms) return CF_ERR_INVALID_ARG;
  e->decode_sms = n;
  return CF_OK;
}

cf_status cf_calibrate_decode_sms(cf_engine* e, const cf_batch* bt, const cf_kv_pool* pool, float frac,
                                  void* stream, int* chosen) {
  if (!e || !bt || !chosen || !(frac > 0.f && frac <= 1.f)) return fail(e, CF_ERR_INVALID_ARG, "bad argument");
  StepChunks ch;
  cf_status st = check_batch(e, bt, &ch);
  if (st != CF_OK) return st;
  if (bt->n_decode == 0) return fail(e, CF_ERR_INVALID_ARG, "no decode requests to calibrate on");
  st = check_pool(e, pool);
  if (st != CF_OK) return st;
  st = pool_maps(e, pool);
  if (st != CF_OK) return st;
  const DecodeArgs da = step_decode_args(e, bt, ch.rows, pool);   // Q rows of the last step's decodes
  int pick = 0;
  st = measure_decode_share(e, da, static_cast<cudaStream_t>(stream), frac, &pick);
  if (st != CF_OK) return st;
  e->auto_sms[bucket_of(bt->n_decode)] = pick;
  e->last_bucket = bucket_of(bt->n_decode);
  *chosen = pick;
  return CF_OK;
}

int cf_calibration_points(cf_engine* e, int* sms, float* ms, int cap) {
  if (!e) return 0;
  int n = 0;
  for (auto& r : e->calib) {
    if (n < cap) {
      sms[n] = r.first;
      ms[n] = r.second;
    }
    ++n;
  }
  return n;
}

cf_status cf_set_profiling(cf_engine* e, int on) {
  if (!e) return CF_ERR_INVALID_ARG;
  if (on && e->ring.empty()) {
    e->ring.resize((size_t)kRing * EV_COUNT);
    for (auto& ev : e->ring)
      if (cudaEventCreate(&ev) != cudaSuccess) return CF_ERR_CUDA;
    e->ring_used.assign(kRing, 0);
    e->ring_has_dec.assign(kRing, 0);
    e->ring_has_pre.assign(kRing, 0);
  }
  e->profiling = on ? 1 : 0;
  return CF_OK;
}

cf_status cf_get_phase_times(cf_engine* e, float* ms, int n, int* steps) {
  if (!e) return CF_ERR_INVALID_ARG;
  for (int s = 0; s < (int)e->ring_used.size(); ++s)
    if (e->ring_used[s]) prof_resolve(e, s);
  for (int i = 0; i < n && i < kPhases; ++i) ms[i] = (float)e->phase_ms[i];
  if (steps) *steps = e->phase_steps;
  for (double& v : e->phase_ms) v = 0.0;
  e->phase_steps = 0;
  return CF_OK;
}

long long cf_launch_count(cf_engine* e) { return e ? e->launches : 0; }

}  // extern "C"
