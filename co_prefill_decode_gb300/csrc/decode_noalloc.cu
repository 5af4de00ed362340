// Decode attention for callers that cannot allocate device memory.
//
// cf_decode_attn keeps its split-K partial results in the workspace that
// cf_create allocates.  Some callers cannot make that allocation: a serving
// runtime that hands all free device memory to its own KV pool at start-up,
// a plugin running inside another framework whose allocator owns the device,
// or a latency-critical loop that must never pay for cudaMalloc's implicit
// device-wide synchronisation.  This entry point runs the same split-K decode
// kernel with its scratch (error word, chunk plan, partial outputs) in a
// fixed-size array compiled into the library, so it allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kScratchBytes of it until the process exits.  In host code
// its name is only a host-side stand-in, so the kernel is given the device
// address that cudaGetSymbolAddress returns for the current device.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace cf {
namespace {

constexpr size_t kScratchBytes = 16u << 20;   // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace
}  // namespace cf

using namespace cf;

extern "C" cf_status cf_decode_attn_noalloc(int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                                            const void* q, long long q_row_stride, const cf_kv_pool* pool, int n,
                                            const int* n_keys, const int* pages, int page_stride, void* out,
                                            long long out_row_stride, int num_sms, void* stream) {
  if (n < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads) return CF_ERR_INVALID_ARG;
  if (n_q_heads / n_kv_heads > 16 || (head_dim != 64 && head_dim != 128) || page_size != kPageSize)
    return CF_ERR_UNSUPPORTED;
  if (n == 0) return CF_OK;
  if (!q || !pool || !pool->k || !pool->v || pool->num_pages <= 0 || !n_keys || !pages || !out || page_stride <= 0)
    return CF_ERR_INVALID_ARG;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out) |
                        reinterpret_cast<uintptr_t>(pool->k) | reinterpret_cast<uintptr_t>(pool->v);
  if ((mis & 15u) || (q_row_stride * 2) % 16 || (out_row_stride * 2) % 16) return CF_ERR_INVALID_ARG;
  if (q_row_stride < (long long)n_q_heads * head_dim || out_row_stride < (long long)n_q_heads * head_dim)
    return CF_ERR_INVALID_ARG;
  const int sms = device_sm_count();
  if (sms <= 0) return CF_ERR_CUDA;
  int ctas = num_sms > 0 ? num_sms : sms;
  if (ctas > sms) ctas = sms;

  // Scratch layout: error word (byte 0) and work-queue counter (byte 128) |
  // chunk plan | (m, l) partials | O partials.  Both words are cleared on the
  // call's stream before the kernel runs, so a call never depends on how the
  // previous one ended.  The keys are cut into chunks planned for the CTAs
  // this call launches, so a smaller num_sms needs less scratch (with all SMs
  // the plan, and so the output, is the one cf_decode_attn makes).
  const int G = n_q_heads / n_kv_heads;
  const long long items = decode_max_items(n, n_kv_heads, ctas);
  const size_t off_plan = 256;
  const size_t off_ml = align256(off_plan + (size_t)(n + 4) * 4);
  const size_t off_o = align256(off_ml + (size_t)items * G * 2 * 4);
  const size_t need = off_o + (size_t)items * G * head_dim * 4;
  if (need > kScratchBytes) return CF_ERR_INVALID_ARG;   // batch too large for the static scratch

  const uint64_t rows = (uint64_t)pool->num_pages * n_kv_heads * page_size;
  if (rows >= (1ull << 31)) return CF_ERR_UNSUPPORTED;
  CUtensorMap tk, tv;
  if (!make_tmap_2d(&tk, pool->k, rows, head_dim, head_dim, 16, 64) ||
      !make_tmap_2d(&tv, pool->v, rows, head_dim, head_dim, 16, 64))
    return CF_ERR_CUDA;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return CF_ERR_CUDA;
  uint8_t* b = static_cast<uint8_t*>(base);
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
  da.Hq = n_q_heads;
  da.Hkv = n_kv_heads;
  da.head_dim = head_dim;
  da.page_size = page_size;
  da.scale_log2 = (float)(1.4426950408889634 / sqrt((double)head_dim));
  da.err = reinterpret_cast<int*>(b);
  da.counter = reinterpret_cast<int*>(b + 128);
  da.plan = reinterpret_cast<int*>(b + off_plan);
  da.part_ml = reinterpret_cast<float*>(b + off_ml);
  da.part_o = reinterpret_cast<float*>(b + off_o);
  da.max_items = items;
  da.plan_ctas = ctas;
  da.wait_ns = 2000000000ull;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(b, 0, 256, s) != cudaSuccess) return CF_ERR_CUDA;
  return launch_decode(tk, tv, da, ctas, s) == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}
