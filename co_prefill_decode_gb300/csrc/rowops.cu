// Row-wise HBM-bound kernels: RMSNorm (with the per-row RoPE table and KV
// slot of the layer step) and the standalone paged KV append.
#include "common.cuh"
#include "internal.h"

namespace cf {

namespace {

constexpr int kPrepThreads = 256;

// One CTA per stacked row.  RMSNorm: xn = x / sqrt(mean(x^2) + eps) * g,
// fp32 reduction, bf16 out.  When the RoPE table is requested, the same CTA
// also writes the row's (cos, sin) pairs at its position and its pool slot:
// row r of chunk i sits at position c_i + r of that chunk's request, decode
// row j at position c_j of its own request (ConfluxServe §4: a chunk appends
// its K/V, each decode extends its own cache).
template <bool IN_F32>
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const __grid_constant__ PrepArgs a) {
  const int row = blockIdx.x;
  const int H = a.H;
  __shared__ float red[kPrepThreads / 32];
  griddep_wait();
  griddep_launch();
  if (a.zero && row == 0 && threadIdx.x == 0) *a.zero = 0u;
  if (a.xn != nullptr) {
  float ss = 0.f;
  // vectorised: 8 elements per step
  if (IN_F32) {
    const float4* x = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.x) + (size_t)row * H);
    for (int i = threadIdx.x; i < H / 4; i += kPrepThreads) {
      const float4 v = x[i];
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
  } else {
    const uint4* x = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.x) + (size_t)row * H);
    for (int i = threadIdx.x; i < H / 8; i += kPrepThreads) {
      const uint4 v = x[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float lo = bf16lo(w[k]), hi = bf16hi(w[k]);
        ss += lo * lo + hi * hi;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < kPrepThreads / 32 ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / H + a.eps);
  uint4* xn = reinterpret_cast<uint4*>(a.xn + (size_t)row * H);
  const uint4* g = reinterpret_cast<const uint4*>(a.gain);
  for (int i = threadIdx.x; i < H / 8; i += kPrepThreads) {
    float v[8];
    if (IN_F32) {
      const float4* x = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.x) + (size_t)row * H);
      const float4 p0 = x[2 * i], p1 = x[2 * i + 1];
      v[0] = p0.x; v[1] = p0.y; v[2] = p0.z; v[3] = p0.w;
      v[4] = p1.x; v[5] = p1.y; v[6] = p1.z; v[7] = p1.w;
    } else {
      const uint4 q = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.x) + (size_t)row * H)[i];
      v[0] = bf16lo(q.x); v[1] = bf16hi(q.x); v[2] = bf16lo(q.y); v[3] = bf16hi(q.y);
      v[4] = bf16lo(q.z); v[5] = bf16hi(q.z); v[6] = bf16lo(q.w); v[7] = bf16hi(q.w);
    }
    const uint4 gg = g[i];
    uint4 o;
    o.x = pack_bf16(v[0] * inv * bf16lo(gg.x), v[1] * inv * bf16hi(gg.x));
    o.y = pack_bf16(v[2] * inv * bf16lo(gg.y), v[3] * inv * bf16hi(gg.y));
    o.z = pack_bf16(v[4] * inv * bf16lo(gg.z), v[5] * inv * bf16hi(gg.z));
    o.w = pack_bf16(v[6] * inv * bf16lo(gg.w), v[7] * inv * bf16hi(gg.w));
    xn[i] = o;
  }
  }
  if (a.rope_cs == nullptr) return;

  // position and pool slot of this row; a replayed graph reads the chunks
  // of the current batch from device memory
  const ChunkRows& cr = a.bdev ? *a.bdev : a.cr;
  const int n_chunks = cr.n;
  const int rows = cr.row0[n_chunks];
  long long pos;
  const int* table;
  int table_len;
  if (row < rows) {
    int i = 0;
    while (i + 1 < n_chunks && cr.row0[i + 1] <= row) ++i;
    const int prefix = cr.prefix[i];
    const int len = cr.row0[i + 1] - cr.row0[i];
    pos = (long long)prefix + (row - cr.row0[i]);
    table = a.pre_pages + (size_t)i * a.pre_stride;
    table_len = (prefix + len + a.page_size - 1) / a.page_size;
  } else {
    const int j = row - rows;
    pos = a.dec_ctx[j];
    table = a.dec_pages + (size_t)j * a.dec_stride;
    table_len = a.dec_stride;
  }
  if (threadIdx.x == 0) {
    int slot = -1;
    const long long pidx = pos / a.page_size;
    if (pos < 0 || pidx >= table_len) {
      set_error(a.err, CF_DEVERR_CONTEXT);
    } else {
      const int page = table[pidx];
      if (page < 0 || page >= a.num_pages)
        set_error(a.err, CF_DEVERR_PAGE);
      else
        slot = page * a.page_size + (int)(pos % a.page_size);
    }
    a.slot[row] = slot;
  }
  // angle = pos * theta^(-2i/d) in double, reduced modulo 2*pi, then sincos
  // (the nearest multiple of 2 pi is found with a multiply by 1 / (2 pi):
  // FP64 division is slow here, and a quotient off by one only moves r by
  // 2 pi, which sincos does not see)
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
  for (int i = threadIdx.x; i < a.half_dim; i += kPrepThreads) {
    const double ang = (double)pos * a.inv_freq[i];
    const double r = ang - rint(ang * inv_two_pi) * two_pi;
    float s, c;
    sincosf((float)r, &s, &c);
    a.rope_cs[(size_t)i * a.cs_ld + row] = make_float2(c, s);
  }
}

// One warp per (row, kv head): d bf16 of K and of V, 16 bytes per lane.
__global__ void kv_append_kernel(const uint4* k, const uint4* v, int n, const int* slots, uint4* kp, uint4* vp,
                                 int num_pages, int Hkv, int d, int ps, int* err) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= n * Hkv) return;
  const int r = gw / Hkv, h = gw % Hkv;
  const int s = slots[r];
  if (s < 0 || s >= num_pages * ps) {
    if (lane == 0) set_error(err, CF_DEVERR_PAGE);
    return;
  }
  const int page = s / ps, off = s % ps;
  const int vec = d / 8;  // uint4 per head row
  const size_t src = ((size_t)r * Hkv + h) * vec;
  const size_t dst = (((size_t)page * Hkv + h) * ps + off) * vec;
  for (int i = lane; i < vec; i += 32) {
    kp[dst + i] = k[src + i];
    vp[dst + i] = v[src + i];
  }
}

}  // namespace

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (a.in_f32)
    return launch_pdl(prep_kernel<true>, dim3(a.T), dim3(kPrepThreads), 0, s, a);
  else
    return launch_pdl(prep_kernel<false>, dim3(a.T), dim3(kPrepThreads), 0, s, a);
  return cudaGetLastError();
}

cudaError_t launch_kv_append(const void* k, const void* v, int n, const int* slots, void* k_pool, void* v_pool,
                             int num_pages, int Hkv, int d, int ps, int* err, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const long long warps = (long long)n * Hkv;
  const int threads = 256;
  const long long blocks = (warps * 32 + threads - 1) / threads;
  kv_append_kernel<<<(unsigned)blocks, threads, 0, s>>>(
      reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v), n, slots,
      reinterpret_cast<uint4*>(k_pool), reinterpret_cast<uint4*>(v_pool), num_pages, Hkv, d, ps, err);
  return cudaGetLastError();
}

}  // namespace cf
