// pa_kv_write.cu -- paged KV write: the step before the decode, which puts the
// keys and values of new tokens into their slots of the paged cache.
//
// What is written follows the vllm.cpp kernel-matrix row KERNEL-KV-CACHE
// (ReshapeAndCache for the K/V pools; ConcatAndCacheMla for the latent ||
// rope-key row of the 576-wide MLA cache, a plain copy whose written bits equal
// the input bits): token t goes to physical page slot_mapping[t] / page_size,
// slot slot_mapping[t] % page_size; a negative slot is a padding token and is
// skipped.  The FP8 variant (row KERNEL-KV-QUANT) stores E4M3 codes of
// value / scale, one float scale per pool.
//
// GB300 mapping: a pure copy, bound by HBM.  Each thread moves one 16-byte
// vector; consecutive threads cover consecutive vectors of one (token, head)
// row, so the reads of the new tokens and the writes into a page are
// coalesced.  The grid is a multiple of the SM count with a grid-stride loop.
#include <cmath>
#include <cstdint>

#include "pa_common.cuh"
#include "pa_decode.h"
#include "pa_launch.h"

namespace pa {

namespace {

// K and V rows: token t, head h, 16-byte vector e of D * 2 bytes.
__global__ void __launch_bounds__(256) kv_write_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                       const int64_t *__restrict__ slots, uint4 *k_pool,
                                                       uint4 *v_pool, long long n_vec, int vec_per_token,
                                                       long long n_slots, uint32_t *status) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec;
       i += (long long)gridDim.x * blockDim.x) {
    const long long t = i / vec_per_token;
    const int e = (int)(i - t * vec_per_token);
    const int64_t s = slots[t];
    if (s < 0) continue;  // padding token
    if (s >= n_slots) {
      if (status && e == 0) atomicOr(status, PA_DEV_BAD_SLOT);
      continue;
    }
    const long long dst = s * (long long)vec_per_token + e;
    k_pool[dst] = k[i];
    v_pool[dst] = v[i];
  }
}

// MLA cache rows of 576 bf16 = 72 vectors: 64 from the latent (512) and 8 from the rope key (64).
__global__ void __launch_bounds__(256) mla_cache_write_kernel(const uint4 *__restrict__ c_lat,
                                                              const uint4 *__restrict__ k_rope,
                                                              const int64_t *__restrict__ slots, uint4 *cache,
                                                              long long n_vec, long long n_slots,
                                                              uint32_t *status) {
  constexpr int ROW = 72, LAT = 64, ROPE = 8;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec;
       i += (long long)gridDim.x * blockDim.x) {
    const long long t = i / ROW;
    const int e = (int)(i - t * ROW);
    const int64_t s = slots[t];
    if (s < 0) continue;
    if (s >= n_slots) {
      if (status && e == 0) atomicOr(status, PA_DEV_BAD_SLOT);
      continue;
    }
    cache[s * ROW + e] = e < LAT ? c_lat[t * LAT + e] : k_rope[t * ROPE + (e - LAT)];
  }
}

// FP8: thread i converts 16 values (two 16-byte bf16 vectors) of k and of v into one 16-byte
// vector of E4M3 codes each: the fp32 quotient x / scale (correctly rounded division), then the
// nearest code (ties to even), magnitudes beyond 448 saturated.
__device__ __forceinline__ uint32_t quant4(uint32_t x0, uint32_t x1, float sc) {
  const float2 a = make_float2(__fdiv_rn(__uint_as_float(x0 << 16), sc), __fdiv_rn(__uint_as_float(x0 & 0xffff0000u), sc));
  const float2 b = make_float2(__fdiv_rn(__uint_as_float(x1 << 16), sc), __fdiv_rn(__uint_as_float(x1 & 0xffff0000u), sc));
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xffffu) | (hi << 16);
}

__device__ __forceinline__ uint4 quant16(uint4 x0, uint4 x1, float sc) {
  return make_uint4(quant4(x0.x, x0.y, sc), quant4(x0.z, x0.w, sc), quant4(x1.x, x1.y, sc), quant4(x1.z, x1.w, sc));
}

__global__ void __launch_bounds__(256) kv_write_fp8_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                           const int64_t *__restrict__ slots, uint4 *k_pool,
                                                           uint4 *v_pool, long long n_vec, int vec_per_token,
                                                           long long n_slots, float k_scale, float v_scale,
                                                           uint32_t *status) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec;
       i += (long long)gridDim.x * blockDim.x) {
    const long long t = i / vec_per_token;
    const int e = (int)(i - t * vec_per_token);
    const int64_t s = slots[t];
    if (s < 0) continue;
    if (s >= n_slots) {
      if (status && e == 0) atomicOr(status, PA_DEV_BAD_SLOT);
      continue;
    }
    const long long dst = s * (long long)vec_per_token + e;
    k_pool[dst] = quant16(k[2 * i], k[2 * i + 1], k_scale);
    v_pool[dst] = quant16(v[2 * i], v[2 * i + 1], v_scale);
  }
}

int grid_for(long long n_vec) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  const long long want = (n_vec + 255) / 256;
  const long long cap = (long long)sms * 8;
  return (int)(want < cap ? want : cap);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

}  // namespace pa

extern "C" int pa_kv_write(const void *k, const void *v, const int64_t *slot_mapping, void *k_pool, void *v_pool,
                           int num_tokens, int num_kv_heads, int head_dim, int page_size, int num_pages,
                           uint32_t *status, cudaStream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || num_pages <= 0)
    return PA_ERR_INVALID_ARGUMENT;
  if (head_dim % 8 != 0 || head_dim > 1024) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_pool || !v_pool) return PA_ERR_INVALID_ARGUMENT;
  if (!pa::aligned16(k) || !pa::aligned16(v) || !pa::aligned16(k_pool) || !pa::aligned16(v_pool) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) || (reinterpret_cast<uintptr_t>(status) & 3u))
    return PA_ERR_MISALIGNED;
  const int vec_per_token = num_kv_heads * head_dim / 8;
  const long long n_vec = (long long)num_tokens * vec_per_token;
  const int grid = pa::grid_for(n_vec);
  if (grid <= 0) return pa::cuda_fail(cudaSuccess);
  pa::note_launches(0);
  if (const cudaError_t ce = pa::profile_mark(true, stream); ce != cudaSuccess) return pa::cuda_fail(ce);
  pa::kv_write_kernel<<<grid, 256, 0, stream>>>(
      static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, static_cast<uint4 *>(k_pool),
      static_cast<uint4 *>(v_pool), n_vec, vec_per_token, (long long)num_pages * page_size, status);
  if (const cudaError_t ce = cudaGetLastError(); ce != cudaSuccess) return pa::cuda_fail(ce);
  pa::note_launches(1);
  if (const cudaError_t ce = pa::profile_mark(false, stream); ce != cudaSuccess) return pa::cuda_fail(ce);
  return PA_OK;
}

extern "C" int pa_kv_write_fp8(const void *k, const void *v, const int64_t *slot_mapping, void *k_pool,
                               void *v_pool, int num_tokens, int num_kv_heads, int head_dim, int page_size,
                               int num_pages, float k_scale, float v_scale, uint32_t *status,
                               cudaStream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || num_pages <= 0)
    return PA_ERR_INVALID_ARGUMENT;
  if (!(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f))
    return PA_ERR_INVALID_ARGUMENT;
  if (head_dim % 16 != 0 || head_dim > 1024) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_pool || !v_pool) return PA_ERR_INVALID_ARGUMENT;
  if (!pa::aligned16(k) || !pa::aligned16(v) || !pa::aligned16(k_pool) || !pa::aligned16(v_pool) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) || (reinterpret_cast<uintptr_t>(status) & 3u))
    return PA_ERR_MISALIGNED;
  const int vec_per_token = num_kv_heads * head_dim / 16;  // 16-byte vectors of codes
  const long long n_vec = (long long)num_tokens * vec_per_token;
  const int grid = pa::grid_for(n_vec);
  if (grid <= 0) return pa::cuda_fail(cudaSuccess);
  pa::note_launches(0);
  if (const cudaError_t ce = pa::profile_mark(true, stream); ce != cudaSuccess) return pa::cuda_fail(ce);
  pa::kv_write_fp8_kernel<<<grid, 256, 0, stream>>>(
      static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, static_cast<uint4 *>(k_pool),
      static_cast<uint4 *>(v_pool), n_vec, vec_per_token, (long long)num_pages * page_size, k_scale, v_scale,
      status);
  if (const cudaError_t ce = cudaGetLastError(); ce != cudaSuccess) return pa::cuda_fail(ce);
  pa::note_launches(1);
  if (const cudaError_t ce = pa::profile_mark(false, stream); ce != cudaSuccess) return pa::cuda_fail(ce);
  return PA_OK;
}

extern "C" int pa_mla_cache_write(const void *c_lat, const void *k_rope, const int64_t *slot_mapping, void *cache,
                                  int num_tokens, int page_size, int num_pages, uint32_t *status,
                                  cudaStream_t stream) {
  if (num_tokens < 0 || page_size <= 0 || num_pages <= 0) return PA_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return PA_OK;
  if (!c_lat || !k_rope || !slot_mapping || !cache) return PA_ERR_INVALID_ARGUMENT;
  if (!pa::aligned16(c_lat) || !pa::aligned16(k_rope) || !pa::aligned16(cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) || (reinterpret_cast<uintptr_t>(status) & 3u))
    return PA_ERR_MISALIGNED;
  const long long n_vec = (long long)num_tokens * 72;
  const int grid = pa::grid_for(n_vec);
  if (grid <= 0) return pa::cuda_fail(cudaSuccess);
  pa::note_launches(0);
  if (const cudaError_t ce = pa::profile_mark(true, stream); ce != cudaSuccess) return pa::cuda_fail(ce);
  pa::mla_cache_write_kernel<<<grid, 256, 0, stream>>>(
      static_cast<const uint4 *>(c_lat), static_cast<const uint4 *>(k_rope), slot_mapping,
      static_cast<uint4 *>(cache), n_vec, (long long)num_pages * page_size, status);
  if (const cudaError_t ce = cudaGetLastError(); ce != cudaSuccess) return pa::cuda_fail(ce);
  pa::note_launches(1);
  if (const cudaError_t ce = pa::profile_mark(false, stream); ce != cudaSuccess) return pa::cuda_fail(ce);
  return PA_OK;
}
