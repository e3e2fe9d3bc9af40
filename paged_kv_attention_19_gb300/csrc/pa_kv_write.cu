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
// GB300 mapping: a pure copy, bound by HBM.  Each thread moves 16-byte vectors,
// two per iteration with all their loads in flight together; consecutive
// threads cover consecutive vectors of one (token, head) row, so the reads of
// the new tokens and the writes into a page are coalesced.  The grid is the SM count times the blocks of the kernel that one
// SM holds at once (one wave), with a grid-stride loop.
#include <cmath>
#include <cstdint>
#include <cstring>

#include <cuda_fp4.h>

#include "pa_common.cuh"
#include "pa_decode.h"
#include "pa_launch.h"

namespace pa {

namespace {

struct Uint4x2 {
  uint4 a, b;
};
__device__ __forceinline__ Uint4x2 make_uint4x2(uint4 a, uint4 b) { return {a, b}; }

// Grid-stride loop over n_vec vectors of vec_per_token per token, U vectors per thread and
// iteration: the loads of all U vectors (load(i, t, e) for vector e of token t, in bounds
// whatever the slot) and of their tokens' slots are issued before any is stored
// (store(slot, e, data): vector e of the row at that slot), so an iteration waits for one memory latency.  The (token, vector) pair
// of each index advances by the grid stride without a division.  A negative slot is a padding
// token; a slot past the pool is skipped and flagged.
template <int U, typename Load, typename Store>
__device__ __forceinline__ void write_loop(long long n_vec, int vec_per_token, const int64_t *__restrict__ slots,
                                           long long n_slots, uint32_t *status, Load load, Store store) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i0 >= n_vec) return;
  const long long dt = stride / vec_per_token;
  const int de = (int)(stride - dt * vec_per_token);
  long long t = i0 / vec_per_token;
  int e = (int)(i0 - t * vec_per_token);
  for (long long i = i0; i < n_vec; i += U * stride) {
    using Data = decltype(load(i, t, e));
    Data d[U];
    long long tu[U];
    int eu[U];
    bool has[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      has[u] = i + u * stride < n_vec;
      tu[u] = has[u] ? t : tu[0];
      eu[u] = has[u] ? e : eu[0];
      d[u] = load(has[u] ? i + u * stride : i, tu[u], eu[u]);
      t += dt;
      e += de;
      if (e >= vec_per_token) {
        e -= vec_per_token;
        ++t;
      }
    }
    int64_t sl[U];
#pragma unroll
    for (int u = 0; u < U; ++u) sl[u] = slots[tu[u]];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!has[u] || sl[u] < 0) continue;
      if (sl[u] >= n_slots) {
        if (status && eu[u] == 0) atomicOr(status, PA_DEV_BAD_SLOT);
        continue;
      }
      store(sl[u], eu[u], d[u]);
    }
  }
}

// K and V rows: token t, head h, 16-byte vector e of D * 2 bytes.
__global__ void __launch_bounds__(256) kv_write_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                       const int64_t *__restrict__ slots, uint4 *k_pool,
                                                       uint4 *v_pool, long long n_vec, int vec_per_token,
                                                       long long n_slots, uint32_t *status) {
  write_loop<2>(
      n_vec, vec_per_token, slots, n_slots, status,
      [&](long long i, long long, int) { return make_uint4x2(k[i], v[i]); },
      [&](long long slot, int e, const Uint4x2 &d) {
        k_pool[slot * vec_per_token + e] = d.a;
        v_pool[slot * vec_per_token + e] = d.b;
      });
}

// MLA cache rows of 576 bf16 = 72 vectors: 64 from the latent (512) and 8 from the rope key (64).
__global__ void __launch_bounds__(256) mla_cache_write_kernel(const uint4 *__restrict__ c_lat,
                                                              const uint4 *__restrict__ k_rope,
                                                              const int64_t *__restrict__ slots, uint4 *cache,
                                                              long long n_vec, long long n_slots,
                                                              uint32_t *status) {
  constexpr int ROW = 72, LAT = 64, ROPE = 8;
  write_loop<2>(
      n_vec, ROW, slots, n_slots, status,
      [&](long long, long long t, int e) { return e < LAT ? c_lat[t * LAT + e] : k_rope[t * ROPE + (e - LAT)]; },
      [&](long long slot, int e, const uint4 &d) { cache[slot * ROW + e] = d; });
}

// FP8: thread i converts 8 values (one 16-byte bf16 vector) of k and of v into 8 bytes of E4M3
// codes each, so that a warp's loads and its stores are both contiguous: the fp32 quotient
// x / scale (correctly rounded division), then the nearest code (ties to even), magnitudes
// beyond 448 saturated.
//
// The correctly rounded quotient a / b is taken in one of three ways (the host picks per scale):
//   * b a normal power of two with a normal reciprocal: the product a * (1 / b), exact;
//   * b in [2^-100, 2^100]: Markstein's correction (P. Markstein, "Computation of elementary
//     functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with
//     y = RN(1 / b), q = RN(a y) is within one ulp of a / b, the remainder r = a - b q is exact
//     (one fma), and RN(q + r y) is RN(a / b) whenever a and the quotient are normal numbers.  A
//     quotient that overflows (q infinite) stays infinite.  Where a or the quotient is subnormal
//     the result may be an ulp off, which changes no code derived from it: the quotient is then
//     below 2^-26 and rounds to the zero code of E4M3 and of E2M1 (its sign is a's), and a block
//     scale derived from it is the zero code;
//   * otherwise the correctly rounded division.
struct Fp8Scale {
  float sc;    // the pool's scale b
  float rcp;   // 1 / b when exact (a power of two), else 0
  float rcpn;  // RN(1 / b) when b and 1 / b are normal and b is not a power of two, else 0
};

__device__ __forceinline__ float markstein_quot(float a, float b, float y) {
  const float q = a * y;
  const float r = fmaf(-q, b, a);
  return fabsf(q) == INFINITY ? q : fmaf(r, y, q);
}

// The same for a quotient known to be finite (no infinite q to keep).
__device__ __forceinline__ float markstein_quot_finite(float a, float b, float y) {
  const float q = a * y;
  return fmaf(fmaf(-q, b, a), y, q);
}

__device__ __forceinline__ float quot(float x, Fp8Scale s) {
  if (s.rcp != 0.f) return x * s.rcp;
  if (s.rcpn != 0.f) return markstein_quot(x, s.sc, s.rcpn);
  return __fdiv_rn(x, s.sc);
}

__device__ __forceinline__ uint32_t quant4(uint32_t x0, uint32_t x1, Fp8Scale s) {
  const float2 a = make_float2(quot(__uint_as_float(x0 << 16), s), quot(__uint_as_float(x0 & 0xffff0000u), s));
  const float2 b = make_float2(quot(__uint_as_float(x1 << 16), s), quot(__uint_as_float(x1 & 0xffff0000u), s));
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xffffu) | (hi << 16);
}

__device__ __forceinline__ uint2 quant8(uint4 x, Fp8Scale s) { return make_uint2(quant4(x.x, x.y, s), quant4(x.z, x.w, s)); }

__global__ void __launch_bounds__(256) kv_write_fp8_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                           const int64_t *__restrict__ slots, uint2 *k_pool,
                                                           uint2 *v_pool, long long n_vec, int vec_per_token,
                                                           long long n_slots, Fp8Scale k_scale,
                                                           Fp8Scale v_scale, uint32_t *status) {
  write_loop<2>(
      n_vec, vec_per_token, slots, n_slots, status,
      [&](long long i, long long, int) { return make_uint4x2(k[i], v[i]); },
      [&](long long slot, int e, const Uint4x2 &d) {
        k_pool[slot * vec_per_token + e] = quant8(d.a, k_scale);
        v_pool[slot * vec_per_token + e] = quant8(d.b, v_scale);
      });
}

// NVFP4: thread i quantizes block i (16 consecutive values of one (token, head) row: two 16-byte
// bf16 vectors) of k and of v into 8 bytes of E2M1 code pairs and one E4M3 scale code, in fp32
// with every step correctly rounded: the scale code of (amax / s) / 6, then each value's code of
// (x / s) / E4M3(scale code).  The thread of a row's block 0 also writes the row's padding.
struct Nvfp4Row {
  int log2_nb;   // blocks per row, head_dim / 16, as a power of two
  int code_off;  // byte offset of the block scales in a row: head_dim / 2
  int row;       // bytes per row (a multiple of 16)
};

// Nearest E2M1 codes of two values (never NaN here): the conversion instruction rounds to nearest
// with ties to the even mantissa bit, saturates at 6 and keeps the sign (a negative value that
// rounds to zero gives the negative-zero code); lo goes to the low nibble.
__device__ __forceinline__ uint32_t e2m1_pair(float lo, float hi) {
  return (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(lo, hi), __NV_E2M1, cudaRoundNearest) & 0xffu;
}

// Value of a non-negative, non-NaN E4M3 code (exact in fp32).
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = c >> 3, m = c & 7u;
  return e == 0 ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

struct Nvfp4Block {
  uint2 codes;
  uint32_t scale;
};

// The value of each non-negative E4M3 scale code and its correctly rounded reciprocal (0 for the
// zero code), tabulated once per thread block.
struct E4m3Table {
  float val[128], rcp[128];
};

__device__ __forceinline__ Nvfp4Block quant_nvfp4(uint4 x0, uint4 x1, Fp8Scale s, const E4m3Table &tab) {
  const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
  // the largest magnitude as bf16 bits: the bits of |x| order like the values, NaN above infinity
  uint32_t m2 = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m2 = __vmaxu2(m2, w[i] & 0x7fff7fffu);
  const uint32_t mh = max(m2 & 0xffffu, m2 >> 16);
  const bool nan = mh > 0x7f80u;
  const float amax = __uint_as_float(mh << 16);
  // x / s for the 16 values, the scale's way of dividing chosen once (it is the same for the launch)
  float y[16];
  if (s.rcp != 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      y[2 * i] = __uint_as_float(w[i] << 16) * s.rcp;
      y[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u) * s.rcp;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      y[2 * i] = quot(__uint_as_float(w[i] << 16), s);
      y[2 * i + 1] = quot(__uint_as_float(w[i] & 0xffff0000u), s);
    }
  }
  Nvfp4Block b;
  if (nan) {
    b.scale = 0x7Fu;
    b.codes = make_uint2(0u, 0u);
    return b;
  }
  // (amax / s) / 6: the second division by Markstein's correction with RN(1 / 6)
  const float qa = quot(amax, s);
  b.scale = (uint32_t)__nv_cvt_float_to_fp8(markstein_quot(qa, 6.f, 1.f / 6.f), __NV_SATFINITE, __NV_E4M3);
  // the code is never NaN here (a NaN block returned above): 0 .. 126
  const float ds = tab.val[b.scale];
  uint32_t c[2] = {0u, 0u};
  if (ds != 0.f) {
    // y / ds by Markstein's correction (ds is normal or an E4M3 subnormal, at least 2^-9, so its
    // reciprocal is normal).  Some y is infinite (an x / s overflowed) only if amax / s is: then the
    // infinite ones stay infinite
    const float r = tab.rcp[b.scale];
    if (fabsf(qa) != INFINITY) {
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const uint32_t pr = e2m1_pair(markstein_quot_finite(y[i], ds, r), markstein_quot_finite(y[i + 1], ds, r));
        c[i >> 3] |= pr << (4 * (i & 7));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const uint32_t pr = e2m1_pair(markstein_quot(y[i], ds, r), markstein_quot(y[i + 1], ds, r));
        c[i >> 3] |= pr << (4 * (i & 7));
      }
    }
  }
  b.codes = make_uint2(c[0], c[1]);
  return b;
}

struct Uint4x4 {
  uint4 k0, k1, v0, v1;
};

__global__ void __launch_bounds__(256, 4) kv_write_nvfp4_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                             const int64_t *__restrict__ slots, uint8_t *k_pool,
                                                             uint8_t *v_pool, long long n_blk, int blk_per_token,
                                                             long long n_slots, Nvfp4Row r, Fp8Scale k_scale,
                                                             Fp8Scale v_scale, uint32_t *status) {
  __shared__ E4m3Table tab;
  if (threadIdx.x < 128) {
    const float x = e4m3_value(threadIdx.x);
    tab.val[threadIdx.x] = x;
    tab.rcp[threadIdx.x] = x != 0.f ? __frcp_rn(x) : 0.f;
  }
  __syncthreads();
  write_loop<1>(
      n_blk, blk_per_token, slots, n_slots, status,
      [&](long long i, long long, int) { return Uint4x4{k[2 * i], k[2 * i + 1], v[2 * i], v[2 * i + 1]}; },
      [&](long long slot, int e, const Uint4x4 &d) {
        const int h = e >> r.log2_nb, blk = e & ((1 << r.log2_nb) - 1);
        const long long row0 = (slot * (blk_per_token >> r.log2_nb) + h) * r.row;
        const Nvfp4Block kb = quant_nvfp4(d.k0, d.k1, k_scale, tab);
        const Nvfp4Block vb = quant_nvfp4(d.v0, d.v1, v_scale, tab);
        *reinterpret_cast<uint2 *>(k_pool + row0 + blk * 8) = kb.codes;
        *reinterpret_cast<uint2 *>(v_pool + row0 + blk * 8) = vb.codes;
        k_pool[row0 + r.code_off + blk] = (uint8_t)kb.scale;
        v_pool[row0 + r.code_off + blk] = (uint8_t)vb.scale;
        if (blk == 0) {
          for (int p = r.code_off + (1 << r.log2_nb); p < r.row; p += 4) {
            *reinterpret_cast<uint32_t *>(k_pool + row0 + p) = 0u;
            *reinterpret_cast<uint32_t *>(v_pool + row0 + p) = 0u;
          }
        }
      });
}

// Blocks of 256 threads for n_vec vectors: at most one wave of the kernel's resident blocks.
template <typename Kernel>
int grid_for(Kernel kernel, long long n_vec) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0) != cudaSuccess || per_sm <= 0) return -1;
  const long long want = (n_vec + 255) / 256;
  const long long cap = (long long)sms * per_sm;
  return (int)(want < cap ? want : cap);
}

// How x / sc is divided (see Fp8Scale): the exact reciprocal of a normal power of two whose
// reciprocal is normal, else RN(1 / sc) for Markstein's correction when sc and 1 / sc are normal,
// else neither (the correctly rounded division).
Fp8Scale fp8_scale(float sc) {
  uint32_t b;
  std::memcpy(&b, &sc, 4);
  const uint32_t e = (b >> 23) & 0xffu;
  const bool pow2 = (b & 0x807fffffu) == 0 && e >= 1 && e <= 253;  // sc = 2^(e - 127), 1 / sc = 2^(127 - e)
  if (pow2) return {sc, 1.0f / sc, 0.f};
  const float y = 1.0f / sc;  // host IEEE division: correctly rounded
  const bool in_range = sc >= 0x1p-100f && sc <= 0x1p100f;
  return {sc, 0.f, in_range ? y : 0.f};
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
  const int grid = pa::grid_for(pa::kv_write_kernel, n_vec);
  if (grid <= 0) return pa::cuda_fail(cudaGetLastError());
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
  const int vec_per_token = num_kv_heads * head_dim / 8;  // 16-byte bf16 vectors, 8 bytes of codes each
  const long long n_vec = (long long)num_tokens * vec_per_token;
  const int grid = pa::grid_for(pa::kv_write_fp8_kernel, n_vec);
  if (grid <= 0) return pa::cuda_fail(cudaGetLastError());
  pa::note_launches(0);
  if (const cudaError_t ce = pa::profile_mark(true, stream); ce != cudaSuccess) return pa::cuda_fail(ce);
  pa::kv_write_fp8_kernel<<<grid, 256, 0, stream>>>(
      static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, static_cast<uint2 *>(k_pool),
      static_cast<uint2 *>(v_pool), n_vec, vec_per_token, (long long)num_pages * page_size,
      pa::fp8_scale(k_scale), pa::fp8_scale(v_scale), status);
  if (const cudaError_t ce = cudaGetLastError(); ce != cudaSuccess) return pa::cuda_fail(ce);
  pa::note_launches(1);
  if (const cudaError_t ce = pa::profile_mark(false, stream); ce != cudaSuccess) return pa::cuda_fail(ce);
  return PA_OK;
}

extern "C" int pa_kv_write_nvfp4(const void *k, const void *v, const int64_t *slot_mapping, void *k_pool,
                                 void *v_pool, int num_tokens, int num_kv_heads, int head_dim, int page_size,
                                 int num_pages, float k_scale, float v_scale, uint32_t *status,
                                 cudaStream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || num_pages <= 0)
    return PA_ERR_INVALID_ARGUMENT;
  if (!(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f))
    return PA_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_pool || !v_pool) return PA_ERR_INVALID_ARGUMENT;
  if (!pa::aligned16(k) || !pa::aligned16(v) || !pa::aligned16(k_pool) || !pa::aligned16(v_pool) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) || (reinterpret_cast<uintptr_t>(status) & 3u))
    return PA_ERR_MISALIGNED;
  const pa::Nvfp4Row r = {head_dim == 64 ? 2 : head_dim == 128 ? 3 : 4, head_dim / 2,
                          (head_dim / 2 + head_dim / 16 + 15) / 16 * 16};
  const int blk_per_token = num_kv_heads << r.log2_nb;
  const long long n_blk = (long long)num_tokens * blk_per_token;
  const int grid = pa::grid_for(pa::kv_write_nvfp4_kernel, n_blk);
  if (grid <= 0) return pa::cuda_fail(cudaGetLastError());
  pa::note_launches(0);
  if (const cudaError_t ce = pa::profile_mark(true, stream); ce != cudaSuccess) return pa::cuda_fail(ce);
  pa::kv_write_nvfp4_kernel<<<grid, 256, 0, stream>>>(
      static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, static_cast<uint8_t *>(k_pool),
      static_cast<uint8_t *>(v_pool), n_blk, blk_per_token, (long long)num_pages * page_size, r,
      pa::fp8_scale(k_scale), pa::fp8_scale(v_scale), status);
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
  const int grid = pa::grid_for(pa::mla_cache_write_kernel, n_vec);
  if (grid <= 0) return pa::cuda_fail(cudaGetLastError());
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
