// pa_common.cuh -- device helpers shared by the decode kernels (sm_103a).
//
// Inline PTX for the Blackwell data movers used by the kernels: mbarrier
// transaction barriers and TMA bulk copies (tensor-map tiles and plain
// contiguous blocks).  Every wait is bounded by the global timer: a wait that
// gives up records PA_DEV_TIMEOUT in the workspace status word and returns
// false instead of spinning forever.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_decode.h"

namespace pa {

// Workspace header, at offset 0 of every workspace.
struct WsHeader {
  uint32_t status;  // PA_DEV_* bits of the last call (written by its combine kernel)
  uint32_t pad[63];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

constexpr unsigned FULL = 0xffffffffu;
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;   // 1 s: far beyond any legal wait (the default limit)
constexpr uint64_t DRAIN_LIMIT_NS = 1000000000ull;  // a wait after a give-up, for copies already in flight

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Per-warpgroup register reallocation (all four warps of a warpgroup execute the same one).  A
// block's warpgroups must stay within the registers the block was launched with: the increases
// wait until the decreases have returned enough.
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking: has the phase of *bar with the given parity completed?  (try_wait above may hold
// the thread for a while before it answers; test_wait answers at once.)
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete; false after WAIT_LIMIT_NS
// (the timeout bit is then set in *status).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
      atomicOr(status, PA_DEV_TIMEOUT);
      return false;
    }
  }
}

// All 32 lanes of a converged warp: wait for phase `parity` of `bar` for at most `limit_ns` of the
// global timer; every lane returns the same result.  A limit of 0 is one non-blocking test.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  if (limit_ns == 0) return __all_sync(FULL, mbar_test(bar, parity));
  if (__all_sync(FULL, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (__all_sync(FULL, mbar_try_wait(bar, parity))) return true;
    if (__any_sync(FULL, global_timer_ns() - t0 > limit_ns)) return false;
  }
}

// One lane's wait for phase `parity` of `bar`, for at most `limit_ns` of the global timer (0: one
// non-blocking test).
__device__ __forceinline__ bool mbar_wait_lane(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  if (limit_ns == 0) return mbar_test(bar, parity);
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// A wait of the split kernels' stage ring under the call's limit (all lanes of a converged warp; the
// result is the same in every lane).  RING_OK: the phase completed within the limit.  RING_LATE: the
// wait passed the limit (PA_DEV_TIMEOUT is recorded) and the phase then completed within the drain
// limit; the warp gives up its work but keeps the ring's protocol (a producer issues no further
// stage, only the end marker, into that slot; a consumer computes nothing more but releases every
// later stage and meets every end-of-piece barrier up to the end marker), so no copy is left in
// flight and no barrier waits for a warp that has left.  RING_FAILED: the drain limit passed too.
enum RingWait { RING_OK = 0, RING_LATE = 1, RING_FAILED = 2 };
__device__ __forceinline__ int ring_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns, uint32_t *status) {
  if (__all_sync(FULL, mbar_wait_lane(bar, parity, limit_ns))) return RING_OK;
  if ((threadIdx.x & 31) == 0) atomicOr(status, PA_DEV_TIMEOUT);
  __syncwarp();
  return mbar_wait_warp(bar, parity, DRAIN_LIMIT_NS) ? RING_LATE : RING_FAILED;
}

// TMA: 4-D tiled copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            int c3, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// TMA: 5-D tiled copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            int c3, int c4, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(bar))
      : "memory");
}

// TMA: 2-D tiled copy global -> shared.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// TMA: 3-D tiled copy global -> shared.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Named barrier among `count` threads (multiple of 32) of the CTA.
__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// 2^x on the SFU (ex2.approx, flush-to-zero); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ldmatrix: four 8x8 b16 matrices; lane 8i + r gives the shared address of row r of matrix i.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte permute: byte i of the result is byte ((sel >> 4 i) & 7) of the pair {hi:lo}.
__device__ __forceinline__ uint32_t prmt(uint32_t lo, uint32_t hi, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(lo), "r"(hi), "r"(sel));
  return r;
}

__device__ __forceinline__ uint2 lds_u2(uint32_t addr) {
  uint2 r;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(addr));
  return r;
}

// Two fp32 -> one bf16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Programmatic dependent launch: wait for the preceding grid / let the next one start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

}  // namespace pa
