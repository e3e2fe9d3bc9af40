// pa_tcgen05.cuh -- the 5th-generation tensor-core instructions (sm_100a / sm_103a) used by the
// MLA attention core: tensor-memory allocation, MMAs with shared-memory and tensor-memory
// operands, completion tracking through mbarriers, tensor-memory loads and stores.
//
// Operand encodings (PTX ISA, tcgen05 "Matrix descriptors" and "Instruction descriptor"):
//  * shared-memory descriptor, 64 bits: start address >> 4 in bits 0-13, leading-dimension byte
//    offset (LBO) >> 4 in bits 16-29, stride-dimension byte offset (SBO) >> 4 in bits 32-45, the
//    fixed value 1 in bits 46-47, base offset 0 in bits 49-51 (every swizzle atom here starts on
//    a 1024-byte boundary), swizzle mode in bits 61-63 (2 = 128-byte swizzle).  With the 128-byte
//    swizzle a row of the operand is 128 bytes and 8 rows form a 1024-byte atom:
//      - K-major (a row holds 64 consecutive K values of one M or N index): SBO = 1024, the
//        distance between 8-row groups; LBO is not used; a K step of 16 bf16 moves the start
//        address by 32 bytes inside the atom.
//      - MN-major (a row holds 64 consecutive M or N values of one K index): LBO = the distance
//        between blocks of 64 M or N values, SBO = 1024, the distance between groups of 8 K rows.
//  * instruction descriptor, 32 bits, kind::f16: D format in bits 4-5 (1 = fp32), A and B formats
//    in bits 7-9 and 10-12 (1 = bf16), A and B major-ness in bits 15 and 16 (1 = MN-major), N >> 3
//    in bits 17-22, M >> 4 in bits 24-28.
// Tensor memory: an address is lane << 16 | column.  The accumulator of an M = 128 MMA holds row i
// in lane i, one fp32 per column.  An A operand read from tensor memory holds two bf16 per column,
// the even K index in the low half.  Warp w of the CTA reaches lanes [32 (w % 4), +32).
//
// These encodings were checked on a GB300 against an fp64 product: a 128 x 576 by 576 x 32 score
// MMA with both operands K-major, a 128 x 32 by 32 x 256 product with B MN-major and A from
// shared memory or from tensor memory, and an A operand copied into tensor memory by tcgen05.cp.
#pragma once

#include <cstdint>

#include "pa_common.cuh"

namespace pa {

__host__ __device__ constexpr uint32_t tc_idesc_bf16(int m, int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ uint64_t tc_sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Warp-wide: ncols (a power of two >= 32) columns of all 128 lanes; the base address is written
// to *dst.  The permit to allocate is given up at once (one allocation per CTA).
__device__ __forceinline__ void tc_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Warp-wide: frees what tc_alloc allocated.
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (tensor memory) = A B (+ D if accumulate), A and B in shared memory.  One thread issues.
__device__ __forceinline__ void tc_mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (tensor memory) = A B (+ D if accumulate), A in tensor memory, B in shared memory.
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Copy of a 128-row x 32-byte matrix from shared memory (described like an MMA operand) into 8
// columns of all 128 lanes; a K-major bf16 operand lands in the layout an A operand read from
// tensor memory has (row i in lane i, two bf16 per column).  One thread issues.
__device__ __forceinline__ void tc_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// One arrival on *bar once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Ordering of tensor-memory accesses around thread synchronisation (barriers, mbarriers).
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Warp-wide: lane l of the warp reads 32 consecutive columns of tensor-memory lane (taddr.lane + l).
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Warp-wide: lane l writes 32 consecutive columns of tensor-memory lane (taddr.lane + l).
__device__ __forceinline__ void tc_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
      "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
      "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
      "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
      "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// Warp-wide: lane l writes 16 consecutive columns of tensor-memory lane (taddr.lane + l).
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&w)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]), "r"(w[9]),
      "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
      : "memory");
}

__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace pa
