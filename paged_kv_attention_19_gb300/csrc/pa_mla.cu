// pa_mla.cu -- MLA absorbed decode (sm_103a): the call sequence and the two projections.
//
// What is computed follows pegainfer PR #938 "warp-cooperative two-pass MLA absorbed
// decode kernel" (Schedule section, steps 1-7) and the vllm.cpp kernel-matrix row
// KERNEL-ATTN-MLA-SPARSE (absorption = two batched contractions around a split-KV decode
// with a fixed ascending merge):
//   1. q_abs = bf16(q_nope . W_UK) || q_rope, and the rounding remainder q_lo  [q_absorb_kernel]
//   2-6. scores over the 576-wide latent || rope cache, online softmax,
//        o_lat = sum_t p_t c_t[0:512], per piece of the balanced partition
//                                                                   [mla_tc_split_kernel]
//   merge of split sequences, ascending, o_lat rounded to bf16, and
//   7. o = W_UV . o_lat; lse += scale * q_lo . o_lat                [mla_uv_kernel]
// Differences from the pages' kernel, all deliberate: scores, probabilities and the
// softmax state stay fp32; the context is walked once with an online max instead of
// twice.  q_lat enters the tensor-core scores rounded to bf16; the rounding's first-order
// effect on the LSE (scale * q_lo . o_lat, up to ~1e-3 for short rows) is added back in step
// 7, its effect on o_lat stays within the output tolerance.  o_lat is rounded to bf16 as the
// operand of step 7.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "pa_gqa_launch.cuh"
#include "pa_mla.h"
#include "pa_mla_tc.cuh"

namespace pa {

constexpr int MLA_NOPE = 128, MLA_QD = 192, MLA_LAT = 512, MLA_C = 576, MLA_V = 128;

// Activation rows in shared memory are padded to 520 bf16 (1040 bytes): the 16-byte offset
// between consecutive rows keeps fragment loads free of bank conflicts.
constexpr int WROW = MLA_LAT + 8;
// Projection weights arrive by TMA in boxes of 64 columns (128 bytes) with the 128-byte swizzle:
// a plane holds one box, rows of 128 bytes, the 16-byte chunk c of row r at c ^ (r & 7).
// q_absorb stages a head's W_UK column quarter (128 rows x 128 columns: 2 planes of 16 KB),
// mla_uv a head's W_UV row half (64 rows x 512 columns: 8 planes of 8 KB).
constexpr int ABS_PARTS = 4, UV_PARTS = 2;
constexpr int ABS_COLS = MLA_LAT / ABS_PARTS;  // 128 latent columns per absorb block
constexpr int UV_ROWS = MLA_V / UV_PARTS;      // 64 output dims per projection block
constexpr int ABS_PLANE = 128 * 128, UV_PLANE = UV_ROWS * 128;
constexpr int ABS_W = (ABS_COLS / 64) * ABS_PLANE;  // 32 KB
constexpr int UV_W = (MLA_LAT / 64) * UV_PLANE;      // 64 KB
// alignment, weights, rows, barrier: each projection kernel asks for its own size, so that the
// absorb kernel's 512 blocks fit 4 to an SM (one wave)
constexpr int ABS_SMEM = 1024 + ABS_W + 16 * WROW * 2 + 16;
constexpr int UV_SMEM = 1024 + UV_W + 16 * WROW * 2 + 16;

// Byte offset of (row, col) in staged weights with planes of `plane` bytes (col a multiple of 8).
__device__ __forceinline__ uint32_t wsw(int plane, int row, int col) {
  return (uint32_t)((col >> 6) * plane + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4));
}

// The projection kernels' weight planes start on a 1024-byte boundary (the swizzle pattern
// repeats every 1024 bytes).
__device__ __forceinline__ uint8_t *proj_weights(uint8_t *raw) {
  return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

// Thread 0 initialises *bar and issues n_box copies of the box at (x0 + 64 i, y) into planes of
// `plane` bytes at w; completion counted on *bar.
__device__ __forceinline__ void stage_weights_issue(uint8_t *w, const CUtensorMap *map, int x0, int y, int n_box,
                                                    int plane, uint64_t *bar) {
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, (uint32_t)(n_box * plane));
    for (int i = 0; i < n_box; ++i) tma_load_2d(w + i * plane, map, x0 + 64 * i, y, bar);
  }
}

// q_lat[b][h][j] = sum_d q_nope[b][h][d] * W_UK[h][d][j] (fp32): q_abs[b][h] = bf16(q_lat) ||
// q_rope (576) and q_lo[b][h] = bf16(q_lat - bf16(q_lat)) (512, for the LSE term of the
// projection kernel).  Block (h, part) of 8 warps computes latent columns [128 part, +128) of
// head h from its W_UK quarter (128 x 128, staged by TMA); the batch rows (16 per tile) are the
// M dimension of m16n8k16 MMAs, warp w producing columns [16 w, 16 w + 16) of the quarter.
__global__ void __launch_bounds__(256) q_absorb_kernel(const __grid_constant__ CUtensorMap tm_w, const uint16_t *q,
                                                       uint16_t *q_abs, uint16_t *q_lo, int B, int H,
                                                       uint32_t *status) {
  extern __shared__ __align__(1024) uint8_t psmem[];
  uint8_t *w = proj_weights(psmem);                                  // W_UK[h][:, quarter]
  uint16_t *qn = reinterpret_cast<uint16_t *>(w + ABS_W);            // [16 rows][WROW] (first 128 used)
  uint64_t *bar = reinterpret_cast<uint64_t *>(qn + 16 * WROW);
  pdl_launch_dependents();  // the split kernel may start its prologue; it waits for q_abs
  const int h = blockIdx.x / ABS_PARTS, part = blockIdx.x % ABS_PARTS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int lm_mat = lane >> 3, lm_row = lane & 7;
  stage_weights_issue(w, &tm_w, part * ABS_COLS, h * MLA_NOPE, ABS_COLS / 64, ABS_PLANE, bar);
  if (part == 0) {
    // the rope part is copied as it is (8 vectors of 16 bytes per row)
    for (int i = tid; i < B * 8; i += 256) {
      const int b = i >> 3, c = i & 7;
      *reinterpret_cast<uint4 *>(q_abs + ((size_t)b * H + h) * MLA_C + MLA_LAT + c * 8) =
          *reinterpret_cast<const uint4 *>(q + ((size_t)b * H + h) * MLA_QD + MLA_NOPE + c * 8);
    }
  }
  for (int m0 = 0; m0 < B; m0 += 16) {
    for (int i = tid; i < 16 * (MLA_NOPE / 8); i += 256) {
      const int r = i / (MLA_NOPE / 8), c = i % (MLA_NOPE / 8);
      const int b = m0 + r;
      *reinterpret_cast<uint4 *>(qn + r * WROW + c * 8) =
          b < B ? *reinterpret_cast<const uint4 *>(q + ((size_t)b * H + h) * MLA_QD + c * 8) : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    // the weights have landed (a wait that gave up ends every thread of the block together)
    if (m0 == 0 && !__syncthreads_and(mbar_wait(bar, 0, status))) return;
    float acc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < MLA_NOPE; k0 += 16) {
      uint32_t af[4], bf[4];
      {
        const int row = (lm_mat & 1) * 8 + lm_row, col = k0 + (lm_mat >> 1) * 8;
        ldmatrix_x4(af, smem_u32(qn + row * WROW + col));
      }
      {
        // W rows k0..k0+15 (k), columns 16 warp .. + 16 of the quarter (two n-tiles), transposed
        const int krow = k0 + (lm_mat & 1) * 8 + lm_row, col = warp * 16 + (lm_mat >> 1) * 8;
        ldmatrix_x4_trans(bf, smem_u32(w) + wsw(ABS_PLANE, krow, col));
      }
      mma_bf16_16816(acc[0], af, bf[0], bf[1]);
      mma_bf16_16816(acc[1], af, bf[2], bf[3]);
    }
    const int r0 = m0 + g, r1 = m0 + g + 8;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = part * ABS_COLS + warp * 16 + nt * 8 + 2 * tq;
      const uint32_t h0 = pack_bf16x2(acc[nt][0], acc[nt][1]), h1 = pack_bf16x2(acc[nt][2], acc[nt][3]);
      const uint32_t l0 = pack_bf16x2(acc[nt][0] - __uint_as_float(h0 << 16), acc[nt][1] - __uint_as_float(h0 & 0xffff0000u));
      const uint32_t l1 = pack_bf16x2(acc[nt][2] - __uint_as_float(h1 << 16), acc[nt][3] - __uint_as_float(h1 & 0xffff0000u));
      if (r0 < B) {
        *reinterpret_cast<uint32_t *>(q_abs + ((size_t)r0 * H + h) * MLA_C + col) = h0;
        *reinterpret_cast<uint32_t *>(q_lo + ((size_t)r0 * H + h) * MLA_LAT + col) = l0;
      }
      if (r1 < B) {
        *reinterpret_cast<uint32_t *>(q_abs + ((size_t)r1 * H + h) * MLA_C + col) = h1;
        *reinterpret_cast<uint32_t *>(q_lo + ((size_t)r1 * H + h) * MLA_LAT + col) = l1;
      }
    }
    __syncthreads();
  }
}

// Arguments of the merge + projection kernel.
struct MlaUvArgs {
  const uint16_t *o_lat;       // [B, 2, H, 256] bf16: halves of o_lat written whole by the split kernel
  const float *part_o;         // [nparts, 2, rs, 256] fp32 partials (normalised) of split sequences
  const float *part_lse;       // [nparts, 2, rs] fp32, log2 units
  const int32_t *seq_first;    // [B, ntile]: -1 whole; else 2 x CTA + slot of the sequence's first piece
  const int32_t *seq_last;     // [B, ntile]: CTA holding its last piece
  const GqaPartDesc *desc;     // [nparts]: status bits of every split CTA
  const int32_t *context_lens;  // [B]
  const uint16_t *q_lo;        // [B, H, 512] bf16: q_lat - bf16(q_lat)
  uint16_t *out;               // [B, H, 128] bf16
  float *lse;                  // [B, H] or null
  uint32_t *status;            // the workspace status word: OR of every CTA's bits
  float scale;
  int B, H, ntile, rs, nparts, hg, max_context_len;
};

// Distributed shared memory of the 2-CTA cluster of the projection kernel.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of this CTA's shared-memory location `local` in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void dsmem_st_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
// All threads of both CTAs: writes before it (shared memory of either CTA) are visible after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Merge of split sequences fused with step 7.  The two blocks (h, part 0) and (h, part 1) of head
// h form a 2-CTA cluster; block part computes o[b][h][v] = sum_j W_UV[h][v][j] o_lat[b][h][j] for
// v in [64 part, +64), 16 batch rows per tile:
//   * before the wait for the split kernel, its W_UV half (64 x 512) is requested by TMA;
//   * o_lat of the tile's 16 rows is assembled as bf16 in both blocks' shared memory, each block
//     producing column half `part` (the sequence (row, tile, half)) and storing it into its own
//     and its partner's shared memory.  A half that one piece covered whole is copied from the
//     split kernel's output; a split one is merged from its fp32 partials (slots of CTAs first,
//     first + hg, ..., last: the sequence's pieces in ascending token order) as an online
//     log-sum-exp merge.  Lane l of warp w owns columns [8 l, +8) of rows w and w + 8, and the
//     loop over partials is outermost, so both rows' loads of a partial (its LSE and values
//     together) are in flight at once;
//   * warp w produces v in [8 w, 8 w + 8) of the half on m16n8k16 MMAs (batch rows as M);
//   * part 0 (which merges column half 0) writes the LSE: the merged one (or the split kernel's,
//     for a whole sequence) plus the first-order term of q_lat's bf16 rounding,
//     scale * (q_lo . o_lat); q_lo and the split kernel's LSE are loaded beside the table lookup.
// Every path through the tile loop passes the same two cluster barriers per tile, so neither block
// waits for one that has left.  Sequence indices from the workspace are range-checked, so a stale
// or partial table never makes a load leave the partial slots.
__global__ void __launch_bounds__(256) mla_uv_kernel(const __grid_constant__ CUtensorMap tm_w, const MlaUvArgs a) {
  extern __shared__ __align__(1024) uint8_t psmem[];
  uint8_t *w = proj_weights(psmem);                                    // W_UV[h][half, :]
  uint16_t *ol = reinterpret_cast<uint16_t *>(w + UV_W);               // [16 rows][WROW]
  uint64_t *bar = reinterpret_cast<uint64_t *>(ol + 16 * WROW);
  __shared__ int32_t s_first[16], s_k[16];  // -1: whole (copy); else 2 x CTA + slot, piece count
  __shared__ float s_lse[16];               // merged LSE (natural log) of split rows; NaN: whole
  const int h = blockIdx.x / UV_PARTS, part = blockIdx.x % UV_PARTS;
  const uint32_t peer = cluster_ctarank() ^ 1u;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int lm_mat = lane >> 3, lm_row = lane & 7;
  const int H = a.H;
  const int rh_head = h % MlaTcCfg::M;         // row of head h in its tile's partial slots
  const int hs = (h / MlaTcCfg::M) * 2 + part;  // the sequence index of column half `part` of head h
  stage_weights_issue(w, &tm_w, 0, h * MLA_V + part * UV_ROWS, MLA_LAT / 64, UV_PLANE, bar);
  __syncthreads();  // the barrier is initialised before any thread waits on it
  pdl_wait();  // the split kernel's outputs, partials, tables and status are final from here on
  if (blockIdx.x == 0 && warp == 0) {
    uint32_t st = 0;
    for (int i = lane; i < a.nparts; i += 32) st |= a.desc[i].status;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) st |= __shfl_xor_sync(FULL, st, o);
    if (lane == 0) *a.status = st;
  }
  const bool do_lse = a.lse && part == 0;
  bool weights_ready = false, ok = true;
  for (int m0 = 0; m0 < a.B; m0 += 16) {
    // ---- where each row's sequence is (one thread per row; the three table loads are
    // independent).  Meanwhile part 0 loads q_lo and the split kernel's LSE of its two rows.
    if (tid < 16) {
      const int b = m0 + tid;
      int first = -1, k = 0;
      if (b < a.B) {
        const size_t si = (size_t)b * a.ntile + hs;
        const int L = a.context_lens[b], f = a.seq_first[si], cl = a.seq_last[si];
        const int c0 = f >> 1;
        if (clamp_len(L, a.max_context_len) > 0 && f >= 0 && c0 < a.nparts && cl >= c0 && cl < a.nparts &&
            (cl - c0) % a.hg == 0) {
          first = f;
          k = (cl - c0) / a.hg + 1;
        }
      }
      s_first[tid] = first;
      s_k[tid] = k;
    }
    uint4 qlo[2][2];  // part 0, warp w: rows 2 w, 2 w + 1; lane l: dims [16 l, 16 l + 16)
    float lse_split[2];
    if (do_lse) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int b = m0 + warp * 2 + q;
        lse_split[q] = -INFINITY;
        qlo[q][0] = qlo[q][1] = make_uint4(0, 0, 0, 0);
        if (b < a.B) {
          const uint16_t *ql = a.q_lo + ((size_t)b * H + h) * MLA_LAT + lane * 16;
          qlo[q][0] = *reinterpret_cast<const uint4 *>(ql);
          qlo[q][1] = *reinterpret_cast<const uint4 *>(ql + 8);
          if (lane == 0) lse_split[q] = a.lse[(size_t)b * H + h];
        }
      }
    }
    __syncthreads();
    // ---- column half `part` of o_lat of the tile, into both blocks' shared memory
    {
      constexpr int NI = 2;
      int fi[NI], ki[NI];
      float mi[NI], zi[NI], acc[NI][8];
      int kmax = 0;
#pragma unroll
      for (int n = 0; n < NI; ++n) {
        const int r = warp + 8 * n;
        fi[n] = m0 + r < a.B ? s_first[r] : -1;
        ki[n] = fi[n] >= 0 ? s_k[r] : 0;
        kmax = max(kmax, ki[n]);
        mi[n] = -INFINITY;
        zi[n] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[n][e] = 0.f;
      }
#pragma unroll 2
      for (int i = 0; i < kmax; ++i) {
#pragma unroll
        for (int n = 0; n < NI; ++n) {
          if (i < ki[n]) {
            const int f = fi[n];
            const size_t pi = i == 0 ? (size_t)f : (size_t)((f >> 1) + i * a.hg) * 2;
            const float l = a.part_lse[pi * a.rs + rh_head];
            const float *po = a.part_o + (pi * a.rs + rh_head) * MlaTcCfg::DVH + lane * 8;
            const float4 x0 = *reinterpret_cast<const float4 *>(po);
            const float4 x1 = *reinterpret_cast<const float4 *>(po + 4);
            if (l != -INFINITY) {  // a partial with no attended key weighs nothing
              const float mn = fmaxf(mi[n], l);
              const float sc = mi[n] == -INFINITY ? 0.f : fast_exp2(mi[n] - mn);
              const float wc = fast_exp2(l - mn);
              mi[n] = mn;
              zi[n] = zi[n] * sc + wc;
              acc[n][0] = acc[n][0] * sc + wc * x0.x;
              acc[n][1] = acc[n][1] * sc + wc * x0.y;
              acc[n][2] = acc[n][2] * sc + wc * x0.z;
              acc[n][3] = acc[n][3] * sc + wc * x0.w;
              acc[n][4] = acc[n][4] * sc + wc * x1.x;
              acc[n][5] = acc[n][5] * sc + wc * x1.y;
              acc[n][6] = acc[n][6] * sc + wc * x1.z;
              acc[n][7] = acc[n][7] * sc + wc * x1.w;
            }
          }
        }
      }
#pragma unroll
      for (int n = 0; n < NI; ++n) {
        const int r = warp + 8 * n, b = m0 + r;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (b < a.B) {
          if (fi[n] < 0) {
            v = *reinterpret_cast<const uint4 *>(a.o_lat + (((size_t)b * 2 + part) * H + h) * MlaTcCfg::DVH + lane * 8);
            if (lane == 0) s_lse[r] = NAN;
          } else {
            const float inv = zi[n] > 0.f ? 1.f / zi[n] : 0.f;
            v.x = pack_bf16x2(acc[n][0] * inv, acc[n][1] * inv);
            v.y = pack_bf16x2(acc[n][2] * inv, acc[n][3] * inv);
            v.z = pack_bf16x2(acc[n][4] * inv, acc[n][5] * inv);
            v.w = pack_bf16x2(acc[n][6] * inv, acc[n][7] * inv);
            if (lane == 0)
              s_lse[r] = (mi[n] == -INFINITY || zi[n] == 0.f) ? -INFINITY : (mi[n] + __log2f(zi[n])) * LN2;
          }
        }
        uint16_t *dst = ol + r * WROW + part * MlaTcCfg::DVH + lane * 8;
        *reinterpret_cast<uint4 *>(dst) = v;
        dsmem_st_v4(dsmem_addr(smem_u32(dst), peer), v);
      }
    }
    cluster_sync();  // both column halves of the tile are in both blocks' shared memory
    if (!weights_ready) {
      // the weights have landed (a wait that gave up makes the whole block skip its output)
      ok = __syncthreads_and(mbar_wait(bar, 0, a.status));
      weights_ready = true;
    }
    if (ok && do_lse) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int r = warp * 2 + q, b = m0 + r;
        if (b >= a.B) break;
        const uint32_t qw[8] = {qlo[q][0].x, qlo[q][0].y, qlo[q][0].z, qlo[q][0].w,
                                qlo[q][1].x, qlo[q][1].y, qlo[q][1].z, qlo[q][1].w};
        float d = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t ow = *reinterpret_cast<const uint32_t *>(ol + r * WROW + lane * 16 + 2 * i);
          d += __uint_as_float(qw[i] << 16) * __uint_as_float(ow << 16) +
               __uint_as_float(qw[i] & 0xffff0000u) * __uint_as_float(ow & 0xffff0000u);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(FULL, d, o);
        if (lane == 0) {
          const float merged = s_lse[r];
          const float l = isnan(merged) ? lse_split[q] : merged;  // a whole sequence's LSE is the split kernel's
          a.lse[(size_t)b * H + h] = l == -INFINITY ? l : l + a.scale * d;
        }
      }
    }
    if (ok) {
      // two accumulators (even and odd k-steps): two independent MMA chains
      float acc[2][4];
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[q2][e] = 0.f;
#pragma unroll 4
      for (int k0 = 0; k0 < MLA_LAT; k0 += 32) {
        uint32_t af0[4], af1[4], bf[4];
        {
          const int row = (lm_mat & 1) * 8 + lm_row, col = k0 + (lm_mat >> 1) * 8;
          ldmatrix_x4(af0, smem_u32(ol + row * WROW + col));
          ldmatrix_x4(af1, smem_u32(ol + row * WROW + col + 16));
        }
        {
          // B = W_UV^T: W rows v (the n index, 8 of them), columns k0 .. k0 + 31 (two k-steps)
          const int vrow = warp * 8 + lm_row, col = k0 + lm_mat * 8;
          ldmatrix_x4(bf, smem_u32(w) + wsw(UV_PLANE, vrow, col));
        }
        mma_bf16_16816(acc[0], af0, bf[0], bf[1]);
        mma_bf16_16816(acc[1], af1, bf[2], bf[3]);
      }
      const int r0 = m0 + g, r1 = m0 + g + 8;
      const int col = part * UV_ROWS + warp * 8 + 2 * tq;
      if (r0 < a.B)
        *reinterpret_cast<uint32_t *>(a.out + ((size_t)r0 * H + h) * MLA_V + col) =
            pack_bf16x2(acc[0][0] + acc[1][0], acc[0][1] + acc[1][1]);
      if (r1 < a.B)
        *reinterpret_cast<uint32_t *>(a.out + ((size_t)r1 * H + h) * MLA_V + col) =
            pack_bf16x2(acc[0][2] + acc[1][2], acc[0][3] + acc[1][3]);
    }
    cluster_sync();  // both blocks are done reading the tile before the next one is written
  }
}

// ----------------------------------------------------------------------------- host side
namespace {

constexpr int kMaxSplits = 4096;                 // largest accepted explicit num_splits (shares)
constexpr int kAutoPartsMax = 256;               // automatic mode: one share per SM, at most this many
constexpr long long kPieceCostBytes = 64 << 10;  // fixed cost of one piece, as cache bytes streamed meanwhile

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int ilog2(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct MlaPlan {
  int ntile, rs, nparts_max;
  size_t off_desc, off_part_lse, off_part_o, off_qabs, off_qlo, off_olat, off_seq, total;
};

// The workspace: header, one descriptor per share, two fp32 partial slots (min(H, 128) heads x 256
// columns) per share, q_abs [B, H, 576], q_lo [B, H, 512] and o_lat [B, 2, H, 256], all bf16, and
// the two int32 tables [B, ntile] that say where each sequence's pieces are.
int mla_shape(int batch, int H, int max_ctx, int P, int num_splits, MlaPlan *pl) {
  if (batch < 0 || H <= 0 || max_ctx < 0 || num_splits < 0) return PA_ERR_INVALID_ARGUMENT;
  if (num_splits > kMaxSplits) return PA_ERR_UNSUPPORTED;
  if (!is_pow2(P) || P < 8 || P > 256) return PA_ERR_UNSUPPORTED;  // a TMA box starts on 1024 bytes
  pl->ntile = 2 * ((H + MlaTcCfg::M - 1) / MlaTcCfg::M);  // (head tile, column half) per row
  pl->rs = H < MlaTcCfg::M ? H : MlaTcCfg::M;
  pl->nparts_max = num_splits > 0 ? num_splits : kAutoPartsMax;
  const size_t np = (size_t)pl->nparts_max, B = (size_t)(batch > 0 ? batch : 1);
  size_t off = sizeof(WsHeader);
  pl->off_desc = off;
  off = round_up(off + np * sizeof(GqaPartDesc), 256);
  pl->off_part_lse = off;
  off = round_up(off + np * 2 * pl->rs * sizeof(float), 256);
  pl->off_part_o = off;
  off = round_up(off + np * 2 * pl->rs * (size_t)MlaTcCfg::DVH * sizeof(float), 256);
  pl->off_qabs = off;
  off = round_up(off + B * (size_t)H * MLA_C * 2, 256);
  pl->off_qlo = off;
  off = round_up(off + B * (size_t)H * MLA_LAT * 2, 256);
  pl->off_olat = off;
  off = round_up(off + B * (size_t)H * MLA_LAT * 2, 256);
  pl->off_seq = off;
  off = round_up(off + 2 * B * (size_t)pl->ntile * sizeof(int32_t), 256);
  pl->total = off;
  return PA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 mla_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D map over the cache [num_pages, P, 576] bf16; box = (64 dims, BH tokens, 1 page), 128-byte swizzle.
bool encode_cache_map(CUtensorMap *m, const void *base, int num_pages, int P, int BH) {
  auto fn = mla_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)MLA_C, (cuuint64_t)P, (cuuint64_t)num_pages};
  cuuint64_t strides[2] = {(cuuint64_t)MLA_C * 2, (cuuint64_t)P * MLA_C * 2};
  cuuint32_t box[3] = {64u, (cuuint32_t)BH, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over projection weights viewed as [H * 128 rows, 512] bf16; box = (64 columns,
// box_rows rows), 128-byte swizzle.
bool encode_weight_map(CUtensorMap *m, const void *base, int H, int box_rows) {
  auto fn = mla_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)MLA_LAT, (cuuint64_t)H * 128};
  cuuint64_t strides[1] = {(cuuint64_t)MLA_LAT * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over q_abs [rows, 576] bf16; box = (64 dims, 128 rows: one head tile), 128-byte swizzle.
bool encode_qabs_map(CUtensorMap *m, const void *base, long long rows) {
  auto fn = mla_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)MLA_C, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)MLA_C * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)MlaTcCfg::M};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count_mla() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return n;
}

}  // namespace

size_t mla_workspace_size(int batch, int num_heads, int max_context_len, int page_size, int num_splits) {
  MlaPlan pl;
  if (mla_shape(batch, num_heads, max_context_len, page_size, num_splits, &pl) != PA_OK) return 0;
  return pl.total;
}

int mla_decode(const void *q, const void *cache, const void *w_uk, const void *w_uv, const int32_t *block_table,
               const int32_t *context_lens, void *out, float *lse, int batch, int H, int page_size, int num_pages,
               int max_pages_per_seq, int max_context_len, float scale, int num_splits, void *workspace,
               size_t workspace_bytes, cudaStream_t stream, cudaEvent_t ev_before, cudaEvent_t ev_after,
               int *launches) {
  using C = MlaTcCfg;
  *launches = 0;
  if (batch == 0) return PA_OK;
  MlaPlan pl;
  int rc = mla_shape(batch, H, max_context_len, page_size, num_splits, &pl);
  if (rc != PA_OK) return rc;
  if (!q || !cache || !w_uk || !w_uv || !block_table || !context_lens || !out || !workspace)
    return PA_ERR_INVALID_ARGUMENT;
  if (num_pages <= 0 || max_pages_per_seq <= 0 || !std::isfinite(scale)) return PA_ERR_INVALID_ARGUMENT;
  if ((long long)max_pages_per_seq * page_size < (long long)max_context_len) return PA_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(cache, 16) || !aligned(w_uk, 16) || !aligned(w_uv, 16) || !aligned(out, 16) ||
      !aligned(workspace, 16) || !aligned(block_table, 4) || !aligned(context_lens, 4) || (lse && !aligned(lse, 4)))
    return PA_ERR_MISALIGNED;
  if (workspace_bytes < pl.total) return PA_ERR_WORKSPACE_TOO_SMALL;
  const int P = page_size;
  const int BH = P < C::ST ? P : C::ST;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  uint16_t *q_abs = reinterpret_cast<uint16_t *>(ws + pl.off_qabs);
  uint16_t *o_lat = reinterpret_cast<uint16_t *>(ws + pl.off_olat);
  uint16_t *q_lo = reinterpret_cast<uint16_t *>(ws + pl.off_qlo);
  int32_t *seq_first = reinterpret_cast<int32_t *>(ws + pl.off_seq);
  int32_t *seq_last = seq_first + (size_t)batch * pl.ntile;
  CUtensorMap tm_c, tm_q, tm_wuk, tm_wuv;
  if (!encode_cache_map(&tm_c, cache, num_pages, P, BH) || !encode_qabs_map(&tm_q, q_abs, (long long)batch * H) ||
      !encode_weight_map(&tm_wuk, w_uk, H, MLA_NOPE) || !encode_weight_map(&tm_wuv, w_uv, H, UV_ROWS))
    return PA_ERR_UNSUPPORTED;
  const int sms = sm_count_mla();
  if (sms <= 0) return pa::cuda_fail(cudaSuccess);
  const int nparts = num_splits > 0 ? num_splits : (sms < kAutoPartsMax ? sms : kAutoPartsMax);

  WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
  GqaPartDesc *desc = reinterpret_cast<GqaPartDesc *>(ws + pl.off_desc);
  float *part_lse = reinterpret_cast<float *>(ws + pl.off_part_lse);
  float *part_o = reinterpret_cast<float *>(ws + pl.off_part_o);

  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    for (const void *k :
         {(const void *)mla_tc_split_kernel, (const void *)q_absorb_kernel, (const void *)mla_uv_kernel}) {
      const int bytes = k == (const void *)mla_tc_split_kernel ? MlaTcSmem::BYTES
                        : k == (const void *)q_absorb_kernel  ? ABS_SMEM
                                                               : UV_SMEM;
      if (const cudaError_t ce = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
          ce != cudaSuccess)
        return pa::cuda_fail(ce);
    }
    configured_device = dev;
  }

  // 1. q_abs
  q_absorb_kernel<<<H * ABS_PARTS, 256, ABS_SMEM, stream>>>(tm_wuk, static_cast<const uint16_t *>(q), q_abs, q_lo, batch, H,
                                                  &hdr->status);
  if (const cudaError_t ce = cudaGetLastError(); ce != cudaSuccess) return pa::cuda_fail(ce);
  ++*launches;

  // 2-6. the attention core
  MlaTcArgs ma;
  ma.block_table = block_table;
  ma.context_lens = context_lens;
  ma.o_lat = o_lat;
  ma.lse = lse;
  ma.part_o = part_o;
  ma.part_lse = part_lse;
  ma.desc = desc;
  ma.seq_first = seq_first;
  ma.seq_last = seq_last;
  ma.batch = batch;
  ma.max_pages_per_seq = max_pages_per_seq;
  ma.num_pages = num_pages;
  ma.max_context_len = max_context_len;
  ma.H = H;
  ma.ntile = pl.ntile;
  ma.rs = pl.rs;
  ma.log2_page = ilog2(P);
  ma.log2_bh = ilog2(BH);
  {
    const long long unit_bytes = (long long)BH * MLA_C * 2;
    ma.piece_cost = (int)((kPieceCostBytes + unit_bytes - 1) / unit_bytes);
  }
  ma.nparts = nparts;
  ma.hg = pl.ntile < nparts ? pl.ntile : nparts;
  ma.qscale = scale * LOG2E;
  if (ev_before) {
    if (const cudaError_t ce = cudaEventRecord(ev_before, stream); ce != cudaSuccess) return pa::cuda_fail(ce);
  }
  {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(nparts), dim3(C::THREADS), MlaTcSmem::BYTES, stream, attr);
    if (const cudaError_t ce = cudaLaunchKernelEx(&cfg, mla_tc_split_kernel, tm_c, tm_q, ma); ce != cudaSuccess) return pa::cuda_fail(ce);
  }
  ++*launches;
  if (ev_after) {
    if (const cudaError_t ce = cudaEventRecord(ev_after, stream); ce != cudaSuccess) return pa::cuda_fail(ce);
  }

  // merge of split sequences and 7. o = W_UV . o_lat
  {
    MlaUvArgs ua;
    ua.o_lat = o_lat;
    ua.part_o = part_o;
    ua.part_lse = part_lse;
    ua.seq_first = seq_first;
    ua.seq_last = seq_last;
    ua.desc = desc;
    ua.context_lens = context_lens;
    ua.q_lo = q_lo;
    ua.out = static_cast<uint16_t *>(out);
    ua.lse = lse;
    ua.status = &hdr->status;
    ua.scale = scale;
    ua.B = batch;
    ua.H = H;
    ua.ntile = pl.ntile;
    ua.rs = pl.rs;
    ua.nparts = nparts;
    ua.hg = ma.hg;
    ua.max_context_len = max_context_len;
    // the two blocks of a head form a cluster (they share the merged o_lat through distributed
    // shared memory); a programmatic dependent of the split kernel like every launch here
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pdl_config(dim3(H * UV_PARTS), dim3(256), UV_SMEM, stream, attr);
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = UV_PARTS;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
    if (const cudaError_t ce = cudaLaunchKernelEx(&cfg, mla_uv_kernel, tm_wuv, ua); ce != cudaSuccess)
      return pa::cuda_fail(ce);
  }
  ++*launches;
  return PA_OK;
}

}  // namespace pa
