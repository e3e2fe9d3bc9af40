// pa_gqa_f8.cuh -- GQA paged decode over an FP8 (E4M3) KV cache: the split-KV
// attention kernel (sm_103a).  The partition, the producer warp, the
// end-of-piece merge and the combine kernel are those of the bf16 kernel
// (pa_gqa.cuh); the consumer warps differ.
//
// What is computed: the decode of pa_gqa.cuh with keys E4M3(code) * k_scale and
// values E4M3(code) * v_scale (vllm.cpp kernel-matrix, row KERNEL-KV-QUANT,
// "FP8": the quantized form of the paged cache, one scale per pool).
//
// GB300 design of the consumers:
//   * a stage holds 32 KB of codes (128 tokens of K and V at head_dim 128), so
//     every byte moved carries twice the tokens of the bf16 kernel and the
//     consumers must run twice as fast per token;
//   * the roles of the MMA operands are swapped against the bf16 kernel: the
//     16 tokens of a group are the M rows and the tile's (head, position)
//     columns the N side (n-tiles of 8), S^T = K Q^T and O^T = V^T P^T.  A
//     group of 8 query heads (Qwen3-32B, Llama-3-8B decode) fills one n8 tile
//     instead of half an m16 tile, so the tensor work per token halves;
//   * the codes widen exactly to f16 in registers (cvt e4m3x2 -> f16x2) right
//     after ldmatrix: K by the plain fragment load with a permuted k order
//     (k slots 2t, 2t + 1 hold dims 4t, 4t + 1 and slots 2t + 8, 2t + 9 dims
//     4t + 2, 4t + 3, matched by the query fragments), V by ldmatrix.trans with
//     a byte permute (each lane then holds two tokens of an even and an odd
//     dim: the M rows of a 16-dim chunk are its even dims 0..7 and odd dims
//     8..15);
//   * the scores' fragment (token rows, column pairs) is turned into the P^T
//     operand (column rows, token pairs) by movmatrix.trans of f16 pairs;
//   * the query is rounded from bf16 to f16 (exact in f16's normal range) and
//     P to f16 as the MMA operand; scores, softmax and accumulation are fp32.
#pragma once

#include "pa_gqa.cuh"

namespace pa {

// NH8_: n-tiles of 8 columns per tile (1: at most 8 (head, position) pairs, 2: up to 16).
template <int D_, int NH8_>
struct GqaF8Cfg {
  static constexpr int D = D_;
  static constexpr bool F8 = true;                 // pools of E4M3 codes
  static constexpr int NH8 = NH8_;
  static constexpr int M = PART_HEADS;             // rows of a partial slot
  static constexpr int MR = 8 * NH8;               // rows per token group in the end-of-piece merge
  static constexpr int ST = D <= 128 ? 128 : 64;   // tokens per stage: 32 KB of K and V
  static constexpr int TW = 16 * NH8;              // tokens per token group (m-tiles of 16)
  static constexpr int NMT = TW / 16;
  static constexpr int TG = ST / TW;               // token groups per stage
  // warps sharing a token group, each owning D / DSPLIT of the P.V rows (and all computing
  // the group's scores); one except where a single warp's registers would not hold its rows
  static constexpr int DSPLIT = (D > 128 && NH8 == 2) ? 2 : 1;
  static constexpr int NCW = TG * DSPLIT;          // consumer warps
  static constexpr int THREADS = (NCW + 1) * 32;   // + producer warp
  static constexpr int CH = D / DSPLIT / 16;       // 16-dim chunks (M tiles of O^T) per warp
  static constexpr int NQ = D / 128;               // 128-byte swizzle planes along D (K, V)
  static constexpr int QNQ = D / 64;               // the same for the bf16 query rows
  static constexpr int PLANE = ST * 128;
  static constexpr int KV_BYTES = NQ * PLANE;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int NS = (229376 / STAGE_BYTES) < 16 ? (229376 / STAGE_BYTES) : 16;  // 224 KB ring
  static_assert(MR * D * 4 * TG <= STAGE_BYTES, "the end-of-piece merge fits the consumed stage");
  static_assert(QNQ * M * 128 <= STAGE_BYTES, "the query rows fit one stage");
  static_assert(D % 128 == 0, "FP8 rows are whole 128-byte planes");
};

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit values held as MMA fragments (lane (g, t): row g,
// columns 2t, 2t + 1) across the warp.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// Two E4M3 codes (bits 0-7: the low result half, bits 8-15: the high one) -> f16x2, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v & 0xffffu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// bf16x2 -> f16x2 (round to nearest even).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  const __half2 h = __floats2half2_rn(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
  return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// MQ: several query positions per row (verify).  NH8: see GqaF8Cfg.
template <int D, bool MQ, int NH8>
__global__ void __launch_bounds__(GqaF8Cfg<D, NH8>::THREADS, 1)
    gqa_f8_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_q, const GqaArgs a) {
  using C = GqaF8Cfg<D, NH8>;
  using S = GqaSmem<C>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
  uint64_t *empty = full + C::NS;
  StageMeta *meta = reinterpret_cast<StageMeta *>(smem + S::OFF_META);
  GqaMisc *misc = reinterpret_cast<GqaMisc *>(smem + S::OFF_MISC);
  uint32_t *status = &misc->status;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  PartitionArgs pargs;
  gqa_setup<C>(smem, &tm_k, &tm_v, &tm_q, a, pargs);

  if (warp == C::NCW) {
    gqa_produce<C>(smem, &tm_k, &tm_v, &tm_q, a, pargs);
  } else {
    // ------------------------------------------------------------ consumers
    const int ct = tid;
    const int g8 = lane >> 2, tq = lane & 3;          // fragment row / column pair
    const int lm_mat = lane >> 3, lm_row = lane & 7;  // ldmatrix: matrix / row this lane addresses
    const int tgrp = warp % C::TG;                    // token group of this warp
    const int dh = warp / C::TG;                      // which part of the P.V rows (dims) it owns
    const int wbase = tgrp * C::TW;                   // first stage token of this warp
    float *sm_ml = reinterpret_cast<float *>(smem + S::OFF_ML);
    const float TAU = 8.f;  // lazy rescale threshold (log2 units): a weight stays below 2^8
    const int bh_tokens = 1 << a.log2_bh;

    // B fragments of Q^T per 16-dim step: [step][n-tile][b0 = dims 4t, 4t + 1; b1 = 4t + 2, 4t + 3]
    uint32_t qb[D / 16][NH8][2];
    float acc[C::CH][NH8][4];  // O^T: [chunk][n-tile]: c0, c1 = even dim x columns 2t, 2t + 1; c2, c3 = odd dim
    float mc[NH8][2], lc[NH8][2];  // running max / sum of this lane's columns 8 n + 2 tq + {0, 1}
    bool cv[NH8][2];               // real column?
    int clo[NH8][2], chi[NH8][2];  // MQ: key bounds [lo, hi) of the column's position
#pragma unroll
    for (int n = 0; n < NH8; ++n)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        mc[n][i] = -INFINITY;
        lc[n][i] = 0.f;
        cv[n][i] = false;
        clo[n][i] = chi[n][i] = 0;
      }
    for (uint32_t j = 0;; ++j) {
      const int s = j % C::NS;
      if (!mbar_wait(&full[s], (j / C::NS) & 1, status)) break;
      const StageMeta &mt = meta[s];
      if (mt.end) break;
      const uint32_t kbase = smem_u32(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
      const uint32_t vbase = kbase + C::KV_BYTES;
      if (mt.first) {
        // a new piece: the columns' validity and bounds, the Q^T fragments (an 8-byte read of
        // the bf16 row of column g8 per 16-dim step, widened to f16), fresh softmax state
#pragma unroll
        for (int n = 0; n < NH8; ++n)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int c = 8 * n + 2 * tq + i;
            if constexpr (MQ) {
              const int iq = c / a.gt;
              cv[n][i] = iq < mt.nq && c % a.gt < mt.ghead;
              clo[n][i] = pos_lo(mt.L, a.Q, mt.i0 + iq, a.window);
              chi[n][i] = pos_hi(mt.L, a.Q, mt.i0 + iq);
            } else {
              cv[n][i] = c < mt.ghead;
            }
            mc[n][i] = -INFINITY;
            lc[n][i] = 0.f;
          }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
          for (int n = 0; n < NH8; ++n) {
            const int row = 8 * n + g8, chunk = 2 * ks + (tq >> 1);
            const uint2 r = lds_u2(kbase + (uint32_t)((chunk >> 3) * (C::M * 128) + (tq & 1) * 8 + row * 128 +
                                                      (((chunk & 7) ^ (row & 7)) << 4)));
            qb[ks][n][0] = bf16x2_to_f16x2(r.x);
            qb[ks][n][1] = bf16x2_to_f16x2(r.y);
          }
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
#pragma unroll
          for (int n = 0; n < NH8; ++n) acc[c][n][0] = acc[c][n][1] = acc[c][n][2] = acc[c][n][3] = 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        continue;
      }

      // ---- S^T = K Q^T: per m-tile of 16 tokens, fragment c0 / c1 = token g8 x columns 2t,
      // 2t + 1, c2 / c3 = token g8 + 8
      float sv[C::NMT][NH8][4];
#pragma unroll
      for (int m = 0; m < C::NMT; ++m)
#pragma unroll
        for (int n = 0; n < NH8; ++n) sv[m][n][0] = sv[m][n][1] = sv[m][n][2] = sv[m][n][3] = 0.f;
#pragma unroll
      for (int m = 0; m < C::NMT; ++m)
#pragma unroll
        for (int ks2 = 0; ks2 < D / 32; ++ks2) {
          // matrices: tokens 0-7 / 8-15 of the m-tile, 16-byte chunks 2 ks2 / 2 ks2 + 1
          uint32_t r[4];
          ldmatrix_x4(r, kbase + kv_off<C>(wbase + 16 * m + (lm_mat & 1) * 8 + lm_row, 2 * ks2 + (lm_mat >> 1)));
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t a4[4] = {e4m3x2_to_f16x2(r[2 * h]), e4m3x2_to_f16x2(r[2 * h + 1]),
                                    e4m3x2_to_f16x2(r[2 * h] >> 16), e4m3x2_to_f16x2(r[2 * h + 1] >> 16)};
#pragma unroll
            for (int n = 0; n < NH8; ++n) mma_f16_16816(sv[m][n], a4, qb[2 * ks2 + h][n][0], qb[2 * ks2 + h][n][1]);
          }
        }
      const bool masked = mt.masked;
      // scale, mask (invalid tokens and columns -> -inf)
#pragma unroll
      for (int m = 0; m < C::NMT; ++m)
#pragma unroll
        for (int n = 0; n < NH8; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            bool valid = cv[n][e & 1];
            if (masked) {
              const int stok = wbase + 16 * m + g8 + (e >> 1) * 8;
              const int ltok = mt.tok0 + stok;
              valid = valid && ltok >= mt.tok_lo && ltok < mt.tok_hi && !((mt.badmask >> (stok / bh_tokens)) & 1u);
              if constexpr (MQ) valid = valid && ltok >= clo[n][e & 1] && ltok < chi[n][e & 1];
            }
            sv[m][n][e] = valid ? sv[m][n][e] * a.qscale : -INFINITY;
          }
      // ---- online softmax per column: max over the tokens of this lane, then over g8
      float x[NH8][2];
      bool up = false;
#pragma unroll
      for (int n = 0; n < NH8; ++n)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          float v = -INFINITY;
#pragma unroll
          for (int m = 0; m < C::NMT; ++m) v = fmaxf(v, fmaxf(sv[m][n][i], sv[m][n][i + 2]));
          v = fmaxf(v, __shfl_xor_sync(FULL, v, 4));
          v = fmaxf(v, __shfl_xor_sync(FULL, v, 8));
          v = fmaxf(v, __shfl_xor_sync(FULL, v, 16));
          x[n][i] = v;
          up = up || v > mc[n][i] + TAU;
        }
      if (__any_sync(FULL, up)) {
#pragma unroll
        for (int n = 0; n < NH8; ++n) {
          float sc[2];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float nm = fmaxf(mc[n][i], x[n][i]);
            sc[i] = (nm == -INFINITY) ? 1.f : fast_exp2(mc[n][i] - nm);
            mc[n][i] = nm;
            lc[n][i] *= sc[i];
          }
#pragma unroll
          for (int c = 0; c < C::CH; ++c) {
            acc[c][n][0] *= sc[0];
            acc[c][n][1] *= sc[1];
            acc[c][n][2] *= sc[0];
            acc[c][n][3] *= sc[1];
          }
        }
      }
      // weights, and P^T as the B operand (per m-tile and n-tile: b0 = tokens 0-7, b1 = 8-15)
      uint32_t pb[C::NMT][NH8][2];
#pragma unroll
      for (int m = 0; m < C::NMT; ++m)
#pragma unroll
        for (int n = 0; n < NH8; ++n) {
          float p[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            p[e] = (sv[m][n][e] == -INFINITY) ? 0.f : fast_exp2(sv[m][n][e] - mc[n][e & 1]);
            lc[n][e & 1] += p[e];  // fp32 weights for the denominator; only the operand is rounded
          }
          pb[m][n][0] = movmatrix_trans(pack_f16x2(p[0], p[1]));
          pb[m][n][1] = movmatrix_trans(pack_f16x2(p[2], p[3]));
        }
      if (masked) {
        // V rows of keys that are not attended may hold anything, NaN included: zero this
        // warp's part of them so that 0 x row stays 0
        uint8_t *vgen = smem + S::OFF_STAGE + s * C::STAGE_BYTES + C::KV_BYTES;
        constexpr int CPW = C::NQ * 8 / C::DSPLIT;  // 16-byte chunks of a row owned by this warp
        for (int e = lane; e < C::TW * CPW; e += 32) {
          const int stok = wbase + e / CPW;
          const int chunk = dh * CPW + e % CPW;
          const int ltok = mt.tok0 + stok;
          if (ltok < mt.tok_lo || ltok >= mt.tok_hi || ((mt.badmask >> (stok / bh_tokens)) & 1u))
            *reinterpret_cast<uint4 *>(vgen + kv_off<C>(stok, chunk)) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      // ---- O^T += V^T P^T: per 16-dim chunk, ldmatrix.trans of the m-tile's tokens 0-7 / 8-15
      // hands lane (g8, t) tokens 2t, 2t + 1 at dims 2 g8, 2 g8 + 1 (bytes: even, odd, even, odd)
#pragma unroll
      for (int m = 0; m < C::NMT; ++m)
#pragma unroll
        for (int c2 = 0; c2 < C::CH; c2 += 2) {
          uint32_t r[4];  // [chunk c2: tokens 0-7, 8-15][chunk c2 + 1: tokens 0-7, 8-15]
          ldmatrix_x4_trans(r, vbase + kv_off<C>(wbase + 16 * m + (lm_mat & 1) * 8 + lm_row,
                                                dh * C::CH + c2 + (lm_mat >> 1)));
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // A rows g8 (even dim) and g8 + 8 (odd dim), k = tokens 2t, 2t + 1 (a0, a1) and
            // 8 + 2t, 9 + 2t (a2, a3)
            const uint32_t ev = prmt(r[2 * h], r[2 * h + 1], 0x6420u), od = prmt(r[2 * h], r[2 * h + 1], 0x7531u);
            const uint32_t a4[4] = {e4m3x2_to_f16x2(ev), e4m3x2_to_f16x2(od), e4m3x2_to_f16x2(ev >> 16),
                                    e4m3x2_to_f16x2(od >> 16)};
#pragma unroll
            for (int n = 0; n < NH8; ++n) mma_f16_16816(acc[c2 + h][n], a4, pb[m][n][0], pb[m][n][1]);
          }
        }

      if (mt.last) {
        // ---- end of a piece: column sums over g8, then merge the token groups
#pragma unroll
        for (int n = 0; n < NH8; ++n)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            float v = lc[n][i];
            v += __shfl_xor_sync(FULL, v, 4);
            v += __shfl_xor_sync(FULL, v, 8);
            v += __shfl_xor_sync(FULL, v, 16);
            lc[n][i] = v;
          }
        named_bar(1, C::NCW * 32);  // all warps are done reading this stage
        float *mg = reinterpret_cast<float *>(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
#pragma unroll
          for (int n = 0; n < NH8; ++n)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int h = 8 * n + 2 * tq + i;                             // merge row = column
              const int d = ((dh * C::CH + c) * 16 + 2 * g8) ^ (4 * (h & 7));  // even dim, then odd
              *reinterpret_cast<float2 *>(mg + (tgrp * C::MR + h) * D + d) = make_float2(acc[c][n][i], acc[c][n][i + 2]);
            }
        if (g8 == 0 && dh == 0) {
#pragma unroll
          for (int n = 0; n < NH8; ++n)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int h = 8 * n + 2 * tq + i;
              sm_ml[(tgrp * C::MR + h) * 2] = mc[n][i];
              sm_ml[(tgrp * C::MR + h) * 2 + 1] = lc[n][i];
            }
        }
        named_bar(1, C::NCW * 32);
        gqa_merge_out<C, MQ>(mg, sm_ml, mt, a, ct, a.vscale);
        fence_proxy_async_smem();  // generic writes to the stage buffer precede its next TMA fill
      } else if (masked) {
        fence_proxy_async_smem();  // the zeroed V rows precede the next TMA fill of this stage
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  gqa_finish<C>(smem, a);
}

}  // namespace pa
