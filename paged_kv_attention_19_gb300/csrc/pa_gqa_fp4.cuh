// pa_gqa_fp4.cuh -- GQA paged decode over an NVFP4 KV cache: the split-KV attention kernel
// (sm_103a).  The partition, the producer warp, the end-of-piece merge and the combine kernel are
// those of the bf16 kernel (pa_gqa.cuh); the consumer warps differ.
//
// What is computed: the decode of pa_gqa.cuh with keys and values read from NVFP4 pool rows
// (vllm.cpp kernel-matrix, row KERNEL-KV-QUANT: "Quantized KV cache, including FP8 and NVFP4"):
// value = e2m1(code) * e4m3(block scale) * pool scale, one block scale per 16 consecutive values.
// A pool row (page slot, KV head) is D / 2 bytes of code pairs (the even dim in the low nibble),
// D / 16 scale codes and zero padding to a multiple of 16 bytes (nvfp4_row_bytes).
//
// GB300 design of the consumers (the rest as in pa_gqa.cuh, one 16-row tile per sequence):
//   * a stage is 64 tokens (32 at head_dim 256) of K rows then V rows, copied by TMA without
//     swizzle: 10 KB at head_dim 128 instead of 32 KB for bf16, so the ring holds 16 stages;
//   * every E2M1 value times an E4M3 scale is a bf16 value (at most 6 significant bits), so the
//     MMAs stay mma.sync m16n8k16 bf16 with the query heads as the M rows and the pool scales
//     applied to the fp32 scores and output;
//   * K: each lane builds its B fragments straight from the codes: one 8-byte load gives a
//     token's 16-dim block, two of its bytes become bf16 pairs through a 256-entry table in
//     shared memory, times the block's scale (bf16x2 multiply, exact);
//   * V: each warp converts its 16 tokens' half rows into a private bf16 tile (2 KB, the 128-byte
//     swizzle of a bf16 stage; rows of keys that are not attended become zeros) and reads its P.V
//     B fragments from it with ldmatrix.trans, as the bf16 kernel reads its stages;
//   * the end-of-piece merge uses an area of its own (a 10 KB stage cannot hold it).
#pragma once

#include "pa_gqa.cuh"

namespace pa {

__host__ __device__ constexpr int nvfp4_row_bytes(int D) { return (D / 2 + D / 16 + 15) / 16 * 16; }

template <int D_>
struct GqaFp4Cfg {
  static constexpr int D = D_;
  static constexpr bool F8 = false;
  static constexpr int ROWB = nvfp4_row_bytes(D);  // bytes of a token's row (codes, scales, padding)
  static constexpr int XSTEP = 0;                  // one plane: the whole row
  static constexpr int M = PART_HEADS;
  static constexpr int MR = M;
  static constexpr int ST = D <= 128 ? 64 : 32;
  static constexpr int TW = 16;
  static constexpr int TG = ST / TW;
  static constexpr int MG = TG;
  static constexpr int DSPLIT = 2;
  static constexpr int NCW = TG * DSPLIT;
  static constexpr int THREADS = (NCW + 1) * 32;
  static constexpr int NT_PV = D / 8 / DSPLIT;
  static constexpr int NACC = 2;
  static constexpr int NQ = 1;
  static constexpr int QNQ = D / 64;
  static constexpr int PLANE = ST * ROWB;
  static constexpr int KV_BYTES = PLANE;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  // shared memory after the ring (GqaSmem's QAREA): the merge area, each consumer warp's bf16 V
  // tile (16 token rows of 128-byte chunks), the code-pair and scale tables
  static constexpr int MERGE_BYTES = MG * MR * D * 4;
  static constexpr int VT_PLANES = (NT_PV + 7) / 8;
  static constexpr int VT_BYTES = VT_PLANES * TW * 128;
  static constexpr int OFF_MERGE = 0, OFF_VT = MERGE_BYTES, OFF_LUTP = OFF_VT + NCW * VT_BYTES,
                       OFF_LUTS = OFF_LUTP + 256 * 4;
  static constexpr int QAREA = OFF_LUTS + 256 * 2;
  static constexpr int NS_FIT = (229376 - QAREA) / STAGE_BYTES;
  static constexpr int NS = NS_FIT < 16 ? NS_FIT : 16;
  static_assert(STAGE_BYTES % 1024 == 0, "stages start on 1024-byte boundaries (the query stage is swizzled)");
  static_assert(QNQ * M * 128 <= STAGE_BYTES, "the query rows fit one stage");
  static_assert(D % 64 == 0, "whole 64-dim planes of query rows");
};

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// bf16 bits of an E2M1 code and of an E4M3 code (both exact: at most 4 significant bits).
__device__ __forceinline__ uint32_t e2m1_bf16(uint32_t c) {
  // magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6
  const uint32_t mag = (c & 7u) == 0 ? 0u : (c & 7u) == 1 ? 0x3F00u : 0x3F80u + (((c & 7u) - 2u) << 6);
  return mag | ((c & 8u) << 12);
}
__device__ __forceinline__ uint32_t e4m3_bf16(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  float v = e == 0 ? (float)m * 0.001953125f : (1.f + (float)m * 0.125f) * __uint_as_float((e + 120u) << 23);
  if (e == 15u && m == 7u) v = __uint_as_float(0x7FC00000u);
  return (__float_as_uint(v) >> 16) | ((c & 0x80u) << 8);
}

// Byte offset of 16-byte chunk c (8 dims of the warp's half of D) of local token row t in a
// warp's V tile: 64-dim planes of 16 rows x 128 bytes, chunk ^ (row & 7) as in a bf16 stage.
__device__ __forceinline__ uint32_t vt_off(int t, int c) {
  return (uint32_t)((c >> 3) * (16 * 128) + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

// MQ: several query positions per row (verify).
template <int D, bool MQ, bool LW>
__global__ void __launch_bounds__(GqaFp4Cfg<D>::THREADS, 1)
    gqa_fp4_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_q, const GqaArgs a) {
  using C = GqaFp4Cfg<D>;
  using S = GqaSmem<C>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
  uint64_t *empty = full + C::NS;
  StageMeta *meta = reinterpret_cast<StageMeta *>(smem + S::OFF_META);
  GqaMisc *misc = reinterpret_cast<GqaMisc *>(smem + S::OFF_MISC);
  uint32_t *status = &misc->status;
  uint8_t *extra = smem + S::OFF_QAREA;
  uint32_t *lut_p = reinterpret_cast<uint32_t *>(extra + C::OFF_LUTP);
  uint16_t *lut_s = reinterpret_cast<uint16_t *>(extra + C::OFF_LUTS);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 256; i += C::THREADS) {
    lut_p[i] = e2m1_bf16((uint32_t)i & 15u) | (e2m1_bf16((uint32_t)i >> 4) << 16);
    lut_s[i] = (uint16_t)e4m3_bf16((uint32_t)i);
  }

  PartitionArgs pargs;
  gqa_setup<C>(smem, &tm_k, &tm_v, &tm_q, a, pargs);  // ends with a CTA barrier: the tables are ready

  if (warp == C::NCW) {
    gqa_produce<C, LW, 1>(smem, &tm_k, &tm_v, &tm_q, a, pargs);
  } else {
    // ------------------------------------------------------------ consumers
    const int ct = tid;
    const int g8 = lane >> 2, tq = lane & 3;
    const int lm_mat = lane >> 3, lm_row = lane & 7;
    const int tgrp = warp % C::TG;
    const int dh = warp / C::TG;
    const int wbase = tgrp * C::TW;
    const int nd0 = dh * C::NT_PV;
    float *sm_ml = reinterpret_cast<float *>(smem + S::OFF_ML);
    uint8_t *vt = extra + C::OFF_VT + warp * C::VT_BYTES;
    const uint32_t vt_u32 = smem_u32(vt);
    float *mg = reinterpret_cast<float *>(extra + C::OFF_MERGE);
    const float TAU = 8.f;
    const int bh_tokens = 1 << a.log2_bh;

    uint32_t qa[D / 16][4];
    float acc[C::NT_PV][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool rv0 = false, rv1 = false;
    int lo0 = 0, hi0 = 0, lo1 = 0, hi1 = 0;
    for (uint32_t j = 0;; ++j) {
      const int s = j % C::NS;
      if constexpr (LW) {
        const int wr = ring_wait(&full[s], (j / C::NS) & 1, a.wait_ns, status);
        if (wr == RING_LATE) gqa_consumer_drain<C, 1>(smem, j, a);
        if (wr != RING_OK) break;
      } else {
        if (!mbar_wait(&full[s], (j / C::NS) & 1, status)) break;
      }
      const StageMeta &mt = meta[s];
      if (mt.end) break;
      const uint8_t *kst = smem + S::OFF_STAGE + s * C::STAGE_BYTES;
      const uint32_t kbase = smem_u32(kst);
      if (mt.first) {
        if constexpr (MQ) {
          const int iq0 = g8 / a.gt, hh0 = g8 % a.gt, iq1 = (g8 + 8) / a.gt, hh1 = (g8 + 8) % a.gt;
          rv0 = iq0 < mt.nq && hh0 < mt.ghead;
          rv1 = iq1 < mt.nq && hh1 < mt.ghead;
          lo0 = pos_lo(mt.L, a.Q, mt.i0 + iq0, a.window);
          hi0 = pos_hi(mt.L, a.Q, mt.i0 + iq0);
          lo1 = pos_lo(mt.L, a.Q, mt.i0 + iq1, a.window);
          hi1 = pos_hi(mt.L, a.Q, mt.i0 + iq1);
        } else {
          rv0 = g8 < mt.ghead;
          rv1 = g8 + 8 < mt.ghead;
        }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int row = (lm_mat & 1) * 8 + lm_row, chunk = 2 * ks + (lm_mat >> 1);
          ldmatrix_x4(qa[ks], kbase + (chunk >> 3) * (C::M * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
        }
#pragma unroll
        for (int n = 0; n < C::NT_PV; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        continue;
      }
      const bool masked = mt.masked;
      auto attended = [&](int stok) {  // a key of the piece that is read (the V rows of others are zeroed)
        const int ltok = mt.tok0 + stok;
        return ltok >= mt.tok_lo && ltok < mt.tok_hi && !((mt.badmask >> (stok / bh_tokens)) & 1u);
      };

      // ---- S = Q K^T for the group's 16 tokens: B fragments from the codes (token g8 of n-tile
      // nt, dims 2 tq, 2 tq + 1 and 8 + 2 tq, 9 + 2 tq of block ks: bytes tq and 4 + tq)
      float sv[2][4];
      {
        float sp[C::NACC][2][4];
#pragma unroll
        for (int q = 0; q < C::NACC; ++q)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) sp[q][nt][0] = sp[q][nt][1] = sp[q][nt][2] = sp[q][nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const uint8_t *row = kst + (wbase + nt * 8 + g8) * C::ROWB;
            const uint2 c8 = *reinterpret_cast<const uint2 *>(row + ks * 8);
            const uint32_t sc = lut_s[row[D / 2 + ks]];
            const uint32_t sc2 = sc | (sc << 16);
            const uint32_t b0 = bf16x2_mul(lut_p[(c8.x >> (8 * tq)) & 255u], sc2);
            const uint32_t b1 = bf16x2_mul(lut_p[(c8.y >> (8 * tq)) & 255u], sc2);
            mma_bf16_16816(sp[ks % C::NACC][nt], qa[ks], b0, b1);
          }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x = sp[0][nt][e];
#pragma unroll
            for (int q = 1; q < C::NACC; ++q) x += sp[q][nt][e];
            sv[nt][e] = x;
          }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float v = sv[nt][e] * a.qscale;
          bool valid = (e < 2) ? rv0 : rv1;
          if (masked) {
            const int stok = wbase + nt * 8 + 2 * tq + (e & 1);
            const int ltok = mt.tok0 + stok;
            valid = valid && attended(stok);
            if constexpr (MQ) valid = valid && ltok >= ((e < 2) ? lo0 : lo1) && ltok < ((e < 2) ? hi0 : hi1);
          }
          sv[nt][e] = valid ? v : -INFINITY;
        }
      // ---- online softmax per head row (rows g8 and g8 + 8)
      float x0 = fmaxf(fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[1][0], sv[1][1]));
      float x1 = fmaxf(fmaxf(sv[0][2], sv[0][3]), fmaxf(sv[1][2], sv[1][3]));
      x0 = fmaxf(x0, __shfl_xor_sync(FULL, x0, 1));
      x0 = fmaxf(x0, __shfl_xor_sync(FULL, x0, 2));
      x1 = fmaxf(x1, __shfl_xor_sync(FULL, x1, 1));
      x1 = fmaxf(x1, __shfl_xor_sync(FULL, x1, 2));
      if (__any_sync(FULL, (x0 > m0 + TAU) || (x1 > m1 + TAU))) {
        const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
        const float a0 = (n0 == -INFINITY) ? 1.f : fast_exp2(m0 - n0);
        const float a1 = (n1 == -INFINITY) ? 1.f : fast_exp2(m1 - n1);
        m0 = n0;
        m1 = n1;
        l0 *= a0;
        l1 *= a1;
#pragma unroll
        for (int n = 0; n < C::NT_PV; ++n) {
          acc[n][0] *= a0;
          acc[n][1] *= a0;
          acc[n][2] *= a1;
          acc[n][3] *= a1;
        }
      }
      uint32_t pa[4];
      {
        float p[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float mr = (e < 2) ? m0 : m1;
            p[nt][e] = (sv[nt][e] == -INFINITY) ? 0.f : fast_exp2(sv[nt][e] - mr);
          }
        pa[0] = pack_bf16x2(p[0][0], p[0][1]);
        pa[1] = pack_bf16x2(p[0][2], p[0][3]);
        pa[2] = pack_bf16x2(p[1][0], p[1][1]);
        pa[3] = pack_bf16x2(p[1][2], p[1][3]);
        l0 += (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
        l1 += (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
      }
      // ---- this warp's V tile: lane (t, hh) converts dims [dh D/2 + hh D/4, + D/4) of local token
      // t, block by block (16 dims: 8 code bytes and one scale), into two 16-byte chunks each
      {
        const int t = lane >> 1, hh = lane & 1;
        const int stok = wbase + t;
        const bool zero = masked && !attended(stok);
        const uint8_t *row = kst + C::KV_BYTES + stok * C::ROWB;
#pragma unroll
        for (int gi = 0; gi < D / 64; ++gi) {
          const int dim0 = dh * (D / 2) + hh * (D / 4) + gi * 16;  // first dim of the block
          const int c0 = (hh * (D / 4) + gi * 16) / 8;              // its first chunk in the tile
          uint4 w0 = make_uint4(0, 0, 0, 0), w1 = make_uint4(0, 0, 0, 0);
          if (!zero) {
            const uint2 c8 = *reinterpret_cast<const uint2 *>(row + dim0 / 2);
            const uint32_t sc = lut_s[row[D / 2 + dim0 / 16]];
            const uint32_t sc2 = sc | (sc << 16);
            w0.x = bf16x2_mul(lut_p[c8.x & 255u], sc2);
            w0.y = bf16x2_mul(lut_p[(c8.x >> 8) & 255u], sc2);
            w0.z = bf16x2_mul(lut_p[(c8.x >> 16) & 255u], sc2);
            w0.w = bf16x2_mul(lut_p[c8.x >> 24], sc2);
            w1.x = bf16x2_mul(lut_p[c8.y & 255u], sc2);
            w1.y = bf16x2_mul(lut_p[(c8.y >> 8) & 255u], sc2);
            w1.z = bf16x2_mul(lut_p[(c8.y >> 16) & 255u], sc2);
            w1.w = bf16x2_mul(lut_p[c8.y >> 24], sc2);
          }
          *reinterpret_cast<uint4 *>(vt + vt_off(t, c0)) = w0;
          *reinterpret_cast<uint4 *>(vt + vt_off(t, c0 + 1)) = w1;
        }
      }
      __syncwarp();
      // ---- O += P V (k = the group's 16 tokens), this warp's columns
      {
        const int t = (lm_mat & 1) * 8 + lm_row;
#pragma unroll
        for (int nd = 0; nd < C::NT_PV; nd += 2) {
          uint32_t b[4];
          ldmatrix_x4_trans(b, vt_u32 + vt_off(t, nd + (lm_mat >> 1)));
          mma_bf16_16816(acc[nd], pa, b[0], b[1]);
          mma_bf16_16816(acc[nd + 1], pa, b[2], b[3]);
        }
      }
      __syncwarp();  // the tile's reads are done before the next stage rewrites it

      if (mt.last) {
        // ---- end of a piece: merge the token groups through the merge area
        l0 += __shfl_xor_sync(FULL, l0, 1);
        l0 += __shfl_xor_sync(FULL, l0, 2);
        l1 += __shfl_xor_sync(FULL, l1, 1);
        l1 += __shfl_xor_sync(FULL, l1, 2);
        named_bar(1, C::NCW * 32);  // the previous piece's merge has read the area
#pragma unroll
        for (int n = 0; n < C::NT_PV; ++n) {
          const int d = ((nd0 + n) * 8 + 2 * tq) ^ (4 * g8);
          *reinterpret_cast<float2 *>(mg + (tgrp * C::M + g8) * D + d) = make_float2(acc[n][0], acc[n][1]);
          *reinterpret_cast<float2 *>(mg + (tgrp * C::M + g8 + 8) * D + d) = make_float2(acc[n][2], acc[n][3]);
        }
        if (tq == 0 && dh == 0) {
          sm_ml[(tgrp * C::M + g8) * 2] = m0;
          sm_ml[(tgrp * C::M + g8) * 2 + 1] = l0;
          sm_ml[(tgrp * C::M + g8 + 8) * 2] = m1;
          sm_ml[(tgrp * C::M + g8 + 8) * 2 + 1] = l1;
        }
        named_bar(1, C::NCW * 32);
        const MergeRows rows = {mt.slot, mt.b, mt.i0, mt.nq, mt.hq0, mt.ghead, 0};
        gqa_merge_out<C, MQ>(mg, sm_ml, rows, a, ct, a.vscale);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  gqa_finish<C>(smem, a);
}

}  // namespace pa
