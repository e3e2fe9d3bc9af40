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
//     every byte moved carries twice the tokens of the bf16 kernel;
//   * the codes go into FP8 tensor-core MMAs (mma.sync m16n8k32 e4m3) as they
//     lie in shared memory: no per-element conversion.  The MMA operand roles
//     are swapped against the bf16 kernel: tokens are the M rows (S^T = K Q^T)
//     and dims the M rows of O^T = V^T P^T, the tile's (head, position) columns
//     the N side in n-tiles of 8, so a group of 8 query heads fills one tile;
//   * K as the A operand is exactly what ldmatrix hands out (4 consecutive
//     codes of one token per register).  V^T comes from ldmatrix.trans of the
//     token rows plus byte permutes, which give each lane the tokens 2t, 2t + 1,
//     8 + 2t, 9 + 2t (then + 16) of one even and one odd dim; the P^T operand
//     is built in that same token order;
//   * the two small operands are split exactly enough into two E4M3 terms:
//     each query column times 2^s (its largest |q| in [128, 256)) is hi + lo
//     (exact for every element above 2^-10 of the column's scale: the bf16
//     query has 8 significant bits, each term 4), and the weights times 128
//     (at most 256, the lazy-rescale bound being 2) are hi + lo within 2^-8
//     relative; each product therefore takes two MMAs.  The 2^-s, k_scale,
//     v_scale and 1/128 factors are applied to the fp32 scores and outputs;
//   * each warp owns 32 tokens of a stage (one k32 of the P.V MMA); for
//     tiles of at most 8 columns two warp sets take turns on a piece's K/V
//     stages, each with its own softmax state, merged with the token groups
//     at the end of the piece: twice the warps in flight, no duplicated work;
//   * scores, softmax and accumulation are fp32.
#pragma once

#include "pa_gqa.cuh"

namespace pa {

// NH8_: n-tiles of 8 columns per tile (1: at most 8 (head, position) pairs, 2: up to 16).
template <int D_, int NH8_>
struct GqaF8Cfg {
  static constexpr int D = D_;
  static constexpr bool F8 = true;                 // pools of E4M3 codes
  static constexpr int ROWB = 128;                 // bytes of a token's row in one plane of a stage
  static constexpr int XSTEP = 128;                // tensor-map x of consecutive planes (one-byte codes)
  static constexpr bool UNIT_MAJOR = false;        // plane-major stage blocks, one copy per plane
  static constexpr int NH8 = NH8_;
  static constexpr int M = PART_HEADS;             // rows of a partial slot
  static constexpr int MR = 8 * NH8;               // rows per token group in the end-of-piece merge
  static constexpr int ST = D <= 128 ? 128 : 64;   // tokens per stage: 32 KB of K and V
  static constexpr int TW = 32;                    // tokens per token group: one k32 of the P.V MMA
  static constexpr int NMT = TW / 16;              // m-tiles of 16 tokens in the score MMA
  static constexpr int TG = ST / TW;               // token groups per stage
  // warps sharing a token group, each owning D / DSPLIT of the O^T rows (and all computing
  // the group's scores); two at head_dim 256 (registers, and four consumer warps instead of two)
  static constexpr int DSPLIT = D > 128 ? 2 : 1;
  // warp sets taking turns on the K/V stages of a piece (each with its own softmax state,
  // merged at the end of the piece): more warps in flight without duplicated work, where the
  // merge area holds the extra groups
  static constexpr int WS = NH8 == 1 ? 2 : 1;
  static constexpr int MG = TG * WS;               // groups merged at the end of a piece
  static constexpr int NCW = TG * DSPLIT * WS;     // consumer warps
  // + producer warp.  With eight consumer warps the block is three warpgroups instead (the
  // producer warp and three idle ones): one producer warp beside them would put three warps on one
  // SM sub-partition and cap every thread at 168 registers, where the producer's warpgroup gives
  // registers back and the consumers' two take them (launch: 384 x 168 = 256 x 208 + 128 x 88).
  static constexpr bool REG_SPLIT = NCW == 8;
  static constexpr int THREADS = REG_SPLIT ? (NCW + 4) * 32 : (NCW + 1) * 32;
  static constexpr int CONSUMER_REGS = 208, PRODUCER_REGS = 88;
  static_assert(!REG_SPLIT || NCW * 32 * CONSUMER_REGS + 128 * PRODUCER_REGS <= THREADS * 168,
                "the register split stays within the launch's registers");
  static constexpr int CH = D / DSPLIT / 16;       // 16-dim chunks (M tiles of O^T) per warp
  static constexpr int NQ = D / 128;               // 128-byte swizzle planes along D (K, V)
  static constexpr int QNQ = D / 64;               // the same for the bf16 query rows
  static constexpr int PLANE = ST * 128;
  static constexpr int KV_BYTES = NQ * PLANE;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int NS = (229376 / STAGE_BYTES) < 16 ? (229376 / STAGE_BYTES) : 16;  // 224 KB ring
  static_assert(MR * D * 4 * MG <= STAGE_BYTES, "the end-of-piece merge fits the consumed stage");
  static_assert(QNQ * M * 128 <= STAGE_BYTES, "the query rows fit one stage");
  static_assert(D % 128 == 0, "FP8 rows are whole 128-byte planes");
  static constexpr int QAREA = 0;                  // no query rows kept outside the ring
};

// D += A(16x32, row) * B(32x8, col), E4M3 inputs (4 per register), fp32 accumulation.  Fragments
// of the 8-bit m16n8k32 shape: a0 / a1 rows g and g + 8 at k = 4t .. 4t + 3, a2 / a3 the same
// rows at k + 16; b0 column g at k = 4t .. 4t + 3, b1 at k + 16 (g = lane / 4, t = lane % 4).
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
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

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// Two-term E4M3 split of an f16 pair x: hi = the nearest codes, lo = the nearest codes of the
// exact f16 remainder x - hi; x = hi + lo within 2^-8 |x|, exactly when each value has at most 8
// significant bits and both terms stay in E4M3's normal range.  2 codes each, x.lo's first.
__device__ __forceinline__ void split_e4m3x2(uint32_t x, uint32_t &hi, uint32_t &lo) {
  __half2_raw xr;
  xr.x = (unsigned short)(x & 0xffffu);
  xr.y = (unsigned short)(x >> 16);
  const __nv_fp8x2_storage_t h = __nv_cvt_halfraw2_to_fp8x2(xr, __NV_SATFINITE, __NV_E4M3);
  const __half2_raw hb = __nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3);
  const __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&xr), *reinterpret_cast<const __half2 *>(&hb));
  hi = (uint32_t)h;
  lo = (uint32_t)__nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw *>(&r), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float bf16x2_absmax(uint32_t v) {
  return fmaxf(fabsf(__uint_as_float(v << 16)), fabsf(__uint_as_float(v & 0xffff0000u)));
}

// 2^s as a float, s in [-126, 127].
__device__ __forceinline__ float pow2f(int s) { return __uint_as_float((uint32_t)(s + 127) << 23); }

// MQ: several query positions per row (verify).  NH8: see GqaF8Cfg.
template <int D, bool MQ, int NH8, bool LW>
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

  if (warp >= C::NCW) {
    if constexpr (C::REG_SPLIT) setmaxnreg_dec<C::PRODUCER_REGS>();
    if (warp == C::NCW) gqa_produce<C, LW, 1>(smem, &tm_k, &tm_v, &tm_q, a, pargs);
  } else {
    if constexpr (C::REG_SPLIT) setmaxnreg_inc<C::CONSUMER_REGS>();
    // ------------------------------------------------------------ consumers
    const int ct = tid;
    const int g8 = lane >> 2, tq = lane & 3;          // fragment row / column pair
    const int lm_mat = lane >> 3, lm_row = lane & 7;  // ldmatrix: matrix / row this lane addresses
    const int tgrp = warp % C::TG;                    // token group of this warp
    const int dh = (warp / C::TG) % C::DSPLIT;        // which part of the O^T rows (dims) it owns
    const int wset = warp / (C::TG * C::DSPLIT);      // warp set: takes K/V stages t = wset mod WS
    const int mgrp = wset * C::TG + tgrp;             // its group in the end-of-piece merge
    const int wbase = tgrp * C::TW;                   // first stage token of this warp
    int kv_t = 0;                                     // K/V stages of the current piece seen so far
    float *sm_ml = reinterpret_cast<float *>(smem + S::OFF_ML);
    // lazy rescale: the running max moves only when a score passes it by TAU (log2 units), so a
    // weight stays at most 2^TAU = 2 and PSCALE x weight at most 256 (E4M3 reaches 448)
    constexpr float TAU = 1.f;
    constexpr float PSCALE = 128.f;
    const int bh_tokens = 1 << a.log2_bh;

    // Q^T B fragments per k32 step (32 dims) and n-tile: [b0 = dims 4t .. +3, b1 = dims 16 + 4t ..
    // + 3] of column g8 times 2^s, high terms then low terms
    uint32_t qh[D / 32][NH8][2], ql[D / 32][NH8][2];
    float acc[C::CH][NH8][4];  // O^T: [chunk][n-tile]: c0, c1 = even dim x columns 2t, 2t + 1; c2, c3 = odd dim
    float mc[NH8][2], lc[NH8][2];  // running max / sum of this lane's columns 8 n + 2 tq + {0, 1}
    float cs[NH8][2];              // score multiplier of the column: qscale x 2^-s
    bool cv[NH8][2];               // real column?
    int clo[NH8][2], chi[NH8][2];  // MQ: key bounds [lo, hi) of the column's position
#pragma unroll
    for (int n = 0; n < NH8; ++n)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        mc[n][i] = -INFINITY;
        lc[n][i] = 0.f;
        cs[n][i] = 0.f;
        cv[n][i] = false;
        clo[n][i] = chi[n][i] = 0;
      }
    for (uint32_t j = 0;; ++j) {
      const int s = j % C::NS;
      if constexpr (LW) {  // the call's limit, and the give-up protocol of ring_wait
        const int wr = ring_wait(&full[s], (j / C::NS) & 1, a.wait_ns, status);
        if (wr == RING_LATE) gqa_consumer_drain<C, 1>(smem, j, a);
        if (wr != RING_OK) break;
      } else {
        if (!mbar_wait(&full[s], (j / C::NS) & 1, status)) break;
      }
      const StageMeta &mt = meta[s];
      if (mt.end) break;
      const uint32_t kbase = smem_u32(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
      const uint32_t vbase = kbase + C::KV_BYTES;
      if (mt.first) {
        // a new piece: the columns' validity and bounds, the split query fragments, fresh state.
        // Lane (g8, tq) reads dims 16 ks + 4 tq .. + 3 of column 8 n + g8's bf16 row (8 bytes).
        auto qaddr = [&](int ks, int row) {
          const int chunk = 2 * ks + (tq >> 1);
          return kbase + (uint32_t)((chunk >> 3) * (C::M * 128) + (tq & 1) * 8 + row * 128 +
                                    (((chunk & 7) ^ (row & 7)) << 4));
        };
#pragma unroll
        for (int n = 0; n < NH8; ++n) {
          const int row = 8 * n + g8;
          float am = 0.f;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint2 r = lds_u2(qaddr(ks, row));
            am = fmaxf(am, fmaxf(bf16x2_absmax(r.x), bf16x2_absmax(r.y)));
          }
          am = fmaxf(am, __shfl_xor_sync(FULL, am, 1));
          am = fmaxf(am, __shfl_xor_sync(FULL, am, 2));
          // s = 7 - floor(log2 am) puts the column's largest |q| in [128, 256); 0 for 0, inf, NaN
          const int e = (int)((__float_as_uint(am) >> 23) & 0xffu);
          const int sh = (e == 0xff || am == 0.f) ? 0 : min(126, max(-126, 134 - e));
          const float f = pow2f(sh);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint2 r = lds_u2(qaddr(ks, row));
            uint32_t h0, l0, h1, l1;  // dims 4tq, +1 / 4tq + 2, +3
            split_e4m3x2(pack_f16x2(__uint_as_float(r.x << 16) * f, __uint_as_float(r.x & 0xffff0000u) * f), h0, l0);
            split_e4m3x2(pack_f16x2(__uint_as_float(r.y << 16) * f, __uint_as_float(r.y & 0xffff0000u) * f), h1, l1);
            qh[ks >> 1][n][ks & 1] = h0 | (h1 << 16);
            ql[ks >> 1][n][ks & 1] = l0 | (l1 << 16);
          }
          // this lane's columns 8 n + 2 tq + i live in lanes 4 (2 tq + i) .. + 3
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int c = 8 * n + 2 * tq + i;
            const int shc = __shfl_sync(FULL, sh, 4 * (2 * tq + i));
            cs[n][i] = a.qscale * pow2f(-shc);
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
        }
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
#pragma unroll
          for (int n = 0; n < NH8; ++n) acc[c][n][0] = acc[c][n][1] = acc[c][n][2] = acc[c][n][3] = 0.f;
        kv_t = 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        continue;
      }
      const bool own = (kv_t++ % C::WS) == wset;
      if (!own && !mt.last) {  // the other set's stage
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        continue;
      }
      const bool masked = mt.masked;
      if (own) {
        // ---- S^T = K Q^T: per m-tile of 16 tokens, fragment c0 / c1 = token g8 x columns 2t,
        // 2t + 1, c2 / c3 = token g8 + 8.  ldmatrix matrices: tokens 0-7 / 8-15 of the m-tile at
        // 16-byte chunks 2 k, 2 k + 1: the A fragment of k32 step k as it is.
        // (high and low query terms in separate accumulators: two independent MMA chains)
        float sv[C::NMT][NH8][4], sl[C::NMT][NH8][4];
#pragma unroll
        for (int m = 0; m < C::NMT; ++m)
#pragma unroll
          for (int n = 0; n < NH8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) sv[m][n][e] = sl[m][n][e] = 0.f;
#pragma unroll
        for (int m = 0; m < C::NMT; ++m)
#pragma unroll
          for (int k = 0; k < D / 32; ++k) {
            uint32_t ak[4];
            ldmatrix_x4(ak, kbase + kv_off<C>(wbase + 16 * m + (lm_mat & 1) * 8 + lm_row, 2 * k + (lm_mat >> 1), a.log2_bh));
#pragma unroll
            for (int n = 0; n < NH8; ++n) {
              mma_e4m3_16832(sv[m][n], ak, qh[k][n][0], qh[k][n][1]);
              mma_e4m3_16832(sl[m][n], ak, ql[k][n][0], ql[k][n][1]);
            }
          }
#pragma unroll
        for (int m = 0; m < C::NMT; ++m)
#pragma unroll
          for (int n = 0; n < NH8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) sv[m][n][e] += sl[m][n][e];
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
              sv[m][n][e] = valid ? sv[m][n][e] * cs[n][e & 1] : -INFINITY;
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
        // weights, and P^T as the B operand of the k32 P.V step: movmatrix.trans turns (token g8,
        // columns 2t, 2t + 1) pairs into (column g8, tokens 2t, 2t + 1) pairs; k slots 4t .. 4t + 3
        // of b0 hold tokens 2t, 2t + 1, 8 + 2t, 9 + 2t of m-tile 0, b1 the same of m-tile 1
        uint32_t ph[NH8][2], pl[NH8][2];
#pragma unroll
        for (int n = 0; n < NH8; ++n)
#pragma unroll
          for (int m = 0; m < C::NMT; ++m) {
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              p[e] = (sv[m][n][e] == -INFINITY) ? 0.f : fast_exp2(sv[m][n][e] - mc[n][e & 1]);
              lc[n][e & 1] += p[e];  // fp32 weights for the denominator; only the operand is rounded
            }
            uint32_t h0, l0, h1, l1;
            split_e4m3x2(movmatrix_trans(pack_f16x2(p[0] * PSCALE, p[1] * PSCALE)), h0, l0);
            split_e4m3x2(movmatrix_trans(pack_f16x2(p[2] * PSCALE, p[3] * PSCALE)), h1, l1);
            ph[n][m] = h0 | (h1 << 16);
            pl[n][m] = l0 | (l1 << 16);
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
              *reinterpret_cast<uint4 *>(vgen + kv_off<C>(stok, chunk, a.log2_bh)) = make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
        }
        // ---- O^T += V^T P^T: per 16-dim chunk, ldmatrix.trans of the group's 32 token rows hands
        // lane (g8, t) tokens 2t, 2t + 1 of each token octet at dims 2 g8 (bytes 0, 2) and 2 g8 + 1
        // (bytes 1, 3); A rows g8 / g8 + 8 are the even / odd dim
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          uint32_t r[4];  // token octets 0-7, 8-15, 16-23, 24-31
          ldmatrix_x4_trans(r, vbase + kv_off<C>(wbase + lane, dh * C::CH + c, a.log2_bh));
          const uint32_t av[4] = {prmt(r[0], r[1], 0x6420u), prmt(r[0], r[1], 0x7531u), prmt(r[2], r[3], 0x6420u),
                                  prmt(r[2], r[3], 0x7531u)};
#pragma unroll
          for (int n = 0; n < NH8; ++n) {
            mma_e4m3_16832(acc[c][n], av, ph[n][0], ph[n][1]);
            mma_e4m3_16832(acc[c][n], av, pl[n][0], pl[n][1]);
          }
        }
      }  // own

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
              const int h = 8 * n + 2 * tq + i;                                 // merge row = column
              const int d = ((dh * C::CH + c) * 16 + 2 * g8) ^ (4 * (h & 7));  // even dim, then odd
              *reinterpret_cast<float2 *>(mg + (mgrp * C::MR + h) * D + d) = make_float2(acc[c][n][i], acc[c][n][i + 2]);
            }
        if (g8 == 0 && dh == 0) {
#pragma unroll
          for (int n = 0; n < NH8; ++n)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int h = 8 * n + 2 * tq + i;
              sm_ml[(mgrp * C::MR + h) * 2] = mc[n][i];
              sm_ml[(mgrp * C::MR + h) * 2 + 1] = lc[n][i];
            }
        }
        named_bar(1, C::NCW * 32);
        const MergeRows rows = {mt.slot, mt.b, mt.i0, mt.nq, mt.hq0, mt.ghead, 0};
        gqa_merge_out<C, MQ>(mg, sm_ml, rows, a, ct, a.vscale / PSCALE);
        fence_proxy_async_smem();  // generic writes to the stage buffer precede its next TMA fill
      } else if (masked && own) {
        fence_proxy_async_smem();  // the zeroed V rows precede the next TMA fill of this stage
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  gqa_finish<C>(smem, a);
}

}  // namespace pa
