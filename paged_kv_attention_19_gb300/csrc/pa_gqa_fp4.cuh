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
//   * a stage is 128 tokens (32 at head_dim 256) of K rows then V rows, copied by TMA without
//     swizzle: 20 KB at head_dim 128;
//   * every E2M1 value times an E4M3 scale is an f16 value (at most 6 significant bits, between
//     2^-10 and 2688 in magnitude), so the MMAs are mma.sync m16n8k16 f16 with fp32 accumulation,
//     the query heads as the M rows, and the pool scales applied to the fp32 scores and output;
//     codes become f16 pairs by the conversion instructions (a byte of two E2M1 codes, a
//     duplicated E4M3 scale code), times the block scale in one f16x2 multiply, exact;
//   * the bf16 query enters as f16 scaled per head row by a power of two (its largest magnitude
//     in [2^14, 2^15)), exact for every element above 2^-29 of that largest one; the scores
//     take the factor back in fp32 with the softmax scale;
//   * P enters the P.V MMA as f16 (11 significant bits, the weights being at most 2^8 under the
//     lazy rescale);
//   * a token group is 32 tokens (16 at head_dim 256) served by two warps; each warp works on
//     the group's 16-token sub-groups side by side (independent chains for the scheduler);
//   * the two warps split the score k-steps: each builds the B fragments of its half of the dims
//     straight from the codes, and the two partial score tiles are exchanged through shared
//     memory and added in one fixed order, so both warps hold the same scores and softmax state
//     and no key is converted twice;
//   * V: each warp converts its tokens' half rows into private f16 tiles (the 128-byte swizzle of
//     a bf16 stage; rows of keys that are not attended become zeros) and reads its P.V B
//     fragments from them with ldmatrix.trans, as the bf16 kernel reads its stages;
//   * the end-of-piece merge uses the V tiles and exchange buffers (free at that point) as its
//     area, with a barrier after it before they are written again.
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
  static constexpr bool UNIT_MAJOR = false;        // (one plane: either order)
  static constexpr int M = PART_HEADS;
  static constexpr int MR = M;
  static constexpr int ST = D <= 128 ? 128 : 32;   // tokens per stage
  static constexpr int TW = D <= 128 ? 32 : 16;    // tokens per token group
  static constexpr int NU = TW / 16;               // 16-token sub-groups per warp
  static constexpr int TG = ST / TW;
  static constexpr int MG = TG;
  static constexpr int DSPLIT = 2;
  static constexpr int NCW = TG * DSPLIT;
  // With eight consumer warps, one producer warp would put three warps on one SM sub-partition and
  // cap every thread at 168 registers (a sub-partition holds 16384).  Instead the block is three
  // warpgroups: the producer's (the producer warp and three idle ones) gives registers back and
  // the consumers' two take them (launch: 384 x 168 = 64512 = 256 x 208 + 128 x 88).
  static constexpr bool REG_SPLIT = NCW == 8;
  static constexpr int THREADS = REG_SPLIT ? (NCW + 4) * 32 : (NCW + 1) * 32;
  static constexpr int CONSUMER_REGS = 208, PRODUCER_REGS = 88;
  static_assert(!REG_SPLIT || NCW * 32 * CONSUMER_REGS + 128 * PRODUCER_REGS <= THREADS * 168,
                "the register split stays within the launch's registers");
  static constexpr int NT_PV = D / 8 / DSPLIT;
  static constexpr int KSH = D / 16 / DSPLIT;      // score k-steps (16-value blocks) per warp
  static constexpr int NACC = KSH >= 2 ? 2 : 1;
  static constexpr int NQ = 1;
  static constexpr int QNQ = D / 64;
  static constexpr int PLANE = ST * ROWB;
  static constexpr int KV_BYTES = PLANE;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  // shared memory after the ring (GqaSmem's QAREA): each consumer warp's f16 V tiles (16 token
  // rows of 128-byte chunks per sub-group) and two partial-score buffers (32 lanes x 8 floats per
  // sub-group), which the end-of-piece merge reuses
  static constexpr int MERGE_BYTES = MG * MR * D * 4;
  static constexpr int VT_PLANES = (NT_PV + 7) / 8;
  static constexpr int VT_BYTES = VT_PLANES * 16 * 128;    // one sub-group's tile
  static constexpr int XBUF_BYTES = NU * 2 * 32 * 16;       // one stage's partial scores of a warp
  static constexpr int WARP_AREA = NU * VT_BYTES + 2 * XBUF_BYTES;
  static constexpr int SHARED_AREA = NCW * WARP_AREA > MERGE_BYTES ? NCW * WARP_AREA : MERGE_BYTES;
  static constexpr int OFF_MERGE = 0, OFF_WARP = 0;
  static constexpr int QAREA = SHARED_AREA;
  static constexpr int NS_FIT = (229376 - QAREA) / STAGE_BYTES;
  static constexpr int NS = NS_FIT < 16 ? NS_FIT : 16;
  static_assert(STAGE_BYTES % 1024 == 0, "stages start on 1024-byte boundaries (the query stage is swizzled)");
  static_assert(QNQ * M * 128 <= STAGE_BYTES, "the query rows fit one stage");
  static_assert(D % 64 == 0, "whole 64-dim planes of query rows");
  static_assert(NS >= 4, "a ring of at least 4 stages");
  static_assert(KSH % 2 == 0, "score k-steps in pairs (16-byte code loads)");
};

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The f16 pair of the two E2M1 codes in byte B of x (the low nibble to the low half).
template <int B>
__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t x) {
  uint32_t r;
  if constexpr (B == 0)
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b0;\n}" : "=r"(r) : "r"(x));
  else if constexpr (B == 1)
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b1;\n}" : "=r"(r) : "r"(x));
  else if constexpr (B == 2)
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b2;\n}" : "=r"(r) : "r"(x));
  else
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b3;\n}" : "=r"(r) : "r"(x));
  return r;
}

// The E4M3 code in byte b of x as an f16 pair (both halves), exact.
__device__ __forceinline__ uint32_t e4m3_f16x2(uint32_t x, int b) {
  const uint32_t d = __byte_perm(x, 0u, (uint32_t)(b | (b << 4)));
  uint32_t r;
  asm("{\n .reg .b16 h0, h1;\n mov.b32 {h0, h1}, %1;\n cvt.rn.f16x2.e4m3x2 %0, h0;\n}" : "=r"(r) : "r"(d));
  return r;
}

__device__ __forceinline__ float bf16_pair_absmax(uint32_t v) {
  return fmaxf(fabsf(__uint_as_float(v << 16)), fabsf(__uint_as_float(v & 0xffff0000u)));
}

__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// D += A(16x16, row) * B(16x8, col), f16 inputs, fp32 accumulation (fragments as for bf16).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Power-of-two exponent s for a query row whose largest magnitude is amax: amax 2^s in [2^14, 2^15)
// (s clamped to [-100, 100]: rows of zeros, subnormals, infinities or NaN).
__device__ __forceinline__ int q_row_shift(float amax) {
  const int e = (int)((__float_as_uint(amax) >> 23) & 255u) - 127;
  const int s = 14 - e;
  return s < -100 ? -100 : (s > 100 ? 100 : s);
}

// 2^s as a float, s in [-126, 127] (exact).
__device__ __forceinline__ float exp2_int(int s) { return __uint_as_float((uint32_t)(s + 127) << 23); }

// The bf16 pair x (low half first) times p2 (a power of two) as an f16 pair.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t x, float p2) {
  return f16x2_of(__uint_as_float(x << 16) * p2, __uint_as_float(x & 0xffff0000u) * p2);
}

// Byte offset of 16-byte chunk c (8 dims of the warp's half of D) of local token row t in a
// warp's V tile: 64-dim planes of 16 rows x 128 bytes, chunk ^ (row & 7) as in a bf16 stage.
__device__ __forceinline__ uint32_t vt_off(int t, int c) {
  return (uint32_t)((c >> 3) * (16 * 128) + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

// A consumer warp whose ring wait at stage j was late (the NVFP4 form of gqa_consumer_drain): it
// computes nothing more but keeps meeting, up to the end marker, every barrier the computing warps
// meet: its token group's score-exchange barrier at each K/V stage and the three end-of-piece
// barriers at each piece's last stage.
template <class C>
__device__ __forceinline__ void fp4_consumer_drain(uint8_t *smem, uint32_t j, int pair_bar) {
  using S = GqaSmem<C>;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
  uint64_t *empty = full + C::NS;
  const StageMeta *meta = reinterpret_cast<const StageMeta *>(smem + S::OFF_META);
  for (bool first_stage = true;; ++j, first_stage = false) {
    const int s = j % C::NS;
    if (!first_stage && !mbar_wait_warp(&full[s], (j / C::NS) & 1, DRAIN_LIMIT_NS)) break;
    const StageMeta &mt = meta[s];
    if (mt.end) break;
    if (!mt.first) named_bar(pair_bar, 64);
    if (mt.last) {
      named_bar(1, C::NCW * 32);
      named_bar(1, C::NCW * 32);
      named_bar(1, C::NCW * 32);
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&empty[s]);
  }
}

// The KSH block-scale codes of a row starting at p (aligned to their size), byte k = block k.
template <int KSH>
__device__ __forceinline__ uint2 load_scales(const uint8_t *p) {
  if constexpr (KSH == 8) return *reinterpret_cast<const uint2 *>(p);
  else if constexpr (KSH == 4) return make_uint2(*reinterpret_cast<const uint32_t *>(p), 0u);
  else return make_uint2(*reinterpret_cast<const uint16_t *>(p), 0u);
}

// MQ: several query positions per row (verify).
template <int D, bool MQ, bool LW>
__global__ void __launch_bounds__(GqaFp4Cfg<D>::THREADS, 1)
    gqa_fp4_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_q, const GqaArgs a) {
  using C = GqaFp4Cfg<D>;
  using S = GqaSmem<C>;
  constexpr int NU = C::NU, KSH = C::KSH;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
  uint64_t *empty = full + C::NS;
  const StageMeta *meta = reinterpret_cast<const StageMeta *>(smem + S::OFF_META);
  GqaMisc *misc = reinterpret_cast<GqaMisc *>(smem + S::OFF_MISC);
  uint32_t *status = &misc->status;
  uint8_t *extra = smem + S::OFF_QAREA;
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
    const int g8 = lane >> 2, tq = lane & 3;
    const int lm_mat = lane >> 3, lm_row = lane & 7;
    const int tgrp = warp % C::TG;
    const int dh = warp / C::TG;        // this warp's half: score k-steps and P.V columns
    const int partner = dh ? warp - C::TG : warp + C::TG;
    const int pair_bar = 2 + tgrp;      // named barrier of the token group's two warps
    const int wbase = tgrp * C::TW;
    const int nd0 = dh * C::NT_PV;
    const int ks0 = dh * KSH;
    float *sm_ml = reinterpret_cast<float *>(smem + S::OFF_ML);
    uint8_t *warea = extra + C::OFF_WARP + warp * C::WARP_AREA;
    uint8_t *vt = warea;                                   // NU tiles
    const uint32_t vt_u32 = smem_u32(vt);
    float4 *xmine = reinterpret_cast<float4 *>(warea + NU * C::VT_BYTES);
    const float4 *xpart =
        reinterpret_cast<const float4 *>(extra + C::OFF_WARP + partner * C::WARP_AREA + NU * C::VT_BYTES);
    float *mg = reinterpret_cast<float *>(extra + C::OFF_MERGE);
    const float TAU = 8.f;
    const int bh_tokens = 1 << a.log2_bh;

    uint32_t qa[KSH][4];      // f16 A fragments of this warp's k-steps, rows scaled by 2^s
    float qs0 = 0.f, qs1 = 0.f;  // score factors of rows g8 and g8 + 8: qscale 2^-s
    float acc[C::NT_PV][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool rv0 = false, rv1 = false;
    int lo0 = 0, hi0 = 0, lo1 = 0, hi1 = 0;
    uint32_t xb = 0;  // exchange buffer of the current stage (0 / 1, alternating)
    for (uint32_t j = 0;; ++j) {
      const int s = j % C::NS;
      if constexpr (LW) {
        const int wr = ring_wait(&full[s], (j / C::NS) & 1, a.wait_ns, status);
        if (wr == RING_LATE) fp4_consumer_drain<C>(smem, j, pair_bar);
        if (wr != RING_OK) break;
      } else {
        if (!mbar_wait(&full[s], (j / C::NS) & 1, status)) break;
      }
      StageMeta mt;
      {
        const uint4 *src = reinterpret_cast<const uint4 *>(&meta[s]);
        uint4 *dst = reinterpret_cast<uint4 *>(&mt);
        dst[0] = src[0];
        dst[1] = src[1];
        dst[2] = src[2];
        dst[3] = src[3];
      }
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
        // each row's largest |q| over all D dims (lane: row lane % 16, half lane / 16 of its
        // chunks), then the rows of this lane's fragments (g8, g8 + 8)
        float qmax;
        {
          const int r = lane & 15, h = lane >> 4;
          float mx = 0.f;
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            const int chunk = h * (D / 16) + c;
            const uint4 v = *reinterpret_cast<const uint4 *>(
                kst + (chunk >> 3) * (C::M * 128) + r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
            mx = fmaxf(mx, fmaxf(bf16_pair_absmax(v.x), bf16_pair_absmax(v.y)));
            mx = fmaxf(mx, fmaxf(bf16_pair_absmax(v.z), bf16_pair_absmax(v.w)));
          }
          qmax = fmaxf(mx, __shfl_xor_sync(FULL, mx, 16));
        }
        const int sh0 = q_row_shift(__shfl_sync(FULL, qmax, g8));
        const int sh1 = q_row_shift(__shfl_sync(FULL, qmax, g8 + 8));
        const float p20 = exp2_int(sh0), p21 = exp2_int(sh1);
        qs0 = a.qscale * exp2_int(-sh0);
        qs1 = a.qscale * exp2_int(-sh1);
#pragma unroll
        for (int k = 0; k < KSH; ++k) {
          const int row = (lm_mat & 1) * 8 + lm_row, chunk = 2 * (ks0 + k) + (lm_mat >> 1);
          uint32_t f[4];
          ldmatrix_x4(f, kbase + (chunk >> 3) * (C::M * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
          // a0, a2: row g8; a1, a3: row g8 + 8
          qa[k][0] = bf16x2_to_f16x2_scaled(f[0], p20);
          qa[k][1] = bf16x2_to_f16x2_scaled(f[1], p21);
          qa[k][2] = bf16x2_to_f16x2_scaled(f[2], p20);
          qa[k][3] = bf16x2_to_f16x2_scaled(f[3], p21);
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

      // ---- this warp's half of S = Q K^T for the group's tokens, sub-group u, n-tile nt: B
      // fragments from the codes (token g8 of the n-tile, dims 2 tq, 2 tq + 1 and 8 + 2 tq,
      // 9 + 2 tq of block ks: bytes tq and 4 + tq of the block's 8 code bytes)
      float sv[NU][2][4];
      {
        float sp[C::NACC][NU][2][4];
#pragma unroll
        for (int q = 0; q < C::NACC; ++q)
#pragma unroll
          for (int u = 0; u < NU; ++u)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) sp[q][u][nt][0] = sp[q][u][nt][1] = sp[q][u][nt][2] = sp[q][u][nt][3] = 0.f;
        // prmt: byte tq of the first code word into byte 0, byte tq of the second into byte 1
        const uint32_t bsel = (uint32_t)tq | ((uint32_t)(tq + 4) << 4);
#pragma unroll
        for (int k = 0; k < KSH; k += 2) {
#pragma unroll
          for (int u = 0; u < NU; ++u)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              const uint8_t *row = kst + (wbase + u * 16 + nt * 8 + g8) * C::ROWB;
              const uint2 scw = load_scales<KSH>(row + D / 2 + ks0);
              const uint4 c16 = *reinterpret_cast<const uint4 *>(row + (ks0 + k) * 8);
#pragma unroll
              for (int kk = 0; kk < 2; ++kk) {
                const int kb = k + kk;  // block index within this warp's half
                const uint32_t sc2 = e4m3_f16x2(kb < 4 ? scw.x : scw.y, kb & 3);
                const uint32_t pr = __byte_perm(kk ? c16.z : c16.x, kk ? c16.w : c16.y, bsel);
                const uint32_t b0 = f16x2_mul(e2m1x2_f16x2<0>(pr), sc2);
                const uint32_t b1 = f16x2_mul(e2m1x2_f16x2<1>(pr), sc2);
                mma_f16_16816(sp[kb % C::NACC][u][nt], qa[kb], b0, b1);
              }
            }
        }
#pragma unroll
        for (int u = 0; u < NU; ++u)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float x = sp[0][u][nt][e];
#pragma unroll
              for (int q = 1; q < C::NACC; ++q) x += sp[q][u][nt][e];
              sv[u][nt][e] = x;
            }
      }
      // ---- exchange the halves with the partner warp; both add them in the order (half 0) + (half 1)
      {
        float4 *xm = xmine + xb * (NU * 64);
#pragma unroll
        for (int u = 0; u < NU; ++u)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
            xm[(u * 2 + nt) * 32 + lane] = make_float4(sv[u][nt][0], sv[u][nt][1], sv[u][nt][2], sv[u][nt][3]);
        named_bar(pair_bar, 64);
        const float4 *xp = xpart + xb * (NU * 64);
#pragma unroll
        for (int u = 0; u < NU; ++u)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const float4 o = xp[(u * 2 + nt) * 32 + lane];
            const float oth[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) sv[u][nt][e] = dh == 0 ? sv[u][nt][e] + oth[e] : oth[e] + sv[u][nt][e];
          }
        xb ^= 1u;
      }
#pragma unroll
      for (int u = 0; u < NU; ++u)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float v = sv[u][nt][e] * ((e < 2) ? qs0 : qs1);
            bool valid = (e < 2) ? rv0 : rv1;
            if (masked) {
              const int stok = wbase + u * 16 + nt * 8 + 2 * tq + (e & 1);
              const int ltok = mt.tok0 + stok;
              valid = valid && attended(stok);
              if constexpr (MQ) valid = valid && ltok >= ((e < 2) ? lo0 : lo1) && ltok < ((e < 2) ? hi0 : hi1);
            }
            sv[u][nt][e] = valid ? v : -INFINITY;
          }
      // ---- online softmax per head row (rows g8 and g8 + 8)
      float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
      for (int u = 0; u < NU; ++u)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          x0 = fmaxf(x0, fmaxf(sv[u][nt][0], sv[u][nt][1]));
          x1 = fmaxf(x1, fmaxf(sv[u][nt][2], sv[u][nt][3]));
        }
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
      uint32_t pa[NU][4];
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        float p[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float mr = (e < 2) ? m0 : m1;
            p[nt][e] = (sv[u][nt][e] == -INFINITY) ? 0.f : fast_exp2(sv[u][nt][e] - mr);
          }
        pa[u][0] = f16x2_of(p[0][0], p[0][1]);
        pa[u][1] = f16x2_of(p[0][2], p[0][3]);
        pa[u][2] = f16x2_of(p[1][0], p[1][1]);
        pa[u][3] = f16x2_of(p[1][2], p[1][3]);
        l0 += (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
        l1 += (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
      }
      // ---- this warp's V tiles: lane (t, hh) converts dims [dh D/2 + hh D/4, + D/4) of token t of
      // each sub-group, block by block (16 dims: 8 code bytes and one scale), into 16-byte chunks
      {
        const int t = lane >> 1, hh = lane & 1;
        constexpr int NB = D / 64;  // blocks per lane and sub-group
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          const int stok = wbase + u * 16 + t;
          const bool zero = masked && !attended(stok);
          const uint8_t *row = kst + C::KV_BYTES + stok * C::ROWB;
          const int dim0 = dh * (D / 2) + hh * (D / 4);  // first dim of the lane's blocks
          uint32_t codes[NB * 2];
          if constexpr (NB == 1) {
            const uint2 c = *reinterpret_cast<const uint2 *>(row + dim0 / 2);
            codes[0] = c.x;
            codes[1] = c.y;
          } else {
#pragma unroll
            for (int q = 0; q < NB / 2; ++q) {
              const uint4 c = *reinterpret_cast<const uint4 *>(row + dim0 / 2 + 16 * q);
              codes[4 * q] = c.x;
              codes[4 * q + 1] = c.y;
              codes[4 * q + 2] = c.z;
              codes[4 * q + 3] = c.w;
            }
          }
          // the lane's NB scale codes: consecutive bytes at an NB-aligned offset
          const uint32_t scw = NB == 1 ? (uint32_t)row[D / 2 + dim0 / 16]
                               : NB == 2 ? (uint32_t)*reinterpret_cast<const uint16_t *>(row + D / 2 + dim0 / 16)
                                         : *reinterpret_cast<const uint32_t *>(row + D / 2 + dim0 / 16);
#pragma unroll
          for (int gi = 0; gi < NB; ++gi) {
            const int c0 = (hh * (D / 4) + gi * 16) / 8;  // the block's first chunk in the tile
            uint4 w0 = make_uint4(0, 0, 0, 0), w1 = make_uint4(0, 0, 0, 0);
            if (!zero) {
              const uint32_t sc2 = e4m3_f16x2(scw, gi);
              const uint32_t cx = codes[2 * gi], cy = codes[2 * gi + 1];
              w0.x = f16x2_mul(e2m1x2_f16x2<0>(cx), sc2);
              w0.y = f16x2_mul(e2m1x2_f16x2<1>(cx), sc2);
              w0.z = f16x2_mul(e2m1x2_f16x2<2>(cx), sc2);
              w0.w = f16x2_mul(e2m1x2_f16x2<3>(cx), sc2);
              w1.x = f16x2_mul(e2m1x2_f16x2<0>(cy), sc2);
              w1.y = f16x2_mul(e2m1x2_f16x2<1>(cy), sc2);
              w1.z = f16x2_mul(e2m1x2_f16x2<2>(cy), sc2);
              w1.w = f16x2_mul(e2m1x2_f16x2<3>(cy), sc2);
            }
            *reinterpret_cast<uint4 *>(vt + u * C::VT_BYTES + vt_off(t, c0)) = w0;
            *reinterpret_cast<uint4 *>(vt + u * C::VT_BYTES + vt_off(t, c0 + 1)) = w1;
          }
        }
      }
      __syncwarp();
      // ---- O += P V (k = each sub-group's 16 tokens), this warp's columns
      {
        const int t = (lm_mat & 1) * 8 + lm_row;
#pragma unroll
        for (int u = 0; u < NU; ++u)
#pragma unroll
          for (int nd = 0; nd < C::NT_PV; nd += 2) {
            uint32_t b[4];
            ldmatrix_x4_trans(b, vt_u32 + u * C::VT_BYTES + vt_off(t, nd + (lm_mat >> 1)));
            mma_f16_16816(acc[nd], pa[u], b[0], b[1]);
            mma_f16_16816(acc[nd + 1], pa[u], b[2], b[3]);
          }
      }
      __syncwarp();  // the tiles' reads are done before the next stage rewrites them

      if (mt.last) {
        // ---- end of a piece: merge the token groups through the warps' areas (all free now)
        l0 += __shfl_xor_sync(FULL, l0, 1);
        l0 += __shfl_xor_sync(FULL, l0, 2);
        l1 += __shfl_xor_sync(FULL, l1, 1);
        l1 += __shfl_xor_sync(FULL, l1, 2);
        named_bar(1, C::NCW * 32);  // every warp is done with its tiles and exchange buffers
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
        named_bar(1, C::NCW * 32);  // the merge has read the area before tiles are written again
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  gqa_finish<C>(smem, a);
}

}  // namespace pa
