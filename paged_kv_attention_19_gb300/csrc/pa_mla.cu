// pa_mla.cu -- MLA absorbed decode (sm_103a).
//
// What is computed follows pegainfer PR #938 "warp-cooperative two-pass MLA
// absorbed decode kernel" (Schedule section, steps 1-7) and the vllm.cpp
// kernel-matrix row KERNEL-ATTN-MLA-SPARSE (absorption = two batched
// contractions around a split-KV decode with a fixed ascending merge):
//   1. q_lat = q_nope . W_UK (128 -> 512), q_rope appended      [q_absorb_kernel]
//   2-6. scores over the 576-wide latent||rope cache, online softmax,
//        o_lat = sum_t p_t c_t[0:512], per page-aligned split     [mla_split_kernel]
//   7. splits merged in ascending order, o = W_UV . o_lat          [mla_out_kernel]
// Differences from the pages' kernel, all deliberate: scores, probabilities
// and q_lat stay fp32 (no bf16 landings); the context is walked once with an
// online max instead of twice; o_lat is rounded to bf16 only as the tensor-
// core operand of step 7.
//
// GB300 mapping:
//   * steps 1 and 7 are dense per-head contractions (M = batch rows) on the
//     tensor cores, bf16 operands, fp32 accumulation (mma.sync m16n8k16).
//   * steps 2-6 run on the CUDA cores in a persistent kernel fed by a TMA
//     producer warp (one 4-D tensor-map copy per page fragment into a ring of
//     36 KB stages).  Every token of a stage is used by all 8 consumer warps;
//     warp w owns 4 heads of the item's 32-head group, lane l owns latent
//     dims [16l, 16l+16) and rope dims [2l, 2l+2), so one 1152-byte token row
//     is read as contiguous 16-byte chunks by the whole warp.  q_lat lives in
//     registers; the 4 partial dots are transpose-reduced across the warp,
//     the owning lane applies the online softmax, and P.V reuses the latent
//     values already in registers.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "pa_plan.cuh"
#include "pa_launch.h"
#include "pa_mla.h"

namespace pa {

constexpr int MLA_NOPE = 128, MLA_QD = 192, MLA_LAT = 512, MLA_C = 576, MLA_V = 128;

struct MlaCfg {
  static constexpr int NCW = 8;
  static constexpr int THREADS = (NCW + 1) * 32;
  static constexpr int HPW = 4;                   // heads per warp
  static constexpr int HG = NCW * HPW;            // heads per work item
  static constexpr int ST = 32;                   // tokens per stage
  static constexpr int ROW_BYTES = MLA_C * 2;     // 1152
  static constexpr int STAGE_BYTES = ST * ROW_BYTES;
  static constexpr int NS = 4;
  static constexpr int MAXBOX = 32;
  static constexpr int OFF_META = NS * STAGE_BYTES;
  static constexpr int OFF_BAR = OFF_META + NS * 64;
  static constexpr int SMEM = OFF_BAR + 2 * NS * 8;
};

struct MlaMeta {
  int32_t end, first, last, masked;
  int32_t b, sub, split, tok0;
  int32_t tok_lo, tok_hi, pad0, pad1;
  uint32_t badmask, pad2, pad3, pad4;
};
static_assert(sizeof(MlaMeta) == 64, "meta is 64 bytes");

struct MlaArgs {
  const uint16_t *q;           // [B, H, 192]
  const int32_t *block_table;
  const float *q_lat;          // [B, H, 512] fp32
  float *part_o;               // [B, H, max_splits, 512]
  float *part_lse;             // [B, H, max_splits] log2 units
  WsHeader *hdr;
  const WorkItem *items;
  const RowInfo *rows;
  int max_pages_per_seq, num_pages, H, page_size, log2_page, max_splits;
  float qscale;                // scale * log2(e)
};

__global__ void __launch_bounds__(MlaCfg::THREADS, 1)
    mla_split_kernel(const __grid_constant__ CUtensorMap tm_c, const MlaArgs a) {
  using C = MlaCfg;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *empty = full + C::NS;
  MlaMeta *meta = reinterpret_cast<MlaMeta *>(smem + C::OFF_META);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NCW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  uint32_t *status = &a.hdr->status;

  if (warp == C::NCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) prefetch_tensormap(&tm_c);
    const int n_items = (int)a.hdr->n_items;
    const int P = a.page_size;
    const int BH = P < C::ST ? P : C::ST;
    const int nbox = C::ST / BH;
    uint32_t j = 0;
    bool ok = true;
    while (ok) {
      int idx = 0;
      if (lane == 0) idx = (int)atomicAdd(&a.hdr->item_counter, 1u);
      idx = __shfl_sync(FULL, idx, 0);
      if (idx >= n_items) {
        const int s = j % C::NS;
        const uint32_t u = j / C::NS;
        if (u > 0) ok = mbar_wait(&empty[s], (u - 1) & 1, status);
        if (ok && lane == 0) {
          meta[s].end = 1;
          mbar_arrive(&full[s]);
        }
        break;
      }
      const WorkItem it = a.items[idx];
      const RowInfo ri = a.rows[it.b];
      const int T0 = it.page_begin * P, T1 = it.page_end * P;
      const int tok_lo = max(ri.lo, T0), tok_hi = min(ri.L, T1);
      const int n_stages = (T1 - T0 + C::ST - 1) / C::ST;
      const int32_t *bt_row = a.block_table + (size_t)it.b * a.max_pages_per_seq;
      for (int t = 0; t < n_stages && ok; ++t, ++j) {
        const int s = j % C::NS;
        const uint32_t u = j / C::NS;
        if (u > 0) ok = mbar_wait(&empty[s], (u - 1) & 1, status);
        if (!ok) break;
        const int tok0 = T0 + t * C::ST;
        bool load = false, isbad = false;
        int phys = 0;
        if (lane < nbox) {
          const int btok = tok0 + lane * BH;
          if (btok < tok_hi && btok + BH > tok_lo) {
            phys = bt_row[btok >> a.log2_page];
            if (phys < 0 || phys >= a.num_pages) {
              isbad = true;
              atomicOr(status, PA_DEV_BAD_PAGE);
            } else {
              load = true;
            }
          }
        }
        const uint32_t bad = __ballot_sync(FULL, isbad);
        const int nvalid = __popc(__ballot_sync(FULL, load));
        if (lane == 0) {
          MlaMeta &m = meta[s];
          m.end = 0;
          m.first = (t == 0);
          m.last = (t == n_stages - 1);
          m.b = it.b;
          m.sub = it.sub;
          m.split = it.split;
          m.tok0 = tok0;
          m.tok_lo = tok_lo;
          m.tok_hi = tok_hi;
          m.badmask = bad;
          m.masked = (tok0 < tok_lo) || (tok0 + C::ST > tok_hi) || bad != 0;
          mbar_arrive_expect_tx(&full[s], (uint32_t)nvalid * (uint32_t)(BH * C::ROW_BYTES));
        }
        __syncwarp();
        if (load) {
          const int btok = tok0 + lane * BH;
          tma_load_4d(smem + s * C::STAGE_BYTES + lane * BH * C::ROW_BYTES, &tm_c, 0, 0, btok & (P - 1), phys,
                      &full[s]);
        }
      }
    }
    if (!ok) {
      const uint32_t first = j > (uint32_t)C::NS ? j - C::NS : 0u;
      for (uint32_t i = first; i < j; ++i) mbar_wait(&full[i % C::NS], (i / C::NS) & 1, status);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int fh = lane >> 3;  // head (of the warp's 4) held after the transpose reduction
  float2 ql[C::HPW][8];      // q_lat, latent dims [16 lane, 16 lane + 16), scaled
  float2 qr[C::HPW];         // q_rope dims [2 lane, 2 lane + 2), scaled
  float2 acc[C::HPW][8];
  float m_run = -INFINITY, l_run = 0.f;
  const float TAU = 8.f;
  int hbase = 0;

  for (uint32_t j = 0;; ++j) {
    const int s = j % C::NS;
    if (!mbar_wait(&full[s], (j / C::NS) & 1, status)) break;
    const MlaMeta &mt = meta[s];
    if (mt.end) break;
    if (mt.first) {
      hbase = mt.sub * C::HG + warp * C::HPW;
      // slot i of q holds head i ^ fh, so that each halving exchange of the
      // transpose reduction keeps slots [0, half) and receives [half, 2 half)
#pragma unroll
      for (int i = 0; i < C::HPW; ++i) {
        const int h = hbase + (i ^ fh);
        if (h < a.H) {
          const float4 *src = reinterpret_cast<const float4 *>(a.q_lat + ((size_t)mt.b * a.H + h) * MLA_LAT + lane * 16);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 v = src[e];
            ql[i][2 * e] = make_float2(v.x * a.qscale, v.y * a.qscale);
            ql[i][2 * e + 1] = make_float2(v.z * a.qscale, v.w * a.qscale);
          }
          const uint32_t rw =
              *reinterpret_cast<const uint32_t *>(a.q + ((size_t)mt.b * a.H + h) * MLA_QD + MLA_NOPE + lane * 2);
          qr[i] = make_float2(__uint_as_float(rw << 16) * a.qscale, __uint_as_float(rw & 0xffff0000u) * a.qscale);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) ql[i][e] = make_float2(0.f, 0.f);
          qr[i] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = make_float2(0.f, 0.f);
      }
      m_run = -INFINITY;
      l_run = 0.f;
    }
    const uint8_t *st = smem + s * C::STAGE_BYTES;
    const int BH = a.page_size < C::ST ? a.page_size : C::ST;
#pragma unroll 2
    for (int t = 0; t < C::ST; ++t) {
      const uint8_t *row = st + t * C::ROW_BYTES;
      uint4 c0 = *reinterpret_cast<const uint4 *>(row + lane * 32);
      uint4 c1 = *reinterpret_cast<const uint4 *>(row + lane * 32 + 16);
      uint32_t cr = *reinterpret_cast<const uint32_t *>(row + MLA_LAT * 2 + lane * 4);
      bool valid = true;
      if (mt.masked) {
        const int ltok = mt.tok0 + t;
        valid = ltok >= mt.tok_lo && ltok < mt.tok_hi && !((mt.badmask >> (t / BH)) & 1u);
        if (!valid) {
          c0 = make_uint4(0, 0, 0, 0);
          c1 = make_uint4(0, 0, 0, 0);
          cr = 0;
        }
      }
      float2 cl[8];
      bf16x8_to_f32(c0, *reinterpret_cast<float2(*)[4]>(&cl[0]));
      bf16x8_to_f32(c1, *reinterpret_cast<float2(*)[4]>(&cl[4]));
      const float2 crf = make_float2(__uint_as_float(cr << 16), __uint_as_float(cr & 0xffff0000u));
      float part[C::HPW];
#pragma unroll
      for (int i = 0; i < C::HPW; ++i) {
        float2 t2 = __fmul2_rn(qr[i], crf);
#pragma unroll
        for (int e = 0; e < 8; ++e) t2 = __ffma2_rn(ql[i][e], cl[e], t2);
        part[i] = t2.x + t2.y;
      }
      // transpose reduction over the 32 lanes: lane keeps head fh = lane / 8
      part[0] += __shfl_xor_sync(FULL, part[2], 16);
      part[1] += __shfl_xor_sync(FULL, part[3], 16);
      part[0] += __shfl_xor_sync(FULL, part[1], 8);
#pragma unroll
      for (int mask = 4; mask >= 1; mask >>= 1) part[0] += __shfl_xor_sync(FULL, part[0], mask);
      const float sc = valid ? part[0] : -INFINITY;
      if (__any_sync(FULL, sc > m_run + TAU)) {
        const float m_new = fmaxf(m_run, sc);
        const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
        l_run *= alpha;
        m_run = m_new;
#pragma unroll
        for (int i = 0; i < C::HPW; ++i) {
          const float al = __shfl_sync(FULL, alpha, 8 * i);
          const float2 a2 = make_float2(al, al);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[i][e] = __fmul2_rn(a2, acc[i][e]);
        }
      }
      const float p = valid ? fast_exp2(sc - m_run) : 0.f;
      l_run += p;
#pragma unroll
      for (int i = 0; i < C::HPW; ++i) {
        const float pi = __shfl_sync(FULL, p, 8 * i);
        const float2 p2 = make_float2(pi, pi);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = __ffma2_rn(p2, cl[e], acc[i][e]);
      }
    }
    if (mt.last) {
#pragma unroll
      for (int i = 0; i < C::HPW; ++i) {
        const int h = hbase + i;
        const float mi = __shfl_sync(FULL, m_run, 8 * i);
        const float li = __shfl_sync(FULL, l_run, 8 * i);
        if (h >= a.H) continue;
        const float inv = li > 0.f ? 1.f / li : 0.f;
        const size_t bh = (size_t)mt.b * a.H + h;
        float4 *dst = reinterpret_cast<float4 *>(a.part_o + (bh * a.max_splits + mt.split) * MLA_LAT + lane * 16);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          dst[e] = make_float4(acc[i][2 * e].x * inv, acc[i][2 * e].y * inv, acc[i][2 * e + 1].x * inv,
                               acc[i][2 * e + 1].y * inv);
        if (lane == 0) a.part_lse[bh * a.max_splits + mt.split] = (li > 0.f) ? mi + __log2f(li) : -INFINITY;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

// ----------------------------------------------------------------------------- tensor-core projections
__device__ __forceinline__ uint32_t pack_u16(uint16_t lo, uint16_t hi) {
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// q_lat[b][h][j] = sum_d q_nope[b][h][d] * W_UK[h][d][j].  Grid (H, 4 chunks of 128 j), 4 warps.
__global__ void __launch_bounds__(128) q_absorb_kernel(const uint16_t *q, const uint16_t *w_uk, float *q_lat, int B,
                                                       int H) {
  __shared__ __align__(16) uint16_t w[MLA_NOPE][128];
  const int h = blockIdx.x, j0 = blockIdx.y * 128;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint16_t *wsrc = w_uk + (size_t)h * MLA_NOPE * MLA_LAT + j0;
  for (int i = tid; i < MLA_NOPE * 16; i += 128) {
    const int d = i >> 4, c = i & 15;
    *reinterpret_cast<uint4 *>(&w[d][c * 8]) = *reinterpret_cast<const uint4 *>(wsrc + (size_t)d * MLA_LAT + c * 8);
  }
  __syncthreads();
  const int g = lane >> 2, tq = lane & 3;
  for (int m0 = 0; m0 < B; m0 += 16) {
    float acc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
    const int r0 = m0 + g, r1 = m0 + g + 8;
    const uint16_t *q0 = q + ((size_t)r0 * H + h) * MLA_QD;
    const uint16_t *q1 = q + ((size_t)r1 * H + h) * MLA_QD;
#pragma unroll
    for (int k0 = 0; k0 < MLA_NOPE; k0 += 16) {
      uint32_t af[4];
      af[0] = r0 < B ? *reinterpret_cast<const uint32_t *>(q0 + k0 + 2 * tq) : 0u;
      af[1] = r1 < B ? *reinterpret_cast<const uint32_t *>(q1 + k0 + 2 * tq) : 0u;
      af[2] = r0 < B ? *reinterpret_cast<const uint32_t *>(q0 + k0 + 8 + 2 * tq) : 0u;
      af[3] = r1 < B ? *reinterpret_cast<const uint32_t *>(q1 + k0 + 8 + 2 * tq) : 0u;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int n = warp * 32 + nt * 8 + g;
        uint32_t bf[2];
        bf[0] = pack_u16(w[k0 + 2 * tq][n], w[k0 + 2 * tq + 1][n]);
        bf[1] = pack_u16(w[k0 + 8 + 2 * tq][n], w[k0 + 9 + 2 * tq][n]);
        mma_bf16_16816(acc[nt], af, bf[0], bf[1]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = j0 + warp * 32 + nt * 8 + 2 * tq;
      if (r0 < B) *reinterpret_cast<float2 *>(q_lat + ((size_t)r0 * H + h) * MLA_LAT + col) = make_float2(acc[nt][0], acc[nt][1]);
      if (r1 < B) *reinterpret_cast<float2 *>(q_lat + ((size_t)r1 * H + h) * MLA_LAT + col) = make_float2(acc[nt][2], acc[nt][3]);
    }
  }
}

struct MlaOutArgs {
  const float *part_o, *part_lse;
  const RowInfo *rows;
  const uint16_t *w_uv;
  uint16_t *out;
  float *lse;
  int B, H, max_splits;
};

// Per head h: merge the splits of o_lat (ascending), round to bf16, then
// o[b][h][v] = sum_j W_UV[h][v][j] o_lat[b][j] on the tensor cores.  4 warps.
__global__ void __launch_bounds__(128) mla_out_kernel(const MlaOutArgs a) {
  __shared__ __align__(16) uint16_t ol[16][MLA_LAT + 8];
  const int h = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  for (int m0 = 0; m0 < a.B; m0 += 16) {
    // ---- merge splits of rows m0..m0+15 (thread owns latent dims 4 tid .. 4 tid + 3)
    for (int rr = 0; rr < 16; ++rr) {
      const int b = m0 + rr;
      float o[4] = {0.f, 0.f, 0.f, 0.f};
      float lse2 = -INFINITY;
      if (b < a.B) {
        const RowInfo ri = a.rows[b];
        const int pages = ri.page_hi - ri.page_lo;
        const int ne = ri.nsplit > 0 ? (pages + ri.chunk - 1) / ri.chunk : 0;
        const size_t bh = (size_t)b * a.H + h;
        const float *pl = a.part_lse + bh * a.max_splits;
        float M = -INFINITY;
        for (int c = 0; c < ne; ++c) M = fmaxf(M, pl[c]);
        if (M != -INFINITY) {
          float Z = 0.f;
          for (int c = 0; c < ne; ++c) {
            const float lc = pl[c];
            if (lc == -INFINITY) continue;
            const float wgt = fast_exp2(lc - M);
            Z += wgt;
            const float4 v = *reinterpret_cast<const float4 *>(a.part_o + (bh * a.max_splits + c) * MLA_LAT + tid * 4);
            o[0] += wgt * v.x;
            o[1] += wgt * v.y;
            o[2] += wgt * v.z;
            o[3] += wgt * v.w;
          }
          const float inv = 1.f / Z;
#pragma unroll
          for (int e = 0; e < 4; ++e) o[e] *= inv;
          lse2 = M + __log2f(Z);
        }
        if (tid == 0 && a.lse) a.lse[bh] = lse2 * LN2;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) ol[rr][tid * 4 + e] = f32_to_bf16_bits(o[e]);
    }
    __syncthreads();
    // ---- o = W_UV . o_lat: warp owns v in [32 warp, 32 warp + 32)
    float acc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
    const uint16_t *wv = a.w_uv + (size_t)h * MLA_V * MLA_LAT;
#pragma unroll 4
    for (int k0 = 0; k0 < MLA_LAT; k0 += 16) {
      uint32_t af[4];
      af[0] = *reinterpret_cast<const uint32_t *>(&ol[g][k0 + 2 * tq]);
      af[1] = *reinterpret_cast<const uint32_t *>(&ol[g + 8][k0 + 2 * tq]);
      af[2] = *reinterpret_cast<const uint32_t *>(&ol[g][k0 + 8 + 2 * tq]);
      af[3] = *reinterpret_cast<const uint32_t *>(&ol[g + 8][k0 + 8 + 2 * tq]);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int v = warp * 32 + nt * 8 + g;
        uint32_t bf[2];
        bf[0] = *reinterpret_cast<const uint32_t *>(wv + (size_t)v * MLA_LAT + k0 + 2 * tq);
        bf[1] = *reinterpret_cast<const uint32_t *>(wv + (size_t)v * MLA_LAT + k0 + 8 + 2 * tq);
        mma_bf16_16816(acc[nt], af, bf[0], bf[1]);
      }
    }
    const int r0 = m0 + g, r1 = m0 + g + 8;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = warp * 32 + nt * 8 + 2 * tq;
      if (r0 < a.B)
        *reinterpret_cast<uint32_t *>(a.out + ((size_t)r0 * a.H + h) * MLA_V + col) =
            pack_u16(f32_to_bf16_bits(acc[nt][0]), f32_to_bf16_bits(acc[nt][1]));
      if (r1 < a.B)
        *reinterpret_cast<uint32_t *>(a.out + ((size_t)r1 * a.H + h) * MLA_V + col) =
            pack_u16(f32_to_bf16_bits(acc[nt][2]), f32_to_bf16_bits(acc[nt][3]));
    }
    __syncthreads();
  }
}

// ----------------------------------------------------------------------------- host side
namespace {

constexpr int kMlaMinChunkTokens = 256;
constexpr int kMlaItemsPerCta = 4;
constexpr int kMaxSplits = 1024;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int ilog2(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct MlaPlan {
  int nhg, max_splits, min_chunk_pages, chunk_align;
  size_t off_rows, off_items, off_qlat, off_part_lse, off_part_o, total;
};

int mla_shape(int batch, int H, int max_ctx, int P, int num_splits, MlaPlan *pl) {
  if (batch < 0 || H <= 0 || max_ctx < 0 || num_splits < 0) return PA_ERR_INVALID_ARGUMENT;
  if (num_splits > kMaxSplits) return PA_ERR_UNSUPPORTED;
  if (!is_pow2(P) || P > 256) return PA_ERR_UNSUPPORTED;
  pl->nhg = (H + MlaCfg::HG - 1) / MlaCfg::HG;
  pl->chunk_align = P >= MlaCfg::ST ? 1 : MlaCfg::ST / P;
  int mcp = kMlaMinChunkTokens / P;
  if (mcp < 1) mcp = 1;
  pl->min_chunk_pages = (int)round_up((size_t)mcp, (size_t)pl->chunk_align);
  const long long max_pages = max_ctx == 0 ? 1 : ((long long)max_ctx + P - 1) / P;
  pl->max_splits = num_splits > 0 ? num_splits : (int)((max_pages + pl->min_chunk_pages - 1) / pl->min_chunk_pages);
  if (pl->max_splits < 1) pl->max_splits = 1;
  const size_t B = (size_t)(batch > 0 ? batch : 1);
  const size_t items = B * (size_t)pl->nhg * (size_t)pl->max_splits;
  if (items > (size_t)INT32_MAX) return PA_ERR_UNSUPPORTED;
  size_t off = sizeof(WsHeader);
  pl->off_rows = off;
  off = round_up(off + B * sizeof(RowInfo), 256);
  pl->off_items = off;
  off = round_up(off + items * sizeof(WorkItem), 256);
  pl->off_qlat = off;
  off = round_up(off + B * (size_t)H * MLA_LAT * sizeof(float), 256);
  pl->off_part_lse = off;
  off = round_up(off + B * (size_t)H * pl->max_splits * sizeof(float), 256);
  pl->off_part_o = off;
  off = round_up(off + B * (size_t)H * pl->max_splits * MLA_LAT * sizeof(float), 256);
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

// [num_pages, P, 576] bf16 viewed as [num_pages][P][9][64]; box = (64, 9, BH tokens, 1 page).
bool encode_cache_map(CUtensorMap *m, const void *base, int num_pages, int P, int BH) {
  auto fn = mla_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {64, 9, (cuuint64_t)P, (cuuint64_t)num_pages};
  cuuint64_t strides[3] = {128, (cuuint64_t)MLA_C * 2, (cuuint64_t)P * MLA_C * 2};
  cuuint32_t box[4] = {64u, 9u, (cuuint32_t)BH, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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
  const int BH = P < MlaCfg::ST ? P : MlaCfg::ST;
  CUtensorMap tm;
  if (!encode_cache_map(&tm, cache, num_pages, P, BH)) return PA_ERR_UNSUPPORTED;
  const int sms = sm_count_mla();
  if (sms <= 0) return PA_ERR_CUDA;

  uint8_t *ws = static_cast<uint8_t *>(workspace);
  WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
  RowInfo *rows = reinterpret_cast<RowInfo *>(ws + pl.off_rows);
  WorkItem *items = reinterpret_cast<WorkItem *>(ws + pl.off_items);
  float *q_lat = reinterpret_cast<float *>(ws + pl.off_qlat);
  float *part_lse = reinterpret_cast<float *>(ws + pl.off_part_lse);
  float *part_o = reinterpret_cast<float *>(ws + pl.off_part_o);
  const long long max_items = (long long)batch * pl.nhg * pl.max_splits;
  const int grid = (int)(max_items < sms ? max_items : sms);

  PlanArgs pa_;
  pa_.context_lens = context_lens;
  pa_.batch = batch;
  pa_.heads_per_row = pl.nhg;
  pa_.page_size = P;
  pa_.log2_page = ilog2(P);
  pa_.window = 0;
  pa_.max_context_len = max_context_len;
  pa_.num_splits = num_splits;
  pa_.max_splits = pl.max_splits;
  pa_.target_items = grid * kMlaItemsPerCta;
  pa_.min_chunk_pages = pl.min_chunk_pages;
  pa_.chunk_align = pl.chunk_align;
  pa_.hdr = hdr;
  pa_.rows = rows;
  pa_.items = items;
  pa_.out = nullptr;  // rows without keys are written by mla_out_kernel
  pa_.lse = nullptr;
  pa_.out_heads = 0;
  pa_.out_dim = 0;
  if (launch_plan(pa_, stream) != cudaSuccess) return PA_ERR_CUDA;
  ++*launches;

  q_absorb_kernel<<<dim3(H, MLA_LAT / 128), 128, 0, stream>>>(static_cast<const uint16_t *>(q),
                                                               static_cast<const uint16_t *>(w_uk), q_lat, batch, H);
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  ++*launches;

  MlaArgs ma;
  ma.q = static_cast<const uint16_t *>(q);
  ma.block_table = block_table;
  ma.q_lat = q_lat;
  ma.part_o = part_o;
  ma.part_lse = part_lse;
  ma.hdr = hdr;
  ma.items = items;
  ma.rows = rows;
  ma.max_pages_per_seq = max_pages_per_seq;
  ma.num_pages = num_pages;
  ma.H = H;
  ma.page_size = P;
  ma.log2_page = ilog2(P);
  ma.max_splits = pl.max_splits;
  ma.qscale = scale * LOG2E;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    if (cudaFuncSetAttribute(mla_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MlaCfg::SMEM) !=
        cudaSuccess)
      return PA_ERR_CUDA;
    configured_device = dev;
  }
  if (ev_before && cudaEventRecord(ev_before, stream) != cudaSuccess) return PA_ERR_CUDA;
  mla_split_kernel<<<grid, MlaCfg::THREADS, MlaCfg::SMEM, stream>>>(tm, ma);
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  ++*launches;
  if (ev_after && cudaEventRecord(ev_after, stream) != cudaSuccess) return PA_ERR_CUDA;

  MlaOutArgs oa;
  oa.part_o = part_o;
  oa.part_lse = part_lse;
  oa.rows = rows;
  oa.w_uv = static_cast<const uint16_t *>(w_uv);
  oa.out = static_cast<uint16_t *>(out);
  oa.lse = lse;
  oa.B = batch;
  oa.H = H;
  oa.max_splits = pl.max_splits;
  mla_out_kernel<<<H, 128, 0, stream>>>(oa);
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  ++*launches;
  return PA_OK;
}

}  // namespace pa
