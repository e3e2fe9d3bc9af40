// pa_gqa.cuh -- GQA paged decode kernels (sm_103a): split-KV attention and combine
// (the work-list planner they consume lives in pa_plan.cu).
//
// Method (what is computed) follows the pages: a query row of length L reads
// its keys through the block table, query heads sharing one KV head are served
// together so each KV page is read once per group (vllm.cpp PR #49 "flip
// decode GQA group-swap default ON", mechanism paragraph: grid batch x
// q_heads -> batch x kv_heads), scores go through an f32 online softmax
// (vllm.cpp PR #425, description), the sequence is split over the machine and
// a separate combine merges the splits in ascending order without atomics
// (vllm.cpp kernel-matrix, rows KERNEL-ATTN-FA2 / KERNEL-ATTN-MLA-SPARSE).
//
// GB300 design (how):
//   * plan kernel (1 CTA): turns context_lens into a list of page-aligned work
//     items (row, KV head, head subgroup, chunk), balanced for the SM count,
//     longest first; resets the dynamic work counter.
//   * split kernel: one persistent CTA per SM.  Warp 8 is a TMA producer: it
//     pulls items from the work counter, reads the block table and issues one
//     4-D tensor-map copy per (page fragment, K or V) into an NS-deep ring of
//     32 KB shared-memory stages, signalling mbarrier transaction counts.
//     Warps 0-7 consume: each stage's tokens are split across the 8 warps;
//     within a warp, LPT = D/8 lanes cover one token row with one 16-byte
//     shared load each, so a warp step covers 32/LPT tokens.  Each lane holds
//     q for all G heads of the group over its 8 dims and computes G partial
//     dot products with packed fp32 FMAs; a transpose-reduction over the LPT
//     lanes (log2 G halving exchanges, then a butterfly) leaves lane r with
//     the full score of head r / (LPT/G).  Online softmax is per warp with a
//     lazy rescale (the running max moves only when a score exceeds it by
//     2^8), probabilities go through a small per-warp shared buffer, and P.V
//     accumulates G x 8 fp32 per lane.  At the end of an item the 8 warps
//     merge through the just-consumed stage buffer and write either the final
//     bf16 output (single-split rows) or an fp32 partial + LSE.
//   * combine kernel: one warp per (row, query head), ascending split order.
#pragma once

#include "pa_common.cuh"

namespace pa {

struct RowInfo {
  int32_t lo, L;            // visible token range [lo, L)
  int32_t page_lo, page_hi; // visible pages [page_lo, page_hi)
  int32_t nsplit;           // splits of this row (0: row has no visible key)
  int32_t chunk;            // pages per split
  int32_t pad[2];
};
static_assert(sizeof(RowInfo) == 32, "row info is 32 bytes");

struct PlanArgs {
  const int32_t *context_lens;
  int batch, heads_per_row;  // heads_per_row: (kv head, subgroup) pairs per row (GQA) or 1 (MLA)
  int page_size, log2_page, window, max_context_len;
  int num_splits;            // 0 = automatic
  int max_splits;            // workspace capacity per row
  int target_items;          // automatic mode: aim for this many items
  int min_chunk_pages;       // automatic mode: smallest chunk
  int chunk_align;           // automatic mode: chunk is a multiple of this
  WsHeader *hdr;
  RowInfo *rows;
  WorkItem *items;
};

struct GqaArgs {
  const uint16_t *q;            // [B, Hq, D] bf16
  const int32_t *block_table;   // [B, max_pages_per_seq]
  uint16_t *out;                // [B, Hq, D] bf16
  float *lse;                   // [B, Hq] or null
  float *part_o;                // [B, Hq, max_splits, D]
  float *part_lse;              // [B, Hq, max_splits], log2 units
  WsHeader *hdr;
  const WorkItem *items;
  const RowInfo *rows;
  int max_pages_per_seq, num_pages;
  int Hq, Hkv, G, nsub;
  int page_size, log2_page;
  int max_splits;
  float qscale;                 // scale * log2(e)
};

template <int D_, int GP_>
struct GqaCfg {
  static constexpr int D = D_;
  static constexpr int GP = GP_;                  // heads per subgroup (padded group)
  static constexpr int LPT = D / 8;               // lanes per token row
  static constexpr int TPW = 32 / LPT;            // tokens per warp step
  static constexpr int DUP = LPT / GP;            // lanes holding the same head after the reduction
  static constexpr int NCW = 8;                   // consumer warps
  static constexpr int THREADS = (NCW + 1) * 32;  // + producer warp
  static constexpr int STAGE_BYTES = 32768;       // K + V of one stage
  static constexpr int ST = STAGE_BYTES / (2 * D * 2);  // tokens per stage
  static constexpr int TOKW = ST / NCW;           // tokens per warp per stage
  static constexpr int STEPS = TOKW / TPW;
  static constexpr int NS = 4;                    // ring depth
  static constexpr int QBYTES = GP * D * 2;
  static constexpr int MAXBOX = 128;              // boxes per stage (page_size >= ST/128)
  static constexpr int HR = (GP * D * 4 * NCW <= STAGE_BYTES) ? GP : STAGE_BYTES / (NCW * D * 4);
  static_assert(GP <= LPT, "group must fit the transpose reduction");
  static_assert(STEPS >= 1 && TOKW % TPW == 0, "stage split");
  static_assert(HR >= 1 && GP % HR == 0, "merge rounds");
};

struct alignas(16) StageMeta {
  int32_t end, first, last, masked;
  int32_t b, g, sub, split;
  int32_t tok0, tok_lo, tok_hi, ghead;  // ghead: number of real heads of the subgroup
  uint32_t badmask[4];                   // bit k: box k of the stage was not loaded (bad page)
};

template <class C>
struct GqaSmem {
  static constexpr int OFF_STAGE = 0;
  static constexpr int OFF_Q = OFF_STAGE + C::NS * C::STAGE_BYTES;
  static constexpr int OFF_P = OFF_Q + C::NS * C::QBYTES;
  static constexpr int OFF_ML = OFF_P + C::NCW * C::TOKW * C::GP * 4;
  static constexpr int OFF_ALPHA = OFF_ML + C::NCW * C::GP * 2 * 4;
  static constexpr int OFF_META = OFF_ALPHA + C::NCW * C::GP * 4;
  static constexpr int OFF_BAR = (OFF_META + C::NS * (int)sizeof(StageMeta) + 15) / 16 * 16;
  static constexpr int BYTES = OFF_BAR + 2 * C::NS * 8;
};

template <int N>
__device__ __forceinline__ void load_f32(const float *p, float (&v)[N]) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
      const float4 t = reinterpret_cast<const float4 *>(p)[i];
      v[4 * i] = t.x;
      v[4 * i + 1] = t.y;
      v[4 * i + 2] = t.z;
      v[4 * i + 3] = t.w;
    }
  } else if constexpr (N == 2) {
    const float2 t = *reinterpret_cast<const float2 *>(p);
    v[0] = t.x;
    v[1] = t.y;
  } else {
    v[0] = p[0];
  }
}

template <int D, int GP>
__global__ void __launch_bounds__(GqaCfg<D, GP>::THREADS, 1)
    gqa_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const GqaArgs a) {
  using C = GqaCfg<D, GP>;
  using S = GqaSmem<C>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
  uint64_t *empty = full + C::NS;
  StageMeta *meta = reinterpret_cast<StageMeta *>(smem + S::OFF_META);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
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
    if (lane == 0) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
    }
    const int n_items = (int)a.hdr->n_items;
    const int P = a.page_size;
    const int BH = P < C::ST ? P : C::ST;  // tokens per box
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
      const int g = it.sub / a.nsub, sub = it.sub % a.nsub;
      const int ghead = min(C::GP, a.G - sub * C::GP);
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
        uint8_t *kdst = smem + S::OFF_STAGE + s * C::STAGE_BYTES;
        uint8_t *vdst = kdst + C::STAGE_BYTES / 2;
        uint32_t bad[4] = {0, 0, 0, 0};
        int nvalid = 0;
        int phys_of[C::MAXBOX / 32];
        bool load_of[C::MAXBOX / 32];
#pragma unroll
        for (int kk = 0; kk < C::MAXBOX / 32; ++kk) {
          const int k = kk * 32 + lane;
          bool load = false, isbad = false;
          int phys = 0;
          if (k < nbox) {
            const int btok = tok0 + k * BH;
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
          phys_of[kk] = phys;
          load_of[kk] = load;
          bad[kk] = __ballot_sync(FULL, isbad);
          nvalid += __popc(__ballot_sync(FULL, load));
        }
        const bool first = (t == 0), last = (t == n_stages - 1);
        if (lane == 0) {
          StageMeta &m = meta[s];
          m.end = 0;
          m.first = first;
          m.last = last;
          m.b = it.b;
          m.g = g;
          m.sub = sub;
          m.split = it.split;
          m.tok0 = tok0;
          m.tok_lo = tok_lo;
          m.tok_hi = tok_hi;
          m.ghead = ghead;
          m.masked = (tok0 < tok_lo) || (tok0 + C::ST > tok_hi) || (bad[0] | bad[1] | bad[2] | bad[3]);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) m.badmask[kk] = bad[kk];
          const uint32_t qbytes = first ? (uint32_t)(ghead * D * 2) : 0u;
          mbar_arrive_expect_tx(&full[s], (uint32_t)nvalid * (uint32_t)(BH * D * 2 * 2) + qbytes);
          if (first) {
            const uint16_t *qsrc = a.q + ((size_t)it.b * a.Hq + (size_t)g * a.G + (size_t)sub * C::GP) * D;
            bulk_load(smem + S::OFF_Q + s * C::QBYTES, qsrc, qbytes, &full[s]);
          }
        }
        __syncwarp();
#pragma unroll
        for (int kk = 0; kk < C::MAXBOX / 32; ++kk) {
          if (load_of[kk]) {
            const int k = kk * 32 + lane;
            const int btok = tok0 + k * BH;
            const int slot = btok & (P - 1);
            tma_load_4d(kdst + k * BH * D * 2, &tm_k, 0, g, slot, phys_of[kk], &full[s]);
            tma_load_4d(vdst + k * BH * D * 2, &tm_v, 0, g, slot, phys_of[kk], &full[s]);
          }
        }
      }
    }
    if (!ok) {
      // A wait gave up: let the copies this warp issued land before the CTA exits.
      const uint32_t first = j > (uint32_t)C::NS ? j - C::NS : 0u;
      for (uint32_t i = first; i < j; ++i) mbar_wait(&full[i % C::NS], (i / C::NS) & 1, status);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int r = lane % C::LPT;   // 16-byte column of the token row
  const int tg = lane / C::LPT;  // token within the warp step
  const int fh = r / C::DUP;     // head held after the transpose reduction
  float *ps = reinterpret_cast<float *>(smem + S::OFF_P) + warp * C::TOKW * C::GP;
  float *sm_ml = reinterpret_cast<float *>(smem + S::OFF_ML);
  float *sm_alpha = reinterpret_cast<float *>(smem + S::OFF_ALPHA) + warp * C::GP;

  float2 qf[C::GP][4];
  float2 acc[C::GP][4];
  float m_run = -INFINITY, l_run = 0.f;
  const float TAU = 8.f;

  for (uint32_t j = 0;; ++j) {
    const int s = j % C::NS;
    if (!mbar_wait(&full[s], (j / C::NS) & 1, status)) break;
    const StageMeta &mt = meta[s];
    if (mt.end) break;
    const uint8_t *kst = smem + S::OFF_STAGE + s * C::STAGE_BYTES;
    const uint8_t *vst = kst + C::STAGE_BYTES / 2;
    if (mt.first) {
      const uint16_t *qs = reinterpret_cast<const uint16_t *>(smem + S::OFF_Q + s * C::QBYTES);
#pragma unroll
      for (int i = 0; i < C::GP; ++i) {
        const int h = i ^ fh;
        if (h < mt.ghead) {
          const uint4 u = *reinterpret_cast<const uint4 *>(qs + h * D + r * 8);
          bf16x8_to_f32(u, qf[i]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            qf[i][e].x *= a.qscale;
            qf[i][e].y *= a.qscale;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) qf[i][e] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][e] = make_float2(0.f, 0.f);
      }
      m_run = -INFINITY;
      l_run = 0.f;
    }

    // ---- scores
    float sc[C::STEPS];
#pragma unroll
    for (int i = 0; i < C::STEPS; ++i) {
      const int tok = warp * C::TOKW + i * C::TPW + tg;
      const uint4 ku = *reinterpret_cast<const uint4 *>(kst + (tok * D + r * 8) * 2);
      float2 kf[4];
      bf16x8_to_f32(ku, kf);
      float part[C::GP];
#pragma unroll
      for (int h = 0; h < C::GP; ++h) {
        float2 t2 = __fmul2_rn(qf[h][0], kf[0]);
        t2 = __ffma2_rn(qf[h][1], kf[1], t2);
        t2 = __ffma2_rn(qf[h][2], kf[2], t2);
        t2 = __ffma2_rn(qf[h][3], kf[3], t2);
        part[h] = t2.x + t2.y;
      }
      // transpose reduction: halve the head set at each exchange
#pragma unroll
      for (int half = C::GP / 2, mask = C::LPT / 2; half >= 1; half >>= 1, mask >>= 1) {
#pragma unroll
        for (int h = 0; h < half; ++h) part[h] += __shfl_xor_sync(FULL, part[h + half], mask);
      }
#pragma unroll
      for (int mask = C::DUP / 2; mask >= 1; mask >>= 1) part[0] += __shfl_xor_sync(FULL, part[0], mask);
      float sv = part[0];
      if (mt.masked) {
        const int ltok = mt.tok0 + tok;
        const int box = tok / (a.page_size < C::ST ? a.page_size : C::ST);
        const bool bad = (mt.badmask[box >> 5] >> (box & 31)) & 1u;
        if (ltok < mt.tok_lo || ltok >= mt.tok_hi || bad) sv = -INFINITY;
      }
      sc[i] = sv;
    }

    // ---- online softmax (per warp, per head fh)
    float tmax = sc[0];
#pragma unroll
    for (int i = 1; i < C::STEPS; ++i) tmax = fmaxf(tmax, sc[i]);
#pragma unroll
    for (int mask = C::LPT; mask < 32; mask <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(FULL, tmax, mask));
    const bool need = tmax > m_run + TAU;
    if (__any_sync(FULL, need)) {
      const float m_new = fmaxf(m_run, tmax);
      const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
      l_run *= alpha;
      m_run = m_new;
      if ((r % C::DUP) == 0 && tg == 0) sm_alpha[fh] = alpha;
      __syncwarp();
      float al[C::GP];
      load_f32<C::GP>(sm_alpha, al);
#pragma unroll
      for (int h = 0; h < C::GP; ++h) {
        const float2 a2 = make_float2(al[h], al[h]);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[h][e] = __fmul2_rn(a2, acc[h][e]);
      }
    }
#pragma unroll
    for (int i = 0; i < C::STEPS; ++i) {
      const float p = (sc[i] == -INFINITY) ? 0.f : fast_exp2(sc[i] - m_run);
      l_run += p;
      if ((r % C::DUP) == 0) ps[(i * C::TPW + tg) * C::GP + fh] = p;
    }
    __syncwarp();

    // ---- P.V
#pragma unroll
    for (int i = 0; i < C::STEPS; ++i) {
      const int tok = warp * C::TOKW + i * C::TPW + tg;
      uint4 vu = *reinterpret_cast<const uint4 *>(vst + (tok * D + r * 8) * 2);
      if (mt.masked) {
        const int ltok = mt.tok0 + tok;
        const int box = tok / (a.page_size < C::ST ? a.page_size : C::ST);
        const bool bad = (mt.badmask[box >> 5] >> (box & 31)) & 1u;
        if (ltok < mt.tok_lo || ltok >= mt.tok_hi || bad) vu = make_uint4(0, 0, 0, 0);
      }
      float2 vf[4];
      bf16x8_to_f32(vu, vf);
      float pv[C::GP];
      load_f32<C::GP>(ps + (i * C::TPW + tg) * C::GP, pv);
#pragma unroll
      for (int h = 0; h < C::GP; ++h) {
        const float2 p2 = make_float2(pv[h], pv[h]);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[h][e] = __ffma2_rn(p2, vf[e], acc[h][e]);
      }
    }
    __syncwarp();

    if (mt.last) {
      // ---- end of item: merge token groups, then the 8 warps
#pragma unroll
      for (int mask = C::LPT; mask < 32; mask <<= 1) {
        l_run += __shfl_xor_sync(FULL, l_run, mask);
#pragma unroll
        for (int h = 0; h < C::GP; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[h][e].x += __shfl_xor_sync(FULL, acc[h][e].x, mask);
            acc[h][e].y += __shfl_xor_sync(FULL, acc[h][e].y, mask);
          }
      }
      named_bar(1, C::NCW * 32);  // every warp is done with this stage's K/V
      float *mg = reinterpret_cast<float *>(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
      if ((r % C::DUP) == 0 && tg == 0) {
        sm_ml[(warp * C::GP + fh) * 2] = m_run;
        sm_ml[(warp * C::GP + fh) * 2 + 1] = l_run;
      }
      const RowInfo ri = a.rows[mt.b];
      const bool direct = ri.nsplit == 1;
      const int hq0 = mt.g * a.G + mt.sub * C::GP;
#pragma unroll
      for (int h0 = 0; h0 < C::GP; h0 += C::HR) {
        if (tg == 0) {
#pragma unroll
          for (int hh = 0; hh < C::HR; ++hh) {
            float4 *dst = reinterpret_cast<float4 *>(mg + ((warp * C::HR + hh) * D + r * 8));
            dst[0] = make_float4(acc[h0 + hh][0].x, acc[h0 + hh][0].y, acc[h0 + hh][1].x, acc[h0 + hh][1].y);
            dst[1] = make_float4(acc[h0 + hh][2].x, acc[h0 + hh][2].y, acc[h0 + hh][3].x, acc[h0 + hh][3].y);
          }
        }
        named_bar(1, C::NCW * 32);
        for (int e = tid; e < C::HR * D; e += C::NCW * 32) {
          const int hh = e / D, d = e % D;
          const int h = h0 + hh;
          if (h >= mt.ghead) continue;
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < C::NCW; ++w) M = fmaxf(M, sm_ml[(w * C::GP + h) * 2]);
          float o = 0.f, lsum = 0.f;
          if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < C::NCW; ++w) {
              const float mw = sm_ml[(w * C::GP + h) * 2];
              const float wgt = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
              lsum += sm_ml[(w * C::GP + h) * 2 + 1] * wgt;
              o += mg[(w * C::HR + hh) * D + d] * wgt;
            }
            o = o / lsum;
          }
          const float lse2 = (M == -INFINITY || lsum == 0.f) ? -INFINITY : M + __log2f(lsum);
          const size_t bh = (size_t)mt.b * a.Hq + hq0 + h;
          if (direct) {
            a.out[bh * D + d] = f32_to_bf16_bits(o);
            if (d == 0 && a.lse) a.lse[bh] = lse2 * LN2;
          } else {
            a.part_o[(bh * a.max_splits + mt.split) * D + d] = o;
            if (d == 0) a.part_lse[bh * a.max_splits + mt.split] = lse2;
          }
        }
        named_bar(1, C::NCW * 32);
      }
      fence_proxy_async_smem();  // generic writes to the stage buffer precede its next TMA fill
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

struct CombineArgs {
  uint16_t *out;
  float *lse;
  const float *part_o;
  const float *part_lse;
  const RowInfo *rows;
  int batch, Hq, D, max_splits;
};

// One warp per (row, query head); splits merged in ascending order.
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= a.batch * a.Hq) return;
  const int b = wid / a.Hq;
  const RowInfo ri = a.rows[b];
  constexpr int PER = D / 32;
  const size_t bh = (size_t)wid;
  if (ri.nsplit == 1) return;  // written by the split kernel
  float o[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) o[e] = 0.f;
  float lse2 = -INFINITY;
  if (ri.nsplit > 1) {
    const int pages = ri.page_hi - ri.page_lo;
    const int ne = (pages + ri.chunk - 1) / ri.chunk;  // non-empty splits
    const float *pl = a.part_lse + bh * a.max_splits;
    float M = -INFINITY;
    for (int c = 0; c < ne; ++c) M = fmaxf(M, pl[c]);
    if (M != -INFINITY) {
      float Z = 0.f;
      for (int c = 0; c < ne; ++c) {
        const float lc = pl[c];
        if (lc == -INFINITY) continue;
        const float w = fast_exp2(lc - M);
        Z += w;
        const float *po = a.part_o + (bh * a.max_splits + c) * D + lane * PER;
#pragma unroll
        for (int e = 0; e < PER; ++e) o[e] += w * po[e];
      }
      const float inv = 1.f / Z;
#pragma unroll
      for (int e = 0; e < PER; ++e) o[e] *= inv;
      lse2 = M + __log2f(Z);
    }
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) a.out[bh * D + lane * PER + e] = f32_to_bf16_bits(o[e]);
  if (lane == 0 && a.lse) a.lse[bh] = lse2 * LN2;
}

}  // namespace pa
