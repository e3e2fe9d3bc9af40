// pa_gqa.cuh -- GQA paged decode, split-KV attention and combine kernels
// (sm_103a), plus the work-list types shared with the planner (pa_plan.cu) and
// the MLA path.
//
// Method (what is computed) follows the pages: a query row of length L reads
// its keys through the block table; the query heads sharing one KV head are
// served together so each KV page is read once per group (vllm.cpp PR #49
// "flip decode GQA group-swap default ON", mechanism paragraph: the decode
// grid becomes batch x kv_heads and the group's heads become the rows of one
// tile); scores go through an f32 online softmax (vllm.cpp PR #425,
// description); the KV sequence is split over the machine and a separate
// combine merges the splits in a fixed ascending order without atomics on the
// data (vllm.cpp kernel-matrix, rows KERNEL-ATTN-FA2 and KERNEL-ATTN-MLA-SPARSE).
//
// GB300 design (how):
//   * one persistent CTA per SM: the last warp is a TMA producer that pulls
//     work items (row, KV head, 16-head subgroup, page-aligned chunk) from a
//     device queue and issues 4-D tensor-map copies of whole page fragments
//     into a ring of shared-memory stages (64 tokens of K and V each), with
//     the 128-byte swizzle so tensor-core fragment loads are bank-conflict
//     free.  Block-table entries are read 32 pages at a time into a register
//     window (lane l holds entry l) with the next window already in flight,
//     and the next item is fetched in dependent steps spread over the current
//     item's stages, so no stage waits on a global load;
//   * the consumer warps take 16 tokens of every stage per token group (four
//     groups per stage; for head_dim <= 128 two warps share a group, both
//     computing its scores and each accumulating half of the P.V columns, so
//     two warps per SM sub-partition hide each other's latency).  The group's
//     (up to 16) query heads are the M rows of mma.sync m16n8k16 bf16 tiles,
//     so S = Q K^T and O += P V cost one tensor-core instruction per 8 tokens
//     x 16 dims.  The online softmax (running max with a lazy rescale, fp32
//     denominator) runs on the CUDA cores; P is rounded to bf16 only as the
//     MMA operand;
//   * at the end of an item the token groups merge through the consumed stage
//     buffer; a single-split row writes the final bf16 output and LSE, a split
//     writes an fp32 partial (normalised output + LSE);
//   * the combine kernel (a programmatic dependent launch, so its launch hides
//     under the split kernel's tail) merges the splits of every row with two
//     or more of them, one warp per (row, query head), in ascending order.
#pragma once

#include "pa_common.cuh"

namespace pa {

struct RowInfo {
  int32_t lo, L;             // visible token range [lo, L)
  int32_t page_lo, page_hi;  // visible pages [page_lo, page_hi)
  int32_t nsplit;            // splits of this row (0: no visible key)
  int32_t chunk;             // pages per split
  int32_t full_off;          // exclusive prefix of full chunks over rows
  int32_t tail_off;          // exclusive prefix of tail chunks over rows
};
static_assert(sizeof(RowInfo) == 32, "row info is 32 bytes");

struct PlanArgs {
  const int32_t *context_lens;
  int batch, heads_per_row;  // (KV head, subgroup) pairs per row (GQA) or head groups (MLA)
  int page_size, log2_page, window, max_context_len;
  int num_splits;            // 0 = automatic
  int max_splits;            // workspace capacity per row
  int target_items;          // automatic mode: aim for this many items
  int min_chunk_pages;       // automatic mode: smallest chunk
  int chunk_align;           // automatic mode: chunk is a multiple of this
  WsHeader *hdr;
  RowInfo *rows;
  WorkItem *items;
  uint16_t *out;             // rows without keys get out = 0, lse = -inf (or null: not written)
  float *lse;
  int out_heads, out_dim;
};

// Non-empty splits of a row.
__device__ __forceinline__ int row_nonempty(const RowInfo &r) {
  const int pages = r.page_hi - r.page_lo;
  return pages > 0 ? (pages + r.chunk - 1) / r.chunk : 0;
}

struct GqaArgs {
  const uint16_t *q;            // [B, Hq, D] bf16
  const int32_t *block_table;   // [B, max_pages_per_seq]
  uint16_t *out;                // [B, Hq, D] bf16
  float *lse;                   // [B, Hq] or null
  float *part_o;                // [B, Hq, max_splits, D]
  float *part_lse;              // [B, Hq, max_splits], log2 units
  WsHeader *hdr;
  const WorkItem *items;
  int max_pages_per_seq, num_pages;
  int Hq, Hkv, G, nsub;
  int page_size, log2_page;
  int max_splits;
  float qscale;                 // scale * log2(e)
};

template <int D_>
struct GqaCfg {
  static constexpr int D = D_;
  static constexpr int M = 16;                     // MMA rows = query heads per subgroup
  static constexpr int TG = 4;                     // token groups per stage
  static constexpr int DSPLIT = D <= 128 ? 2 : 1;  // warps sharing a token group (each: D / DSPLIT of P.V)
  static constexpr int NCW = TG * DSPLIT;          // consumer warps
  static constexpr int THREADS = (NCW + 1) * 32;   // + producer warp
  static constexpr int TW = 16;                    // tokens per token group per stage
  static constexpr int ST = TG * TW;               // tokens per stage
  static constexpr int NT_PV = D / 8 / DSPLIT;     // P.V n-tiles per warp
  static constexpr int NQ = D / 64;                // 128-byte swizzle planes along D
  static constexpr int PLANE = ST * 128;           // bytes of one plane (ST rows x 64 dims)
  static constexpr int KV_BYTES = NQ * PLANE;      // K (or V) of one stage
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int NS = (196608 / STAGE_BYTES) < 8 ? (196608 / STAGE_BYTES) : 8;
  static constexpr int QBYTES = M * D * 2;
  static constexpr int NACC = 2;                   // independent QK accumulators
  static_assert(M * D * 4 * TG <= STAGE_BYTES, "merge area fits in one stage");
};

struct alignas(16) StageMeta {
  int32_t end, first, last, masked;
  int32_t b, g, sub, split;
  int32_t tok0, tok_lo, tok_hi, ghead;  // ghead: real heads of the subgroup
  uint32_t badmask;                     // bit k: box k of the stage was not loaded
  int32_t nsplit, ne, pad0;             // splits / non-empty splits of the item's row
};

template <class C>
struct GqaSmem {
  static constexpr int OFF_STAGE = 0;
  static constexpr int OFF_Q = OFF_STAGE + C::NS * C::STAGE_BYTES;
  static constexpr int OFF_ML = OFF_Q + C::NS * C::QBYTES;
  static constexpr int OFF_META = OFF_ML + C::TG * C::M * 2 * 4;
  static constexpr int OFF_BAR = OFF_META + C::NS * (int)sizeof(StageMeta);
  static constexpr int USED = OFF_BAR + 2 * C::NS * 8;
  static constexpr int BYTES = USED + 1024;  // slack to align the base to 1024 bytes
};

// Byte offset of 16-byte chunk `chunk` (along D) of token row `tok` in a
// stage's K or V block: planes of 64 dims, 128-byte rows, chunk ^ (row & 7)
// (the TMA 128-byte swizzle; every box starts on a 1024-byte boundary).
template <class C>
__device__ __forceinline__ uint32_t kv_off(int tok, int chunk) {
  return (uint32_t)((chunk >> 3) * C::PLANE + tok * 128 + (((chunk & 7) ^ (tok & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(GqaCfg<D>::THREADS, 1)
    gqa_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const GqaArgs a) {
  using C = GqaCfg<D>;
  using S = GqaSmem<C>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the 128-byte swizzle pattern repeats every 1024 bytes: start the stages on such a boundary
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
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
  if (warp == C::NCW && lane == 0) {
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }
  __syncthreads();
  pdl_wait();               // the plan written by the previous kernel is visible from here on
  pdl_launch_dependents();  // the combine kernel may be scheduled; it waits for this grid to finish
  uint32_t *status = &a.hdr->status;

  if (warp == C::NCW) {
    // ------------------------------------------------------------ producer
    const int n_items = (int)a.hdr->n_items;
    const int P = a.page_size;
    const int BH = P < C::ST ? P : C::ST;  // tokens per box
    const int nbox = C::ST / BH;
    uint32_t j = 0;
    bool ok = true;
    // next-item fetch: 0 idle, 1 ticket taken, 2 descriptor loaded, 3 first window loaded
    int pstate = 0;
    uint32_t nticket = 0;
    int nidx = 0, nwin = 0;
    WorkItem nit = {};
    auto step = [&]() {
      if (pstate == 0) {
        if (lane == 0) nticket = atomicAdd(&a.hdr->item_counter, 1u);
        pstate = 1;
      } else if (pstate == 1) {
        nidx = __shfl_sync(FULL, (int)nticket, 0);
        if (nidx < n_items) nit = a.items[nidx];
        pstate = 2;
      } else if (pstate == 2) {
        if (nidx < n_items) {
          const int np = nit.page_end - nit.page_begin;
          nwin = lane < np ? a.block_table[(size_t)nit.b * a.max_pages_per_seq + nit.page_begin + lane] : 0;
        }
        pstate = 3;
      }
    };
    step();
    step();
    step();
    while (ok) {
      if (nidx >= n_items) {
        const int s = j % C::NS;
        const uint32_t u = j / C::NS;
        if (u > 0) ok = mbar_wait(&empty[s], (u - 1) & 1, status);
        if (ok && lane == 0) {
          meta[s].end = 1;
          mbar_arrive(&full[s]);
        }
        break;
      }
      const WorkItem it = nit;
      int cwin = nwin;  // block-table window `wi` of this item
      int wi = 0;
      pstate = 0;
      step();  // take the next ticket right away
      const int g = it.sub / a.nsub, sub = it.sub % a.nsub;
      const int ghead = min(C::M, a.G - sub * C::M);
      const int npages = it.page_end - it.page_begin;
      const int T0 = it.page_begin * P, T1 = it.page_end * P;
      const int tok_lo = it.tok_lo, tok_hi = it.tok_hi;
      const int n_stages = (T1 - T0 + C::ST - 1) / C::ST;
      const int32_t *bt_item = a.block_table + (size_t)it.b * a.max_pages_per_seq + it.page_begin;
      int fwin = (lane + 32 < npages) ? bt_item[32 + lane] : 0;  // window wi + 1, in flight
      const int nsplit = it.splits >> 16, ne = it.splits & 0xffff;
      for (int t = 0; t < n_stages && ok; ++t, ++j) {
        const int s = j % C::NS;
        const uint32_t u = j / C::NS;
        if (u > 0) ok = mbar_wait(&empty[s], (u - 1) & 1, status);
        if (!ok) break;
        const int tok0 = T0 + t * C::ST;
        // the pages of one stage never straddle a 32-page window
        const int pwin = ((tok0 - T0) >> a.log2_page) >> 5;
        while (wi < pwin) {
          cwin = fwin;
          ++wi;
          const int nxt = 32 * (wi + 1) + lane;
          fwin = nxt < npages ? bt_item[nxt] : 0;
        }
        bool load = false, isbad = false;
        const int btok = tok0 + lane * BH;
        const int pi = (btok - T0) >> a.log2_page;  // page index within the item
        const int phys = __shfl_sync(FULL, cwin, pi & 31);
        if (lane < nbox && btok < tok_hi && btok + BH > tok_lo) {
          if (phys < 0 || phys >= a.num_pages) {
            isbad = true;
            atomicOr(status, PA_DEV_BAD_PAGE);
          } else {
            load = true;
          }
        }
        const uint32_t bad = __ballot_sync(FULL, isbad);
        const int nvalid = __popc(__ballot_sync(FULL, load));
        const bool first = (t == 0), last = (t == n_stages - 1);
        uint8_t *kdst = smem + S::OFF_STAGE + s * C::STAGE_BYTES;
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
          m.badmask = bad;
          m.nsplit = nsplit;
          m.ne = ne;
          m.masked = (tok0 < tok_lo) || (tok0 + C::ST > tok_hi) || bad != 0;
          const uint32_t qbytes = first ? (uint32_t)(ghead * D * 2) : 0u;
          mbar_arrive_expect_tx(&full[s], (uint32_t)nvalid * (uint32_t)(BH * D * 2 * 2) + qbytes);
          if (first) {
            const uint16_t *qsrc = a.q + ((size_t)it.b * a.Hq + (size_t)g * a.G + (size_t)sub * C::M) * D;
            bulk_load(smem + S::OFF_Q + s * C::QBYTES, qsrc, qbytes, &full[s]);
          }
        }
        __syncwarp();
        if (load) {
          const int slot = btok & (P - 1);
#pragma unroll
          for (int dq = 0; dq < C::NQ; ++dq) {
            uint8_t *dst = kdst + dq * C::PLANE + lane * BH * 128;
            tma_load_4d(dst, &tm_k, dq * 64, g, slot, phys, &full[s]);
            tma_load_4d(dst + C::KV_BYTES, &tm_v, dq * 64, g, slot, phys, &full[s]);
          }
        }
        // advance the next-item fetch at stages ~n/3 and ~2n/3, so each dependent load has a
        // third of the item's stages to land before its value is needed
        if (pstate < 3 && (t + 1) * 3 >= pstate * n_stages) step();
      }
      while (pstate < 3) step();
    }
    if (!ok) {
      // A wait gave up: let the copies this warp issued land before the CTA exits.
      const uint32_t first = j > (uint32_t)C::NS ? j - C::NS : 0u;
      for (uint32_t i = first; i < j; ++i) mbar_wait(&full[i % C::NS], (i / C::NS) & 1, status);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ct = tid;                               // consumer thread index
  const int g8 = lane >> 2, tq = lane & 3;          // MMA fragment row / column pair
  const int lm_mat = lane >> 3, lm_row = lane & 7;  // ldmatrix: matrix / row this lane addresses
  const int tgrp = warp % C::TG;                    // token group of this warp
  const int dh = warp / C::TG;                      // which 1/DSPLIT of the P.V columns it owns
  const int wbase = tgrp * C::TW;                   // first stage token of this warp
  const int nd0 = dh * C::NT_PV;                    // first P.V n-tile of this warp
  float *sm_ml = reinterpret_cast<float *>(smem + S::OFF_ML);
  const float TAU = 8.f;

  uint32_t qa[D / 16][4];   // Q A-fragments (rows = heads)
  float acc[C::NT_PV][4];   // O C-fragments of this warp's columns: [n-tile][row g8 x2, row g8+8 x2]
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  int ghead = 0;

  for (uint32_t j = 0;; ++j) {
    const int s = j % C::NS;
    if (!mbar_wait(&full[s], (j / C::NS) & 1, status)) break;
    const StageMeta &mt = meta[s];
    if (mt.end) break;
    const uint32_t kbase = smem_u32(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
    const uint32_t vbase = kbase + C::KV_BYTES;
    if (mt.first) {
      ghead = mt.ghead;
      const uint16_t *qs = reinterpret_cast<const uint16_t *>(smem + S::OFF_Q + s * C::QBYTES);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int c0 = ks * 16 + 2 * tq;
        qa[ks][0] = g8 < ghead ? *reinterpret_cast<const uint32_t *>(qs + g8 * D + c0) : 0u;
        qa[ks][1] = g8 + 8 < ghead ? *reinterpret_cast<const uint32_t *>(qs + (g8 + 8) * D + c0) : 0u;
        qa[ks][2] = g8 < ghead ? *reinterpret_cast<const uint32_t *>(qs + g8 * D + c0 + 8) : 0u;
        qa[ks][3] = g8 + 8 < ghead ? *reinterpret_cast<const uint32_t *>(qs + (g8 + 8) * D + c0 + 8) : 0u;
      }
#pragma unroll
      for (int n = 0; n < C::NT_PV; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
    }

    // ---- S = Q K^T for the group's 16 tokens (two n-tiles of 8); the k-steps are
    // spread over NACC independent accumulators so no long chain of dependent MMAs forms
    float sv[2][4];
    {
      float sp[C::NACC][2][4];
#pragma unroll
      for (int q = 0; q < C::NACC; ++q)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) sp[q][nt][0] = sp[q][nt][1] = sp[q][nt][2] = sp[q][nt][3] = 0.f;
#pragma unroll
      for (int ks2 = 0; ks2 < D / 32; ++ks2) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          uint32_t b[4];
          ldmatrix_x4(b, kbase + kv_off<C>(wbase + nt * 8 + lm_row, 4 * ks2 + lm_mat));
          mma_bf16_16816(sp[(2 * ks2) % C::NACC][nt], qa[2 * ks2], b[0], b[1]);
          mma_bf16_16816(sp[(2 * ks2 + 1) % C::NACC][nt], qa[2 * ks2 + 1], b[2], b[3]);
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
    const bool masked = mt.masked;
    const int bh_tokens = a.page_size < C::ST ? a.page_size : C::ST;
    // scale, mask (invalid tokens and padded head rows -> -inf)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float v = sv[nt][e] * a.qscale;
        const int row = (e < 2) ? g8 : g8 + 8;
        bool valid = row < ghead;
        if (masked) {
          const int stok = wbase + nt * 8 + 2 * tq + (e & 1);
          const int ltok = mt.tok0 + stok;
          valid = valid && ltok >= mt.tok_lo && ltok < mt.tok_hi && !((mt.badmask >> (stok / bh_tokens)) & 1u);
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
      // the denominator (and so the LSE) sums the fp32 weights; only the MMA operand is rounded
      l0 += (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
      l1 += (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
    }
    if (masked) {
      // V rows of keys that are not attended (outside [lo, L), unloaded boxes) may hold
      // anything, NaN included: zero this warp's columns of them so that 0 x row stays 0.
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
    // ---- O += P V (k = the group's 16 tokens), this warp's columns
    {
      const int tok = wbase + (lm_mat & 1) * 8 + lm_row;
#pragma unroll
      for (int nd = 0; nd < C::NT_PV; nd += 2) {
        uint32_t b[4];
        ldmatrix_x4_trans(b, vbase + kv_off<C>(tok, nd0 + nd + (lm_mat >> 1)));
        mma_bf16_16816(acc[nd], pa, b[0], b[1]);
        mma_bf16_16816(acc[nd + 1], pa, b[2], b[3]);
      }
    }

    if (mt.last) {
      // ---- end of item: merge the token groups through this stage's buffer
      l0 += __shfl_xor_sync(FULL, l0, 1);
      l0 += __shfl_xor_sync(FULL, l0, 2);
      l1 += __shfl_xor_sync(FULL, l1, 1);
      l1 += __shfl_xor_sync(FULL, l1, 2);
      named_bar(1, C::NCW * 32);  // all warps are done reading this stage
      float *mg = reinterpret_cast<float *>(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
      // merge-area column of (head h, dim d) is d ^ (4 (h & 7)): rows of one fragment hit distinct banks
#pragma unroll
      for (int n = 0; n < C::NT_PV; ++n) {
        const int d = ((nd0 + n) * 8 + 2 * tq) ^ (4 * g8);
        *reinterpret_cast<float2 *>(mg + (tgrp * C::M + g8) * D + d) = make_float2(acc[n][0], acc[n][1]);
        *reinterpret_cast<float2 *>(mg + (tgrp * C::M + g8 + 8) * D + d) = make_float2(acc[n][2], acc[n][3]);
      }
      if (tq == 0 && dh == 0) {  // both column halves of a token group hold the same (m, l)
        sm_ml[(tgrp * C::M + g8) * 2] = m0;
        sm_ml[(tgrp * C::M + g8) * 2 + 1] = l0;
        sm_ml[(tgrp * C::M + g8 + 8) * 2] = m1;
        sm_ml[(tgrp * C::M + g8 + 8) * 2 + 1] = l1;
      }
      named_bar(1, C::NCW * 32);
      const bool direct = mt.nsplit == 1;
      const int hq0 = mt.g * a.G + mt.sub * C::M;
      // per head: weight of each token group, exp2(m_w - M) / sum_w l_w exp2(m_w - M)
      if (ct < ghead) {
        const int h = ct;
        float mw[C::TG], lw[C::TG], M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::TG; ++w) {
          mw[w] = sm_ml[(w * C::M + h) * 2];
          lw[w] = sm_ml[(w * C::M + h) * 2 + 1];
          M = fmaxf(M, mw[w]);
        }
        float L = 0.f, wt[C::TG];
#pragma unroll
        for (int w = 0; w < C::TG; ++w) {
          wt[w] = (mw[w] == -INFINITY) ? 0.f : fast_exp2(mw[w] - M);
          L += lw[w] * wt[w];
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const float lse2 = (M == -INFINITY || L == 0.f) ? -INFINITY : M + __log2f(L);
        const size_t bh = (size_t)mt.b * a.Hq + hq0 + h;
        if (direct) {
          if (a.lse) a.lse[bh] = lse2 * LN2;
        } else {
          a.part_lse[bh * a.max_splits + mt.split] = lse2;
        }
        // each thread only rewrites the m-slots of its own head, which only it reads
#pragma unroll
        for (int w = 0; w < C::TG; ++w) sm_ml[(w * C::M + h) * 2] = wt[w] * inv;
      }
      named_bar(1, C::NCW * 32);
      for (int e = ct; e < ghead * D; e += C::NCW * 32) {
        const int h = e / D, d = e % D;
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < C::TG; ++w) o += mg[(w * C::M + h) * D + (d ^ (4 * (h & 7)))] * sm_ml[(w * C::M + h) * 2];
        const size_t bh = (size_t)mt.b * a.Hq + hq0 + h;
        if (direct) {
          a.out[bh * D + d] = f32_to_bf16_bits(o);
        } else {
          a.part_o[(bh * a.max_splits + mt.split) * D + d] = o;
        }
      }
      named_bar(1, C::NCW * 32);
      fence_proxy_async_smem();  // generic writes to the stage buffer precede its next TMA fill
    } else if (masked) {
      fence_proxy_async_smem();  // the zeroed V rows precede the next TMA fill of this stage
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
  int batch, Hq, max_splits;
};

// One warp per (row, query head) with >= 2 splits: weights exp2(lse_c - M) for
// every non-empty split c (one lane each), then o = sum_c w_c o_c / sum_c w_c
// in ascending c, each lane owning D/32 consecutive dims.
template <int D>
__global__ void __launch_bounds__(128) gqa_combine_kernel(const CombineArgs a) {
  __shared__ float s_w[4][1024 + 1];
  pdl_wait();  // the split kernel's partials are visible from here on
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wid = blockIdx.x * 4 + warp;
  if (wid >= a.batch * a.Hq) return;
  const RowInfo ri = a.rows[wid / a.Hq];
  if (ri.nsplit <= 1) return;  // written by the split kernel or the planner
  const int ne = row_nonempty(ri);
  const size_t bh = (size_t)wid;
  const float *pl = a.part_lse + bh * a.max_splits;
  float *w = s_w[warp];
  float M = -INFINITY;
  for (int c = lane; c < ne; c += 32) M = fmaxf(M, pl[c]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, o));
  float Z = 0.f;
  for (int c = lane; c < ne; c += 32) {
    const float lc = pl[c];
    const float wc = (lc == -INFINITY || M == -INFINITY) ? 0.f : fast_exp2(lc - M);
    w[c] = wc;
    Z += wc;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) Z += __shfl_xor_sync(FULL, Z, o);
  __syncwarp();
  constexpr int PER = D / 32;  // 2, 4 or 8 consecutive dims per lane
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  // every split c < ne was written (finite), so the loads need no guard and stay independent
  const float *po = a.part_o + bh * a.max_splits * D + lane * PER;
#pragma unroll 16
  for (int c = 0; c < ne; ++c) {
    const float wc = w[c];
    if constexpr (PER == 2) {
      const float2 x = *reinterpret_cast<const float2 *>(po + (size_t)c * D);
      acc[0] += wc * x.x;
      acc[1] += wc * x.y;
    } else {
#pragma unroll
      for (int e = 0; e < PER; e += 4) {
        const float4 x = *reinterpret_cast<const float4 *>(po + (size_t)c * D + e);
        acc[e] += wc * x.x;
        acc[e + 1] += wc * x.y;
        acc[e + 2] += wc * x.z;
        acc[e + 3] += wc * x.w;
      }
    }
  }
  const float inv = Z > 0.f ? 1.f / Z : 0.f;
  uint32_t *dst = reinterpret_cast<uint32_t *>(a.out + bh * D + lane * PER);
#pragma unroll
  for (int e = 0; e < PER; e += 2) dst[e / 2] = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
  if (lane == 0 && a.lse) a.lse[bh] = (M == -INFINITY || Z == 0.f) ? -INFINITY : (M + __log2f(Z)) * LN2;
}

}  // namespace pa
