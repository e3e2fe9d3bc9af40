// pa_mla_tc.cuh -- MLA absorbed decode, attention core on the tensor cores (sm_103a).
//
// What is computed follows pegainfer PR #938 "warp-cooperative two-pass MLA absorbed
// decode kernel" (Schedule section, steps 2-6): for each head, scores over the 576-wide
// latent || rope cache row of every visible token, softmax, and o_lat = sum_t p_t c_t[0:512].
// The query arrives from the absorb kernel as q_abs = bf16(q_lat) || q_rope (576 values per
// head).  The rounding of q_lat moves each score by scale * lo . c_t (lo = q_lat - bf16(q_lat)),
// which shifts the LSE by scale * lo . o_lat to first order (up to ~1e-3 for a short row); the
// projection kernel adds that term back, which leaves ~1e-6.
//
// GB300 mapping: the absorbed core is multi-query attention with one 576-wide KV row per
// token shared by all heads, so it runs on the split-KV machinery of the GQA kernel
// (pa_partition.cuh): a sequence is (row, tile of 16 heads), the 8 tiles of a row form a
// CTA group that streams the same cache pages at about the same time (DRAM once, L2 for
// the others), and the per-piece partials are merged by the GQA combine kernel (D = 512).
//   * producer warp: TMA copies of 32-token stages (9 planes of 64 dims x 32 tokens, 128-byte
//     swizzle, 36 KB) into a 5-stage ring, plus one query stage per piece (9 planes of 16
//     heads), which the consumers copy into a query area;
//   * 8 consumer warps = 2 token groups (16 tokens each) x 4 quarters: for the scores each
//     warp of a group contracts its quarter of the 576 dims (9 k-steps of m16n8k16,
//     the 16 heads as M rows, query fragments read from the piece's query area); the four
//     partial score tiles meet in shared memory and every warp of the group sums them in
//     the same order, so all four hold identical scores and softmax state.  For P.V each warp
//     owns 128 of the 512 latent columns (V is the first 512 dims of the same cache row);
//   * end of a piece: the two token groups merge pairwise through the consumed stage buffer.
#pragma once

#include "pa_gqa.cuh"
#include "pa_partition.cuh"

namespace pa {

struct MlaTcArgs {
  const int32_t *block_table;   // [B, max_pages_per_seq]
  const int32_t *context_lens;  // [B]
  uint16_t *o_lat;              // [B, H, 512] bf16: o_lat of whole-sequence pieces
  float *lse;                   // [B, H] or null
  float *part_o;                // [nparts, 2, 16, 512] fp32
  float *part_lse;              // [nparts, 2, 16] fp32, log2 units
  GqaPartDesc *desc;            // [nparts]
  int batch, max_pages_per_seq, num_pages, max_context_len;
  int H, ntile;                 // heads, tiles of 16 heads
  int log2_page, log2_bh, piece_cost, nparts, hg;
  float qscale;                 // scale * log2(e)
};

struct MlaTcCfg {
  static constexpr int M = PART_HEADS;        // heads per tile (MMA rows)
  static constexpr int DQK = 576, DV = 512;
  static constexpr int NQK = DQK / 64;        // 9 swizzle planes per cache row
  static constexpr int ST = 32;               // tokens per stage
  static constexpr int TW = 16;               // tokens per token group
  static constexpr int TG = ST / TW;          // 2
  static constexpr int DSPLIT = 4;            // warps per token group
  static constexpr int NCW = TG * DSPLIT;     // 8 consumer warps
  static constexpr int THREADS = (NCW + 1) * 32;
  static constexpr int KSW = DQK / 16 / DSPLIT;  // score k-steps per warp: 9
  static constexpr int NT_PV = DV / 8 / DSPLIT;  // P.V n-tiles per warp: 16
  static constexpr int PLANE = ST * 128;         // 4 KB
  static constexpr int STAGE_BYTES = NQK * PLANE;  // 36 KB
  static constexpr int QPLANE = M * 128;         // 2 KB
  static constexpr int NS = 5;
  static constexpr int SPART = TG * DSPLIT * 32 * 8 * 4;  // partial scores: per warp 32 lanes x 8 floats
  static_assert(QPLANE * NQK <= STAGE_BYTES, "the query stage fits a ring slot");
  static_assert(DSPLIT * M * (DV / DSPLIT) * 4 <= STAGE_BYTES, "pairwise merge area fits a stage");
};

struct MlaTcMisc {
  uint32_t status;
  int32_t pad[3];
  GqaPartDesc desc;
  PartitionState part;
};

struct MlaTcSmem {
  using C = MlaTcCfg;
  static constexpr int OFF_STAGE = 0;
  static constexpr int OFF_Q = OFF_STAGE + C::NS * C::STAGE_BYTES;   // the piece's query rows
  static constexpr int OFF_SP = OFF_Q + C::NQK * C::QPLANE;           // 2 buffers of partial scores
  static constexpr int OFF_ML = OFF_SP + 2 * C::SPART;
  static constexpr int OFF_META = OFF_ML + C::M * 2 * 4 * 2;
  static constexpr int OFF_BAR = OFF_META + C::NS * (int)sizeof(StageMeta);
  static constexpr int OFF_MISC = OFF_BAR + 2 * C::NS * 8;
  static constexpr int USED = OFF_MISC + (int)sizeof(MlaTcMisc);
  static constexpr int BYTES = USED + 1024;
  static_assert(BYTES <= 232448, "fits the 227 KB opt-in shared memory of one CTA");
};

__device__ __forceinline__ uint32_t mla_off(int plane_bytes, int row, int chunk) {
  return (uint32_t)((chunk >> 3) * plane_bytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

__global__ void __launch_bounds__(MlaTcCfg::THREADS, 1)
    mla_tc_split_kernel(const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_q,
                        const MlaTcArgs a) {
  using C = MlaTcCfg;
  using S = MlaTcSmem;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
  uint64_t *empty = full + C::NS;
  StageMeta *meta = reinterpret_cast<StageMeta *>(smem + S::OFF_META);
  MlaTcMisc *misc = reinterpret_cast<MlaTcMisc *>(smem + S::OFF_MISC);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NCW);
    }
    fence_mbar_init();
    misc->status = 0;
  }
  if (warp == C::NCW && lane == 0) {
    prefetch_tensormap(&tm_c);
    prefetch_tensormap(&tm_q);
  }
  __syncthreads();
  pdl_wait();               // q_abs, written by the absorb kernel, is visible from here on
  pdl_launch_dependents();  // the combine kernel may be scheduled; it waits for this grid to finish
  uint32_t *status = &misc->status;

  PartitionArgs pargs;
  pargs.context_lens = a.context_lens;
  pargs.batch = a.batch;
  pargs.max_context_len = a.max_context_len;
  pargs.Q = 1;
  pargs.window = 0;
  pargs.log2_bh = a.log2_bh;
  pargs.piece_cost = a.piece_cost;
  pargs.nparts = a.nparts;
  pargs.hg = a.hg;
  pargs.hs = a.ntile;
  partition_prologue<C::THREADS>(pargs, &misc->part, status);
  zero_empty_rows<C::THREADS>(pargs, a.o_lat, a.lse, a.H * C::DV, a.H);
  __syncthreads();

  if (warp == C::NCW) {
    // ------------------------------------------------------------ producer
    const int P = 1 << a.log2_page;
    const int nbox = C::ST >> a.log2_bh;
    uint32_t j = 0;
    bool ok = true;
    int npieces = 0;
    Piece last_piece = {};
    bool first_ends = false;
    PieceWalker walker(pargs, &misc->part, lane);
    auto piece_window = [&](const Piece &p) {
      const int pb = (p.ub << a.log2_bh) >> a.log2_page;
      const int pe = (((p.ue << a.log2_bh) - 1) >> a.log2_page) + 1;
      return lane < pe - pb ? a.block_table[(size_t)p.b * a.max_pages_per_seq + pb + lane] : 0;
    };
    Piece cur = {}, nxt = {};
    bool has_cur = walker.take(cur);
    int cwin0 = 0, nwin0 = 0;
    bool has_next = false;
    if (has_cur) {
      cwin0 = piece_window(cur);
      has_next = walker.take(nxt);
      if (has_next) nwin0 = piece_window(nxt);
    }
    while (has_cur && ok) {
      const int h0 = cur.hs * C::M;
      const int nh = min(C::M, a.H - h0);
      const int slot = (cur.starts && cur.ends) ? -1 : (npieces == 0 ? 0 : 1);
      const int T0 = cur.ub << a.log2_bh;
      const int tok_lo = max(cur.lo, T0), tok_hi = min(cur.L, cur.ue << a.log2_bh);
      const int n_stages = (cur.ue - cur.ub + nbox - 1) / nbox;
      const int pb = T0 >> a.log2_page;
      const int npages = ((((cur.ue << a.log2_bh) - 1) >> a.log2_page) + 1) - pb;
      const int32_t *bt_piece = a.block_table + (size_t)cur.b * a.max_pages_per_seq + pb;
      int cwin = cwin0, wi = 0;
      int fwin = (lane + 32 < npages) ? bt_piece[32 + lane] : 0;
      {
        // the query stage: q_abs rows b * H + h0 .. + 16 (rows past H are masked)
        const int s = j % C::NS;
        const uint32_t u = j / C::NS;
        if (u > 0) ok = mbar_wait(&empty[s], (u - 1) & 1, status);
        if (!ok) break;
        if (lane == 0) {
          StageMeta &m = meta[s];
          m.end = 0;
          m.first = 1;
          m.last = 0;
          m.b = cur.b;
          m.hq0 = h0;
          m.ghead = nh;
          mbar_arrive_expect_tx(&full[s], (uint32_t)(C::NQK * C::QPLANE));
          uint8_t *qdst = smem + S::OFF_STAGE + s * C::STAGE_BYTES;
#pragma unroll
          for (int dq = 0; dq < C::NQK; ++dq)
            tma_load_2d(qdst + dq * C::QPLANE, &tm_q, dq * 64, cur.b * a.H + h0, &full[s]);
        }
        __syncwarp();
        ++j;
      }
      for (int t = 0; t < n_stages && ok; ++t, ++j) {
        const int s = j % C::NS;
        const uint32_t u = j / C::NS;
        if (u > 0) ok = mbar_wait(&empty[s], (u - 1) & 1, status);
        if (!ok) break;
        const int unit0 = cur.ub + t * nbox;
        const int tok0 = unit0 << a.log2_bh;
        const int pwin = ((tok0 >> a.log2_page) - pb) >> 5;
        while (wi < pwin) {
          cwin = fwin;
          ++wi;
          const int nx = 32 * (wi + 1) + lane;
          fwin = nx < npages ? bt_piece[nx] : 0;
        }
        const int unit = unit0 + lane;
        const int btok = unit << a.log2_bh;
        const int prel = (btok >> a.log2_page) - pb;
        const int phys = __shfl_sync(FULL, cwin, prel & 31);
        bool load = false, isbad = false;
        if (lane < nbox && unit < cur.ue) {
          if (phys < 0 || phys >= a.num_pages) {
            isbad = true;
            atomicOr(status, PA_DEV_BAD_PAGE);
          } else {
            load = true;
          }
        }
        const uint32_t bad = __ballot_sync(FULL, isbad);
        const int nvalid = __popc(__ballot_sync(FULL, load));
        const bool last = (t == n_stages - 1);
        uint8_t *kdst = smem + S::OFF_STAGE + s * C::STAGE_BYTES;
        if (lane == 0) {
          StageMeta &m = meta[s];
          m.end = 0;
          m.first = 0;
          m.last = last;
          m.b = cur.b;
          m.hq0 = h0;
          m.ghead = nh;
          m.slot = slot;
          m.tok0 = tok0;
          m.tok_lo = tok_lo;
          m.tok_hi = tok_hi;
          m.badmask = bad;
          m.masked = (tok0 < tok_lo) || (tok0 + C::ST > tok_hi) || bad != 0;
          mbar_arrive_expect_tx(&full[s], (uint32_t)nvalid * (uint32_t)((C::DQK * 2) << a.log2_bh));
        }
        __syncwarp();
        if (load) {
          const int pslot = btok & (P - 1);
          uint8_t *dst = kdst + (lane << a.log2_bh) * 128;
#pragma unroll
          for (int dq = 0; dq < C::NQK; ++dq) tma_load_3d(dst + dq * C::PLANE, &tm_c, dq * 64, pslot, phys, &full[s]);
        }
      }
      if (!ok) break;
      if (npieces == 0) first_ends = cur.ends;
      if (npieces < (int)DESC_PIECES) ++npieces;
      last_piece = cur;
      has_cur = has_next;
      if (!has_cur) break;
      cur = nxt;
      cwin0 = nwin0;
      has_next = walker.take(nxt);
      if (has_next) nwin0 = piece_window(nxt);
    }
    if (ok) {
      const int s = j % C::NS;
      const uint32_t u = j / C::NS;
      if (u > 0) ok = mbar_wait(&empty[s], (u - 1) & 1, status);
      if (ok && lane == 0) {
        meta[s].end = 1;
        mbar_arrive(&full[s]);
      }
    }
    if (!ok) {
      const uint32_t first = j > (uint32_t)C::NS ? j - C::NS : 0u;
      for (uint32_t i = first; i < j; ++i) mbar_wait(&full[i % C::NS], (i / C::NS) & 1, status);
    }
    if (lane == 0) {
      misc->desc.last_b = last_piece.b;
      misc->desc.last_hs = last_piece.hs;
      misc->desc.flags = (uint32_t)npieces | (last_piece.starts ? DESC_LAST_STARTS : 0u) |
                         (last_piece.ends ? DESC_LAST_ENDS : 0u) | (first_ends ? DESC_FIRST_ENDS : 0u);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int g8 = lane >> 2, tq = lane & 3;
    const int lm_mat = lane >> 3, lm_row = lane & 7;
    const int tgrp = warp % C::TG;           // token group
    const int dq4 = warp / C::TG;            // quarter: score dims [144 dq4, +144), P.V columns [128 dq4, +128)
    const int wbase = tgrp * C::TW;
    const int nd0 = dq4 * C::NT_PV;
    float *sm_ml = reinterpret_cast<float *>(smem + S::OFF_ML);
    float *spart = reinterpret_cast<float *>(smem + S::OFF_SP);
    const float TAU = 8.f;
    const int bh_tokens = 1 << a.log2_bh;

    const uint32_t qarea = smem_u32(smem + S::OFF_Q);
    float acc[C::NT_PV][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool rv0 = false, rv1 = false;

    for (uint32_t j = 0;; ++j) {
      const int s = j % C::NS;
      if (!mbar_wait(&full[s], (j / C::NS) & 1, status)) break;
      const StageMeta &mt = meta[s];
      if (mt.end) break;
      const uint32_t cbase = smem_u32(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
      if (mt.first) {
        // a new piece: its query rows into the query area (every warp finished the previous
        // piece's scores before the merge barrier of its last stage)
        rv0 = g8 < mt.ghead;
        rv1 = g8 + 8 < mt.ghead;
        {
          const uint4 *src = reinterpret_cast<const uint4 *>(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
          uint4 *dst = reinterpret_cast<uint4 *>(smem + S::OFF_Q);
          for (int e = tid; e < C::NQK * C::QPLANE / 16; e += C::NCW * 32) dst[e] = src[e];
        }
        named_bar(1, C::NCW * 32);
#pragma unroll
        for (int n = 0; n < C::NT_PV; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        continue;
      }
      // ---- partial scores over this warp's 144 dims, for the group's 16 tokens (2 n-tiles);
      // even and odd k-steps go to separate accumulators (two independent chains per n-tile)
      float sp[2][4], sq[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sp[nt][e] = sq[nt][e] = 0.f;
#pragma unroll
      for (int k = 0; k < C::KSW; ++k) {
        const int ks = dq4 * C::KSW + k;
        // matrices: (tokens 0-7, dims 0-7), (tokens 0-7, dims 8-15), (tokens 8-15, ...) of the k-step
        uint32_t qa[4], b[4];
        ldmatrix_x4(qa, qarea + mla_off(C::QPLANE, (lm_mat & 1) * 8 + lm_row, 2 * ks + (lm_mat >> 1)));
        const int tok = wbase + (lm_mat >> 1) * 8 + lm_row, chunk = 2 * ks + (lm_mat & 1);
        ldmatrix_x4(b, cbase + mla_off(C::PLANE, tok, chunk));
        if (k & 1) {
          mma_bf16_16816(sq[0], qa, b[0], b[1]);
          mma_bf16_16816(sq[1], qa, b[2], b[3]);
        } else {
          mma_bf16_16816(sp[0], qa, b[0], b[1]);
          mma_bf16_16816(sp[1], qa, b[2], b[3]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sp[nt][e] += sq[nt][e];
      float *myp = spart + (j & 1) * (C::SPART / 4) + (size_t)(tgrp * C::DSPLIT + dq4) * 32 * 8;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) myp[(nt * 4 + e) * 32 + lane] = sp[nt][e];
      named_bar(2 + tgrp, C::DSPLIT * 32);  // the group's four partials are written
      float sv[2][4];
      {
        const float *gp = spart + (j & 1) * (C::SPART / 4) + (size_t)(tgrp * C::DSPLIT) * 32 * 8;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x = 0.f;
#pragma unroll
            for (int w = 0; w < C::DSPLIT; ++w) x += gp[(size_t)w * 32 * 8 + (nt * 4 + e) * 32 + lane];
            sv[nt][e] = x;
          }
      }
      const bool masked = mt.masked;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float v = sv[nt][e] * a.qscale;
          bool valid = (e < 2) ? rv0 : rv1;
          if (masked) {
            const int stok = wbase + nt * 8 + 2 * tq + (e & 1);
            const int ltok = mt.tok0 + stok;
            valid = valid && ltok >= mt.tok_lo && ltok < mt.tok_hi && !((mt.badmask >> (stok / bh_tokens)) & 1u);
          }
          sv[nt][e] = valid ? v : -INFINITY;
        }
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
      if (masked) {
        // cache rows of keys that are not attended may hold anything (NaN included): zero this
        // warp's latent columns of them (every warp of the group has read its score dims)
        uint8_t *vgen = smem + S::OFF_STAGE + s * C::STAGE_BYTES;
        constexpr int CPW = C::DV / 8 / C::DSPLIT;  // 16-byte chunks of a row owned by this warp: 16
        for (int e = lane; e < C::TW * CPW; e += 32) {
          const int stok = wbase + e / CPW;
          const int chunk = dq4 * CPW + e % CPW;
          const int ltok = mt.tok0 + stok;
          if (ltok < mt.tok_lo || ltok >= mt.tok_hi || ((mt.badmask >> (stok / bh_tokens)) & 1u))
            *reinterpret_cast<uint4 *>(vgen + mla_off(C::PLANE, stok, chunk)) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      // ---- O += P V over this warp's 128 latent columns
      {
        const int tok = wbase + (lm_mat & 1) * 8 + lm_row;
#pragma unroll
        for (int nd = 0; nd < C::NT_PV; nd += 2) {
          uint32_t b[4];
          ldmatrix_x4_trans(b, cbase + mla_off(C::PLANE, tok, nd0 + nd + (lm_mat >> 1)));
          mma_bf16_16816(acc[nd], pa, b[0], b[1]);
          mma_bf16_16816(acc[nd + 1], pa, b[2], b[3]);
        }
      }

      if (mt.last) {
        // ---- end of a piece: token group 1 hands (acc, m, l) to group 0 through this stage
        l0 += __shfl_xor_sync(FULL, l0, 1);
        l0 += __shfl_xor_sync(FULL, l0, 2);
        l1 += __shfl_xor_sync(FULL, l1, 1);
        l1 += __shfl_xor_sync(FULL, l1, 2);
        named_bar(1, C::NCW * 32);  // all warps are done reading this stage
        float *mg = reinterpret_cast<float *>(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
        // area of quarter dq4: 16 rows x 128 columns; column c of row r at c ^ (4 (r & 7))
        float *mq = mg + dq4 * C::M * (C::DV / C::DSPLIT);
        if (tgrp == 1) {
#pragma unroll
          for (int n = 0; n < C::NT_PV; ++n) {
            const int c = (n * 8 + 2 * tq) ^ (4 * g8);
            *reinterpret_cast<float2 *>(mq + g8 * (C::DV / C::DSPLIT) + c) = make_float2(acc[n][0], acc[n][1]);
            *reinterpret_cast<float2 *>(mq + (g8 + 8) * (C::DV / C::DSPLIT) + c) = make_float2(acc[n][2], acc[n][3]);
          }
          if (tq == 0 && dq4 == 0) {
            sm_ml[g8 * 2] = m0;
            sm_ml[g8 * 2 + 1] = l0;
            sm_ml[(g8 + 8) * 2] = m1;
            sm_ml[(g8 + 8) * 2 + 1] = l1;
          }
        }
        named_bar(1, C::NCW * 32);
        if (tgrp == 0) {
          const float om0 = sm_ml[g8 * 2], ol0 = sm_ml[g8 * 2 + 1];
          const float om1 = sm_ml[(g8 + 8) * 2], ol1 = sm_ml[(g8 + 8) * 2 + 1];
          const float M0 = fmaxf(m0, om0), M1 = fmaxf(m1, om1);
          const float wa0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - M0), wb0 = om0 == -INFINITY ? 0.f : fast_exp2(om0 - M0);
          const float wa1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M1), wb1 = om1 == -INFINITY ? 0.f : fast_exp2(om1 - M1);
          const float L0 = l0 * wa0 + ol0 * wb0, L1 = l1 * wa1 + ol1 * wb1;
          const float i0 = L0 > 0.f ? 1.f / L0 : 0.f, i1 = L1 > 0.f ? 1.f / L1 : 0.f;
          const int slot = mt.slot;
          const size_t pi = (size_t)blockIdx.x * 2 + (slot > 0 ? 1 : 0);
          const size_t bh0 = (size_t)mt.b * a.H + mt.hq0 + g8, bh1 = bh0 + 8;
#pragma unroll
          for (int n = 0; n < C::NT_PV; ++n) {
            const int c = (n * 8 + 2 * tq) ^ (4 * g8);
            const float2 x0v = *reinterpret_cast<const float2 *>(mq + g8 * (C::DV / C::DSPLIT) + c);
            const float2 x1v = *reinterpret_cast<const float2 *>(mq + (g8 + 8) * (C::DV / C::DSPLIT) + c);
            const float o00 = (acc[n][0] * wa0 + x0v.x * wb0) * i0, o01 = (acc[n][1] * wa0 + x0v.y * wb0) * i0;
            const float o10 = (acc[n][2] * wa1 + x1v.x * wb1) * i1, o11 = (acc[n][3] * wa1 + x1v.y * wb1) * i1;
            const int col = (nd0 + n) * 8 + 2 * tq;
            if (slot < 0) {
              if (rv0) *reinterpret_cast<uint32_t *>(a.o_lat + bh0 * C::DV + col) = pack_bf16x2(o00, o01);
              if (rv1) *reinterpret_cast<uint32_t *>(a.o_lat + bh1 * C::DV + col) = pack_bf16x2(o10, o11);
            } else {
              *reinterpret_cast<float2 *>(a.part_o + (pi * C::M + g8) * C::DV + col) = make_float2(o00, o01);
              *reinterpret_cast<float2 *>(a.part_o + (pi * C::M + g8 + 8) * C::DV + col) = make_float2(o10, o11);
            }
          }
          if (tq == 0 && dq4 == 0) {
            const float s0 = (M0 == -INFINITY || L0 == 0.f) ? -INFINITY : M0 + __log2f(L0);
            const float s1 = (M1 == -INFINITY || L1 == 0.f) ? -INFINITY : M1 + __log2f(L1);
            if (slot < 0) {
              if (a.lse && rv0) a.lse[bh0] = s0 * LN2;
              if (a.lse && rv1) a.lse[bh1] = s1 * LN2;
            } else {
              a.part_lse[pi * C::M + g8] = s0;
              a.part_lse[pi * C::M + g8 + 8] = s1;
            }
          }
        }
        fence_proxy_async_smem();
      } else if (masked) {
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }

  __syncthreads();
  if (tid == 0) {
    GqaPartDesc d = misc->desc;
    d.status = misc->status;
    a.desc[blockIdx.x] = d;
  }
  if ((misc->desc.flags & DESC_PIECES) == 0) {
    for (int e = tid; e < C::M * C::DV; e += C::THREADS) a.part_o[(size_t)blockIdx.x * 2 * C::M * C::DV + e] = 0.f;
    for (int h = tid; h < C::M; h += C::THREADS) a.part_lse[(size_t)blockIdx.x * 2 * C::M + h] = -INFINITY;
  }
}

}  // namespace pa
