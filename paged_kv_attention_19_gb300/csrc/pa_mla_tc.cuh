// pa_mla_tc.cuh -- MLA absorbed decode, attention core on the 5th-generation tensor cores (sm_103a).
//
// What is computed follows pegainfer PR #938 "warp-cooperative two-pass MLA absorbed
// decode kernel" (Schedule section, steps 2-6): for each head, scores over the 576-wide
// latent || rope cache row of every visible token, softmax, and o_lat = sum_t p_t c_t[0:512].
// The query arrives from the absorb kernel as q_abs = bf16(q_lat) || q_rope (576 values per
// head).  The rounding of q_lat moves each score by scale * lo . c_t (lo = q_lat - bf16(q_lat)),
// which shifts the LSE by scale * lo . o_lat to first order (up to ~1e-3 for a short row); the
// projection kernel adds that term back, which leaves ~1e-6.
//
// GB300 mapping.  The absorbed core is multi-query attention: one 576-wide cache row per token,
// shared by all heads.  A tile of 128 heads is the M dimension of tcgen05 MMAs (one head per
// tensor-memory lane), so every cache row a CTA stages serves all the tile's heads at once.  The
// fp32 o_lat of 128 heads x 512 columns would fill the whole tensor memory, so a sequence is
// (row, head tile, half of the 512 latent columns): the two halves of a tile are the CTA group
// of the split-KV partition (pa_partition.cuh), stream the same cache pages at about the same
// time (DRAM once, L2 for the other) and each compute the full scores.
//
// An MMA instruction costs about the same issue time for N = 32 as for N = 128, so the score MMAs
// take 64 tokens at once (N = 64).  Shared memory cannot hold the tile's 144 KB of query rows next
// to a ring of 72 KB stages, so the query is split: 5 of its 9 planes of 64 dims stay in shared
// memory (A operand from shared memory), the other 4 are copied into tensor memory by tcgen05.cp
// once per piece (A operand from tensor memory).  Query and cache planes are held in the same
// order (mla_plane_at): positions 0-4 the planes only the scores read, positions 5-8 this half's
// latent columns.  A ring slot is two parts with their own barriers: part A (positions 0-4) is
// reloaded as soon as the stage's first 20 score MMAs have completed, part B (positions 5-8, the
// V operand) once its P.V has; the scores of the next stage in the slot start on part A.  Per CTA:
//   * warp 0, producer: per piece the query positions 0-4 into the query area and positions 5-8
//     into a ring slot (a "query stage"), then TMA copies of 64-token stages (9 planes of 64 dims
//     x 64 tokens, 128-byte swizzle, 72 KB) into the 2-slot ring, part A then part B;
//   * warp 1, one thread issues the tensor-core work from a polling loop: the tcgen05.cp of a query
//     stage, the 36 score MMAs of a stage (S = Q C^T, M = 128 heads, N = 64 tokens, K = 576) into
//     one of two score buffers, 20 on part A and 16 on part B, and, as soon as a stage's
//     probabilities are in tensor memory, its P.V (P: 128 x 64 bf16 written over the stage's own
//     scores, V: positions 5-8, MN-major, N = 256) into the O columns.  With both operands in shared memory a
//     score MMA reads 6 KB, so the MMAs keep the shared-memory port busy and every mbarrier test
//     or shared-memory access of this thread waits behind them: the loop makes few of them;
//   * warps 2-5, softmax: one thread per head row reads its 64 scores, keeps the fp32 running max
//     and sum (rescaling its O row in tensor memory only when the max grows by more than 2^8),
//     writes the probabilities as bf16 over the scores, and at the end of a piece reads O, divides
//     by the sum and stores o_lat (or an fp32 partial) and the LSE.
// Tensor-memory columns: scores (then P) 0-127 (two buffers of 64), query positions 5-8 128-255, O 256-511.
#pragma once

#include <type_traits>

#include "pa_gqa.cuh"
#include "pa_partition.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

struct MlaTcArgs {
  const int32_t *block_table;   // [B, max_pages_per_seq]
  const int32_t *context_lens;  // [B]
  uint16_t *o_lat;              // [B, 2, H, 256] bf16: the two column halves of o_lat, whole-sequence pieces
  float *lse;                   // [B, H] or null
  float *part_o;                // [nparts, 2, RS, 256] fp32
  float *part_lse;              // [nparts, 2, RS] fp32, log2 units
  GqaPartDesc *desc;            // [nparts]
  int32_t *seq_first;           // [B, ntile]: -1 whole piece; else 2 x CTA + slot of the first piece
  int32_t *seq_last;            // [B, ntile]: CTA holding the last piece of a split sequence
  int batch, max_pages_per_seq, num_pages, max_context_len;
  int H, ntile, rs;             // heads; sequences per row (2 x head tiles); rows per partial slot
  int log2_page, log2_bh, piece_cost, nparts, hg;
  float qscale;                 // scale * log2(e)
};

struct MlaTcCfg {
  static constexpr int M = 128;                   // heads per tile: MMA rows, tensor-memory lanes
  static constexpr int DQK = 576, DV = 512, DVH = DV / 2;
  static constexpr int NQK = DQK / 64;            // 9 swizzle planes per cache row
  static constexpr int NQS = 5;                   // query planes in shared memory; the rest in tensor memory
  static constexpr int NA = 5;                    // stage positions read by the scores only (part A)
  static constexpr int ST = 64;                   // tokens per stage: N of the score MMA, K of P.V
  static constexpr int NS = 2;                    // slots in the ring
  static constexpr int PLANE = ST * 128;          // 8 KB
  static constexpr int STAGE_BYTES = NQK * PLANE; // 72 KB
  static constexpr int QPLANE = M * 128;          // 16 KB
  static constexpr int QS_BYTES = NQS * QPLANE;   // 80 KB: positions 0-4
  static constexpr int QT_BYTES = (NQK - NQS) * QPLANE;  // 64 KB: positions 5-8, through a ring slot
  static constexpr int SOFTMAX_WARPS = 4;
  static constexpr int THREADS = (2 + SOFTMAX_WARPS) * 32;
  static constexpr uint32_t TM_S = 0, TM_QT = 128, TM_O = 256, TM_COLS = 512;
  static constexpr float TAU = 8.f;               // lazy rescale threshold (log2 units)
  static constexpr uint32_t IDESC_S = tc_idesc_bf16(M, ST, false);
  static constexpr uint32_t IDESC_PV = tc_idesc_bf16(M, DVH, true);
  static_assert(NQK == 9 && NA == 5 && NQS == NA && DVH == 4 * 64,
                "positions 0-4: score-only planes (query in shared memory), 5-8: this half's V planes");
  static_assert((ST & (ST - 1)) == 0, "a stage holds a whole number of TMA boxes of a power-of-two token count");
  static_assert(QT_BYTES <= STAGE_BYTES, "the query positions 5-8 fit a ring slot");
  static_assert(2 * ST + (NQK - NQS) * 4 * 8 + DVH <= (int)TM_COLS, "tensor-memory budget");
};

// The 64-column plane of a cache row (or of a query row) held at stage position p by the CTA of
// column half hv: positions 0-4 the planes that only the scores read (the other half's latent
// columns, then the rope columns), positions 5-8 this half's latent columns in order.
__device__ __forceinline__ int mla_plane_at(int p, int hv) {
  if (p >= MlaTcCfg::NA) return 4 * hv + (p - MlaTcCfg::NA);
  return hv ? (p < 4 ? p : 8) : 4 + p;
}

struct MlaTcMisc {
  uint32_t status;
  uint32_t tmem;   // base address of the tensor-memory allocation
  int32_t pad[2];
  GqaPartDesc desc;
  PartitionState part;
};

struct MlaTcSmem {
  using C = MlaTcCfg;
  static constexpr int OFF_Q = 0;                                      // the piece's query positions 0-4
  static constexpr int OFF_STAGE = OFF_Q + C::QS_BYTES;
  static constexpr int OFF_META = OFF_STAGE + C::NS * C::STAGE_BYTES;  // per ring slot
  static constexpr int OFF_SMETA = OFF_META + C::NS * (int)sizeof(StageMeta);  // per cache stage, mod 4
  // full_a[NS], full_b[NS], empty_a[NS], empty_b[NS], q_full, q_empty, s_full[2], sbuf_free[2],
  // p_full, pv_done, o_free, drain
  static constexpr int OFF_BAR = OFF_SMETA + 4 * (int)sizeof(StageMeta);
  static constexpr int NBAR = 4 * C::NS + 10;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int USED = OFF_MISC + (int)sizeof(MlaTcMisc);
  static constexpr int BYTES = USED + 1024;
  static_assert(BYTES <= 232448, "fits the 227 KB opt-in shared memory of one CTA");
};

// StageMeta fields as used here: nq = 1 marks a query stage; aux = the ring slot of the stage.  The
// producer writes a stage's record twice: into its ring slot's meta, read by the issuing thread
// when the stage starts, and into smeta[t % 4] for cache stage t, read by the softmax warps.  A
// slot's meta is rewritten once the stage's part-A MMAs have completed, which can be before the
// softmax reaches the stage; smeta[t % 4] is rewritten for stage t + 4 only after the issuing
// thread has started a stage whose score buffer needed the softmax of stage t done (or, through a
// query stage, the scores of a stage that started after it).
__global__ void __launch_bounds__(MlaTcCfg::THREADS, 1)
    mla_tc_split_kernel(const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_q,
                        const MlaTcArgs a) {
  using C = MlaTcCfg;
  using S = MlaTcSmem;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
  uint64_t *full_a = bars, *full_b = bars + C::NS, *empty_a = bars + 2 * C::NS, *empty_b = bars + 3 * C::NS;
  uint64_t *q_full = bars + 4 * C::NS, *q_empty = q_full + 1;
  uint64_t *s_full = q_full + 2, *sbuf_free = s_full + 2;
  uint64_t *p_full = sbuf_free + 2, *pv_done = p_full + 1, *o_free = p_full + 2, *drain = p_full + 3;
  StageMeta *meta = reinterpret_cast<StageMeta *>(smem + S::OFF_META);
  StageMeta *smeta = reinterpret_cast<StageMeta *>(smem + S::OFF_SMETA);
  MlaTcMisc *misc = reinterpret_cast<MlaTcMisc *>(smem + S::OFF_MISC);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full_a[s], 1);
      mbar_init(&full_b[s], 1);
      mbar_init(&empty_a[s], 1);
      mbar_init(&empty_b[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 2);  // the scores' commit and the issuing thread's arrive
      mbar_init(&sbuf_free[i], 1);
    }
    mbar_init(p_full, C::SOFTMAX_WARPS);
    mbar_init(pv_done, 1);
    mbar_init(o_free, C::SOFTMAX_WARPS);
    mbar_init(drain, 1);
    fence_mbar_init();
    misc->status = 0;
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_c);
    prefetch_tensormap(&tm_q);
  }
  if (warp == 1) tc_alloc(&misc->tmem, C::TM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem;
  // Only the query rows come from the absorb kernel: the producer waits for it (griddepcontrol)
  // just before their first copy, so the partition and the first cache stage overlap its tail.
  pdl_launch_dependents();  // the projection kernel may stage its weights; it waits for this grid to finish
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const int P = 1 << a.log2_page;
    const int nbox = C::ST >> a.log2_bh;
    uint32_t j = 0;   // ring slots issued
    uint32_t kq = 0;  // pieces whose query was issued
    bool ok = true;
    bool pre_pending = false;  // ring index 1 was issued ahead of ring index 0
    bool a_only = false;       // ring index j has its part A in flight but not its part B
    uint32_t tcs = 0;          // cache stages issued: the next one's record goes to smeta[tcs % 4]
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
      const int h0 = (cur.hs >> 1) * C::M, hv = cur.hs & 1;
      const int nh = min(C::M, a.H - h0);
      const int slot = (cur.starts && cur.ends) ? -1 : (npieces == 0 ? 0 : 1);
      if (lane == 0) {
        // where the projection kernel finds the sequence: written directly (whole piece), or
        // merged from the partial slots of CTAs first, first + hg, ..., last
        const size_t si = (size_t)cur.b * a.ntile + cur.hs;
        if (cur.starts)
          a.seq_first[si] = slot < 0 ? -1 : (int32_t)blockIdx.x * 2 + slot;
        else if (cur.ends)
          a.seq_last[si] = (int32_t)blockIdx.x;
      }
      const int T0 = cur.ub << a.log2_bh;
      const int tok_lo = max(cur.lo, T0), tok_hi = min(cur.L, cur.ue << a.log2_bh);
      const int n_stages = (cur.ue - cur.ub + nbox - 1) / nbox;
      const int pb = T0 >> a.log2_page;
      const int npages = ((((cur.ue << a.log2_bh) - 1) >> a.log2_page) + 1) - pb;
      const int32_t *bt_piece = a.block_table + (size_t)cur.b * a.max_pages_per_seq + pb;
      int cwin = cwin0, wi = 0;
      int fwin = (lane + 32 < npages) ? bt_piece[32 + lane] : 0;
      // cache stage t of the piece into ring index jj: part A (positions 0-4) once the slot's
      // previous part-A scores have completed, part B (positions 5-8) once its previous P.V has
      auto issue_stage = [&](int t, uint32_t jj) -> bool {
        const int s = jj % C::NS;
        const uint32_t u = jj / C::NS;
        if (u > 0 && !mbar_wait(&empty_a[s], (u - 1) & 1, status)) return false;
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
        uint8_t *kdst = smem + S::OFF_STAGE + s * C::STAGE_BYTES;
        if (lane == 0) {
          StageMeta m;
          m.end = 0;
          m.nq = 0;
          m.aux = s;
          m.L = 0;
          m.first = t == 0;
          m.last = t == n_stages - 1;
          m.b = cur.b;
          m.hq0 = h0;
          m.ghead = nh;
          m.i0 = hv;
          m.slot = slot;
          m.tok0 = tok0;
          m.tok_lo = tok_lo;
          m.tok_hi = tok_hi;
          m.badmask = bad;
          m.masked = (tok0 < tok_lo) || (tok0 + C::ST > tok_hi) || bad != 0;
          meta[s] = m;
          smeta[tcs & 3] = m;
          mbar_arrive_expect_tx(&full_a[s], (uint32_t)nvalid * (uint32_t)((C::NA * 128) << a.log2_bh));
        }
        __syncwarp();
        ++tcs;
        const int pslot = btok & (P - 1);
        uint8_t *dst = kdst + (lane << a.log2_bh) * 128;
        if (load) {
#pragma unroll
          for (int dq = 0; dq < C::NA; ++dq)
            tma_load_3d(dst + dq * C::PLANE, &tm_c, mla_plane_at(dq, hv) * 64, pslot, phys, &full_a[s]);
        }
        if (u > 0 && !mbar_wait(&empty_b[s], (u - 1) & 1, status)) {
          a_only = true;
          return false;
        }
        if (lane == 0)
          mbar_arrive_expect_tx(&full_b[s], (uint32_t)nvalid * (uint32_t)(((C::NQK - C::NA) * 128) << a.log2_bh));
        __syncwarp();
        if (load) {
#pragma unroll
          for (int dq = C::NA; dq < C::NQK; ++dq)
            tma_load_3d(dst + dq * C::PLANE, &tm_c, mla_plane_at(dq, hv) * 64, pslot, phys, &full_b[s]);
        }
        return true;
      };
      // The ring holds the piece's query stage, then its cache stages.  The first piece's first
      // cache stage (ring index 1) is issued before the wait for the absorb kernel.
      const bool early = kq == 0;
      if (early) {
        ok = issue_stage(0, j + 1);
        pre_pending = ok;
        pdl_wait();  // q_abs is visible from here on
      }
      if (ok) {
        // the tile's query, its planes in this half's stage order: positions 0-4 into the query
        // area, positions 5-8 into ring index j (both parts of the slot, counted on full_a; full_b
        // completes empty); all are free once the previous piece's score MMAs have completed
        if (kq > 0) ok = mbar_wait(q_empty, (kq - 1) & 1, status);
        const int s = j % C::NS;
        const uint32_t u = j / C::NS;
        if (ok && u > 0) ok = mbar_wait(&empty_a[s], (u - 1) & 1, status);
        if (ok && u > 0) ok = mbar_wait(&empty_b[s], (u - 1) & 1, status);
        if (ok && lane == 0) {
          StageMeta &m = meta[s];
          m.end = 0;
          m.nq = 1;
          mbar_arrive_expect_tx(q_full, (uint32_t)C::QS_BYTES);
#pragma unroll
          for (int dq = 0; dq < C::NQS; ++dq)
            tma_load_2d(smem + S::OFF_Q + dq * C::QPLANE, &tm_q, mla_plane_at(dq, hv) * 64, cur.b * a.H + h0, q_full);
          mbar_arrive_expect_tx(&full_a[s], (uint32_t)C::QT_BYTES);
          uint8_t *qt = smem + S::OFF_STAGE + s * C::STAGE_BYTES;
#pragma unroll
          for (int dq = C::NQS; dq < C::NQK; ++dq)
            tma_load_2d(qt + (dq - C::NQS) * C::QPLANE, &tm_q, mla_plane_at(dq, hv) * 64, cur.b * a.H + h0,
                        &full_a[s]);
          mbar_arrive(&full_b[s]);
        }
        __syncwarp();
        if (ok) {
          ++kq;
          j += early ? 2 : 1;
          pre_pending = false;
        }
      }
      for (int t = early ? 1 : 0; t < n_stages && ok; ++t) {
        ok = issue_stage(t, j);
        if (ok) ++j;
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
      // the end marker: only its metadata, read when the slot's part A is next consumed
      const int s = j % C::NS;
      const uint32_t u = j / C::NS;
      if (u > 0) ok = mbar_wait(&empty_a[s], (u - 1) & 1, status);
      if (ok && lane == 0) {
        meta[s].end = 1;
        meta[s].nq = 0;
        smeta[tcs & 3].end = 1;
        mbar_arrive(&full_a[s]);
      }
    }
    if (!ok) {
      // copies still in flight land before the CTA exits
      const uint32_t first = j > (uint32_t)C::NS ? j - C::NS : 0u;
      for (uint32_t i = first; i < j; ++i) {
        mbar_wait(&full_a[i % C::NS], (i / C::NS) & 1, status);
        mbar_wait(&full_b[i % C::NS], (i / C::NS) & 1, status);
      }
      if (a_only) mbar_wait(&full_a[j % C::NS], (j / C::NS) & 1, status);
      if (pre_pending) {
        mbar_wait(&full_a[1 % C::NS], 0, status);
        mbar_wait(&full_b[1 % C::NS], 0, status);
      }
      if (kq > 0) mbar_wait(q_full, (kq - 1) & 1, status);
    }
    if (lane == 0) {
      misc->desc.last_b = last_piece.b;
      misc->desc.last_hs = last_piece.hs;
      misc->desc.flags = (uint32_t)npieces | (last_piece.starts ? DESC_LAST_STARTS : 0u) |
                         (last_piece.ends ? DESC_LAST_ENDS : 0u) | (first_ends ? DESC_FIRST_ENDS : 0u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ tensor-core issue (one thread)
    // A polling loop over the events the tensor-core work waits for.  P.V of the oldest stage goes
    // first (it frees part B of a ring slot and a score buffer).  A stage starts once its part A
    // has landed, and its 20 part-A score MMAs go out in the same iteration; its 16 part-B MMAs
    // go out together once part B has landed.
    // The metadata of a stage is read once, as two 16-byte words; what P.V needs of it stays in
    // registers; the softmax warps read their copy in smeta.
    if (lane == 0) {
      const uint64_t qd0 = tc_sdesc_sw128(smem_u32(smem + S::OFF_Q), 16, 1024);
      const uint32_t stage0 = smem_u32(smem + S::OFF_STAGE);
      uint32_t r = 0;     // ring slot consumed next
      uint32_t js = 0;    // stage whose scores are issued next
      uint32_t jp = 0;    // stage whose P.V is issued next (jp <= js)
      uint32_t kq = 0;    // query stages copied (q_empty phases awaited: one per earlier piece)
      uint32_t kf = 0;    // pieces whose first scores were issued (q_full phases)
      uint32_t npp = 0;   // pieces whose first P.V was issued (o_free phases: one per earlier piece)
      uint32_t rs0 = 0, rs1 = 0;  // ring slots of the stages in score buffers 0 and 1
      int spass = 0;      // scores of stage js due next: 0 none (stage not started), 1 part A, 2 part B
      uint32_t ru = 0;    // ring index of stage js once started
      bool last_js = false, ended = false;
      uint32_t pvfirst = 0;  // bit b: the stage in score buffer b is a piece's first
      uint64_t idle_since = 0;
      while (!(ended && jp == js)) {
        bool progress = false;
        if (jp < js && mbar_test(p_full, jp & 1)) {
          const int bp = jp & 1;
          const bool first = (pvfirst >> bp) & 1u;
          if (!first || npp == 0 || mbar_test(o_free, (npp - 1) & 1)) {
            tc_fence_after();
            if (first) ++npp;
            const uint32_t sp = bp ? rs1 : rs0;
            const uint64_t vd = tc_sdesc_sw128(stage0 + sp * C::STAGE_BYTES + C::NA * C::PLANE, C::PLANE, 1024);
#pragma unroll
            for (int kk = 0; kk < C::ST / 16; ++kk)
              tc_mma_ts(tmem + C::TM_O, tmem + C::TM_S + bp * C::ST + 8 * kk, vd + (uint64_t)((kk * 16 * 128) >> 4),
                        C::IDESC_PV, (first && kk == 0) ? 0u : 1u);
            tc_commit(&empty_b[sp]);
            tc_commit(pv_done);
            tc_commit(&sbuf_free[bp]);
            ++jp;
            progress = true;
          }
        }
        if (!progress && spass == 0 && !ended && mbar_test(&full_a[r % C::NS], (r / C::NS) & 1)) {
          const int s = r % C::NS;
          const int4 mf = *reinterpret_cast<const int4 *>(&meta[s].end);      // end, first, last, masked
          const int4 mg = *reinterpret_cast<const int4 *>(&meta[s].badmask);  // badmask, i0, nq, aux
          const int sb = js & 1;
          const bool buf_free = js < 2 || mbar_test(&sbuf_free[sb], ((js >> 1) - 1) & 1);
          if (mg.z) {
            // a query stage: positions 5-8 into tensor memory once the previous piece's scores are done
            if (kq == 0 || mbar_test(q_empty, (kq - 1) & 1)) {
              tc_fence_after();
              const uint64_t td0 = tc_sdesc_sw128(stage0 + s * C::STAGE_BYTES, 16, 1024);
#pragma unroll
              for (int p = 0; p < C::NQK - C::NQS; ++p)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  tc_cp_128x256b(tmem + C::TM_QT + (p * 4 + kk) * 8, td0 + (uint64_t)((p * C::QPLANE + 32 * kk) >> 4));
              tc_commit(&empty_a[s]);
              tc_commit(&empty_b[s]);
              ++kq;
              ++r;
              progress = true;
            }
          } else if (mf.x) {
            if (buf_free) {
              tc_fence_after();
              mbar_arrive(&s_full[sb]);  // the softmax warps stop at this stage
              mbar_arrive(&s_full[sb]);
              ended = true;
              progress = true;
            }
          } else if (buf_free && (!mf.y || mbar_test(q_full, kf & 1))) {
            tc_fence_after();
            if (mf.y) ++kf;
            pvfirst = (pvfirst & ~(1u << sb)) | ((uint32_t)(mf.y != 0) << sb);
            if (sb) rs1 = s; else rs0 = s;
            mbar_arrive(&s_full[sb]);  // the phase completes with the scores' commit
            last_js = mf.z != 0;
            spass = 1;
            ru = r;
            ++r;
            progress = true;
          }
        }
        if (spass == 2 && mbar_test(&full_b[ru % C::NS], (ru / C::NS) & 1)) {
          // part B: positions NA-8, query operand in tensor memory
          tc_fence_after();
          const int sb = js & 1;
          const uint64_t cd0 = tc_sdesc_sw128(stage0 + (sb ? rs1 : rs0) * C::STAGE_BYTES, 16, 1024);
          const uint32_t dS = tmem + C::TM_S + sb * C::ST;
#pragma unroll
          for (int p = C::NA; p < C::NQK; ++p)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_ts(dS, tmem + C::TM_QT + ((p - C::NQS) * 4 + kk) * 8,
                        cd0 + (uint64_t)((p * C::PLANE + 32 * kk) >> 4), C::IDESC_S, 1u);
          tc_commit(&s_full[sb]);
          if (last_js) tc_commit(q_empty);  // the query may be replaced by the next piece's
          spass = 0;
          ++js;
          progress = true;
        }
        if (spass == 1) {  // in the iteration that started the stage
          // part A: positions 0 to NA-1, query operand in shared memory; compile-time offsets
          const int sb = js & 1;
          const uint32_t sr = sb ? rs1 : rs0;
          const uint64_t cd0 = tc_sdesc_sw128(stage0 + sr * C::STAGE_BYTES, 16, 1024);
          const uint32_t dS = tmem + C::TM_S + sb * C::ST;
#pragma unroll
          for (int p = 0; p < C::NA; ++p)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_ss(dS, qd0 + (uint64_t)((p * C::QPLANE + 32 * kk) >> 4),
                        cd0 + (uint64_t)((p * C::PLANE + 32 * kk) >> 4), C::IDESC_S, (p | kk) != 0 ? 1u : 0u);
          tc_commit(&empty_a[sr]);  // part A may be reloaded once these have completed
          spass = 2;
          progress = true;
        }
        if (progress) {
          idle_since = 0;
        } else {
          const uint64_t now = global_timer_ns();
          if (idle_since == 0) {
            idle_since = now;
          } else if (now - idle_since > WAIT_LIMIT_NS) {
            atomicOr(status, PA_DEV_TIMEOUT);
            break;
          }
        }
      }
      // every operation this thread issued has completed before the tensor memory is released
      tc_commit(drain);
      mbar_wait(drain, 0, status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax and output
    const int q4 = warp & 3;                      // lanes [32 q4, +32) of the tensor memory
    const int row = 32 * q4 + lane;               // head row of the tile
    const int ts = tid - 64;                      // 0 .. 127
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
    const int bh_tokens = 1 << a.log2_bh;
    float m = -INFINITY, l = 0.f;
    for (uint32_t j = 0;; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(&s_full[sb], (j >> 1) & 1, status)) break;
      tc_fence_after();
      const StageMeta &mt = smeta[j & 3];
      if (mt.end) break;
      const int rslot = mt.aux;
      const bool first = mt.first, last = mt.last, masked = mt.masked;
      const int tok0 = mt.tok0, tok_lo = mt.tok_lo, tok_hi = mt.tok_hi;
      const uint32_t badmask = mt.badmask;
      const int b = mt.b, h0 = mt.hq0, nh = mt.ghead, hv = mt.i0, slot = mt.slot;
      if (first) {
        m = -INFINITY;
        l = 0.f;
      }
      auto visible = [&](int t) {
        const int lt = tok0 + t;
        return lt >= tok_lo && lt < tok_hi && !((badmask >> (t / bh_tokens)) & 1u);
      };
      const uint32_t tS = tl + C::TM_S + sb * C::ST;
      float x[C::ST];
      tc_ld32(tS, *reinterpret_cast<float(*)[32]>(&x[0]));
      tc_ld32(tS + 32, *reinterpret_cast<float(*)[32]>(&x[32]));
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < C::ST; ++i) {
        const float v = x[i] * a.qscale;
        x[i] = (!masked || visible(i)) ? v : -INFINITY;
        mx = fmaxf(mx, x[i]);
      }
      // the previous stage's P.V has completed: O may be rescaled
      if (j > 0 && !mbar_wait(pv_done, (j - 1) & 1, status)) break;
      tc_fence_after();
      if (__any_sync(FULL, m != -INFINITY && mx > m + C::TAU)) {
        const float mn = fmaxf(m, mx);
        const float alpha = m == -INFINITY ? 0.f : fast_exp2(m - mn);
        m = mn;
        l *= alpha;
#pragma unroll 1
        for (int c = 0; c < C::DVH; c += 32) {
          float o[32];
          tc_ld32(tl + C::TM_O + c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tc_st32(tl + C::TM_O + c, o);
        }
        tc_wait_st();
      } else if (m == -INFINITY) {
        m = mx;  // nothing attended yet in this piece: O is zero or is overwritten by the first P.V
      }
      // the probabilities, as bf16 pairs (even token in the low half), over the stage's scores
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float x0 = x[32 * h + 2 * c], x1 = x[32 * h + 2 * c + 1];
          const float p0 = x0 == -INFINITY ? 0.f : fast_exp2(x0 - m);
          const float p1 = x1 == -INFINITY ? 0.f : fast_exp2(x1 - m);
          l += p0 + p1;
          w[c] = pack_bf16x2(p0, p1);
        }
        tc_st16(tS + 16 * h, w);
      }
      tc_wait_st();
      if (masked) {
        // cache rows of keys that are not attended may hold anything (NaN included): zero their
        // latent columns of this half before P.V reads them
        uint8_t *st = smem + S::OFF_STAGE + rslot * C::STAGE_BYTES + C::NA * C::PLANE;
        for (int e = ts; e < C::ST * 32; e += C::SOFTMAX_WARPS * 32) {
          const int t = e >> 5, ch = e & 31;
          if (!visible(t))
            *reinterpret_cast<uint4 *>(st + (ch >> 3) * C::PLANE + t * 128 + (((ch & 7) ^ (t & 7)) << 4)) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      if (last) {
        // ---- end of a piece: O / l of this row, and the LSE
        if (!mbar_wait(pv_done, j & 1, status)) break;
        tc_fence_after();
        const bool rv = row < nh;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const float lse2 = (m == -INFINITY || l == 0.f) ? -INFINITY : m + __log2f(l);
        const size_t pi = (size_t)blockIdx.x * 2 + (slot > 0 ? 1 : 0);
        uint16_t *orow = a.o_lat + (((size_t)b * 2 + hv) * a.H + h0 + row) * C::DVH;
        float *prow = a.part_o + (pi * a.rs + row) * C::DVH;
#pragma unroll 1
        for (int c = 0; c < C::DVH; c += 32) {
          float o[32];
          tc_ld32(tl + C::TM_O + c, o);
          if (rv) {
            if (slot < 0) {
#pragma unroll
              for (int i = 0; i < 32; i += 8) {
                uint4 v;
                v.x = pack_bf16x2(o[i] * inv, o[i + 1] * inv);
                v.y = pack_bf16x2(o[i + 2] * inv, o[i + 3] * inv);
                v.z = pack_bf16x2(o[i + 4] * inv, o[i + 5] * inv);
                v.w = pack_bf16x2(o[i + 6] * inv, o[i + 7] * inv);
                *reinterpret_cast<uint4 *>(orow + c + i) = v;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4 *>(prow + c + i) =
                    make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free);
        if (rv) {
          if (slot < 0) {
            if (a.lse && hv == 0) a.lse[(size_t)b * a.H + h0 + row] = lse2 * LN2;
          } else {
            a.part_lse[pi * a.rs + row] = lse2;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tc_dealloc(tmem, C::TM_COLS);
  if (tid == 0) {
    GqaPartDesc d = misc->desc;
    d.status = misc->status;
    a.desc[blockIdx.x] = d;
  }
  if ((misc->desc.flags & DESC_PIECES) == 0) {
    // a CTA whose range held no visible key can still lie between two pieces of a sequence: the
    // merge walks over its slot 0, which must weigh nothing
    float *po = a.part_o + (size_t)blockIdx.x * 2 * a.rs * C::DVH;
    for (int e = tid; e < a.rs * C::DVH; e += C::THREADS) po[e] = 0.f;
    for (int h = tid; h < a.rs; h += C::THREADS) a.part_lse[(size_t)blockIdx.x * 2 * a.rs + h] = -INFINITY;
  }
}

}  // namespace pa
