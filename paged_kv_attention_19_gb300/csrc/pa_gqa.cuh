// pa_gqa.cuh -- GQA paged decode: the split-KV attention kernel and the split
// combine kernel (sm_103a).
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
//   * static, balanced partition.  A sequence is (row, KV head, tile), a tile
//     being up to 16 query rows of the KV head (a 16-head subgroup, or
//     positions x heads for verify); its visible keys are cut into units of
//     one TMA box (min(page, stage) tokens).  The CTAs (one per SM by
//     default) form groups of HG = KV heads x tiles per KV head; each group
//     takes an equal share of the rows' total cost (units plus a fixed cost
//     per piece) and CTA r of a group serves sequence r of those rows, so the
//     group's CTAs stream the same pages at about the same time (DRAM once,
//     L2 for the rest).  Each CTA finds its range from the context lengths in
//     a short prologue: no planner launch, no work queue, no atomics,
//     identical from run to run.  A range is a list of pieces (maximal runs of
//     one sequence); only its first and last piece can be part of a sequence
//     that another CTA also touches, so a CTA leaves at most two partials;
//   * the last warp is a TMA producer: it walks the CTA's pieces, keeps 32
//     block-table entries in a register window (the next window and the next
//     piece's first window already in flight), and issues a stage of the
//     piece's query rows (a 3-D tensor-map box) and then 4-D tensor-map
//     copies of page fragments into a ring of shared-memory stages (K and V
//     of 64 tokens, 32 for head_dim 256) with the 128-byte swizzle, so the
//     tensor-core fragment loads are bank-conflict free.  The ring takes all
//     of shared memory (224 KB) to keep ~200 KB of copies in flight per SM;
//   * the consumer warps take 16 tokens of every stage per token group; two
//     warps share a group, both computing its scores and each accumulating
//     half of the P.V columns.  The tile's (up to 16) query rows are the M
//     rows of mma.sync m16n8k16 bf16 tiles, read with ldmatrix from the query
//     stage into registers at the start of a piece, so S = Q K^T and
//     O += P V cost one tensor-core instruction per 8 tokens x 16 dims.  The
//     online softmax (running max with a lazy rescale, fp32 denominator) runs
//     on the CUDA cores; P is rounded to bf16 only as the MMA operand;
//   * at the end of a piece the token groups merge through the consumed stage
//     buffer; a piece that covers its whole sequence writes the final bf16
//     output and LSE, any other writes an fp32 partial (normalised output +
//     LSE) to one of the CTA's two slots;
//   * the setup, the producer, the end-of-piece merge and the epilogue are
//     device functions shared with the FP8 kernel (pa_gqa_f8.cuh);
//   * the combine kernel (a programmatic dependent launch, so its launch hides
//     under the split kernel's tail) merges every split sequence over the
//     CTAs that hold its pieces, in ascending order, one warp per row.
#pragma once

#include <type_traits>

#include "pa_common.cuh"
#include "pa_partition.cuh"

namespace pa {

// What each split CTA leaves for the combine kernel.
struct GqaPartDesc {
  int32_t last_b;   // row of the CTA's last piece
  int32_t last_hs;  // sequence of the last piece in its row (kv_head * nseqh + tile pair)
  uint32_t flags;   // bits 0-15: pieces of the CTA (saturating); DESC_* bits
  uint32_t status;  // PA_DEV_* bits seen by the CTA
};
static_assert(sizeof(GqaPartDesc) == 16, "descriptor is 16 bytes");
constexpr uint32_t DESC_PIECES = 0xffffu;
constexpr uint32_t DESC_LAST_STARTS = 1u << 16;  // the last piece begins its sequence
constexpr uint32_t DESC_LAST_ENDS = 1u << 17;    // the last piece ends its sequence
constexpr uint32_t DESC_FIRST_ENDS = 1u << 18;   // the first piece ends its sequence
constexpr int PART_HEADS = 16;                   // MMA rows of one tile (a 16-head subgroup)
constexpr int PART_ROWS = 2 * PART_HEADS;        // rows of a partial slot: up to two tiles

struct GqaArgs {
  const uint16_t *q;            // [B, Hq, D] bf16
  const int32_t *block_table;   // [B, max_pages_per_seq]
  const int32_t *context_lens;  // [B]
  uint16_t *out;                // [B, Hq, D] bf16
  float *lse;                   // [B, Hq] or null
  float *part_o;                // [nparts, 2, 16, D] fp32
  float *part_lse;              // [nparts, 2, 16] fp32, log2 units
  GqaPartDesc *desc;            // [nparts]
  int32_t *seq_first;           // [B, sequences per row]: -1 whole piece; else 2 x CTA + slot of the first piece
  int32_t *seq_last;            // [B, sequences per row]: CTA holding the last piece of a split sequence
  int batch, max_pages_per_seq, num_pages, max_context_len, window;
  int Hq, Hkv, G, nsub;
  int Q;                        // query positions per row (1: decode; > 1: verify, causal within them)
  int gt, qt, ntile;            // a tile of MMA rows: qt positions x gt heads; ntile tiles per KV head
  int mt, nseqh;                // tiles per sequence (1 or 2) and sequences per KV head (ntile / mt, rounded up)
  int log2_page, log2_bh;       // page size and tokens per unit (TMA box), as powers of two
  int unit_copy;                // 1: the unit-major kernel (GqaUnitCfg) and a 5-D pool map
  int piece_cost;               // partition cost of starting a piece, in units
  int nparts;                   // CTAs (shares); groups of hg consecutive CTAs
  int hg;                       // CTAs per group: min(Hkv * nseqh, nparts)
  float qscale;                 // scale * log2(e) (FP8: times the keys' scale)
  float vscale;                 // FP8: the values' scale; 1 for bf16 pools
  unsigned long long wait_ns;   // limit of a stage-ring wait (global-timer ns) before the CTA gives up
};

// Layout of the bf16 split kernel: stage ring, token groups, consumer warps.  The FP8
// kernel (pa_gqa_f8.cuh) has its own configuration with the same members.
template <int D_>
struct GqaCfg {
  static constexpr int D = D_;
  static constexpr bool F8 = false;                // pools of bf16 values
  static constexpr int ROWB = 128;                 // bytes of a token's row in one plane of a stage
  static constexpr int XSTEP = 64;                 // tensor-map x of consecutive planes (bf16 values)
  // A stage's K (and V) block is plane-major: its NQ planes of ST 128-byte rows (see kv_off).
  static constexpr bool UNIT_MAJOR = false;
  static constexpr int M = PART_HEADS;             // MMA rows = query heads per subgroup
  static constexpr int MR = M;                     // rows per token group in the end-of-piece merge
  static constexpr int ST = D <= 128 ? 64 : 32;    // tokens per stage
  static constexpr int TW = 16;                    // tokens per token group per stage
  static constexpr int TG = ST / TW;               // token groups per stage
  static constexpr int MG = TG;                    // groups merged at the end of a piece
  static constexpr int DSPLIT = 2;                 // warps sharing a token group (each: D / 2 of P.V)
  static constexpr int NCW = TG * DSPLIT;          // consumer warps
  // + producer warp.  With eight consumer warps the block is three warpgroups instead (the
  // producer warp and three idle ones): one producer warp beside them would put three warps on one
  // SM sub-partition and cap every thread at 168 registers, where the producer's warpgroup gives
  // registers back and the consumers' two take them (launch: 384 x 168 = 256 x 208 + 128 x 88).
  static constexpr bool REG_SPLIT = NCW == 8;
  static constexpr int THREADS = REG_SPLIT ? (NCW + 4) * 32 : (NCW + 1) * 32;
  static constexpr int CONSUMER_REGS = 208, PRODUCER_REGS = 88;
  static_assert(!REG_SPLIT || NCW * 32 * CONSUMER_REGS + 128 * PRODUCER_REGS <= THREADS * 168,
                "the register split stays within the launch's registers");
  static constexpr int NT_PV = D / 8 / DSPLIT;     // P.V n-tiles per warp
  static constexpr int NQ = D / 64;                // 128-byte swizzle planes along D
  static constexpr int QNQ = NQ;                   // the same for the query rows
  static constexpr int PLANE = ST * 128;           // bytes of one plane (ST rows x 128 bytes)
  static constexpr int KV_BYTES = NQ * PLANE;      // K (or V) of one stage
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int NS = (229376 / STAGE_BYTES) < 16 ? (229376 / STAGE_BYTES) : 16;  // 224 KB ring
  static constexpr int NACC = 2;                   // independent QK accumulators
  static constexpr int QAREA = 0;                  // query rows kept outside the ring (none)
  static_assert(MR * D * 4 * MG <= STAGE_BYTES, "the end-of-piece merge fits the consumed stage");
};

// Unit-major stage blocks (decode over pages of fewer than 32 tokens, head_dim 128 and 256): per
// unit (one box of BH tokens) its NQ planes of BH 128-byte rows, so that one 5-D copy brings all
// planes of a unit.  A copy costs the producer about the same whatever its size, and the
// plane-major order takes NQ copies per unit (16 per stage at page 16, head_dim 128).
template <int D_>
struct GqaUnitCfg : GqaCfg<D_> {
  static constexpr bool UNIT_MAJOR = true;
};

// Two 16-row tiles per sequence (gqa_consume_pair): the piece's query rows of both tiles are copied
// out of their ring stage into an area of their own, which takes one stage of the ring.
template <int D_>
struct GqaPairCfg : GqaCfg<D_> {
  using B = GqaCfg<D_>;
  static constexpr int QAREA = 2 * B::QNQ * B::M * 128;  // both tiles' rows, 128-byte swizzled planes
  static constexpr int NS = (229376 - QAREA) / B::STAGE_BYTES;
  static_assert(QAREA <= B::STAGE_BYTES, "a query stage holds both tiles' rows");
};

struct alignas(16) StageMeta {
  int32_t end, first, last, masked;  // first: a stage holding the piece's query rows only
  int32_t b, hq0, ghead, slot;  // slot: -1 = whole sequence (final output), else partial slot 0 / 1
  int32_t tok0, tok_lo, tok_hi, L;  // L: the row's length (query position i attends below L - Q + 1 + i)
  uint32_t badmask;             // bit k: box k of the stage was not loaded
  int32_t i0, nq, aux;          // the (first) tile's positions [i0, i0 + nq); ghead: its heads; aux: GQA: the
                                // sequence (hs of the piece), MLA score buffers: the ring slot of the stage
};
static_assert(sizeof(StageMeta) == 64, "stage meta is 64 bytes");

// Small shared state of a CTA outside the ring.
struct GqaMisc {
  uint32_t status;
  int32_t pad[3];
  GqaPartDesc desc;
  PartitionState part;
};

template <class C>
struct GqaSmem {
  static constexpr int OFF_STAGE = 0;
  static constexpr int OFF_QAREA = OFF_STAGE + C::NS * C::STAGE_BYTES;  // 1024-byte aligned like the stages
  static constexpr int OFF_ML = OFF_QAREA + C::QAREA;
  static constexpr int OFF_META = OFF_ML + C::MG * C::M * 2 * 4;
  static constexpr int OFF_BAR = OFF_META + C::NS * (int)sizeof(StageMeta);
  static constexpr int OFF_MISC = OFF_BAR + 2 * C::NS * 8;
  static constexpr int USED = OFF_MISC + (int)sizeof(GqaMisc);
  static constexpr int BYTES = USED + 1024;  // slack to align the base to 1024 bytes
  static_assert(BYTES <= 232448, "fits the 227 KB opt-in shared memory of one CTA");
};

// Byte offset of 16-byte chunk `chunk` (along D) of token row `tok` in a stage's K or V block of
// 128-byte rows, chunk ^ (row & 7) (the TMA 128-byte swizzle; every plane of a box starts on a
// 1024-byte boundary since a unit holds at least 8 tokens).  Plane-major (C::UNIT_MAJOR false):
// the stage's planes of 64 dims one after the other.  Unit-major: per unit of 2^lbh tokens its
// planes one after the other (the two orders agree when a unit is the whole stage).
template <class C>
__device__ __forceinline__ uint32_t kv_off(int tok, int chunk, int lbh) {
  if constexpr (C::UNIT_MAJOR && C::NQ > 1) {
    constexpr int LNQ = C::NQ == 4 ? 2 : 1;
    const int row = ((tok >> lbh) << (lbh + LNQ)) + ((chunk >> 3) << lbh) + (tok & ((1 << lbh) - 1));
    return (uint32_t)(row * 128 + (((chunk & 7) ^ (tok & 7)) << 4));
  } else {
    return (uint32_t)((chunk >> 3) * C::PLANE + tok * 128 + (((chunk & 7) ^ (tok & 7)) << 4));
  }
}

// Tile t of a KV head's query rows: positions [i0, i0 + nq), heads [h0, h0 + nh) of the
// group (h0 relative to the group's first head).  MMA row r is position i0 + r / gt, head
// h0 + r % gt; it is a real row when r / gt < nq and r % gt < nh.
struct Tile {
  int i0, nq, h0, nh;
};
__device__ __forceinline__ Tile tile_of(int t, int G, int nsub, int Q, int qt) {
  Tile x;
  if (G < 16) {
    x.i0 = t * qt;
    x.nq = min(qt, Q - x.i0);
    x.h0 = 0;
    x.nh = G;
  } else {
    x.i0 = t / nsub;
    x.nq = 1;
    x.h0 = (t % nsub) * 16;
    x.nh = min(16, G - x.h0);
  }
  return x;
}

// ---------------------------------------------------------------------------
// Parts shared by the bf16 and FP8 split kernels.  C: the kernel's configuration
// (ring geometry, consumer warp count, merge rows).

// Barriers, tensor-map prefetch, the programmatic-launch wait and the partition
// prologue (this CTA's range); rows with no visible key get their zero output.
template <class C>
__device__ __forceinline__ void gqa_setup(uint8_t *smem, const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                                          const CUtensorMap *tm_q, const GqaArgs &a, PartitionArgs &pargs) {
  using S = GqaSmem<C>;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
  uint64_t *empty = full + C::NS;
  GqaMisc *misc = reinterpret_cast<GqaMisc *>(smem + S::OFF_MISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NCW);
    }
    fence_mbar_init();
    misc->status = 0;
  }
  if (warp == C::NCW && lane == 0) {
    prefetch_tensormap(tm_k);
    prefetch_tensormap(tm_v);
    prefetch_tensormap(tm_q);
  }
  __syncthreads();
  pdl_wait();               // inputs written by the stream's previous kernel are visible from here on
  pdl_launch_dependents();  // the combine kernel may be scheduled; it waits for this grid to finish
  pargs.context_lens = a.context_lens;
  pargs.batch = a.batch;
  pargs.max_context_len = a.max_context_len;
  pargs.Q = a.Q;
  pargs.window = a.window;
  pargs.log2_bh = a.log2_bh;
  pargs.piece_cost = a.piece_cost;
  pargs.nparts = a.nparts;
  pargs.hg = a.hg;
  pargs.hs = a.Hkv * a.nseqh;  // sequences per row: KV heads x tile groups
  partition_prologue<C::THREADS>(pargs, &misc->part, &misc->status);
  zero_empty_rows<C::THREADS>(pargs, a.out, a.lse, a.Q * a.Hq * C::D, a.Q * a.Hq);
  __syncthreads();
}

// The producer warp: walks the CTA's pieces and fills the stage ring (a stage of the piece's
// query rows, then its K/V stages), ends with an end marker.  LW: its waits for a free slot take
// the call's limit (a.wait_ns) and follow the give-up protocol of ring_wait (a late wait: no
// further stage, the end marker once the slot is free); otherwise they are bounded at 1 s.  The
// consumers' waits follow the same rule.
template <class C, bool LW, int MT>
__device__ __forceinline__ void gqa_produce(uint8_t *smem, const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                                            const CUtensorMap *tm_q, const GqaArgs &a, const PartitionArgs &pargs) {
  using S = GqaSmem<C>;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
  uint64_t *empty = full + C::NS;
  StageMeta *meta = reinterpret_cast<StageMeta *>(smem + S::OFF_META);
  GqaMisc *misc = reinterpret_cast<GqaMisc *>(smem + S::OFF_MISC);
  uint32_t *status = &misc->status;
  const int lane = threadIdx.x & 31;
  const int P = 1 << a.log2_page;
  const int nbox = C::ST >> a.log2_bh;  // boxes (units) per stage
  uint32_t j = 0;
  bool ok = true;
  bool stop = false;  // LW: a wait passed the call's limit: no more stages, straight to the end marker
  // a wait for a free slot: RING_OK, RING_LATE (LW only) or RING_FAILED
  auto slot_wait = [&](int s, uint32_t parity) -> int {
    if constexpr (LW) return ring_wait(&empty[s], parity, a.wait_ns, status);
    else return mbar_wait(&empty[s], parity, status) ? RING_OK : RING_FAILED;
  };
  int npieces = 0;
  Piece last_piece = {};
  bool first_ends = false;
  PieceWalker walker(pargs, &misc->part, lane);
  auto take_piece = [&](Piece &pc) { return walker.take(pc); };
  // block-table window 0 of a piece (lane l: entry l of its first page)
  auto piece_window = [&](const Piece &p) {
    const int pb = (p.ub << a.log2_bh) >> a.log2_page;
    const int pe = (((p.ue << a.log2_bh) - 1) >> a.log2_page) + 1;
    return lane < pe - pb ? a.block_table[(size_t)p.b * a.max_pages_per_seq + pb + lane] : 0;
  };
  Piece cur = {}, nxt = {};
  bool has_cur = take_piece(cur);
  int cwin0 = 0, nwin0 = 0;
  bool has_next = false;
  if (has_cur) {
    cwin0 = piece_window(cur);
    has_next = take_piece(nxt);
    if (has_next) nwin0 = piece_window(nxt);
  }
  while (has_cur && ok && !stop) {
    // ---- emit the stages of `cur`
    const int g = cur.hs / a.nseqh;
    const int t0 = (cur.hs % a.nseqh) * MT;                     // the sequence's first tile
    const bool two = MT == 2 && t0 + 1 < a.ntile;                // and a second one
    const Tile tl = tile_of(t0, a.G, a.nsub, a.Q, a.qt);
    const Tile tlz = two ? tile_of(t0 + 1, a.G, a.nsub, a.Q, a.qt) : tl;  // the last tile
    const int hq0 = g * a.G + tl.h0;
    // the sequence's tightest key bounds: its first position ends first, its last starts last
    const int hi_min = pos_hi(cur.L, a.Q, tl.i0), lo_max = pos_lo(cur.L, a.Q, tlz.i0 + tlz.nq - 1, a.window);
    const int slot = (cur.starts && cur.ends) ? -1 : (npieces == 0 ? 0 : 1);
    if (lane == 0) {
      // where the combine kernel finds the sequence: written whole (one piece), or merged from the
      // partial slots of CTAs first, first + hg, ..., last
      const size_t si = (size_t)cur.b * pargs.hs + cur.hs;
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
    int fwin = (lane + 32 < npages) ? bt_piece[32 + lane] : 0;  // window 1, in flight
    {
      // the piece's query rows: a stage of their own (a qt x gt box of (position, head) rows
      // from position i0 and head hq0; rows of other heads or positions are masked by the
      // consumers)
      const int s = j % C::NS;
      const uint32_t u = j / C::NS;
      if (u > 0) {
        const int wr = slot_wait(s, (u - 1) & 1);
        ok = wr != RING_FAILED;
        stop = wr == RING_LATE;
      }
      if (!ok || stop) break;
      if (lane == 0) {
        StageMeta &m = meta[s];
        m.end = 0;
        m.first = 1;
        m.last = 0;
        m.b = cur.b;
        m.hq0 = hq0;
        m.ghead = tl.nh;
        m.i0 = tl.i0;
        m.nq = tl.nq;
        m.aux = cur.hs;
        m.L = cur.L;
        mbar_arrive_expect_tx(&full[s], (uint32_t)(C::QNQ * a.gt * a.qt * 128 * (two ? 2 : 1)));
        uint8_t *qdst = smem + S::OFF_STAGE + s * C::STAGE_BYTES;
#pragma unroll
        for (int dq = 0; dq < C::QNQ; ++dq)
          tma_load_3d(qdst + dq * (C::M * 128), tm_q, dq * 64, hq0, cur.b * a.Q + tl.i0, &full[s]);
        if (two) {  // the second tile's rows follow the first's planes
#pragma unroll
          for (int dq = 0; dq < C::QNQ; ++dq)
            tma_load_3d(qdst + (C::QNQ + dq) * (C::M * 128), tm_q, dq * 64, g * a.G + tlz.h0,
                        cur.b * a.Q + tlz.i0, &full[s]);
        }
      }
      __syncwarp();
      ++j;
    }
    for (int t = 0; t < n_stages && ok; ++t, ++j) {
      const int s = j % C::NS;
      const uint32_t u = j / C::NS;
      if (u > 0) {
        const int wr = slot_wait(s, (u - 1) & 1);
        ok = wr != RING_FAILED;
        stop = wr == RING_LATE;
      }
      if (!ok || stop) break;
      const int unit0 = cur.ub + t * nbox;
      const int tok0 = unit0 << a.log2_bh;
      // the pages of one stage never straddle a 32-page window (nbox divides 32)
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
        m.hq0 = hq0;
        m.ghead = tl.nh;
        m.i0 = tl.i0;
        m.nq = tl.nq;
        m.aux = cur.hs;
        m.L = cur.L;
        m.slot = slot;
        m.tok0 = tok0;
        m.tok_lo = tok_lo;
        m.tok_hi = tok_hi;
        m.badmask = bad;
        m.masked = (tok0 < max(tok_lo, lo_max)) || (tok0 + C::ST > min(tok_hi, hi_min)) || bad != 0;
        mbar_arrive_expect_tx(&full[s], (uint32_t)nvalid * (uint32_t)((C::NQ * C::ROWB * 2) << a.log2_bh));
      }
      __syncwarp();
      if (load) {
        const int pslot = btok & (P - 1);
        if constexpr (C::UNIT_MAJOR && C::NQ > 1) {
          // one copy per unit and pool: (64 dims, the unit's tokens, all planes, head g, page)
          uint8_t *dst = kdst + (lane << a.log2_bh) * (C::NQ * C::ROWB);
          tma_load_5d(dst, tm_k, 0, pslot, 0, g, phys, &full[s]);
          tma_load_5d(dst + C::KV_BYTES, tm_v, 0, pslot, 0, g, phys, &full[s]);
        } else {
          uint8_t *dst = kdst + (lane << a.log2_bh) * C::ROWB;
#pragma unroll
          for (int dq = 0; dq < C::NQ; ++dq) {
            const int x = dq * C::XSTEP;  // C::ROWB bytes of the row per plane
            tma_load_4d(dst + dq * C::PLANE, tm_k, x, g, pslot, phys, &full[s]);
            tma_load_4d(dst + dq * C::PLANE + C::KV_BYTES, tm_v, x, g, pslot, phys, &full[s]);
          }
        }
      }
    }
    if (!ok || stop) break;
    if (npieces == 0) first_ends = cur.ends;
    if (npieces < (int)DESC_PIECES) ++npieces;
    last_piece = cur;
    has_cur = has_next;
    if (!has_cur) break;
    cur = nxt;
    cwin0 = nwin0;
    has_next = take_piece(nxt);
    if (has_next) nwin0 = piece_window(nxt);
  }
  if (ok) {
    // end marker (after a late wait too, into the slot that wait was for, which is free by then:
    // the consumers finish the stages already issued and leave)
    const int s = j % C::NS;
    const uint32_t u = j / C::NS;
    if (u > 0 && !stop) ok = slot_wait(s, (u - 1) & 1) != RING_FAILED;
    if (ok && lane == 0) {
      meta[s].end = 1;
      mbar_arrive(&full[s]);
    }
  }
  if (!ok) {
    // A wait gave up: let the copies this warp issued land before the CTA exits.
    const uint32_t first = j > (uint32_t)C::NS ? j - C::NS : 0u;
    for (uint32_t i = first; i < j; ++i) mbar_wait(&full[i % C::NS], (i / C::NS) & 1, status);
  }
  if (lane == 0) {
    misc->desc.last_b = last_piece.b;
    misc->desc.last_hs = last_piece.hs;
    misc->desc.flags = (uint32_t)npieces | (last_piece.starts ? DESC_LAST_STARTS : 0u) |
                       (last_piece.ends ? DESC_LAST_ENDS : 0u) | (first_ends ? DESC_FIRST_ENDS : 0u);
  }
}

// End of a piece, after each of the C::MG groups has put its (m, l) in sm_ml and its unnormalised
// output rows in the merge area mg ([group][row][D] fp32, column of (row h, dim d) at
// d ^ (4 (h & 7))): each thread takes 4 consecutive dims of one row and merges the groups
// with weights exp2(m_w - M) / sum_w l_w exp2(m_w - M); a piece that covers its sequence writes
// bf16 out and the LSE, any other an fp32 partial (times oscale / L either way).
// The rows one merge writes: a tile of the piece's sequence (positions [i0, i0 + nq), heads
// [hq0, hq0 + nh)) and where its rows start in a partial slot.
struct MergeRows {
  int slot, b, i0, nq, hq0, nh, prow0;
};

template <class C, bool MQ>
__device__ __forceinline__ void gqa_merge_out(const float *mg, const float *sm_ml, const MergeRows &mt,
                                              const GqaArgs &a, int ct, float oscale) {
  constexpr int D = C::D;
  const int slot = mt.slot;
  const size_t pi = (size_t)blockIdx.x * 2 + (slot > 0 ? 1 : 0);  // partial slot (when slot >= 0)
  const int nrows = MQ ? mt.nq * a.gt : mt.nh;
  for (int e = ct; e < nrows * (D / 4); e += C::NCW * 32) {
    const int h = e / (D / 4), d4 = (e % (D / 4)) * 4;  // h: the MMA row
    if (MQ && h % a.gt >= mt.nh) continue;             // not a head of this tile
    float mw[C::MG], M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::MG; ++w) {
      mw[w] = sm_ml[(w * C::MR + h) * 2];
      M = fmaxf(M, mw[w]);
    }
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < C::MG; ++w) {
      const float wt = (mw[w] == -INFINITY) ? 0.f : fast_exp2(mw[w] - M);
      L += sm_ml[(w * C::MR + h) * 2 + 1] * wt;
      const float4 x = *reinterpret_cast<const float4 *>(mg + (w * C::MR + h) * D + (d4 ^ (4 * (h & 7))));
      o.x += wt * x.x;
      o.y += wt * x.y;
      o.z += wt * x.z;
      o.w += wt * x.w;
    }
    const float inv = L > 0.f ? oscale / L : 0.f;
    const size_t bh = MQ ? ((size_t)mt.b * a.Q + mt.i0 + h / a.gt) * a.Hq + mt.hq0 + h % a.gt
                         : (size_t)mt.b * a.Hq + mt.hq0 + h;
    if (slot < 0) {
      uint2 v;
      v.x = pack_bf16x2(o.x * inv, o.y * inv);
      v.y = pack_bf16x2(o.z * inv, o.w * inv);
      *reinterpret_cast<uint2 *>(a.out + bh * D + d4) = v;
    } else {
      *reinterpret_cast<float4 *>(a.part_o + (pi * PART_ROWS + mt.prow0 + h) * D + d4) =
          make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
    }
    if (d4 == 0) {
      const float lse2 = (M == -INFINITY || L == 0.f) ? -INFINITY : M + __log2f(L);
      if (slot < 0) {
        if (a.lse) a.lse[bh] = lse2 * LN2;
      } else {
        a.part_lse[pi * PART_ROWS + mt.prow0 + h] = lse2;
      }
    }
  }
}

// A consumer warp whose ring wait at stage j was late (it has completed since): it computes nothing
// more, but releases this and every later stage and meets both end-of-piece barriers of every
// piece's last stage, up to the end marker, as the warps still computing do.
template <class C, int MT>
__device__ __forceinline__ void gqa_consumer_drain(uint8_t *smem, uint32_t j, const GqaArgs &a) {
  using S = GqaSmem<C>;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
  uint64_t *empty = full + C::NS;
  const StageMeta *meta = reinterpret_cast<const StageMeta *>(smem + S::OFF_META);
  for (bool first_stage = true;; ++j, first_stage = false) {
    const int s = j % C::NS;
    if (!first_stage && !mbar_wait_warp(&full[s], (j / C::NS) & 1, DRAIN_LIMIT_NS)) break;
    const StageMeta &mt = meta[s];
    if (mt.end) break;
    if (mt.last) {  // one merge round (two barriers) per tile of the sequence
      const bool two = MT == 2 && (mt.aux % a.nseqh) * MT + 1 < a.ntile;
      for (int r = 0; r < (two ? 2 : 1); ++r) {
        named_bar(1, C::NCW * 32);
        named_bar(1, C::NCW * 32);
      }
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&empty[s]);
  }
}

// Descriptor of the CTA's pieces for the combine kernel; an idle CTA leaves slot 0 empty
// (lse -inf, output 0), so a merge that spans it adds nothing.
template <class C>
__device__ __forceinline__ void gqa_finish(uint8_t *smem, const GqaArgs &a) {
  using S = GqaSmem<C>;
  constexpr int D = C::D;
  GqaMisc *misc = reinterpret_cast<GqaMisc *>(smem + S::OFF_MISC);
  const int tid = threadIdx.x;
  __syncthreads();
  if (tid == 0) {
    GqaPartDesc d = misc->desc;
    d.status = misc->status;
    a.desc[blockIdx.x] = d;
  }
  if ((misc->desc.flags & DESC_PIECES) == 0) {
    for (int e = tid; e < PART_ROWS * D; e += C::THREADS) a.part_o[(size_t)blockIdx.x * 2 * PART_ROWS * D + e] = 0.f;
    for (int h = tid; h < PART_ROWS; h += C::THREADS) a.part_lse[(size_t)blockIdx.x * 2 * PART_ROWS + h] = -INFINITY;
  }
}

// Consumers of sequences of two 16-row tiles (MT = 2, configuration GqaPairCfg).  Warp w serves
// tile w / TG over token group w % TG of every stage: it computes that tile's scores of the group's
// 16 tokens and accumulates all D columns of its P.V (where the one-tile consumers split the columns
// between two warps that both compute the scores), so the two warps of a token group read each K
// and V fragment of the stage, one per tile, and no score is computed twice.  At the start of a
// piece the consumers copy both tiles' query rows out of their ring stage into the query area
// (the stage goes back at once: a ring stage held for a whole piece would be needed again before
// the piece's end) and read the A fragments from there at every stage.  The end of a piece merges
// the tiles one after the other through the consumed stage.
template <class C, bool MQ, bool LW>
__device__ __forceinline__ void gqa_consume_pair(uint8_t *smem, const GqaArgs &a) {
  using S = GqaSmem<C>;
  constexpr int D = C::D;
  constexpr int NTF = D / 8;                 // P.V n-tiles: all columns of the tile
  constexpr int QOFF1 = C::QNQ * C::M * 128;  // the second tile's rows in a query stage / the area
  static_assert(C::NCW == 2 * C::TG, "one warp per (tile, token group)");
  static_assert(C::QAREA == 2 * QOFF1, "the query area holds both tiles");
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
  uint64_t *empty = full + C::NS;
  const StageMeta *meta = reinterpret_cast<const StageMeta *>(smem + S::OFF_META);
  GqaMisc *misc = reinterpret_cast<GqaMisc *>(smem + S::OFF_MISC);
  uint32_t *status = &misc->status;
  float *sm_ml = reinterpret_cast<float *>(smem + S::OFF_ML);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ct = tid;
  const int g8 = lane >> 2, tq = lane & 3;          // MMA fragment row / column pair
  const int lm_mat = lane >> 3, lm_row = lane & 7;  // ldmatrix: matrix / row this lane addresses
  const int tgrp = warp % C::TG;                    // token group of this warp
  const int x = warp / C::TG;                       // the tile it serves
  const int wbase = tgrp * C::TW;                   // first stage token of this warp
  const float TAU = 8.f;
  const int bh_tokens = 1 << a.log2_bh;
  const int lbh = a.log2_bh;  // tokens per unit, log2 (the stage layout of kv_off)
  const uint32_t qarea = smem_u32(smem + S::OFF_QAREA) + x * QOFF1;
  // one QK accumulator per n-tile: the tile's 64 P.V accumulators fill the registers (two
  // accumulators spilled and were 2 us slower on the 4-position verify workload)
  constexpr int NACC = 1;

  float acc[NTF][4];  // O C-fragments of the tile: [n-tile][row g8 x2, row g8+8 x2]
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  bool rv0 = false, rv1 = false;  // this thread's fragment rows (g8, g8 + 8): real rows?
  int lo0 = 0, hi0 = 0, lo1 = 0, hi1 = 0;  // their key bounds [lo, hi)
  bool two = false;     // the piece's sequence has a second tile (the same in every warp)
  bool active = false;  // this warp's tile is in it
  bool late = false;    // LW: a wait was late; from then on only the ring's protocol is kept
  for (uint32_t j = 0;; ++j) {
    const int s = j % C::NS;
    if constexpr (LW) {
      const int wr = ring_wait(&full[s], (j / C::NS) & 1, late ? DRAIN_LIMIT_NS : a.wait_ns, status);
      if (wr == RING_FAILED) break;
      late = late || wr == RING_LATE;
    } else {
      if (!mbar_wait(&full[s], (j / C::NS) & 1, status)) break;
    }
    const StageMeta &mt = meta[s];
    if (mt.end) break;
    const uint32_t kbase = smem_u32(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
    const uint32_t vbase = kbase + C::KV_BYTES;
    const int t0 = (mt.aux % a.nseqh) * 2;
    if (mt.first) {
      // a new piece: both tiles' query rows into the query area (every warp passed the previous
      // piece's merge, the last reads of the area, before this stage), fresh softmax state
      two = t0 + 1 < a.ntile;
      active = x == 0 || two;
      if (!late) {
        const uint4 *src = reinterpret_cast<const uint4 *>(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
        uint4 *dst = reinterpret_cast<uint4 *>(smem + S::OFF_QAREA);
        for (int e = ct; e < C::QAREA / 16; e += C::NCW * 32) dst[e] = src[e];
        const Tile tl = tile_of(active ? t0 + x : t0, a.G, a.nsub, a.Q, a.qt);
        if constexpr (MQ) {
          const int iq0 = g8 / a.gt, hh0 = g8 % a.gt, iq1 = (g8 + 8) / a.gt, hh1 = (g8 + 8) % a.gt;
          rv0 = active && iq0 < tl.nq && hh0 < tl.nh;
          rv1 = active && iq1 < tl.nq && hh1 < tl.nh;
          lo0 = pos_lo(mt.L, a.Q, tl.i0 + iq0, a.window);
          hi0 = pos_hi(mt.L, a.Q, tl.i0 + iq0);
          lo1 = pos_lo(mt.L, a.Q, tl.i0 + iq1, a.window);
          hi1 = pos_hi(mt.L, a.Q, tl.i0 + iq1);
        } else {  // one position: row r is head r of the tile
          rv0 = active && g8 < tl.nh;
          rv1 = active && g8 + 8 < tl.nh;
        }
#pragma unroll
        for (int n = 0; n < NTF; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
      }
      named_bar(1, C::NCW * 32);  // the area is complete before any warp reads it
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      continue;
    }
    const bool masked = mt.masked;
    if (active && !late) {
      // ---- S = Q K^T of this tile for the group's 16 tokens (two n-tiles of 8)
      float sv[2][4];
      {
        float sp[NACC][2][4];
#pragma unroll
        for (int q = 0; q < NACC; ++q)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) sp[q][nt][0] = sp[q][nt][1] = sp[q][nt][2] = sp[q][nt][3] = 0.f;
#pragma unroll
        for (int ks2 = 0; ks2 < D / 32; ++ks2) {
          uint32_t qf[2][4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int ks = 2 * ks2 + h;
            const int row = (lm_mat & 1) * 8 + lm_row, chunk = 2 * ks + (lm_mat >> 1);
            ldmatrix_x4(qf[h], qarea + (chunk >> 3) * (C::M * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
          }
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            uint32_t b[4];
            ldmatrix_x4(b, kbase + kv_off<C>(wbase + nt * 8 + lm_row, 4 * ks2 + lm_mat, lbh));
            mma_bf16_16816(sp[(2 * ks2) % NACC][nt], qf[0], b[0], b[1]);
            mma_bf16_16816(sp[(2 * ks2 + 1) % NACC][nt], qf[1], b[2], b[3]);
          }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float v = sp[0][nt][e];
#pragma unroll
            for (int q = 1; q < NACC; ++q) v += sp[q][nt][e];
            sv[nt][e] = v;
          }
      }
      // scale, mask (invalid tokens and padded rows -> -inf)
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
            if constexpr (MQ) valid = valid && ltok >= ((e < 2) ? lo0 : lo1) && ltok < ((e < 2) ? hi0 : hi1);
          }
          sv[nt][e] = valid ? v : -INFINITY;
        }
      // ---- online softmax per row (rows g8 and g8 + 8)
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
        for (int n = 0; n < NTF; ++n) {
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
        // V rows of keys that are not attended may hold anything, NaN included: zero them (all
        // columns of the group's rows; the other tile's warp of the group writes the same zeros)
        // so that 0 x row stays 0
        uint8_t *vgen = smem + S::OFF_STAGE + s * C::STAGE_BYTES + C::KV_BYTES;
        constexpr int CPR = C::NQ * 8;  // 16-byte chunks of a row
        for (int e = lane; e < C::TW * CPR; e += 32) {
          const int stok = wbase + e / CPR;
          const int chunk = e % CPR;
          const int ltok = mt.tok0 + stok;
          if (ltok < mt.tok_lo || ltok >= mt.tok_hi || ((mt.badmask >> (stok / bh_tokens)) & 1u))
            *reinterpret_cast<uint4 *>(vgen + kv_off<C>(stok, chunk, lbh)) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      // ---- O += P V (k = the group's 16 tokens), all columns
      {
        const int tok = wbase + (lm_mat & 1) * 8 + lm_row;
#pragma unroll
        for (int nd = 0; nd < NTF; nd += 2) {
          uint32_t b[4];
          ldmatrix_x4_trans(b, vbase + kv_off<C>(tok, nd + (lm_mat >> 1), lbh));
          mma_bf16_16816(acc[nd], pa, b[0], b[1]);
          mma_bf16_16816(acc[nd + 1], pa, b[2], b[3]);
        }
      }
    }

    if (mt.last) {
      // ---- end of a piece: the tiles one after the other, through this stage's buffer
      float *mg = reinterpret_cast<float *>(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
      const int g = mt.aux / a.nseqh;
      if (active && !late) {
        l0 += __shfl_xor_sync(FULL, l0, 1);
        l0 += __shfl_xor_sync(FULL, l0, 2);
        l1 += __shfl_xor_sync(FULL, l1, 1);
        l1 += __shfl_xor_sync(FULL, l1, 2);
      }
      for (int xr = 0; xr < (two ? 2 : 1); ++xr) {
        named_bar(1, C::NCW * 32);  // all warps are done reading this stage (or the last merge)
        if (x == xr && !late) {
#pragma unroll
          for (int n = 0; n < NTF; ++n) {
            const int d = (n * 8 + 2 * tq) ^ (4 * g8);
            *reinterpret_cast<float2 *>(mg + (tgrp * C::M + g8) * D + d) = make_float2(acc[n][0], acc[n][1]);
            *reinterpret_cast<float2 *>(mg + (tgrp * C::M + g8 + 8) * D + d) = make_float2(acc[n][2], acc[n][3]);
          }
          if (tq == 0) {
            sm_ml[(tgrp * C::M + g8) * 2] = m0;
            sm_ml[(tgrp * C::M + g8) * 2 + 1] = l0;
            sm_ml[(tgrp * C::M + g8 + 8) * 2] = m1;
            sm_ml[(tgrp * C::M + g8 + 8) * 2 + 1] = l1;
          }
        }
        named_bar(1, C::NCW * 32);
        if (!late) {
          const Tile tl = tile_of(t0 + xr, a.G, a.nsub, a.Q, a.qt);
          const MergeRows rows = {mt.slot, mt.b, tl.i0, tl.nq, g * a.G + tl.h0, tl.nh, xr * C::M};
          gqa_merge_out<C, MQ>(mg, sm_ml, rows, a, ct, 1.f);
        }
      }
      // no CTA barrier before the release: every warp arrives on the stage's empty barrier
      // after its own reads, and the producer refills the stage only once all have arrived
      fence_proxy_async_smem();  // generic writes to the stage buffer precede its next TMA fill
    } else if (masked) {
      fence_proxy_async_smem();  // the zeroed V rows precede the next TMA fill of this stage
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

// MQ: several query positions per row (verify); false compiles the decode-only row logic.
// LW: the stage ring's waits take the call's limit (see gqa_produce).
// MT: tiles per sequence.  With MT = 2 a sequence is a pair of 16-row tiles of one KV head (32
// (position, head) rows: verify with more than 16 rows per KV head, or more than 16 heads per
// group): each K or V fragment a warp loads from the stage feeds the MMAs of both tiles, so a page
// crosses shared memory once for all of the head's rows.
// UM: unit-major stage blocks (GqaUnitCfg; one-tile sequences).
template <int D, int MT, bool UM = false>
using GqaCfgOf = std::conditional_t<MT == 2, GqaPairCfg<D>, std::conditional_t<UM, GqaUnitCfg<D>, GqaCfg<D>>>;

template <int D, bool MQ, bool LW, int MT, bool UM = false>
__global__ void __launch_bounds__(GqaCfg<D>::THREADS, 1)
    gqa_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_q, const GqaArgs a) {
  using C = GqaCfgOf<D, MT, UM>;
  static_assert(!UM || MT == 1, "unit-major stage blocks serve one-tile sequences");
  using S = GqaSmem<C>;
  static_assert(MT == 1 || MT == 2, "one or two tiles per sequence");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the 128-byte swizzle pattern repeats every 1024 bytes: start the stages on such a boundary
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
    if (warp == C::NCW) gqa_produce<C, LW, MT>(smem, &tm_k, &tm_v, &tm_q, a, pargs);
  } else {
    if constexpr (C::REG_SPLIT) setmaxnreg_inc<C::CONSUMER_REGS>();
    if constexpr (MT == 2) {
      gqa_consume_pair<C, MQ, LW>(smem, a);
    } else {
      // ------------------------------------------------------------ consumers
      const int ct = tid;                               // consumer thread index
      const int g8 = lane >> 2, tq = lane & 3;          // MMA fragment row / column pair
      const int lm_mat = lane >> 3, lm_row = lane & 7;  // ldmatrix: matrix / row this lane addresses
      const int tgrp = warp % C::TG;                    // token group of this warp
      const int dh = warp / C::TG;                      // which half of the P.V columns it owns
      const int wbase = tgrp * C::TW;                   // first stage token of this warp
      const int nd0 = dh * C::NT_PV;                    // first P.V n-tile of this warp
      float *sm_ml = reinterpret_cast<float *>(smem + S::OFF_ML);
      const float TAU = 8.f;
      const int bh_tokens = 1 << a.log2_bh;
      const int lbh = a.log2_bh;  // tokens per unit, log2 (the stage layout of kv_off)

      uint32_t qa[D / 16][4];  // Q A-fragments (rows = heads)
      float acc[C::NT_PV][4];  // O C-fragments of this warp's columns: [n-tile][row g8 x2, row g8+8 x2]
      float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
      // this thread's two fragment rows (g8, g8 + 8): real row?, key bounds [lo, hi) of its position
      bool rv0 = false, rv1 = false;
      int lo0 = 0, hi0 = 0, lo1 = 0, hi1 = 0;
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
          // a new piece: its query rows into the A-fragments (ldmatrix from the 128-byte
          // swizzled planes of 16 rows x 64 dims), fresh softmax state, and the stage goes back
          if constexpr (MQ) {
            const int iq0 = g8 / a.gt, hh0 = g8 % a.gt, iq1 = (g8 + 8) / a.gt, hh1 = (g8 + 8) % a.gt;
            rv0 = iq0 < mt.nq && hh0 < mt.ghead;
            rv1 = iq1 < mt.nq && hh1 < mt.ghead;
            lo0 = pos_lo(mt.L, a.Q, mt.i0 + iq0, a.window);
            hi0 = pos_hi(mt.L, a.Q, mt.i0 + iq0);
            lo1 = pos_lo(mt.L, a.Q, mt.i0 + iq1, a.window);
            hi1 = pos_hi(mt.L, a.Q, mt.i0 + iq1);
          } else {  // one position: row r is head r, and the piece's bounds are the row's
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

        // ---- S = Q K^T for the group's 16 tokens (two n-tiles of 8); the k-steps are spread
        // over NACC independent accumulators so no long chain of dependent MMAs forms
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
              ldmatrix_x4(b, kbase + kv_off<C>(wbase + nt * 8 + lm_row, 4 * ks2 + lm_mat, lbh));
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
        // scale, mask (invalid tokens and padded head rows -> -inf)
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
              *reinterpret_cast<uint4 *>(vgen + kv_off<C>(stok, chunk, lbh)) = make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
        }
        // ---- O += P V (k = the group's 16 tokens), this warp's columns
        {
          const int tok = wbase + (lm_mat & 1) * 8 + lm_row;
  #pragma unroll
          for (int nd = 0; nd < C::NT_PV; nd += 2) {
            uint32_t b[4];
            ldmatrix_x4_trans(b, vbase + kv_off<C>(tok, nd0 + nd + (lm_mat >> 1), lbh));
            mma_bf16_16816(acc[nd], pa, b[0], b[1]);
            mma_bf16_16816(acc[nd + 1], pa, b[2], b[3]);
          }
        }

        if (mt.last) {
          // ---- end of a piece: merge the token groups through this stage's buffer
          l0 += __shfl_xor_sync(FULL, l0, 1);
          l0 += __shfl_xor_sync(FULL, l0, 2);
          l1 += __shfl_xor_sync(FULL, l1, 1);
          l1 += __shfl_xor_sync(FULL, l1, 2);
          named_bar(1, C::NCW * 32);  // all warps are done reading this stage
          float *mg = reinterpret_cast<float *>(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
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
          const MergeRows rows = {mt.slot, mt.b, mt.i0, mt.nq, mt.hq0, mt.ghead, 0};
          gqa_merge_out<C, MQ>(mg, sm_ml, rows, a, ct, 1.f);
          // no CTA barrier before the release: every warp arrives on the stage's empty barrier
          // after its own reads, and the producer refills the stage only once all have arrived
          fence_proxy_async_smem();  // generic writes to the stage buffer precede its next TMA fill
        } else if (masked) {
          fence_proxy_async_smem();  // the zeroed V rows precede the next TMA fill of this stage
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
    }
  }
  gqa_finish<C>(smem, a);
}

struct CombineArgs {
  uint16_t *out;
  float *lse;
  const float *part_o;
  const float *part_lse;
  const GqaPartDesc *desc;
  const int32_t *seq_first, *seq_last;  // where each sequence's pieces are (written by the split kernel)
  const int32_t *context_lens;
  uint32_t *status;  // the workspace status word: OR of every CTA's bits
  int Hq, G, nsub, nparts, hg;
  int Q, gt, qt, ntile, mt, nseqh;
  int hs, max_context_len;  // sequences per row; the call's bound on the context lengths
  int nblocks;              // batch x hs: one block per sequence
};

// One block per sequence (row b, sequence q of the row).  A sequence that one piece covered was
// written by the split kernel; a split one is merged here from the partial slots of CTAs first,
// first + hg, ..., last (its pieces in ascending token order; a CTA in between whose range held no
// visible key left an empty slot, lse -inf, that weighs nothing).  Warp w handles row w of the
// sequence's slots, i.e. MMA row w % 16 of its tile w / 16, each lane owning D/32 dims: an online
// log-sum-exp merge (running max, rescaled sum and accumulator).  The partials (LSE and values) of
// up to four pieces are loaded together before any of them is merged, so after the table lookup a
// sequence of at most four pieces costs one trip to L2.  The indices read from the tables are
// range-checked.
constexpr int COMBINE_THREADS = PART_ROWS * 32;  // the largest block: two tiles
template <int D>
__global__ void __launch_bounds__(COMBINE_THREADS) gqa_combine_kernel(const CombineArgs a) {
  pdl_wait();               // the split kernel's partials, tables and descriptors are visible from here on
  pdl_launch_dependents();  // a following kernel may stage its inputs
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && warp == 0) {
    uint32_t st = 0;
    for (int i = lane; i < a.nparts; i += 32) st |= a.desc[i].status;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) st |= __shfl_xor_sync(FULL, st, o);
    if (lane == 0) *a.status = st;
  }
  const int b = blockIdx.x / a.hs, q = blockIdx.x % a.hs;
  const size_t si = (size_t)b * a.hs + q;
  const int L = a.context_lens[b], f = a.seq_first[si], cl = a.seq_last[si];
  const int c0 = f >> 1;
  if (clamp_len(L, a.max_context_len) == 0 || f < 0 || c0 >= a.nparts || cl < c0 || cl >= a.nparts ||
      (cl - c0) % a.hg != 0)
    return;  // an empty row, a sequence written whole, or (only if the split kernel gave up) a stale entry
  const int k = (cl - c0) / a.hg + 1;  // pieces
  const int g = q / a.nseqh;
  const int h = warp;                                // the row of the partial slots
  const int t = (q % a.nseqh) * a.mt + h / PART_HEADS;  // its tile
  if (t >= a.ntile) return;                          // a sequence with one tile of two
  const Tile tl = tile_of(t, a.G, a.nsub, a.Q, a.qt);
  const int r = h % PART_HEADS;  // the MMA row of the tile
  if (r >= tl.nq * a.gt || r % a.gt >= tl.nh) return;
  constexpr int PER = D / 32;  // 2, 4 or 8 consecutive dims per lane
  constexpr int CHUNK = 4;     // pieces whose partials are loaded together (one trip to L2)
  float M = -INFINITY, Z = 0.f, acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  for (int i0 = 0; i0 < k; i0 += CHUNK) {
    float lc[CHUNK], x[CHUNK][PER];
#pragma unroll
    for (int u = 0; u < CHUNK; ++u) {
      const int i = i0 + u;
      lc[u] = -INFINITY;
#pragma unroll
      for (int e = 0; e < PER; ++e) x[u][e] = 0.f;
      if (i < k) {
        const size_t pi = i == 0 ? (size_t)f : (size_t)(c0 + i * a.hg) * 2;
        lc[u] = a.part_lse[pi * PART_ROWS + h];
        const float *po = a.part_o + (pi * PART_ROWS + h) * D + lane * PER;
        if constexpr (PER == 2) {
          const float2 v = *reinterpret_cast<const float2 *>(po);
          x[u][0] = v.x;
          x[u][1] = v.y;
        } else {
#pragma unroll
          for (int e = 0; e < PER; e += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(po + e);
            x[u][e] = v.x;
            x[u][e + 1] = v.y;
            x[u][e + 2] = v.z;
            x[u][e + 3] = v.w;
          }
        }
      }
    }
    // the online merge in ascending piece order, as before
#pragma unroll
    for (int u = 0; u < CHUNK; ++u) {
      const float l = lc[u];
      if (l != -INFINITY) {
        const float mn = fmaxf(M, l);
        const float sc = M == -INFINITY ? 0.f : fast_exp2(M - mn);
        const float wc = fast_exp2(l - mn);
        M = mn;
        Z = Z * sc + wc;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = acc[e] * sc + wc * x[u][e];
      }
    }
  }
  const float inv = Z > 0.f ? 1.f / Z : 0.f;
  const size_t bh = ((size_t)b * a.Q + tl.i0 + r / a.gt) * a.Hq + g * a.G + tl.h0 + r % a.gt;
  uint32_t *dst = reinterpret_cast<uint32_t *>(a.out + bh * D + lane * PER);
#pragma unroll
  for (int e = 0; e < PER; e += 2) dst[e / 2] = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
  if (lane == 0 && a.lse) a.lse[bh] = (M == -INFINITY || Z == 0.f) ? -INFINITY : (M + __log2f(Z)) * LN2;
}

}  // namespace pa
