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
//   * static, balanced partition.  The visible keys of every (row, KV head,
//     16-head subgroup) sequence are cut into units of one TMA box (min(page,
//     stage) tokens).  All units, flattened row by row, are divided into
//     `nparts` equal contiguous ranges, one per CTA (one CTA per SM by
//     default), so every SM streams the same number of KV bytes.  Each CTA
//     finds its range from the context lengths in a short prologue: no
//     planner launch, no work queue, no atomics, identical from run to run.
//     A range is a list of pieces (maximal runs of one sequence); only its
//     first and last piece can be part of a sequence that another CTA also
//     touches, so a CTA leaves at most two partial results;
//   * the last warp is a TMA producer: it walks the CTA's pieces, keeps 32
//     block-table entries in a register window (the next window and the next
//     piece's first window already in flight), and issues 4-D tensor-map
//     copies of page fragments into a ring of shared-memory stages (K and V
//     of 64 tokens, 32 for head_dim 256) with the 128-byte swizzle, so the
//     tensor-core fragment loads are bank-conflict free.  The ring takes all
//     of shared memory (224 KB) to keep ~200 KB of copies in flight per SM;
//   * the consumer warps take 16 tokens of every stage per token group; two
//     warps share a group, both computing its scores and each accumulating
//     half of the P.V columns.  The group's (up to 16) query heads are the M
//     rows of mma.sync m16n8k16 bf16 tiles, so S = Q K^T and O += P V cost one
//     tensor-core instruction per 8 tokens x 16 dims.  The online softmax
//     (running max with a lazy rescale, fp32 denominator) runs on the CUDA
//     cores; P is rounded to bf16 only as the MMA operand.  Q is read from
//     global memory into registers at the start of a piece (the producer has
//     prefetched it to L2), so no shared memory is spent on it;
//   * at the end of a piece the token groups merge through the consumed stage
//     buffer; a piece that covers its whole sequence writes the final bf16
//     output and LSE, any other writes an fp32 partial (normalised output +
//     LSE) to one of the CTA's two slots;
//   * the combine kernel (a programmatic dependent launch, so its launch hides
//     under the split kernel's tail) merges every split sequence over the
//     CTAs that hold its pieces, in ascending order.
#pragma once

#include "pa_common.cuh"
#include "pa_partition.cuh"

namespace pa {

// What each split CTA leaves for the combine kernel.
struct GqaPartDesc {
  int32_t last_b;   // row of the CTA's last piece
  int32_t last_hs;  // KV head x tile (kv_head * ntile + tile) of the last piece
  uint32_t flags;   // bits 0-15: pieces of the CTA (saturating); DESC_* bits
  uint32_t status;  // PA_DEV_* bits seen by the CTA
};
static_assert(sizeof(GqaPartDesc) == 16, "descriptor is 16 bytes");
constexpr uint32_t DESC_PIECES = 0xffffu;
constexpr uint32_t DESC_LAST_STARTS = 1u << 16;  // the last piece begins its sequence
constexpr uint32_t DESC_LAST_ENDS = 1u << 17;    // the last piece ends its sequence
constexpr uint32_t DESC_FIRST_ENDS = 1u << 18;   // the first piece ends its sequence
constexpr int PART_HEADS = 16;                   // heads per partial slot (one subgroup)

struct GqaArgs {
  const uint16_t *q;            // [B, Hq, D] bf16
  const int32_t *block_table;   // [B, max_pages_per_seq]
  const int32_t *context_lens;  // [B]
  uint16_t *out;                // [B, Hq, D] bf16
  float *lse;                   // [B, Hq] or null
  float *part_o;                // [nparts, 2, 16, D] fp32
  float *part_lse;              // [nparts, 2, 16] fp32, log2 units
  GqaPartDesc *desc;            // [nparts]
  int batch, max_pages_per_seq, num_pages, max_context_len, window;
  int Hq, Hkv, G, nsub;
  int Q;                        // query positions per row (1: decode; > 1: verify, causal within them)
  int gt, qt, ntile;            // a tile of MMA rows: qt positions x gt heads; ntile tiles per KV head
  int log2_page, log2_bh;       // page size and tokens per unit (TMA box), as powers of two
  int piece_cost;               // partition cost of starting a piece, in units
  int nparts;                   // CTAs (shares); groups of hg consecutive CTAs
  int hg;                       // CTAs per group: min(Hkv * ntile, nparts)
  float qscale;                 // scale * log2(e) (FP8: times the keys' scale)
  float vscale;                 // FP8: the values' scale; 1 for bf16 pools
};

// F8_: the pools hold FP8 E4M3 codes (one byte per value) instead of bf16.
template <int D_, bool F8_ = false>
struct GqaCfg {
  static constexpr int D = D_;
  static constexpr bool F8 = F8_;
  static constexpr int M = PART_HEADS;             // MMA rows = query heads per subgroup
  // tokens per stage: 32 KB of K and V (16 KB for bf16 head_dim 256)
  static constexpr int ST = F8 ? (D <= 128 ? 128 : 64) : (D <= 128 ? 64 : 32);
  static constexpr int TW = F8 ? 32 : 16;          // tokens per token group per stage (one MMA k-extent)
  static constexpr int TG = ST / TW;               // token groups per stage
  // warps sharing a token group, each computing its scores and D / DSPLIT of the P.V columns
  static constexpr int DSPLIT = (F8 && D <= 128) ? 1 : 2;
  static constexpr int NCW = TG * DSPLIT;          // consumer warps
  static constexpr int THREADS = (NCW + 1) * 32;   // + producer warp
  static constexpr int NTT = TW / 8;               // score n-tiles (8 tokens) per warp
  static constexpr int NT_PV = D / 8 / DSPLIT;     // P.V n-tiles (8 dims) per warp
  static constexpr int NQ = F8 ? D / 128 : D / 64;  // 128-byte swizzle planes along D (K, V)
  static constexpr int QNQ = D / 64;               // the same for the bf16 query rows
  static constexpr int PLANE = ST * 128;           // bytes of one plane (ST rows x 128 bytes)
  static constexpr int KV_BYTES = NQ * PLANE;      // K (or V) of one stage
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int NS = (229376 / STAGE_BYTES) < 16 ? (229376 / STAGE_BYTES) : 16;  // 224 KB ring
  static constexpr int NACC = F8 ? 1 : 2;          // independent QK accumulators per n-tile
  static_assert(M * D * 4 * TG <= STAGE_BYTES, "the end-of-piece merge fits the consumed stage");
  static_assert(QNQ * M * 128 <= STAGE_BYTES, "the query rows fit one stage");
  static_assert(!F8 || D % 128 == 0, "FP8 rows are whole 128-byte planes");
};

struct alignas(16) StageMeta {
  int32_t end, first, last, masked;  // first: a stage holding the piece's query rows only
  int32_t b, hq0, ghead, slot;  // slot: -1 = whole sequence (final output), else partial slot 0 / 1
  int32_t tok0, tok_lo, tok_hi, L;  // L: the row's length (query position i attends below L - Q + 1 + i)
  uint32_t badmask;             // bit k: box k of the stage was not loaded
  int32_t i0, nq, pad0;         // the tile's positions [i0, i0 + nq); ghead: its heads
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
  static constexpr int OFF_ML = OFF_STAGE + C::NS * C::STAGE_BYTES;
  static constexpr int OFF_META = OFF_ML + C::TG * C::M * 2 * 4;
  static constexpr int OFF_BAR = OFF_META + C::NS * (int)sizeof(StageMeta);
  static constexpr int OFF_MISC = OFF_BAR + 2 * C::NS * 8;
  static constexpr int USED = OFF_MISC + (int)sizeof(GqaMisc);
  static constexpr int BYTES = USED + 1024;  // slack to align the base to 1024 bytes
  static_assert(BYTES <= 232448, "fits the 227 KB opt-in shared memory of one CTA");
};

// Byte offset of 16-byte chunk `chunk` (along D) of token row `tok` in a
// stage's K or V block: planes of 64 dims, 128-byte rows, chunk ^ (row & 7)
// (the TMA 128-byte swizzle; every box starts on a 1024-byte boundary).
template <class C>
__device__ __forceinline__ uint32_t kv_off(int tok, int chunk) {
  return (uint32_t)((chunk >> 3) * C::PLANE + tok * 128 + (((chunk & 7) ^ (tok & 7)) << 4));
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

// MQ: several query positions per row (verify); false compiles the decode-only row logic.
// F8: FP8 E4M3 pools; keys and values widen to f16 (exact) for f16 MMAs, the query too.
template <int D, bool MQ, bool F8 = false>
__global__ void __launch_bounds__(GqaCfg<D, F8>::THREADS, 1)
    gqa_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_q, const GqaArgs a) {
  using C = GqaCfg<D, F8>;
  using S = GqaSmem<C>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the 128-byte swizzle pattern repeats every 1024 bytes: start the stages on such a boundary
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
  uint64_t *empty = full + C::NS;
  StageMeta *meta = reinterpret_cast<StageMeta *>(smem + S::OFF_META);
  GqaMisc *misc = reinterpret_cast<GqaMisc *>(smem + S::OFF_MISC);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int HS = a.Hkv * a.ntile;  // sequences per row: KV heads x tiles
  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NCW);
    }
    fence_mbar_init();
    misc->status = 0;
  }
  if (warp == C::NCW && lane == 0) {
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_q);
  }
  __syncthreads();
  pdl_wait();               // inputs written by the stream's previous kernel are visible from here on
  pdl_launch_dependents();  // the combine kernel may be scheduled; it waits for this grid to finish
  uint32_t *status = &misc->status;

  // ---------------------------------------------- prologue: this CTA's range
  PartitionArgs pargs;
  pargs.context_lens = a.context_lens;
  pargs.batch = a.batch;
  pargs.max_context_len = a.max_context_len;
  pargs.Q = a.Q;
  pargs.window = a.window;
  pargs.log2_bh = a.log2_bh;
  pargs.piece_cost = a.piece_cost;
  pargs.nparts = a.nparts;
  pargs.hg = a.hg;
  pargs.hs = HS;
  partition_prologue<C::THREADS>(pargs, &misc->part, status);
  zero_empty_rows<C::THREADS>(pargs, a.out, a.lse, a.Q * a.Hq * D, a.Q * a.Hq);
  __syncthreads();

  if (warp == C::NCW) {
    // ------------------------------------------------------------ producer
    const int P = 1 << a.log2_page;
    const int nbox = C::ST >> a.log2_bh;  // boxes (units) per stage
    uint32_t j = 0;
    bool ok = true;
    int npieces = 0;
    Piece last_piece = {};
    bool first_ends = false;
    PieceWalker walker(pargs, &misc->part, lane);
    auto take_piece = [&](Piece &pc) { return walker.take(pc); };
    auto tile = [&](const Piece &p) { return tile_of(p.hs % a.ntile, a.G, a.nsub, a.Q, a.qt); };
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
    while (has_cur && ok) {
      // ---- emit the stages of `cur`
      const int g = cur.hs / a.ntile;
      const Tile tl = tile(cur);
      const int hq0 = g * a.G + tl.h0;
      // the tile's tightest key bounds: its first position ends first, its last starts last
      const int hi_min = pos_hi(cur.L, a.Q, tl.i0), lo_max = pos_lo(cur.L, a.Q, tl.i0 + tl.nq - 1, a.window);
      const int slot = (cur.starts && cur.ends) ? -1 : (npieces == 0 ? 0 : 1);
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
        if (u > 0) ok = mbar_wait(&empty[s], (u - 1) & 1, status);
        if (!ok) break;
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
          m.L = cur.L;
          mbar_arrive_expect_tx(&full[s], (uint32_t)(C::QNQ * a.gt * a.qt * 128));
          uint8_t *qdst = smem + S::OFF_STAGE + s * C::STAGE_BYTES;
#pragma unroll
          for (int dq = 0; dq < C::QNQ; ++dq)
            tma_load_3d(qdst + dq * (C::M * 128), &tm_q, dq * 64, hq0, cur.b * a.Q + tl.i0, &full[s]);
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
          m.L = cur.L;
          m.slot = slot;
          m.tok0 = tok0;
          m.tok_lo = tok_lo;
          m.tok_hi = tok_hi;
          m.badmask = bad;
          m.masked = (tok0 < max(tok_lo, lo_max)) || (tok0 + C::ST > min(tok_hi, hi_min)) || bad != 0;
          mbar_arrive_expect_tx(&full[s], (uint32_t)nvalid * (uint32_t)((D * (F8 ? 1 : 2) * 2) << a.log2_bh));
        }
        __syncwarp();
        if (load) {
          const int pslot = btok & (P - 1);
          uint8_t *dst = kdst + (lane << a.log2_bh) * 128;
#pragma unroll
          for (int dq = 0; dq < C::NQ; ++dq) {
            const int x = dq * (F8 ? 128 : 64);  // 128 bytes of the row per plane
            tma_load_4d(dst + dq * C::PLANE, &tm_k, x, g, pslot, phys, &full[s]);
            tma_load_4d(dst + dq * C::PLANE + C::KV_BYTES, &tm_v, x, g, pslot, phys, &full[s]);
          }
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
      has_next = take_piece(nxt);
      if (has_next) nwin0 = piece_window(nxt);
    }
    if (ok) {
      // end marker
      const int s = j % C::NS;
      const uint32_t u = j / C::NS;
      if (u > 0) ok = mbar_wait(&empty[s], (u - 1) & 1, status);
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
  } else {
    // ------------------------------------------------------------ consumers
    const int ct = tid;                               // consumer thread index
    const int g8 = lane >> 2, tq = lane & 3;          // MMA fragment row / column pair
    const int lm_mat = lane >> 3, lm_row = lane & 7;  // ldmatrix: matrix / row this lane addresses
    const int tgrp = warp % C::TG;                    // token group of this warp
    const int dh = warp / C::TG;                      // which part of the P.V columns it owns
    const int wbase = tgrp * C::TW;                   // first stage token of this warp
    const int nd0 = dh * C::NT_PV;                    // first P.V n-tile of this warp
    float *sm_ml = reinterpret_cast<float *>(smem + S::OFF_ML);
    // lazy rescale: the running max moves only when a score passes it by TAU (log2 units), so
    // a weight never exceeds 2^TAU (FP8: 2, so that PSCALE x weight stays within E4M3's 448)
    constexpr float TAU = F8 ? 1.f : 8.f;
    constexpr float PSCALE = 128.f;  // FP8: weights enter the P.V MMA as PSCALE x p
    const int bh_tokens = 1 << a.log2_bh;

    // Q A-fragments (rows = heads).  bf16: one per k16 step.  FP8: one per k32 step for the
    // high terms ([0, D/32)) and for the low terms ([D/32, D/16)).
    uint32_t qa[D / 16][4];
    float acc[C::NT_PV][4];  // O C-fragments of this warp's columns: [n-tile][row g8 x2, row g8+8 x2]
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float qs0 = a.qscale, qs1 = a.qscale;  // score multipliers of rows g8 / g8 + 8
    // this thread's two fragment rows (g8, g8 + 8): real row?, key bounds [lo, hi) of its position
    bool rv0 = false, rv1 = false;
    int lo0 = 0, hi0 = 0, lo1 = 0, hi1 = 0;
    for (uint32_t j = 0;; ++j) {
      const int s = j % C::NS;
      if (!mbar_wait(&full[s], (j / C::NS) & 1, status)) break;
      const StageMeta &mt = meta[s];
      if (mt.end) break;
      const uint32_t kbase = smem_u32(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
      const uint32_t vbase = kbase + C::KV_BYTES;
      if (mt.first) {
        // a new piece: its query rows into the A-fragments (from the 128-byte swizzled planes of
        // 16 rows x 64 dims), fresh softmax state, and the stage goes back
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
        const uint32_t qbase = kbase;
        if constexpr (F8) {
          // Each row times 2^s (s: its largest |q| lands in [128, 256)) is split into two E4M3
          // terms, q 2^s = hi + lo, exact for every element above 2^-10 of the row's scale; the
          // scores come out times 2^s, taken back in the row's multiplier.  Lane (g8, tq) holds
          // dims 16 ks + 4 tq .. + 3 of its rows for every 16-dim step ks (an 8-byte read).
          auto qaddr = [&](int ks, int row) {
            const int chunk = 2 * ks + (tq >> 1);
            return qbase + (uint32_t)((chunk >> 3) * (C::M * 128) + (tq & 1) * 8 + row * 128 +
                                      (((chunk & 7) ^ (row & 7)) << 4));
          };
          float am0 = 0.f, am1 = 0.f;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint2 r0 = lds_u2(qaddr(ks, g8)), r1 = lds_u2(qaddr(ks, g8 + 8));
            am0 = fmaxf(am0, fmaxf(bf16x2_absmax(r0.x), bf16x2_absmax(r0.y)));
            am1 = fmaxf(am1, fmaxf(bf16x2_absmax(r1.x), bf16x2_absmax(r1.y)));
          }
          am0 = fmaxf(am0, __shfl_xor_sync(FULL, am0, 1));
          am0 = fmaxf(am0, __shfl_xor_sync(FULL, am0, 2));
          am1 = fmaxf(am1, __shfl_xor_sync(FULL, am1, 1));
          am1 = fmaxf(am1, __shfl_xor_sync(FULL, am1, 2));
          auto row_shift = [](float am) {  // 7 - floor(log2 am) in [-126, 126]; 0 for 0, inf, NaN
            const int e = (int)((__float_as_uint(am) >> 23) & 0xffu);
            if (e == 0xff || am == 0.f) return 0;
            return min(126, max(-126, 134 - e));
          };
          const int s0 = row_shift(am0), s1 = row_shift(am1);
          const float f0 = pow2f(s0), f1 = pow2f(s1);
          qs0 = a.qscale * pow2f(-s0);
          qs1 = a.qscale * pow2f(-s1);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint2 r0 = lds_u2(qaddr(ks, g8)), r1 = lds_u2(qaddr(ks, g8 + 8));
            uint32_t h[4], l[4];  // [row g8: dims 4tq,+1 | +2,+3][row g8 + 8: the same]
            split_e4m3x2(f32x2_to_f16x2_raw(__uint_as_float(r0.x << 16) * f0, __uint_as_float(r0.x & 0xffff0000u) * f0),
                         h[0], l[0]);
            split_e4m3x2(f32x2_to_f16x2_raw(__uint_as_float(r0.y << 16) * f0, __uint_as_float(r0.y & 0xffff0000u) * f0),
                         h[1], l[1]);
            split_e4m3x2(f32x2_to_f16x2_raw(__uint_as_float(r1.x << 16) * f1, __uint_as_float(r1.x & 0xffff0000u) * f1),
                         h[2], l[2]);
            split_e4m3x2(f32x2_to_f16x2_raw(__uint_as_float(r1.y << 16) * f1, __uint_as_float(r1.y & 0xffff0000u) * f1),
                         h[3], l[3]);
            const int kj = ks >> 1, hk = (ks & 1) * 2;  // k32 step; a0/a1 (first half) or a2/a3
            qa[kj][hk] = h[0] | (h[1] << 16);
            qa[kj][hk + 1] = h[2] | (h[3] << 16);
            qa[D / 32 + kj][hk] = l[0] | (l[1] << 16);
            qa[D / 32 + kj][hk + 1] = l[2] | (l[3] << 16);
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const int row = (lm_mat & 1) * 8 + lm_row, chunk = 2 * ks + (lm_mat >> 1);
            ldmatrix_x4(qa[ks], qbase + (chunk >> 3) * (C::M * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
          }
        }
#pragma unroll
        for (int n = 0; n < C::NT_PV; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        continue;
      }

      // ---- S = Q K^T for the group's TW tokens (n-tiles of 8); the k-steps are spread over
      // NACC independent accumulators so no long chain of dependent MMAs forms
      float sv[C::NTT][4];
      {
        float sp[C::NACC][C::NTT][4];
#pragma unroll
        for (int q = 0; q < C::NACC; ++q)
#pragma unroll
          for (int nt = 0; nt < C::NTT; ++nt) sp[q][nt][0] = sp[q][nt][1] = sp[q][nt][2] = sp[q][nt][3] = 0.f;
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
          for (int ks2 = 0; ks2 < D / (F8 ? 64 : 32); ++ks2) {
            // four 16-byte chunks of the group's tokens 8 nt .. 8 nt + 7
            uint32_t b[4];
            ldmatrix_x4(b, kbase + kv_off<C>(wbase + nt * 8 + lm_row, 4 * ks2 + lm_mat));
            if constexpr (F8) {  // chunks 4 ks2, +1: k32 step 2 ks2; chunks +2, +3: step 2 ks2 + 1
              mma_e4m3_16832(sp[0][nt], qa[2 * ks2], b[0], b[1]);
              mma_e4m3_16832(sp[0][nt], qa[D / 32 + 2 * ks2], b[0], b[1]);
              mma_e4m3_16832(sp[0][nt], qa[2 * ks2 + 1], b[2], b[3]);
              mma_e4m3_16832(sp[0][nt], qa[D / 32 + 2 * ks2 + 1], b[2], b[3]);
            } else {
              mma_bf16_16816(sp[(2 * ks2) % C::NACC][nt], qa[2 * ks2], b[0], b[1]);
              mma_bf16_16816(sp[(2 * ks2 + 1) % C::NACC][nt], qa[2 * ks2 + 1], b[2], b[3]);
            }
          }
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt)
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
      for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float v = sv[nt][e] * ((e < 2) ? qs0 : qs1);
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
      float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < C::NTT; ++nt) {
        x0 = fmaxf(x0, fmaxf(sv[nt][0], sv[nt][1]));
        x1 = fmaxf(x1, fmaxf(sv[nt][2], sv[nt][3]));
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
      // P as the A operand of the P.V MMA.  bf16: one k16 step.  FP8: one k32 step, high terms
      // pa[0..3] and low terms pa[4..7] of PSCALE x p, k slot 4 tq + i of a0 / a1 holding token
      // {2tq, 2tq + 1, 8 + 2tq, 9 + 2tq}[i] (a2 / a3: the same + 16): the token order in which
      // the V operand below is loaded, and the order the score fragments already have.
      uint32_t pa[F8 ? 8 : 4];
      {
        float p[C::NTT][4];
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float mr = (e < 2) ? m0 : m1;
            p[nt][e] = (sv[nt][e] == -INFINITY) ? 0.f : fast_exp2(sv[nt][e] - mr);
          }
        if constexpr (F8) {
          uint32_t h[C::NTT][2], l[C::NTT][2];  // per n-tile: row g8 pair, row g8 + 8 pair
#pragma unroll
          for (int nt = 0; nt < C::NTT; ++nt) {
            split_e4m3x2(f32x2_to_f16x2_raw(p[nt][0] * PSCALE, p[nt][1] * PSCALE), h[nt][0], l[nt][0]);
            split_e4m3x2(f32x2_to_f16x2_raw(p[nt][2] * PSCALE, p[nt][3] * PSCALE), h[nt][1], l[nt][1]);
          }
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            pa[r] = h[0][r] | (h[1][r] << 16);
            pa[2 + r] = h[2][r] | (h[3][r] << 16);
            pa[4 + r] = l[0][r] | (l[1][r] << 16);
            pa[6 + r] = l[2][r] | (l[3][r] << 16);
          }
        } else {
          pa[0] = pack_bf16x2(p[0][0], p[0][1]);
          pa[1] = pack_bf16x2(p[0][2], p[0][3]);
          pa[2] = pack_bf16x2(p[1][0], p[1][1]);
          pa[3] = pack_bf16x2(p[1][2], p[1][3]);
        }
        // the denominator (and so the LSE) sums the fp32 weights; only the MMA operand is rounded
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt) {
          l0 += p[nt][0] + p[nt][1];
          l1 += p[nt][2] + p[nt][3];
        }
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
      // ---- O += P V (k = the group's tokens), this warp's columns
      if constexpr (F8) {
        // per 16-dim chunk: ldmatrix.trans of the group's 32 token rows hands lane (g8, tq) the
        // bytes of tokens 2tq, 2tq + 1 (r[0]), 8 + 2tq, 9 + 2tq (r[1]), and the same + 16 (r[2],
        // r[3]), at dims 2 g8 and 2 g8 + 1 of the chunk; the byte permutes gather the even dim
        // (n-tile 2 cc) and the odd one (n-tile 2 cc + 1) in the k order of P
        constexpr int CH = D / C::DSPLIT / 16;
        const uint32_t ph[4] = {pa[0], pa[1], pa[2], pa[3]}, pl[4] = {pa[4], pa[5], pa[6], pa[7]};
#pragma unroll
        for (int cc = 0; cc < CH; ++cc) {
          uint32_t r[4];
          ldmatrix_x4_trans(r, vbase + kv_off<C>(wbase + lane, dh * CH + cc));
          const uint32_t b0e = prmt(r[0], r[1], 0x6420u), b0o = prmt(r[0], r[1], 0x7531u);
          const uint32_t b1e = prmt(r[2], r[3], 0x6420u), b1o = prmt(r[2], r[3], 0x7531u);
          mma_e4m3_16832(acc[2 * cc], ph, b0e, b1e);
          mma_e4m3_16832(acc[2 * cc + 1], ph, b0o, b1o);
          mma_e4m3_16832(acc[2 * cc], pl, b0e, b1e);
          mma_e4m3_16832(acc[2 * cc + 1], pl, b0o, b1o);
        }
      } else {
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
        // ---- end of a piece: merge the token groups through this stage's buffer
        l0 += __shfl_xor_sync(FULL, l0, 1);
        l0 += __shfl_xor_sync(FULL, l0, 2);
        l1 += __shfl_xor_sync(FULL, l1, 1);
        l1 += __shfl_xor_sync(FULL, l1, 2);
        named_bar(1, C::NCW * 32);  // all warps are done reading this stage
        // merge area: 16 rows x D fp32 per token group; the column of (head h, dim d) is
        // d ^ (4 (h & 7)), so the rows of one fragment hit distinct banks
        float *mg = reinterpret_cast<float *>(smem + S::OFF_STAGE + s * C::STAGE_BYTES);
        if constexpr (F8) {
          // n-tiles 2 cc / 2 cc + 1 hold dims 16 c + 4 tq + {0, 2} / {1, 3}, c = the chunk
          constexpr int CH = D / C::DSPLIT / 16;
#pragma unroll
          for (int cc = 0; cc < CH; ++cc) {
            const int d = ((dh * CH + cc) * 16 + 4 * tq) ^ (4 * g8);
            *reinterpret_cast<float4 *>(mg + (tgrp * C::M + g8) * D + d) =
                make_float4(acc[2 * cc][0], acc[2 * cc + 1][0], acc[2 * cc][1], acc[2 * cc + 1][1]);
            *reinterpret_cast<float4 *>(mg + (tgrp * C::M + g8 + 8) * D + d) =
                make_float4(acc[2 * cc][2], acc[2 * cc + 1][2], acc[2 * cc][3], acc[2 * cc + 1][3]);
          }
        } else {
#pragma unroll
          for (int n = 0; n < C::NT_PV; ++n) {
            const int d = ((nd0 + n) * 8 + 2 * tq) ^ (4 * g8);
            *reinterpret_cast<float2 *>(mg + (tgrp * C::M + g8) * D + d) = make_float2(acc[n][0], acc[n][1]);
            *reinterpret_cast<float2 *>(mg + (tgrp * C::M + g8 + 8) * D + d) = make_float2(acc[n][2], acc[n][3]);
          }
        }
        if (tq == 0 && dh == 0) {  // all column parts of a token group hold the same (m, l)
          sm_ml[(tgrp * C::M + g8) * 2] = m0;
          sm_ml[(tgrp * C::M + g8) * 2 + 1] = l0;
          sm_ml[(tgrp * C::M + g8 + 8) * 2] = m1;
          sm_ml[(tgrp * C::M + g8 + 8) * 2 + 1] = l1;
        }
        named_bar(1, C::NCW * 32);
        // each thread: 4 consecutive dims of one row; token-group weights
        // exp2(m_w - M) / sum_w l_w exp2(m_w - M), computed by every thread of the row
        const int slot = mt.slot;
        const size_t pi = (size_t)blockIdx.x * 2 + (slot > 0 ? 1 : 0);  // partial slot (when slot >= 0)
        const int nrows = MQ ? mt.nq * a.gt : mt.ghead;
        for (int e = ct; e < nrows * (D / 4); e += C::NCW * 32) {
          const int h = e / (D / 4), d4 = (e % (D / 4)) * 4;  // h: the MMA row
          if (MQ && h % a.gt >= mt.ghead) continue;          // not a head of this tile
          float mw[C::TG], M = -INFINITY;
#pragma unroll
          for (int w = 0; w < C::TG; ++w) {
            mw[w] = sm_ml[(w * C::M + h) * 2];
            M = fmaxf(M, mw[w]);
          }
          float L = 0.f;
          float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int w = 0; w < C::TG; ++w) {
            const float wt = (mw[w] == -INFINITY) ? 0.f : fast_exp2(mw[w] - M);
            L += sm_ml[(w * C::M + h) * 2 + 1] * wt;
            const float4 x = *reinterpret_cast<const float4 *>(mg + (w * C::M + h) * D + (d4 ^ (4 * (h & 7))));
            o.x += wt * x.x;
            o.y += wt * x.y;
            o.z += wt * x.z;
            o.w += wt * x.w;
          }
          // FP8: the values' scale over the weights' PSCALE, else 1
          const float inv = L > 0.f ? (F8 ? a.vscale / (PSCALE * L) : 1.f / L) : 0.f;
          const size_t bh = MQ ? ((size_t)mt.b * a.Q + mt.i0 + h / a.gt) * a.Hq + mt.hq0 + h % a.gt
                               : (size_t)mt.b * a.Hq + mt.hq0 + h;
          if (slot < 0) {
            uint2 v;
            v.x = pack_bf16x2(o.x * inv, o.y * inv);
            v.y = pack_bf16x2(o.z * inv, o.w * inv);
            *reinterpret_cast<uint2 *>(a.out + bh * D + d4) = v;
          } else {
            *reinterpret_cast<float4 *>(a.part_o + (pi * C::M + h) * D + d4) =
                make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
          }
          if (d4 == 0) {
            const float lse2 = (M == -INFINITY || L == 0.f) ? -INFINITY : M + __log2f(L);
            if (slot < 0) {
              if (a.lse) a.lse[bh] = lse2 * LN2;
            } else {
              a.part_lse[pi * C::M + h] = lse2;
            }
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

  __syncthreads();
  if (tid == 0) {
    GqaPartDesc d = misc->desc;
    d.status = misc->status;
    a.desc[blockIdx.x] = d;
  }
  if ((misc->desc.flags & DESC_PIECES) == 0) {
    // no work: leave slot 0 empty (lse -inf, output 0), so a merge that spans this CTA adds nothing
    for (int e = tid; e < C::M * D; e += C::THREADS) a.part_o[(size_t)blockIdx.x * 2 * C::M * D + e] = 0.f;
    for (int h = tid; h < C::M; h += C::THREADS) a.part_lse[(size_t)blockIdx.x * 2 * C::M + h] = -INFINITY;
  }
}

struct CombineArgs {
  uint16_t *out;
  float *lse;
  const float *part_o;
  const float *part_lse;
  const GqaPartDesc *desc;
  uint32_t *status;  // the workspace status word: OR of every CTA's bits
  int Hq, G, nsub, nparts, hg;
  int Q, gt, qt, ntile;
};

// One block per split CTA c.  Block c merges the sequence that CTA c's last
// piece begins, if that piece does not also end it: the sequence's pieces are
// CTA c's slot (1 if the CTA has several pieces, else 0) and slot 0 of CTAs
// c + hg, c + 2 hg, ... (the same head in the following groups) up to the
// first one whose first piece ends the sequence.
// Warp w handles heads w, w + 4, ...: weights exp2(lse_k - M), then
// o = sum_k w_k o_k / sum_k w_k in ascending k, each lane owning D/32 dims.
template <int D>
__global__ void __launch_bounds__(128) gqa_combine_kernel(const CombineArgs a) {
  pdl_wait();               // the split kernel's partials and descriptors are visible from here on
  pdl_launch_dependents();  // a following kernel (MLA: the W_UV projection) may stage its inputs
  const int c = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (c == 0 && warp == 0) {
    uint32_t s = 0;
    for (int i = lane; i < a.nparts; i += 32) s |= a.desc[i].status;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) s |= __shfl_xor_sync(FULL, s, o);
    if (lane == 0) *a.status = s;
  }
  const GqaPartDesc d0 = a.desc[c];
  const uint32_t np = d0.flags & DESC_PIECES;
  if (np == 0 || !(d0.flags & DESC_LAST_STARTS) || (d0.flags & DESC_LAST_ENDS)) return;
  // the later pieces of the sequence are in CTAs c + hg, c + 2 hg, ... (same head, next groups)
  int k = -1;  // pieces: CTA c + i hg holds piece i, i < k
  for (int base = 1; c + base * a.hg < a.nparts && k < 0; base += 32) {
    const int i = c + (base + lane) * a.hg;
    bool hit = false;
    if (i < a.nparts) {
      const uint32_t f = a.desc[i].flags;
      hit = (f & DESC_PIECES) != 0 && (f & DESC_FIRST_ENDS) != 0;
    }
    const uint32_t m = __ballot_sync(FULL, hit);
    if (m) k = base + __ffs(m);
  }
  if (k < 0) return;  // not reachable for a consistent partition
  const int first_slot = np >= 2 ? 1 : 0;
  const int g = d0.last_hs / a.ntile;
  const Tile tl = tile_of(d0.last_hs % a.ntile, a.G, a.nsub, a.Q, a.qt);
  const int hq0 = g * a.G + tl.h0;
  constexpr int PER = D / 32;  // 2, 4 or 8 consecutive dims per lane
  for (int h = warp; h < tl.nq * a.gt; h += 4) {  // h: the MMA row
    if (h % a.gt >= tl.nh) continue;
    float M = -INFINITY;
    for (int i = lane; i < k; i += 32) {
      const size_t pi = i == 0 ? (size_t)c * 2 + first_slot : (size_t)(c + i * a.hg) * 2;
      M = fmaxf(M, a.part_lse[pi * PART_HEADS + h]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, o));
    float Z = 0.f;
    for (int i = lane; i < k; i += 32) {
      const size_t pi = i == 0 ? (size_t)c * 2 + first_slot : (size_t)(c + i * a.hg) * 2;
      const float l = a.part_lse[pi * PART_HEADS + h];
      Z += (l == -INFINITY || M == -INFINITY) ? 0.f : fast_exp2(l - M);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) Z += __shfl_xor_sync(FULL, Z, o);
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
#pragma unroll 4
    for (int i = 0; i < k; ++i) {
      const size_t pi = i == 0 ? (size_t)c * 2 + first_slot : (size_t)(c + i * a.hg) * 2;
      const float l = a.part_lse[pi * PART_HEADS + h];
      const float wc = (l == -INFINITY || M == -INFINITY) ? 0.f : fast_exp2(l - M);
      const float *po = a.part_o + (pi * PART_HEADS + h) * D + lane * PER;
      if constexpr (PER == 2) {
        const float2 x = *reinterpret_cast<const float2 *>(po);
        acc[0] += wc * x.x;
        acc[1] += wc * x.y;
      } else {
#pragma unroll
        for (int e = 0; e < PER; e += 4) {
          const float4 x = *reinterpret_cast<const float4 *>(po + e);
          acc[e] += wc * x.x;
          acc[e + 1] += wc * x.y;
          acc[e + 2] += wc * x.z;
          acc[e + 3] += wc * x.w;
        }
      }
    }
    const float inv = Z > 0.f ? 1.f / Z : 0.f;
    const size_t bh = ((size_t)d0.last_b * a.Q + tl.i0 + h / a.gt) * a.Hq + hq0 + h % a.gt;
    uint32_t *dst = reinterpret_cast<uint32_t *>(a.out + bh * D + lane * PER);
#pragma unroll
    for (int e = 0; e < PER; e += 2) dst[e / 2] = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
    if (lane == 0 && a.lse) a.lse[bh] = (M == -INFINITY || Z == 0.f) ? -INFINITY : (M + __log2f(Z)) * LN2;
  }
}

}  // namespace pa
