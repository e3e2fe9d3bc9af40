// pa_partition.cuh -- the static, cost-balanced work partition shared by the split-KV
// kernels (GQA in pa_gqa.cuh, MLA in pa_mla_tc.cuh).
//
// A sequence is one (row, head tile) of a row's query rows; its keys are cut into
// units of one TMA box.  The CTAs form NG groups of HG = min(HS, nparts) consecutive
// CTAs (HS: sequences per row); CTA r of a group serves the sequences r, r + HG, ... of
// every row.  A row's column cost is w_b = n_b + piece_cost units (0 when n_b == 0); the
// column axis (rows in order) is cut into NG equal ranges, one per group, so the HG CTAs
// of a group stream the same pages (each its own tile) at about the same time and every
// CTA streams the same cost.  A position inside the first piece_cost units of a row maps
// to no key: those units stand for the fixed cost of a piece (its query stage, the merge
// at its end).  With NG >= 2 each CTA serves exactly one sequence per row (HG == HS);
// with NG == 1 every piece is a whole sequence.
#pragma once

#include "pa_common.cuh"

namespace pa {

__device__ __forceinline__ int clamp_len(int L, int max_len) { return min(max(L, 0), max_len); }

// Keys of query position i of a row of length L holding Q new tokens: [lo, hi) with
// hi = L - Q + 1 + i (the position itself included) and lo = max(0, hi - window) under a window.
__device__ __forceinline__ int pos_hi(int L, int Q, int i) { return max(L - Q + 1 + i, 0); }
__device__ __forceinline__ int pos_lo(int L, int Q, int i, int window) {
  return window > 0 ? max(pos_hi(L, Q, i) - window, 0) : 0;
}

// Units of a row of length L that some of its Q query positions attend to:
// [*u_lo, u_lo + return value), the union of the positions' key ranges.
__device__ __forceinline__ int row_units(int L, int Q, int window, int log2_bh, int *u_lo) {
  const int lo = window > 0 ? max(L - Q + 1 - window, 0) : 0;
  *u_lo = lo >> log2_bh;
  return L > 0 ? ((L + (1 << log2_bh) - 1) >> log2_bh) - *u_lo : 0;
}

// Block-wide sum / exclusive scan of 64-bit values (all threads of the CTA take part).
__device__ __forceinline__ long long block_sum64(long long v, long long *warp_part) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  if (lane == 0) warp_part[warp] = v;
  __syncthreads();
  long long t = 0;
  for (int w = 0; w < nw; ++w) t += warp_part[w];
  __syncthreads();
  return t;
}

__device__ __forceinline__ long long block_scan64(long long v, long long *excl, long long *warp_part) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(FULL, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_part[warp] = x;
  __syncthreads();
  long long before = 0, t = 0;
  for (int w = 0; w < nw; ++w) {
    if (w < warp) before += warp_part[w];
    t += warp_part[w];
  }
  __syncthreads();
  *excl = before + x - v;
  return t;
}

struct PartitionArgs {
  const int32_t *context_lens;
  int batch, max_context_len, Q, window, log2_bh, piece_cost;
  int nparts, hg, hs;  // CTAs, CTAs per group, sequences per row
};

// Shared state the prologue leaves for the producer (in shared memory).
struct PartitionState {
  int32_t found_b;       // row holding the group's first column, -1: no work
  int32_t pad;
  long long found_off;   // column offset of that position inside the row
  long long x_begin, x_end;
  long long warp_part[10];
};

__device__ __forceinline__ int seq_cost(const PartitionArgs &p, int L, int *n_out) {
  int ul;
  const int n = row_units(L, p.Q, p.window, p.log2_bh, &ul);
  *n_out = n;
  return n > 0 ? n + p.piece_cost : 0;
}

// All threads of the CTA: this CTA's column range and where it starts.  Context lengths
// outside [0, max_context_len] are clamped and set PA_DEV_BAD_LEN in *status.
template <int THREADS>
__device__ void partition_prologue(const PartitionArgs &p, PartitionState *ps, uint32_t *status) {
  const int tid = threadIdx.x;
  if (tid == 0) ps->found_b = -1;
  __syncthreads();
  const int NG = p.nparts / p.hg;
  const int grp = (int)blockIdx.x / p.hg;
  const bool member = grp < NG;  // CTAs past the last full group get no work
  long long W = 0;               // total column cost
  if (p.batch <= THREADS) {
    // one pass: every row in one thread
    long long v = 0;
    if (tid < p.batch) {
      const int L0 = p.context_lens[tid];
      if (L0 < 0 || L0 > p.max_context_len) atomicOr(status, PA_DEV_BAD_LEN);
      int n;
      v = seq_cost(p, clamp_len(L0, p.max_context_len), &n);
    }
    long long ex;
    W = block_scan64(v, &ex, ps->warp_part);
    const long long xb = (long long)grp * W / NG, xe = ((long long)grp + 1) * W / NG;
    if (member && v > 0 && xb >= ex && xb < ex + v && xb < xe) {
      ps->found_b = tid;
      ps->found_off = xb - ex;
    }
  } else {
    long long local = 0;
    for (int b = tid; b < p.batch; b += THREADS) {
      const int L0 = p.context_lens[b];
      if (L0 < 0 || L0 > p.max_context_len) atomicOr(status, PA_DEV_BAD_LEN);
      int n;
      local += seq_cost(p, clamp_len(L0, p.max_context_len), &n);
    }
    W = block_sum64(local, ps->warp_part);
    const long long xb = (long long)grp * W / NG, xe = ((long long)grp + 1) * W / NG;
    if (member && xb < xe) {
      long long base = 0;
      for (int b0 = 0; b0 < p.batch; b0 += THREADS) {
        const int b = b0 + tid;
        long long v = 0;
        if (b < p.batch) {
          int n;
          v = seq_cost(p, clamp_len(p.context_lens[b], p.max_context_len), &n);
        }
        long long ex;
        const long long tot = block_scan64(v, &ex, ps->warp_part);
        if (v > 0 && xb >= base + ex && xb < base + ex + v) {
          ps->found_b = b;
          ps->found_off = xb - base - ex;
        }
        base += tot;
        __syncthreads();
        if (ps->found_b >= 0) break;
      }
    }
  }
  if (tid == 0) {
    ps->x_begin = member ? (long long)grp * W / NG : 0;
    ps->x_end = member ? ((long long)grp + 1) * W / NG : 0;
  }
  __syncthreads();
}

// One piece: units [ub, ue) of sequence (b, hs); lo / L: the row's key range for position 0
// and its length.
struct Piece {
  int b, hs, ub, ue, lo, L;
  bool starts, ends;
};

// The producer warp's walk over its CTA's pieces (all lanes call every method together).
struct PieceWalker {
  const PartitionArgs &p;
  int lane, hr, b_first, in_first;
  long long span, R;  // column cost of the range; cost still to walk for it_hs
  int rb, lwin;       // lane l holds the clamped length of row rb + l
  int it_hs, it_b, it_in;

  __device__ PieceWalker(const PartitionArgs &pa_, const PartitionState *ps, int lane_)
      : p(pa_), lane(lane_) {
    hr = (int)blockIdx.x % p.hg;
    b_first = max(ps->found_b, 0);
    in_first = ps->found_b >= 0 ? (int)ps->found_off : 0;
    span = ps->found_b >= 0 ? ps->x_end - ps->x_begin : 0;
    R = span;
    rb = b_first;
    lwin = rb + lane < p.batch ? clamp_len(p.context_lens[rb + lane], p.max_context_len) : 0;
    it_hs = hr;
    it_b = b_first;
    it_in = in_first;
  }

  __device__ int len_of(int row) {
    if (row < rb || row >= rb + 32) {
      rb = row;
      lwin = rb + lane < p.batch ? clamp_len(p.context_lens[rb + lane], p.max_context_len) : 0;
    }
    return __shfl_sync(FULL, lwin, row - rb);
  }

  // The next piece that holds at least one key; false once the range is walked for every
  // sequence of this CTA.
  __device__ bool take(Piece &pc) {
    while (true) {
      if (R == 0) {
        it_hs += p.hg;
        if (span == 0 || it_hs >= p.hs) return false;
        R = span;
        it_b = b_first;
        it_in = in_first;
      }
      const int L = len_of(it_b);
      int n;
      const int w = seq_cost(p, L, &n);
      const int take = (int)min((long long)(w - it_in), R);
      const int u0 = max(0, it_in - p.piece_cost), u1 = max(0, it_in + take - p.piece_cost);
      const int b = it_b;
      R -= take;
      it_in += take;
      if (it_in == w && R > 0) {
        it_in = 0;
        int nn;
        do {
          ++it_b;
        } while (it_b < p.batch - 1 && seq_cost(p, len_of(it_b), &nn) == 0);
      }
      if (u1 > u0) {
        int ul;
        row_units(L, p.Q, p.window, p.log2_bh, &ul);
        pc.b = b;
        pc.hs = it_hs;
        pc.L = L;
        pc.lo = pos_lo(L, p.Q, 0, p.window);
        pc.ub = ul + u0;
        pc.ue = ul + u1;
        pc.starts = u0 == 0;
        pc.ends = u1 == n;
        return true;
      }
    }
  }
};

// Rows without a visible key (b = blockIdx.x mod nparts): `row_elems` bf16 zeros of out and
// `row_lse` values -inf of lse (if not null).  All threads.
template <int THREADS>
__device__ void zero_empty_rows(const PartitionArgs &p, uint16_t *out, float *lse, int row_elems, int row_lse) {
  for (int b = blockIdx.x; b < p.batch; b += p.nparts) {
    int ul;
    if (row_units(clamp_len(p.context_lens[b], p.max_context_len), p.Q, p.window, p.log2_bh, &ul) != 0) continue;
    uint4 *o = reinterpret_cast<uint4 *>(out + (size_t)b * row_elems);
    for (int e = threadIdx.x; e < row_elems / 8; e += THREADS) o[e] = make_uint4(0, 0, 0, 0);
    if (lse)
      for (int h = threadIdx.x; h < row_lse; h += THREADS) lse[(size_t)b * row_lse + h] = -INFINITY;
  }
}

}  // namespace pa
