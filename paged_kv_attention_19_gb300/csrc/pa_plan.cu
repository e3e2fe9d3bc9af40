// pa_plan.cu -- the work-list planner of the MLA split-KV kernel.
//
// Turns the device-resident context lengths into page-aligned work items
// without a host round trip.  Automatic mode picks one chunk length so the
// machine sees about `target_items` items (never fewer than
// `min_chunk_pages` pages each); a fixed num_splits cuts every row into that
// many chunks.  Items are placed by prefix sums (no atomics, so the list is
// identical from run to run): first every full-length chunk, row by row, then
// the shorter tail chunks, so the dynamic queue of the split kernel ends with
// short work.  The planner also resets the queue cursor and writes the output
// of rows that have no key to attend (out = 0, lse = -inf).
#include "pa_plan.cuh"
#include "pa_launch.h"

namespace pa {

namespace {

// Exclusive block-wide scan of one value per thread (blockDim.x == 1024); returns the block total.
__device__ int block_exclusive_scan(int v, int *excl, int *s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FULL, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
  const int total = s_warp[31];
  __syncthreads();
  *excl = before;
  return total;
}

constexpr int kPlanSmemRows = 1024;  // batches up to this size keep the row table in shared memory

}  // namespace

// One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) plan_kernel(const PlanArgs a) {
  pdl_launch_dependents();  // the split kernel may start its prologue; it waits for our writes
  __shared__ unsigned long long s_total;
  __shared__ int s_maxpages, s_chunk, s_warp[32];
  __shared__ RowInfo s_rows[kPlanSmemRows];
  const bool in_smem = a.batch <= kPlanSmemRows;
  RowInfo *rows = in_smem ? s_rows : a.rows;  // working copy (global only for very large batches)
  const int tid = threadIdx.x;
  if (tid == 0) {
    a.hdr->status = 0;
    s_total = 0;
    s_maxpages = 0;
  }
  __syncthreads();
  const int P = a.page_size;
  // pass 1: visible range of every row
  unsigned long long local = 0;
  int localmax = 0;
  for (int b = tid; b < a.batch; b += blockDim.x) {
    int L = a.context_lens[b];
    if (L < 0 || L > a.max_context_len) {
      atomicOr(&a.hdr->status, PA_DEV_BAD_LEN);
      L = min(max(L, 0), a.max_context_len);
    }
    const int lo = (a.window > 0 && L > a.window) ? L - a.window : 0;
    RowInfo r;
    r.lo = lo;
    r.L = L;
    r.page_lo = lo >> a.log2_page;
    r.page_hi = (L + P - 1) >> a.log2_page;
    r.nsplit = 0;
    r.chunk = 1;
    r.full_off = r.tail_off = 0;
    rows[b] = r;
    const int pages = r.page_hi - r.page_lo;
    local += (unsigned long long)pages;
    localmax = max(localmax, pages);
  }
  // reduce within each warp first: one shared-memory atomic per warp, not per thread
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    local += __shfl_xor_sync(FULL, local, o);
    localmax = max(localmax, __shfl_xor_sync(FULL, localmax, o));
  }
  if ((tid & 31) == 0) {
    atomicAdd(&s_total, local);
    atomicMax(&s_maxpages, localmax);
  }
  __syncthreads();
  if (tid == 0) {
    long long chunk = 0;  // fixed num_splits: per row
    if (a.num_splits <= 0) {
      const long long work = (long long)s_total * a.heads_per_row;
      chunk = (work + a.target_items - 1) / max(a.target_items, 1);
      chunk = max(chunk, (long long)a.min_chunk_pages);
      chunk = max(chunk, (long long)((s_maxpages + a.max_splits - 1) / a.max_splits));
      chunk = (chunk + a.chunk_align - 1) / a.chunk_align * a.chunk_align;
      chunk = max(chunk, 1ll);
    }
    s_chunk = (int)chunk;
    a.hdr->chunk_pages = (uint32_t)chunk;
  }
  __syncthreads();
  // pass 2: split counts and the prefix offsets of full / tail chunks (1024 rows per round)
  int full_base = 0, tail_base = 0;
  for (int b0 = 0; b0 < a.batch; b0 += blockDim.x) {
    const int b = b0 + tid;
    int nfull = 0, ntail = 0;
    RowInfo r;
    if (b < a.batch) {
      r = rows[b];
      const int pages = r.page_hi - r.page_lo;
      if (pages == 0) {
        r.nsplit = 0;
        r.chunk = 1;
      } else if (a.num_splits > 0) {
        r.nsplit = a.num_splits;
        r.chunk = (pages + a.num_splits - 1) / a.num_splits;
      } else {
        r.chunk = s_chunk;
        r.nsplit = (pages + r.chunk - 1) / r.chunk;
      }
      if (pages > 0) {
        nfull = pages / r.chunk;
        ntail = (pages % r.chunk) ? 1 : 0;
      }
    }
    int fex, tex;
    const int ftot = block_exclusive_scan(nfull, &fex, s_warp);
    const int ttot = block_exclusive_scan(ntail, &tex, s_warp);
    if (b < a.batch) {
      r.full_off = full_base + fex;
      r.tail_off = tail_base + tex;
      rows[b] = r;
      if (in_smem) a.rows[b] = r;  // the table the split and combine kernels read
    }
    full_base += ftot;
    tail_base += ttot;
  }
  __syncthreads();
  // pass 3: emit items; warp w handles rows w, w + 32, ...; positions are prefix-determined
  const int hpr = a.heads_per_row;
  const int lane = tid & 31, warp = tid >> 5;
  const int n_full_items = full_base * hpr;
  for (int b = warp; b < a.batch; b += 32) {
    const RowInfo r = rows[b];
    const int pages = r.page_hi - r.page_lo;
    if (pages == 0) {
      if (a.out) {  // no key: out = 0, lse = -inf for every head of the row
        const int n = a.out_heads * a.out_dim;
        uint16_t *o = a.out + (size_t)b * n;
        for (int e = lane; e < n; e += 32) o[e] = 0;
        if (a.lse)
          for (int h = lane; h < a.out_heads; h += 32) a.lse[(size_t)b * a.out_heads + h] = -INFINITY;
      }
      continue;
    }
    const int nfull = pages / r.chunk;
    const int n = nfull * hpr;
    const int ne = nfull + ((pages % r.chunk) ? 1 : 0);
    const int splits = (r.nsplit << 16) | ne;
    for (int e = lane; e < n; e += 32) {
      const int c = e / hpr, sub = e % hpr;
      WorkItem it;
      it.b = b;
      it.sub = sub;
      it.split = c;
      it.page_begin = r.page_lo + c * r.chunk;
      it.page_end = it.page_begin + r.chunk;
      it.tok_lo = max(r.lo, it.page_begin * P);
      it.tok_hi = min(r.L, it.page_end * P);
      it.splits = splits;
      a.items[(size_t)r.full_off * hpr + e] = it;
    }
    if (pages % r.chunk) {
      for (int sub = lane; sub < hpr; sub += 32) {
        WorkItem it;
        it.b = b;
        it.sub = sub;
        it.split = nfull;
        it.page_begin = r.page_lo + nfull * r.chunk;
        it.page_end = r.page_hi;
        it.tok_lo = max(r.lo, it.page_begin * P);
        it.tok_hi = min(r.L, it.page_end * P);
        it.splits = splits;
        a.items[(size_t)n_full_items + (size_t)r.tail_off * hpr + sub] = it;
      }
    }
  }
  if (tid == 0) {
    a.hdr->n_items = (uint32_t)((full_base + tail_base) * hpr);
    a.hdr->item_counter = 0;
  }
}

cudaError_t launch_plan(const PlanArgs &a, cudaStream_t stream) {
  plan_kernel<<<1, 1024, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pa
