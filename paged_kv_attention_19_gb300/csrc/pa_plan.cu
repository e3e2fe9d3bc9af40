// pa_plan.cu -- the work-list planner shared by the GQA and MLA split-KV kernels.
//
// Turns the device-resident context lengths into page-aligned work items
// without a host round trip: automatic mode picks one chunk length so that
// the machine sees about `target_items` items (never fewer than
// `min_chunk_pages` pages each), a fixed num_splits cuts every row into that
// many chunks.  Items are written longest-first (all full chunks, then the
// shorter tails) so the dynamic queue of the split kernel ends with short work.
#include "pa_gqa.cuh"
#include "pa_launch.h"

namespace pa {

// One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) plan_kernel(const PlanArgs a) {
  __shared__ unsigned long long s_total;
  __shared__ int s_maxpages, s_chunk;
  __shared__ unsigned s_nfull, s_ntail, s_cur_full, s_cur_tail;
  const int tid = threadIdx.x;
  if (tid == 0) {
    a.hdr->status = 0;
    s_total = 0;
    s_maxpages = 0;
    s_nfull = s_ntail = 0;
    s_cur_full = s_cur_tail = 0;
  }
  __syncthreads();
  const int P = a.page_size;
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
    r.pad[0] = r.pad[1] = 0;
    a.rows[b] = r;
    const int pages = r.page_hi - r.page_lo;
    local += (unsigned long long)pages;
    localmax = max(localmax, pages);
  }
  atomicAdd(&s_total, local);
  atomicMax(&s_maxpages, localmax);
  __syncthreads();
  if (tid == 0) {
    long long chunk;
    if (a.num_splits > 0) {
      chunk = 0;  // per row
    } else {
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
  // pass 2: split counts; count full and tail chunks
  unsigned nfull = 0, ntail = 0;
  for (int b = tid; b < a.batch; b += blockDim.x) {
    RowInfo r = a.rows[b];
    const int pages = r.page_hi - r.page_lo;
    int chunk, nsplit;
    if (pages == 0) {
      nsplit = 0;
      chunk = 1;
    } else if (a.num_splits > 0) {
      nsplit = a.num_splits;
      chunk = (pages + a.num_splits - 1) / a.num_splits;
    } else {
      chunk = s_chunk;
      nsplit = (pages + chunk - 1) / chunk;
    }
    r.nsplit = nsplit;
    r.chunk = chunk;
    a.rows[b] = r;
    if (pages > 0) {
      nfull += (unsigned)(pages / chunk);
      ntail += (pages % chunk) ? 1u : 0u;
    }
  }
  atomicAdd(&s_nfull, nfull * (unsigned)a.heads_per_row);
  atomicAdd(&s_ntail, ntail * (unsigned)a.heads_per_row);
  __syncthreads();
  // pass 3: emit items, full chunks first (longest-first order)
  const unsigned n_full_total = s_nfull;
  const unsigned total_work = (unsigned)a.batch * (unsigned)a.heads_per_row;
  for (unsigned w = tid; w < total_work; w += blockDim.x) {
    const int b = (int)(w / (unsigned)a.heads_per_row);
    const int sub = (int)(w % (unsigned)a.heads_per_row);
    const RowInfo r = a.rows[b];
    const int pages = r.page_hi - r.page_lo;
    if (pages == 0) continue;
    const int nonempty = (pages + r.chunk - 1) / r.chunk;
    for (int c = 0; c < nonempty; ++c) {
      WorkItem it;
      it.b = b;
      it.sub = sub;
      it.split = c;
      it.page_begin = r.page_lo + c * r.chunk;
      it.page_end = min(r.page_hi, it.page_begin + r.chunk);
      it.pad[0] = it.pad[1] = it.pad[2] = 0;
      const bool full = (it.page_end - it.page_begin) == r.chunk;
      const unsigned pos = full ? atomicAdd(&s_cur_full, 1u) : n_full_total + atomicAdd(&s_cur_tail, 1u);
      a.items[pos] = it;
    }
  }
  __syncthreads();
  if (tid == 0) {
    a.hdr->n_items = s_nfull + s_ntail;
    a.hdr->item_counter = 0;
  }
}

cudaError_t launch_plan(const PlanArgs &a, cudaStream_t stream) {
  plan_kernel<<<1, 1024, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pa
