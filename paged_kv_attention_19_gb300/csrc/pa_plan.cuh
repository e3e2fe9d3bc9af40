// pa_plan.cuh -- work-list types of the MLA split-KV path: the per-row table
// and the arguments of the planner (pa_plan.cu) that turns device-resident
// context lengths into page-aligned work items.
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
  int batch, heads_per_row;  // head groups per row
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

}  // namespace pa
