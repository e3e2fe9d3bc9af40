// pa_mla.h -- host entry of the MLA absorbed decode path (internal).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

size_t mla_workspace_size(int batch, int num_heads, int max_context_len, int page_size, int num_splits);

int mla_decode(const void *q, const void *cache, const void *w_uk, const void *w_uv, const int32_t *block_table,
               const int32_t *context_lens, void *out, float *lse, int batch, int num_heads, int page_size,
               int num_pages, int max_pages_per_seq, int max_context_len, float scale, int num_splits,
               void *workspace, size_t workspace_bytes, cudaStream_t stream, cudaEvent_t ev_before,
               cudaEvent_t ev_after, int *launches);

}  // namespace pa
