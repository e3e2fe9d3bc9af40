// pa_noalloc.cu -- GQA paged decode for callers that cannot allocate device memory.
//
// pa_decode_gqa needs a caller-provided device workspace.  Some callers have
// no way to provide one at call time: an inference engine that handed all
// device memory to its own pool at start-up, a plug-in whose host framework
// gives it only the input and output pointers, or a latency-critical path
// that must not pay for cudaMalloc (which can synchronise the device).  For
// them, pa_decode_gqa_noalloc runs the same decode with the workspace placed
// in the fixed-size device array below, which every GPU that loads this
// library holds until the process exits.
#include <mutex>

#include "pa_decode.h"
#include "pa_launch.h"

namespace {

// The built-in scratch.  In host code this name is only a stand-in for the
// device array, never a device address: host code must use the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_pa_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
int scratch_address(void **out) {
  int dev = 0;
  if (const cudaError_t ce = cudaGetDevice(&dev); ce != cudaSuccess) return pa::cuda_fail(ce);
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (const cudaError_t ce = cudaGetSymbolAddress(&p, g_pa_scratch); ce != cudaSuccess || p == nullptr)
      return pa::cuda_fail(ce);
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" int pa_decode_gqa_noalloc(const void *q, const void *k_pool, const void *v_pool,
                                     const int32_t *block_table, const int32_t *context_lens, void *out,
                                     float *lse, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                     int page_size, int num_pages, int max_pages_per_seq, int max_context_len,
                                     float scale, int window, int num_splits, cudaStream_t stream) {
  const size_t need = pa_workspace_size(PA_KIND_GQA, batch, num_q_heads, num_kv_heads, head_dim, max_context_len,
                                        page_size, num_splits);
  if (need == 0 || batch == 0) {
    // invalid shape (or empty batch): the regular entry point reports it, before any device work
    return pa_decode_gqa(q, k_pool, v_pool, block_table, context_lens, out, lse, batch, num_q_heads, num_kv_heads,
                         head_dim, page_size, num_pages, max_pages_per_seq, max_context_len, scale, window,
                         num_splits, nullptr, 0, stream);
  }
  if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE_TOO_SMALL;
  void *scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != PA_OK) return rc;
  return pa_decode_gqa(q, k_pool, v_pool, block_table, context_lens, out, lse, batch, num_q_heads, num_kv_heads,
                       head_dim, page_size, num_pages, max_pages_per_seq, max_context_len, scale, window, num_splits,
                       scratch, (size_t)PA_NOALLOC_SCRATCH_BYTES, stream);
}
