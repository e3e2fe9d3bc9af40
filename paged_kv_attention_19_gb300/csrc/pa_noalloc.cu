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
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_decode.h"
#include "pa_launch.h"

namespace {

// The built-in scratch.  In host code this name is only a stand-in for the
// device array, never a device address: host code must use the address that
// cudaGetSymbolAddress returns in the current context.
static __device__ __align__(256) unsigned char g_pa_scratch[PA_NOALLOC_SCRATCH_BYTES];

// The array's address is looked up once per CUDA context and cached under the
// context's unique ID (cuCtxGetId: never reused within a process), so a
// context created later on the same device -- after cudaDeviceReset, or a
// caller's own non-primary context -- gets a fresh lookup, never a stale address.
constexpr int kCacheSlots = 64;
struct ScratchSlot {
  unsigned long long ctx_id;
  void *ptr;
};
std::mutex g_mu;
ScratchSlot g_cache[kCacheSlots] = {};
int g_next_slot = 0;

struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxFns &ctx_fns() {
  static CtxFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return fns;
}

// Unique ID of the calling thread's current context; 0 if none is current yet.
int current_ctx_id(unsigned long long *id) {
  const CtxFns &f = ctx_fns();
  if (!f.get_current || !f.get_id) return pa::cuda_fail(cudaErrorNotSupported);
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS) return pa::cuda_fail(cudaErrorContextIsDestroyed);
  *id = 0;
  if (ctx && f.get_id(ctx, id) != CUDA_SUCCESS) return pa::cuda_fail(cudaErrorContextIsDestroyed);
  return PA_OK;
}

// Device address of the scratch in the current context (looked up on the first call in a
// context, then cached).
int scratch_address(void **out) {
  unsigned long long id = 0;
  int rc = current_ctx_id(&id);
  if (rc != PA_OK) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  if (id != 0) {
    for (const ScratchSlot &e : g_cache)
      if (e.ctx_id == id) {
        *out = e.ptr;
        return PA_OK;
      }
  }
  void *p = nullptr;
  if (const cudaError_t ce = cudaGetSymbolAddress(&p, g_pa_scratch); ce != cudaSuccess || p == nullptr)
    return pa::cuda_fail(ce);
  if (id == 0) {  // no context was current: the lookup made the device's primary context current
    rc = current_ctx_id(&id);
    if (rc != PA_OK) return rc;
  }
  if (id != 0) {
    g_cache[g_next_slot] = {id, p};
    g_next_slot = (g_next_slot + 1) % kCacheSlots;
  }
  *out = p;
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
