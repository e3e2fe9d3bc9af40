// pa_gqa_d64.cu -- head_dim 64 instantiations of the GQA split-KV and combine kernels.
#include "pa_gqa_launch.cuh"

namespace pa {

cudaError_t launch_gqa_split_d64(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                                 const GqaArgs &a, cudaStream_t stream) {
  return launch_split_any<64>(grid, tm_k, tm_v, tm_q, a, stream);
}

cudaError_t launch_gqa_combine_d64(const CombineArgs &a, cudaStream_t stream) { return launch_combine<64>(a, stream); }

}  // namespace pa
