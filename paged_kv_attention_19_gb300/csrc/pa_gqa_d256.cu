// pa_gqa_d256.cu -- head_dim 256 instantiations of the GQA split-KV and combine kernels.
#include "pa_gqa_launch.cuh"

namespace pa {

cudaError_t launch_gqa_split_d256(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                                 const GqaArgs &a, cudaStream_t stream) {
  return launch_split_any<256>(grid, tm_k, tm_v, tm_q, a, stream);
}

cudaError_t launch_gqa_combine_d256(const CombineArgs &a, cudaStream_t stream) { return launch_combine<256>(a, stream); }

}  // namespace pa
