// pa_gqa_d128.cu -- head_dim 128 instantiations of the GQA split-KV and combine kernels.
#include "pa_gqa_launch.cuh"

namespace pa {

cudaError_t launch_gqa_split_d128(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                                 const GqaArgs &a, cudaStream_t stream) {
  return launch_split_any<128>(grid, tm_k, tm_v, tm_q, a, stream);
}

cudaError_t launch_gqa_combine_d128(const CombineArgs &a, cudaStream_t stream) { return launch_combine<128>(a, stream); }

}  // namespace pa
