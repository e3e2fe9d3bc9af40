// pa_gqa_fp8.cu -- instantiations of the FP8 E4M3 split-KV kernel (head_dim 128 and 256; the
// combine kernel is the bf16 pools' one: partials are fp32 either way).
#include "pa_gqa_launch.cuh"

namespace pa {

cudaError_t launch_gqa_split_fp8_d128(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                      const CUtensorMap &tm_q, const GqaArgs &a, cudaStream_t stream) {
  return launch_f8_split_any<128>(grid, tm_k, tm_v, tm_q, a, stream);
}

cudaError_t launch_gqa_split_fp8_d256(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                      const CUtensorMap &tm_q, const GqaArgs &a, cudaStream_t stream) {
  return launch_f8_split_any<256>(grid, tm_k, tm_v, tm_q, a, stream);
}

}  // namespace pa
