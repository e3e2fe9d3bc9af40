// pa_launch.h -- host-side launchers of the kernel instantiations (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {
struct GqaArgs;
struct PlanArgs;
struct CombineArgs;

cudaError_t launch_plan(const PlanArgs &a, cudaStream_t stream);
cudaError_t launch_gqa_split_d64(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                                  const GqaArgs &a,
                                 cudaStream_t stream);
cudaError_t launch_gqa_split_d128(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                                  const GqaArgs &a,
                                  cudaStream_t stream);
cudaError_t launch_gqa_split_d256(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                                  const GqaArgs &a,
                                  cudaStream_t stream);
cudaError_t launch_gqa_combine_d64(const CombineArgs &a, cudaStream_t stream);
cudaError_t launch_gqa_combine_d128(const CombineArgs &a, cudaStream_t stream);
cudaError_t launch_gqa_combine_d256(const CombineArgs &a, cudaStream_t stream);
}  // namespace pa
