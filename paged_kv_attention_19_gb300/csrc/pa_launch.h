// pa_launch.h -- host-side launchers of the kernel instantiations (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {
struct GqaArgs;
struct CombineArgs;
struct PlanArgs;

// Shared-memory bytes and thread count of the split kernel for (D, GP).
int gqa_split_smem_bytes(int D, int GP);
int gqa_split_threads();
int gqa_stage_tokens(int D);

cudaError_t launch_plan(const PlanArgs &a, cudaStream_t stream);
cudaError_t launch_gqa_split(int D, int GP, int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                             const GqaArgs &a, cudaStream_t stream);
cudaError_t launch_gqa_combine(int D, const CombineArgs &a, cudaStream_t stream);
}  // namespace pa
