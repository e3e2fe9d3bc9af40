// pa_launch.h -- host-side launchers of the kernel instantiations (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {
// Bookkeeping of the profiling hook and launch counter of the C ABI (pa_api.cu).
void note_launches(int n);
cudaError_t profile_mark(bool before, cudaStream_t stream);
// Records e (or the thread's last CUDA error, if e is cudaSuccess) as the CUDA error behind
// a PA_ERR_CUDA return, and returns PA_ERR_CUDA.
int cuda_fail(cudaError_t e);

struct GqaArgs;
struct CombineArgs;

cudaError_t launch_gqa_split_d64(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                                  const GqaArgs &a,
                                 cudaStream_t stream);
cudaError_t launch_gqa_split_d128(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                                  const GqaArgs &a,
                                  cudaStream_t stream);
cudaError_t launch_gqa_split_d256(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                                  const GqaArgs &a,
                                  cudaStream_t stream);
// FP8 E4M3 pools (head_dim 128 and 256)
cudaError_t launch_gqa_split_fp8_d128(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                      const CUtensorMap &tm_q, const GqaArgs &a, cudaStream_t stream);
cudaError_t launch_gqa_split_fp8_d256(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                      const CUtensorMap &tm_q, const GqaArgs &a, cudaStream_t stream);
// NVFP4 pools (head_dim 64, 128 or 256)
cudaError_t launch_gqa_split_nvfp4(int D, int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                   const CUtensorMap &tm_q, const GqaArgs &a, cudaStream_t stream);
cudaError_t launch_gqa_combine_d64(const CombineArgs &a, cudaStream_t stream);
cudaError_t launch_gqa_combine_d128(const CombineArgs &a, cudaStream_t stream);
cudaError_t launch_gqa_combine_d256(const CombineArgs &a, cudaStream_t stream);
}  // namespace pa
