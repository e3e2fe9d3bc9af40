// pa_gqa_d256.cu -- head_dim 256 instantiations of the GQA split-KV and combine kernels and their launchers.
#include "pa_gqa.cuh"
#include "pa_launch.h"

namespace pa {

namespace {
// Both kernels are launched as programmatic dependents of the kernel before them: the
// combine kernel's launch overlaps the split kernel's tail and waits (griddepcontrol.wait)
// before reading its output; the split kernel reads nothing an earlier kernel of the call wrote.
cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, int smem, cudaStream_t stream, cudaLaunchAttribute *attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}
}  // namespace

cudaError_t launch_gqa_split_d256(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                                  const GqaArgs &a, cudaStream_t stream) {
  using C = GqaCfg<256>;
  constexpr int smem = GqaSmem<C>::BYTES;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gqa_split_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(C::THREADS), smem, stream, attr);
  return cudaLaunchKernelEx(&cfg, gqa_split_kernel<256>, tm_k, tm_v, tm_q, a);
}

cudaError_t launch_gqa_combine_d256(const CombineArgs &a, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(a.nparts), dim3(128), 0, stream, attr);
  return cudaLaunchKernelEx(&cfg, gqa_combine_kernel<256>, a);
}

}  // namespace pa
