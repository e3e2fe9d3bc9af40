// pa_gqa_d64.cu -- head_dim 64 instantiations of the GQA split-KV and combine kernels.
#include "pa_gqa.cuh"
#include "pa_launch.h"

namespace pa {

template <int GP>
static cudaError_t launch_split_gp(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                   const GqaArgs &a, cudaStream_t stream) {
  using C = GqaCfg<64, GP>;
  constexpr int smem = GqaSmem<C>::BYTES;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gqa_split_kernel<64, GP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  gqa_split_kernel<64, GP><<<grid, C::THREADS, smem, stream>>>(tm_k, tm_v, a);
  return cudaGetLastError();
}

cudaError_t launch_gqa_split_d64(int GP, int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                 const GqaArgs &a, cudaStream_t stream) {
  switch (GP) {
    case 1: return launch_split_gp<1>(grid, tm_k, tm_v, a, stream);
    case 2: return launch_split_gp<2>(grid, tm_k, tm_v, a, stream);
    case 4: return launch_split_gp<4>(grid, tm_k, tm_v, a, stream);
    case 8: return launch_split_gp<8>(grid, tm_k, tm_v, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

int gqa_split_smem_bytes_d64(int GP) {
  switch (GP) {
    case 1: return GqaSmem<GqaCfg<64, 1>>::BYTES;
    case 2: return GqaSmem<GqaCfg<64, 2>>::BYTES;
    case 4: return GqaSmem<GqaCfg<64, 4>>::BYTES;
    case 8: return GqaSmem<GqaCfg<64, 8>>::BYTES;
    default: return 0;
  }
}

cudaError_t launch_gqa_combine_d64(const CombineArgs &a, cudaStream_t stream) {
  const int warps = a.batch * a.Hq;
  const int blocks = (warps + 7) / 8;
  combine_kernel<64><<<blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pa
