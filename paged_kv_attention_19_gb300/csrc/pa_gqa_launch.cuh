// pa_gqa_launch.cuh -- host launchers of the GQA split-KV and combine kernels, instantiated
// once per head_dim by pa_gqa_d{64,128,256}.cu and, for FP8 pools, by pa_gqa_fp8.cu (one
// translation unit each, built in parallel).
#pragma once

#include "pa_gqa.cuh"
#include "pa_gqa_f8.cuh"
#include "pa_launch.h"

namespace pa {

// Both kernels are launched as programmatic dependents of the kernel before them: the
// combine kernel's launch overlaps the split kernel's tail and waits (griddepcontrol.wait)
// before reading its output; the split kernel waits the same way before it reads its inputs.
inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, int smem, cudaStream_t stream,
                                     cudaLaunchAttribute *attr) {
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

// One launch of split kernel `kernel` with configuration C (the shared-memory opt-in is made
// once per device and kernel: one static per instantiation).
template <class C, auto kernel>
cudaError_t launch_split_kernel(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                                const GqaArgs &a, cudaStream_t stream) {
  constexpr int smem = GqaSmem<C>::BYTES;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(C::THREADS), smem, stream, attr);
  return cudaLaunchKernelEx(&cfg, kernel, tm_k, tm_v, tm_q, a);
}

// Q == 1 (decode) runs the kernel compiled without the per-position row logic; a wait limit other
// than the default runs the instantiation whose producer takes it as an argument (LW).
template <int D, bool LW, int MT>
cudaError_t launch_split_mt(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                            const GqaArgs &a, cudaStream_t stream) {
  using C = GqaCfgOf<D, MT>;
  if constexpr (MT == 1 && D > 64) {
    if (a.unit_copy)  // decode over small pages: the unit-major kernel (its pool maps are 5-D)
      return launch_split_kernel<GqaCfgOf<D, 1, true>, gqa_split_kernel<D, false, LW, 1, true>>(grid, tm_k, tm_v,
                                                                                              tm_q, a, stream);
  }
  return a.Q > 1 ? launch_split_kernel<C, gqa_split_kernel<D, true, LW, MT>>(grid, tm_k, tm_v, tm_q, a, stream)
                 : launch_split_kernel<C, gqa_split_kernel<D, false, LW, MT>>(grid, tm_k, tm_v, tm_q, a, stream);
}

// Tiles paired in one sequence (a.mt == 2) exist for head_dim up to 128.
template <int D, bool LW>
cudaError_t launch_split_lw(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                            const GqaArgs &a, cudaStream_t stream) {
  if constexpr (D <= 128) {
    if (a.mt == 2) return launch_split_mt<D, LW, 2>(grid, tm_k, tm_v, tm_q, a, stream);
  }
  return launch_split_mt<D, LW, 1>(grid, tm_k, tm_v, tm_q, a, stream);
}

template <int D>
cudaError_t launch_split_any(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                             const GqaArgs &a, cudaStream_t stream) {
  return a.wait_ns == WAIT_LIMIT_NS ? launch_split_lw<D, false>(grid, tm_k, tm_v, tm_q, a, stream)
                                    : launch_split_lw<D, true>(grid, tm_k, tm_v, tm_q, a, stream);
}

// FP8 pools: NH8 = 1 when a tile has at most 8 (head, position) columns, else 2.
template <int D, int NH8, bool LW>
cudaError_t launch_f8_split_lw(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                               const GqaArgs &a, cudaStream_t stream) {
  using C = GqaF8Cfg<D, NH8>;
  return a.Q > 1 ? launch_split_kernel<C, gqa_f8_split_kernel<D, true, NH8, LW>>(grid, tm_k, tm_v, tm_q, a, stream)
                 : launch_split_kernel<C, gqa_f8_split_kernel<D, false, NH8, LW>>(grid, tm_k, tm_v, tm_q, a, stream);
}

template <int D, int NH8>
cudaError_t launch_f8_split(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                            const GqaArgs &a, cudaStream_t stream) {
  return a.wait_ns == WAIT_LIMIT_NS ? launch_f8_split_lw<D, NH8, false>(grid, tm_k, tm_v, tm_q, a, stream)
                                    : launch_f8_split_lw<D, NH8, true>(grid, tm_k, tm_v, tm_q, a, stream);
}

template <int D>
cudaError_t launch_f8_split_any(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                                const GqaArgs &a, cudaStream_t stream) {
  return a.gt * a.qt <= 8 ? launch_f8_split<D, 1>(grid, tm_k, tm_v, tm_q, a, stream)
                          : launch_f8_split<D, 2>(grid, tm_k, tm_v, tm_q, a, stream);
}

template <int D>
cudaError_t launch_combine(const CombineArgs &a, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)a.nblocks), dim3(a.mt * PART_HEADS * 32), 0, stream, attr);
  return cudaLaunchKernelEx(&cfg, gqa_combine_kernel<D>, a);
}

}  // namespace pa
