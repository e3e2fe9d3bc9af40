// pa_gqa_nvfp4.cu -- instantiations of the NVFP4 split-KV kernel (head_dim 64, 128 and 256; the
// combine kernel is the bf16 pools' one: partials are fp32 either way).
#include "pa_gqa_fp4.cuh"
#include "pa_gqa_launch.cuh"

namespace pa {

namespace {

template <int D, bool LW>
cudaError_t launch_fp4_split_lw(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                                const GqaArgs &a, cudaStream_t stream) {
  using C = GqaFp4Cfg<D>;
  return a.Q > 1 ? launch_split_kernel<C, gqa_fp4_split_kernel<D, true, LW>>(grid, tm_k, tm_v, tm_q, a, stream)
                 : launch_split_kernel<C, gqa_fp4_split_kernel<D, false, LW>>(grid, tm_k, tm_v, tm_q, a, stream);
}

template <int D>
cudaError_t launch_fp4_split(int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                             const GqaArgs &a, cudaStream_t stream) {
  return a.wait_ns == WAIT_LIMIT_NS ? launch_fp4_split_lw<D, false>(grid, tm_k, tm_v, tm_q, a, stream)
                                    : launch_fp4_split_lw<D, true>(grid, tm_k, tm_v, tm_q, a, stream);
}

}  // namespace

cudaError_t launch_gqa_split_nvfp4(int D, int grid, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                   const CUtensorMap &tm_q, const GqaArgs &a, cudaStream_t stream) {
  switch (D) {
    case 64: return launch_fp4_split<64>(grid, tm_k, tm_v, tm_q, a, stream);
    case 128: return launch_fp4_split<128>(grid, tm_k, tm_v, tm_q, a, stream);
    default: return launch_fp4_split<256>(grid, tm_k, tm_v, tm_q, a, stream);
  }
}

}  // namespace pa
