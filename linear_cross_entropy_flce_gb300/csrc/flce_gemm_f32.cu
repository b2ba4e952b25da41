// Instantiations and launcher of the tcgen05 GEMM with the EPI_F32 epilogue.
#include "flce_gemm.cuh"
#include "flce_internal.h"

namespace flce {

namespace {

template <int kCta>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                   const GemmParams& p, int grid, cudaStream_t stream) {
  auto kern = flce_gemm_kernel<EPI_F32, kCta, 0>;
  constexpr size_t smem = TileCfg<kCta>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCta;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, b, c, p);
}

}  // namespace

cudaError_t launch_gemm_f32(int cta_group, const CUtensorMap& a, const CUtensorMap& b,
                            const CUtensorMap& c, const GemmParams& p, int grid,
                            cudaStream_t stream) {
  if (cta_group != 2) return cudaErrorInvalidValue;  // only the pair kernel is built
  return launch<2>(a, b, c, p, grid, stream);
}

}  // namespace flce
