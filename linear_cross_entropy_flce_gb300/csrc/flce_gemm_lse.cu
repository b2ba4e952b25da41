// Instantiations and launcher of the tcgen05 GEMM with the EPI_LSE epilogue.
#include "flce_gemm.cuh"
#include "flce_internal.h"

namespace flce {

namespace {

template <int kCta, int kFp8>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, int grid,
                   cudaStream_t stream) {
  auto kern = flce_gemm_kernel<EPI_LSE, kCta, kFp8>;
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
  const CUtensorMap unused = {};  // the LSE epilogue writes no tiles
  return cudaLaunchKernelEx(&cfg, kern, a, b, unused, p);
}

}  // namespace

cudaError_t launch_gemm_lse(int cta_group, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmParams& p, int grid, cudaStream_t stream, int fp8) {
  if (cta_group != 2) return cudaErrorInvalidValue;  // only the pair kernel is built
  return fp8 ? launch<2, 1>(a, b, p, grid, stream) : launch<2, 0>(a, b, p, grid, stream);
}

}  // namespace flce
