// Instantiation and launcher of the tcgen05 GEMM with the EPI_GRAD epilogue.
#include "flce_gemm.cuh"
#include "flce_internal.h"

namespace flce {

cudaError_t launch_gemm_grad(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                             int grid, cudaStream_t stream) {
  auto kern = flce_gemm_kernel<EPI_GRAD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, kSmemBytes, stream>>>(a, b, p);
  return cudaGetLastError();
}

}  // namespace flce
