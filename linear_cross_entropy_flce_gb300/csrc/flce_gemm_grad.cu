// Instantiations of the tcgen05 GEMM with the EPI_GRAD epilogue (bf16 and E4M3
// operands). One translation unit per epilogue, so that they compile in parallel.
#include "flce_gemm.cuh"
#include "flce_internal.h"

namespace flce {

cudaError_t launch_gemm_grad(int cta_group, const CUtensorMap& a, const CUtensorMap& b,
                             const CUtensorMap& c, const GemmParams& p, int grid,
                             cudaStream_t stream, int fp8) {
  if (cta_group != 2) return cudaErrorInvalidValue;  // only the pair kernel is built
  GemmArgs g{};
  g.a = a;
  g.b = b;
  g.c = c;
  g.p = p;
  return fp8 ? launch_gemm<EPI_GRAD, 2, 1, 0>(g, g, grid, stream)
             : launch_gemm<EPI_GRAD, 2, 0, 0>(g, g, grid, stream);
}

}  // namespace flce
