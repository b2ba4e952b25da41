// Instantiations of the tcgen05 GEMM with the EPI_F32 epilogue: 256 x 256 tiles
// with two TMEM accumulators, 256 x 512 tiles with one (wide), and the wide form
// carrying two products in one launch. One translation unit per epilogue, so that
// they compile in parallel.
#include "flce_gemm.cuh"
#include "flce_internal.h"

namespace flce {

cudaError_t launch_gemm_f32(int cta_group, const CUtensorMap& a, const CUtensorMap& b,
                            const CUtensorMap& c, const GemmParams& p, int grid,
                            cudaStream_t stream, int wide) {
  if (cta_group != 2) return cudaErrorInvalidValue;  // only the pair kernel is built
  GemmArgs g{};
  g.a = a;
  g.b = b;
  g.c = c;
  g.p = p;
  return wide ? launch_gemm<EPI_F32, 2, 0, 1>(g, g, grid, stream)
              : launch_gemm<EPI_F32, 2, 0, 0>(g, g, grid, stream);
}

cudaError_t launch_gemm_f32_pair(int cta_group, const GemmArgs& first, const GemmArgs& second,
                                 int grid, cudaStream_t stream) {
  if (cta_group != 2) return cudaErrorInvalidValue;  // only the pair kernel is built
  return launch_gemm<EPI_F32, 2, 0, 1, 2>(first, second, grid, stream);
}

}  // namespace flce
