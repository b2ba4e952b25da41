// Internal launch interface shared by the host API and the kernel translation
// units of the library. Not part of the public C ABI (include/flce.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "flce_gemm_params.h"

namespace flce {

// cta_group 2: grid/2 clusters of two CTAs (the kernel template also has a
// one-CTA form, cta_group 1, which is not built; other values fail).
// fp8 = 1: E4M3 operands (kind::f8f6f4) scaled in the epilogue by the product of
// the device scales p.acc_scale_h, p.acc_scale_w.
// c is the output map of the epilogue's TMA stores (unused by the LSE epilogue):
// bf16 G for the gradient GEMM; fp32 (or bf16 for OUT_STORE_BF16) for the F32 one.
// wide = 1 (F32 only): 256 x 512 tiles (TileCfg<2, 1>); p.n_blocks then counts
// 512-column tiles.
cudaError_t launch_gemm_lse(int cta_group, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmParams& p, int grid, cudaStream_t stream, int fp8);
cudaError_t launch_gemm_grad(int cta_group, const CUtensorMap& a, const CUtensorMap& b,
                             const CUtensorMap& c, const GemmParams& p, int grid,
                             cudaStream_t stream, int fp8);
cudaError_t launch_gemm_f32(int cta_group, const CUtensorMap& a, const CUtensorMap& b,
                            const CUtensorMap& c, const GemmParams& p, int grid,
                            cudaStream_t stream, int wide);

// Two products of 256 x 512 tiles and the fp32 epilogue in one launch: the units of
// `first` (its p.num_units) are dealt to the pairs before those of `second`. Both
// only read what earlier launches wrote, and their outputs do not overlap.
cudaError_t launch_gemm_f32_pair(int cta_group, const GemmArgs& first, const GemmArgs& second,
                                 int grid, cudaStream_t stream);

// Per-token merge of the vocabulary-range partials into lse and the per-token
// negative log-likelihood, and (gstat not null) per token (max, 1 / sum exp,
// 1 - p of the target, 0) for the gradient epilogue.
// part is [splits][part_stride][128] (max, sum exp over every id but the target's)
// pairs; zt holds the target logits.
cudaError_t launch_lse_merge(const float2* part, const float* zt, const int32_t* labels, int N,
                             int V, int part_stride, int splits, int ignore_index, float* lse,
                             float* nll, float4* gstat, cudaStream_t stream);

// Vocabulary shard [v_lo, v_hi): per token the shard's max m, sum of exp(z - m)
// and the target logit when the label lies in the shard (else 0).
cudaError_t launch_shard_merge(const float2* part, const float* zt, const int32_t* labels, int N,
                               int v_lo, int v_hi, int part_stride, int splits, int ignore_index,
                               float* m, float* s, float* zt_out, cudaStream_t stream);

// One-block deterministic reduction: label validation, n_valid, the loss (nll may
// be null: the loss is then 0 and only n, the scale and the label check count) and
// the gradient scale grad_scale / n (or / normalizer, or 1 for "sum").
cudaError_t launch_loss_reduce(const float* nll, const int32_t* labels, int N, int V,
                               int ignore_index, int reduction, float grad_scale,
                               float normalizer, float* loss, float* scale, int32_t* n_valid,
                               int32_t* status, cudaStream_t stream);

// Cross-entropy over given logits: label count and gradient scale (one block),
// then the row pass (lse, per-token loss, optional gradient; bf16 = 1 for bf16
// logits and gradient, 0 for fp32). g may equal z (in place, same row stride).
cudaError_t launch_ce_count(const int32_t* labels, int N, int V, int ignore_index, int reduction,
                            float grad_scale, float normalizer, float* scale, int32_t* status,
                            cudaStream_t stream);
cudaError_t launch_ce_rows(int bf16, const void* z, int64_t ld_bytes, const int32_t* labels,
                           int N, int V, int ignore_index, const float* scale, float* lse,
                           float* nll, void* g, int64_t gld_bytes, int sms, int32_t* status,
                           int64_t timeout_ns, cudaStream_t stream);

// dst[i] = bf16(src[i]) (round to nearest even), n a multiple of 8, both 16-byte aligned.
cudaError_t launch_f32_to_bf16(const float* src, uint16_t* dst, int64_t n, int sms,
                               cudaStream_t stream);

// E4M3 per-tensor quantisation of bf16 x [n] (n % 8 == 0): out[1] = amax,
// out[0] = scale, q = e4m3(x / scale).
cudaError_t launch_quantize_e4m3(const uint16_t* x, int64_t n, uint8_t* q, float* out, int sms,
                                 cudaStream_t stream);

// x (bf16 if bf16, else fp32; bytes a multiple of 16) *= *scale, in place.
cudaError_t launch_scale(void* x, int64_t bytes, int bf16, const float* scale, int sms,
                         cudaStream_t stream);

}  // namespace flce
