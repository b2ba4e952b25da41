// Per-token merge of the forward pass's vocabulary-range partials, and the
// one-block deterministic loss reduction.
//
// The merge is the combination rule of the online log-sum-exp ("Liger Kernel:
// Fused Triton Kernels for LLM Training", The Architecture, 1. step 3): for
// partials (m_u, s_u) with s_u = sum exp(z - m_u) over disjoint vocabulary
// ranges, M = max_u m_u and lse = M + log(sum_u s_u exp(m_u - M)). The loss is
// the mean over non-ignored tokens of lse_i - z_{i,y_i} (same section, steps
// 4-5; the mean of the page's simulation and of PyTorch's reduction="mean").
#include <cmath>

#include "flce_internal.h"

namespace flce {

namespace {

__device__ __forceinline__ float ex2f_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The partial sums leave out the target's own term (LSE epilogue), so per token
//   S_o = sum over the other ids of exp(z - M),  e_t = exp(z_target - M),
//   lse = M + log(S_o + e_t),  NLL = log(1 + S_o / e_t) (lse - z_t once e_t < 2^-60),
//   1 - p = S_o / (S_o + e_t),
// none of them a difference of nearly equal numbers when p is close to 1. With
// gstat, (M, 1 / S, 1 - p, 0) is stored for the gradient epilogue.
__global__ void lse_merge_kernel(const float2* __restrict__ part, const float* __restrict__ zt,
                                 const int32_t* __restrict__ labels, int N, int V, int part_stride,
                                 int splits, int ignore_index, float* __restrict__ lse,
                                 float* __restrict__ nll, float4* __restrict__ gstat) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N) return;
  const int r = i / BM, l = i - (i / BM) * BM;
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, part[(static_cast<int64_t>(s) * part_stride + r) * BM + l].x);
  float So = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float2 pr = part[(static_cast<int64_t>(s) * part_stride + r) * BM + l];
    So += pr.y * ex2f_approx((pr.x - M) * kLog2e);
  }
  const int y = labels[i];
  const bool valid = y != ignore_index && y >= 0 && y < V;
  const float zy = valid ? zt[i] : -INFINITY;
  const float et = valid ? ex2f_approx((zy - M) * kLog2e) : 0.f;
  const float S = So + et;
  const float L = M + logf(S);
  lse[i] = L;
  // e_t < 2^-60 (the target more than 41 below the max): lse - z_t has no
  // cancellation, and S_o / e_t, with S_o at most V < 2^30, cannot overflow above it
  nll[i] = !valid ? 0.f : (et >= 0x1p-60f ? log1pf(So / et) : L - zy);
  if (gstat != nullptr) gstat[i] = make_float4(M, 1.f / S, So / S, 0.f);
}

// One vocabulary shard (ids [v_lo, v_hi) of a vocabulary split over several
// calls): the per-token merge of the shard's vocabulary-range partials into its
// (max, sum of exponentials), and the target logit when the token's label lies
// in the shard (else 0), so that the shards combine by max, rescaled sum and sum.
__global__ void shard_merge_kernel(const float2* __restrict__ part, const float* __restrict__ zt,
                                   const int32_t* __restrict__ labels, int N, int v_lo, int v_hi,
                                   int part_stride, int splits, int ignore_index,
                                   float* __restrict__ m_out, float* __restrict__ s_out,
                                   float* __restrict__ zt_out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N) return;
  const int r = i / BM, l = i - (i / BM) * BM;
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, part[(static_cast<int64_t>(s) * part_stride + r) * BM + l].x);
  float S = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float2 pr = part[(static_cast<int64_t>(s) * part_stride + r) * BM + l];
    S += pr.y * ex2f_approx((pr.x - M) * kLog2e);
  }
  const int y = labels[i];
  const bool here = y != ignore_index && y >= v_lo && y < v_hi;
  // the partial sums leave out the target's term: the shard's sum includes it
  if (here) S += ex2f_approx((zt[i] - M) * kLog2e);
  m_out[i] = M;
  s_out[i] = S;
  zt_out[i] = here ? zt[i] : 0.f;
}

constexpr int kReduceThreads = 1024;

__global__ void __launch_bounds__(kReduceThreads)
    loss_reduce_kernel(const float* __restrict__ nll, const int32_t* __restrict__ labels, int N,
                       int V, int ignore_index, int reduction, float grad_scale, float normalizer,
                       float* loss, float* scale, int32_t* n_valid_out, int32_t* status) {
  __shared__ double s_sum[kReduceThreads];
  __shared__ int s_cnt[kReduceThreads];
  __shared__ int s_bad[kReduceThreads];
  const int t = threadIdx.x;
  double acc = 0.0;
  int cnt = 0, bad = 0;
  for (int i = t; i < N; i += kReduceThreads) {
    const int y = labels[i];
    if (y == ignore_index) continue;
    if (y < 0 || y >= V) {
      bad = 1;
      continue;
    }
    ++cnt;
    if (nll != nullptr) acc += static_cast<double>(nll[i]);
  }
  s_sum[t] = acc;
  s_cnt[t] = cnt;
  s_bad[t] = bad;
  __syncthreads();
  for (int w = kReduceThreads / 2; w > 0; w >>= 1) {
    if (t < w) {
      s_sum[t] += s_sum[t + w];
      s_cnt[t] += s_cnt[t + w];
      s_bad[t] |= s_bad[t + w];
    }
    __syncthreads();
  }
  if (t == 0) {
    const double total = s_sum[0];
    const int n = s_cnt[0];
    double l, sc;
    if (reduction == 1) {  // sum
      l = total;
      sc = grad_scale;
    } else if (normalizer > 0.f) {
      l = total / normalizer;
      sc = grad_scale / static_cast<double>(normalizer);
    } else if (n > 0) {
      l = total / n;
      sc = grad_scale / static_cast<double>(n);
    } else {
      l = 0.0;
      sc = 0.0;
    }
    *loss = static_cast<float>(l);
    *scale = static_cast<float>(sc);
    *n_valid_out = n;
    if (s_bad[0] && status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, 8);
  }
}

// x *= *scale over n16 16-byte vectors (bf16 or fp32), in place. Every thread
// reads the scale first and leaves at once when it is exactly 1.
template <int kBf16>
__global__ void scale_kernel(uint4* __restrict__ x, int64_t n16, const float* __restrict__ scale) {
  const float sc = *scale;
  if (sc == 1.0f) return;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
    uint4 v = x[i];
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if constexpr (kBf16) {
        const float lo = __uint_as_float(w[k] << 16) * sc;
        const float hi = __uint_as_float(w[k] & 0xFFFF0000u) * sc;
        uint32_t r;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        w[k] = r;
      } else {
        w[k] = __float_as_uint(__uint_as_float(w[k]) * sc);
      }
    }
    x[i] = v;
  }
}

// dst = bf16(src), round to nearest even, 8 elements (two 16-byte loads, one
// 16-byte store) per thread and step: the last step of an fp32 accumulator that
// the GEMM epilogue built by TMA reduce-adds (dH across vocabulary chunks, dW
// across token blocks).
__global__ void f32_to_bf16_kernel(const float4* __restrict__ src, uint4* __restrict__ dst,
                                   int64_t n8) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 a = src[2 * i], b = src[2 * i + 1];
    uint4 o;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.x) : "f"(a.y), "f"(a.x));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.y) : "f"(a.w), "f"(a.z));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.z) : "f"(b.y), "f"(b.x));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.w) : "f"(b.w), "f"(b.z));
    dst[i] = o;
  }
}

// ---- per-tensor E4M3 quantisation -----------------------------------------------

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// amax over |x|: grid-stride over 8-element vectors, four independent 16-byte
// loads in flight per thread, warp then block max, one atomicMax per block on the
// bits of a non-negative float (ordered like the value). Plain loads, so that a
// tensor smaller than L2 is still there for the quantising pass.
__device__ __forceinline__ float absmax8(uint4 v, float m) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    m = fmaxf(m, fabsf(bf16_bits_to_float(w[k] & 0xFFFFu)));
    m = fmaxf(m, fabsf(bf16_bits_to_float(w[k] >> 16)));
  }
  return m;
}

__global__ void amax_kernel(const uint4* __restrict__ x, int64_t n8, unsigned int* amax_bits) {
  __shared__ float s_w[32];
  float m = 0.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n8; i += 4 * stride) {
    const uint4 a = x[i], b = x[i + stride], c = x[i + 2 * stride], d = x[i + 3 * stride];
    m = absmax8(d, absmax8(c, absmax8(b, absmax8(a, m))));
  }
  for (; i < n8; i += stride) m = absmax8(x[i], m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) s_w[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < static_cast<int>(blockDim.x >> 5) ? s_w[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) atomicMax(amax_bits, __float_as_uint(m));
  }
}

// Two fp32 values to two E4M3 bytes (round to nearest even, saturating), low byte
// first; a zero result is +0.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  uint32_t b = r;
  if ((b & 0x007Fu) == 0) b &= 0xFF00u;
  if ((b & 0x7F00u) == 0) b &= 0x00FFu;
  return b;
}

// Eight bf16 values times inv to eight E4M3 bytes.
__device__ __forceinline__ uint2 quant8(uint4 v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t b[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    b[k] = e4m3x2(__fmul_rn(bf16_bits_to_float(w[k] & 0xFFFFu), inv),
                  __fmul_rn(bf16_bits_to_float(w[k] >> 16), inv));
  return make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
}

// q = e4m3(x * inv) with inv = 448 / amax (double, rounded to fp32 and capped at the
// largest finite fp32, which only an amax below about 1.3e-36 reaches; 1 if
// amax == 0); block 0 stores scale = amax / 448 (double, rounded to fp32; 1 if
// amax == 0) next to the amax. One multiply per element instead of an IEEE divide.
__global__ void quantize_e4m3_kernel(const uint4* __restrict__ x, int64_t n8, uint2* __restrict__ q,
                                     float* out) {
  const float amax = __ldcg(out + 1);
  const float inv = amax > 0.f ? static_cast<float>(fmin(448.0 / static_cast<double>(amax),
                                                         3.4028234663852886e38))
                               : 1.f;
  if (blockIdx.x == 0 && threadIdx.x == 0)
    out[0] = amax > 0.f ? static_cast<float>(static_cast<double>(amax) / 448.0) : 1.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n8; i += 4 * stride) {
    const uint4 a = __ldcs(x + i), b = __ldcs(x + i + stride), c = __ldcs(x + i + 2 * stride),
                d = __ldcs(x + i + 3 * stride);
    q[i] = quant8(a, inv);
    q[i + stride] = quant8(b, inv);
    q[i + 2 * stride] = quant8(c, inv);
    q[i + 3 * stride] = quant8(d, inv);
  }
  for (; i < n8; i += stride) q[i] = quant8(__ldcs(x + i), inv);
}

}  // namespace

cudaError_t launch_quantize_e4m3(const uint16_t* x, int64_t n, uint8_t* q, float* out, int sms,
                                 cudaStream_t stream) {
  const int64_t n8 = n / 8;
  cudaError_t e = cudaMemsetAsync(out + 1, 0, sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int threads = 256;
  const int64_t want = (n8 + threads - 1) / threads;
  const int grid = static_cast<int>(want < static_cast<int64_t>(sms) * 8 ? want : static_cast<int64_t>(sms) * 8);
  amax_kernel<<<grid, threads, 0, stream>>>(reinterpret_cast<const uint4*>(x), n8,
                                            reinterpret_cast<unsigned int*>(out + 1));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  quantize_e4m3_kernel<<<grid, threads, 0, stream>>>(reinterpret_cast<const uint4*>(x), n8,
                                                     reinterpret_cast<uint2*>(q), out);
  return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* src, uint16_t* dst, int64_t n, int sms,
                               cudaStream_t stream) {
  const int64_t n8 = n / 8;
  if (n8 <= 0) return cudaSuccess;
  const int threads = 256;
  const int64_t want = (n8 + threads - 1) / threads;
  const int grid = static_cast<int>(want < static_cast<int64_t>(sms) * 8 ? want : static_cast<int64_t>(sms) * 8);
  f32_to_bf16_kernel<<<grid, threads, 0, stream>>>(reinterpret_cast<const float4*>(src),
                                                   reinterpret_cast<uint4*>(dst), n8);
  return cudaGetLastError();
}

cudaError_t launch_scale(void* x, int64_t bytes, int bf16, const float* scale, int sms,
                         cudaStream_t stream) {
  const int64_t n16 = bytes / 16;
  if (n16 <= 0) return cudaSuccess;
  const int threads = 256;
  const int64_t want = (n16 + threads - 1) / threads;
  const int grid = static_cast<int>(want < static_cast<int64_t>(sms) * 8 ? want : static_cast<int64_t>(sms) * 8);
  if (bf16)
    scale_kernel<1><<<grid, threads, 0, stream>>>(static_cast<uint4*>(x), n16, scale);
  else
    scale_kernel<0><<<grid, threads, 0, stream>>>(static_cast<uint4*>(x), n16, scale);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const float2* part, const float* zt, const int32_t* labels, int N,
                             int V, int part_stride, int splits, int ignore_index, float* lse,
                             float* nll, float4* gstat, cudaStream_t stream) {
  const int threads = 256;
  lse_merge_kernel<<<(N + threads - 1) / threads, threads, 0, stream>>>(
      part, zt, labels, N, V, part_stride, splits, ignore_index, lse, nll, gstat);
  return cudaGetLastError();
}

cudaError_t launch_shard_merge(const float2* part, const float* zt, const int32_t* labels, int N,
                               int v_lo, int v_hi, int part_stride, int splits, int ignore_index,
                               float* m, float* s, float* zt_out, cudaStream_t stream) {
  const int threads = 256;
  shard_merge_kernel<<<(N + threads - 1) / threads, threads, 0, stream>>>(
      part, zt, labels, N, v_lo, v_hi, part_stride, splits, ignore_index, m, s, zt_out);
  return cudaGetLastError();
}

cudaError_t launch_loss_reduce(const float* nll, const int32_t* labels, int N, int V,
                               int ignore_index, int reduction, float grad_scale,
                               float normalizer, float* loss, float* scale, int32_t* n_valid,
                               int32_t* status, cudaStream_t stream) {
  loss_reduce_kernel<<<1, kReduceThreads, 0, stream>>>(nll, labels, N, V, ignore_index, reduction,
                                                       grad_scale, normalizer, loss, scale,
                                                       n_valid, status);
  return cudaGetLastError();
}

}  // namespace flce
