// Cross-entropy over a given logits matrix Z [N, V] (fp32 or bf16): the
// unfused loss that fused linear cross-entropy replaces ("GPU MODE lecture 28"
// notes, cross-entropy section: the loss takes logits.view(-1, vocab) and labels
// with reduction="mean"). It is a bandwidth-bound pass: the logits are read
// once for the online log-sum-exp and, for the gradient, the same row is read
// again (from L2) and dZ = (softmax - onehot) * scale is written, in place when
// the caller passes the logits as the gradient buffer.
//
// Kernels:
//   ce_count_kernel : one block; n_valid, label check, gradient scale.
//   ce_rows_staged_kernel : rows of 64-880 KB. Persistent clusters of 1-8 CTAs,
//                     one row per cluster at a time, each CTA's slice (at most
//                     110 KB) copied into shared memory by the bulk-copy engine,
//                     double-buffered so that the next row's slice streams in
//                     while this one is reduced and its gradient written. Both
//                     passes read shared memory: one DRAM read and one write per
//                     element.
//   ce_rows_kernel  : other rows. Persistent clusters of 1-8 CTAs, one row per
//                     cluster at a time, each CTA streaming a ~128 KB slice with
//                     16-byte vector loads; the gradient pass re-reads its slice
//                     (from L2 when the live rows fit in it).
// Both merge per-thread running (max, sum exp) across the block and then across
// the cluster, then form lse and the per-token loss: the staged kernel by
// asynchronous stores of each CTA's (max, sum exp, target logit) into every
// CTA's shared memory, counted on the receiver's mbarrier (so the previous row's
// gradient stores need not drain first); the streamed kernel through distributed
// shared memory reads after one cluster barrier per row.
// The loss itself is formed by loss_reduce_kernel (flce_reduce.cu).
#include <cmath>
#include <cstdint>

#include "flce_internal.h"

namespace flce {

namespace {

constexpr int kCeThreads = 512;
constexpr int kMaxCeCluster = 8;  // CTAs per row at most (portable cluster size)
constexpr int kCountThreads = 1024;

__device__ __forceinline__ float ex2a(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Element-wise maximum of two bf16 pairs (exact); -inf in both halves.
constexpr uint32_t kBf16NegInf2 = 0xFF80FF80u;
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 16-byte vector of logits: 4 fp32 or 8 bf16, widened to fp32.
template <int kBf16>
struct Vec16;

template <>
struct Vec16<0> {
  static constexpr int E = 4;
  __device__ static void load(const void* p, float (&x)[4]) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  }
  __device__ static void store(void* p, const float (&x)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  }
  __device__ static float load1(const void* p) { return __ldcg(reinterpret_cast<const float*>(p)); }
  __device__ static void store1(void* p, float v) { *reinterpret_cast<float*>(p) = v; }
};

template <>
struct Vec16<1> {
  static constexpr int E = 8;
  __device__ static void load(const void* p, float (&x)[8]) {
    const uint4 v = __ldcg(reinterpret_cast<const uint4*>(p));
    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
    x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
  }
  __device__ static void store(void* p, const float (&x)[8]) {
    *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]),
                                              pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
  }
  __device__ static float load1(const void* p) {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
  }
  __device__ static void store1(void* p, float v) {
    *reinterpret_cast<uint16_t*>(p) = static_cast<uint16_t>(pack_bf16(v, 0.f) & 0xFFFFu);
  }
};

// (m, s) with s = sum exp(z - m): merge two partial states.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  s = s * ex2a((m - mn) * kLog2e) + s2 * ex2a((m2 - mn) * kLog2e);
  m = mn;
}

// A row's merged (max M, sum S_o of exp(z - M) over every id but the target's,
// target logit z_t) to what the gradient pass and the loss need, with no
// difference of nearly equal numbers when p of the target is close to 1.
// row_grad, before the gradient pass: e_t = exp(z_t - M), S = S_o + e_t, and
// dZ = exp(z - M) * a off the target, -scale * q at it, with a = scale / S and
// q = S_o / S (1 - p). row_loss, after it (only the CTA that writes the loss):
// lse = M + log S and NLL = log1p(S_o / e_t), or lse - z_t once e_t < 2^-60,
// where that has no cancellation and S_o / e_t could overflow.
struct RowStat {
  float M, So, zt, et, S, a, q;
  bool valid;
};

__device__ __forceinline__ RowStat row_grad(float M, float So, float zt, bool valid,
                                            float scale) {
  RowStat r;
  r.M = M;
  r.So = So;
  r.zt = zt;
  r.valid = valid;
  r.et = valid ? ex2a((zt - M) * kLog2e) : 0.f;
  r.S = So + r.et;
  float inv;   // S >= 1 (the row's maximum term is 1): the hardware reciprocal, within 1 ulp
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(r.S));
  r.a = (valid ? scale : 0.f) * inv;
  r.q = So * inv;
  return r;
}

__device__ __forceinline__ void row_loss(const RowStat& r, float& lse, float& nll) {
  lse = r.M + logf(r.S);
  nll = !r.valid ? 0.f : (r.et >= 0x1p-60f ? log1pf(r.So / r.et) : lse - r.zt);
}

__global__ void __launch_bounds__(kCountThreads)
    ce_count_kernel(const int32_t* __restrict__ labels, int N, int V, int ignore_index,
                    int reduction, float grad_scale, float normalizer, float* scale,
                    int32_t* status) {
  __shared__ int s_cnt[kCountThreads];
  __shared__ int s_bad[kCountThreads];
  const int t = threadIdx.x;
  int cnt = 0, bad = 0;
  for (int i = t; i < N; i += kCountThreads) {
    const int y = labels[i];
    if (y == ignore_index) continue;
    if (y < 0 || y >= V) bad = 1;
    else ++cnt;
  }
  s_cnt[t] = cnt;
  s_bad[t] = bad;
  __syncthreads();
  for (int w = kCountThreads / 2; w > 0; w >>= 1) {
    if (t < w) {
      s_cnt[t] += s_cnt[t + w];
      s_bad[t] |= s_bad[t + w];
    }
    __syncthreads();
  }
  if (t == 0) {
    const int n = s_cnt[0];
    double sc;
    if (reduction == 1) sc = grad_scale;
    else if (normalizer > 0.f) sc = grad_scale / static_cast<double>(normalizer);
    else sc = n > 0 ? grad_scale / static_cast<double>(n) : 0.0;
    *scale = static_cast<float>(sc);
    if (s_bad[0] && status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, 8);
  }
}

__device__ __forceinline__ uint32_t cta_rank_in_cluster() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t ctas_in_cluster() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Stores v into `local`'s copy in CTA `rank` of the cluster and counts its 16
// bytes on that CTA's mbarrier `bar_local` (the same offset in the peer): the
// receiver learns of the data by waiting on its own barrier, with no fence over
// this thread's other (global) stores.
__device__ __forceinline__ void st_async_f4(const float4* local, uint64_t* bar_local, uint32_t rank,
                                            float4 v) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(bar_local));
  uint32_t ra, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(b), "r"(rank));
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(ra),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(rb)
      : "memory");
}

__device__ __forceinline__ float2 ld_dsmem_f2(const float2* local, uint32_t rank) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(r) : "memory");
  return v;
}

// One row per cluster of CTAs: CTA r of the cluster streams its slice of the
// row's 16-byte vectors, the block merges its (max, sum exp), the cluster
// exchanges the per-CTA pairs through distributed shared memory (one cluster
// barrier per row; pair slots alternate between rows), every CTA forms lse, and
// each CTA writes the gradient of its own slice, which it re-reads from L2.
template <int kBf16, bool kGrad>
__global__ void __launch_bounds__(kCeThreads)
    ce_rows_kernel(const uint8_t* z, int64_t ld_bytes,  // may alias g (in place)
                   const int32_t* __restrict__ labels, int N, int V, int ignore_index,
                   const float* __restrict__ scale_ptr, float* __restrict__ lse_out,
                   float* __restrict__ nll_out, uint8_t* g, int64_t gld_bytes) {
  using VT = Vec16<kBf16>;
  constexpr int E = VT::E;
  constexpr int kElt = kBf16 ? 2 : 4;
  constexpr int kUnroll = 32 / E;  // 32 values (8 or 4 16-byte loads) in flight per thread
  __shared__ float2 s_red[kCeThreads / 32];
  __shared__ float2 s_part[2];  // this CTA's (max, sum exp), alternating between rows
  __shared__ float s_zmax, s_a, s_q;  // the row's max, scale / sum, 1 - p of the target
  __shared__ int s_y;  // target id, -1 when the token is ignored
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const float scale = kGrad ? *scale_ptr : 0.f;
  const int nvec = V / E;
  const int crank = static_cast<int>(cta_rank_in_cluster());
  const int csize = static_cast<int>(ctas_in_cluster());
  const int cluster = static_cast<int>(blockIdx.x) / csize;
  const int nclusters = static_cast<int>(gridDim.x) / csize;
  const int per = (nvec + csize - 1) / csize;   // vectors per CTA slice
  const int v0 = min(nvec, crank * per), v1 = min(nvec, v0 + per);
  const bool last = crank == csize - 1;        // also owns the scalar tail

  int it = 0;
  int yl_next = cluster < N ? labels[cluster] : 0;  // each row's label is read a row ahead
  for (int row = cluster; row < N; row += nclusters, ++it) {
    const uint8_t* zr = z + static_cast<int64_t>(row) * ld_bytes;
    const int yl = yl_next;
    if (row + nclusters < N) yl_next = labels[row + nclusters];
    const int yt = (yl != ignore_index && yl >= 0 && yl < V) ? yl : -1;  // target, or -1
    float m = -INFINITY, s = 0.f;
    // pass 1: running max (the target included) and sum of exponentials (the
    // target's term left out) over this CTA's slice
    int v = v0 + tid;
    for (; v + (kUnroll - 1) * kCeThreads < v1; v += kUnroll * kCeThreads) {
      float x[kUnroll][E];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        VT::load(zr + static_cast<int64_t>(v + u * kCeThreads) * 16, x[u]);
      float cm = m;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
#pragma unroll
        for (int e = 0; e < E; ++e) cm = fmaxf(cm, x[u][e]);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int base = (v + u * kCeThreads) * E;
        if (static_cast<unsigned>(yt - base) < static_cast<unsigned>(E)) {
#pragma unroll
          for (int e = 0; e < E; ++e)
            if (base + e == yt) x[u][e] = -INFINITY;
        }
      }
      const float ms = cm * kLog2e;
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
#pragma unroll
        for (int e = 0; e < E; ++e) acc += ex2a(fmaf(x[u][e], kLog2e, -ms));
      s = s * ex2a((m - cm) * kLog2e) + acc;
      m = cm;
    }
    for (; v < v1; v += kCeThreads) {
      float x[E];
      VT::load(zr + static_cast<int64_t>(v) * 16, x);
      float cm = m;
#pragma unroll
      for (int e = 0; e < E; ++e) cm = fmaxf(cm, x[e]);
      const int base = v * E;
      if (static_cast<unsigned>(yt - base) < static_cast<unsigned>(E)) {
#pragma unroll
        for (int e = 0; e < E; ++e)
          if (base + e == yt) x[e] = -INFINITY;
      }
      const float ms = cm * kLog2e;
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc += ex2a(fmaf(x[e], kLog2e, -ms));
      s = s * ex2a((m - cm) * kLog2e) + acc;
      m = cm;
    }
    if (last) {
      for (int i = nvec * E + tid; i < V; i += kCeThreads) {
        const float x = VT::load1(zr + static_cast<int64_t>(i) * kElt);
        lse_merge(m, s, x, i == yt ? 0.f : 1.f);
      }
    }
    // block merge: warp shuffles, then the first warp
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      lse_merge(m, s, m2, s2);
    }
    if (lane == 0) s_red[warp] = make_float2(m, s);
    __syncthreads();
    if (warp == 0) {
      float2 r = lane < kCeThreads / 32 ? s_red[lane] : make_float2(-INFINITY, 0.f);
      m = r.x;
      s = r.y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        lse_merge(m, s, m2, s2);
      }
      if (lane == 0) s_part[it & 1] = make_float2(m, s);
    }
    // The target logit is read before the cluster barrier: after it, peers may
    // overwrite their slices with the gradient (in place).
    float zt = 0.f;
    if (tid == 0 && yt >= 0) zt = VT::load1(zr + static_cast<int64_t>(yt) * kElt);
    // cluster merge through distributed shared memory
    cluster_barrier();
    RowStat rs;
    if (tid == 0) {
      float M = -INFINITY, S = 0.f;
      for (int r = 0; r < csize; ++r) {
        const float2 pr = ld_dsmem_f2(&s_part[it & 1], static_cast<uint32_t>(r));
        lse_merge(M, S, pr.x, pr.y);
      }
      rs = row_grad(M, S, zt, yt >= 0, scale);
      s_zmax = M;
      s_a = rs.a;
      s_q = rs.q;
      s_y = yt;
    }
    __syncthreads();
    if (tid == 0 && crank == 0) {  // the loss, off the gradient pass's critical path
      float lse, nll;
      row_loss(rs, lse, nll);
      if (lse_out != nullptr) lse_out[row] = lse;
      nll_out[row] = nll;
    }
    if constexpr (kGrad) {
      // pass 2: dZ = (exp(z - lse) - [v = y]) * scale over this CTA's slice, as
      // exp(z - M) * scale / S off the target and -scale * (1 - p) at it
      const float zmax = s_zmax, a = s_a;
      const int y = s_y;
      const float gt = y >= 0 ? -scale * s_q : 0.f;
      uint8_t* gr = g + static_cast<int64_t>(row) * gld_bytes;
      for (int w = v0 + tid; w < v1; w += kCeThreads) {
        float x[E];
        VT::load(zr + static_cast<int64_t>(w) * 16, x);
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] = ex2a((x[e] - zmax) * kLog2e) * a;
        const int base = w * E;
        if (static_cast<unsigned>(y - base) < static_cast<unsigned>(E)) {
#pragma unroll
          for (int e = 0; e < E; ++e)
            if (base + e == y) x[e] = gt;
        }
        VT::store(gr + static_cast<int64_t>(w) * 16, x);
      }
      if (last) {
        for (int i = nvec * E + tid; i < V; i += kCeThreads) {
          float x = ex2a((VT::load1(zr + static_cast<int64_t>(i) * kElt) - zmax) * kLog2e) * a;
          if (i == y) x = gt;
          VT::store1(gr + static_cast<int64_t>(i) * kElt, x);
        }
      }
    }
    __syncthreads();  // s_red and the row's values in shared memory are reused
  }
  // No CTA leaves while a peer may still read its s_part through the cluster.
  cluster_barrier();
}

// ---- shared-memory staged variant ---------------------------------------------

// Slices of at most 110 KB with one CTA per SM (fp32 rows of 501 KB on clusters
// of 5 rather than 6: more clusters resident, one barrier fewer per row), or
// (bf16 rows, whose passes carry twice the exponentials per byte) at most 56 KB
// with two CTAs per SM, so that one CTA's reduction overlaps the other's
// gradient writes.
constexpr int kSliceOne = 110 * 1024;
constexpr int kSliceTwo = 56 * 1024;
constexpr int kBulkPiece = 16 * 1024;      // bytes per bulk copy instruction

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool wait_phase_bounded(uint32_t bar, uint32_t parity,
                                                   uint64_t timeout_ns) {
  uint32_t done = 0;
  uint64_t t0 = 0;
  for (int i = 0;; ++i) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if (i == 0) t0 = globaltimer_ns();
    else if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// One row per cluster of CTAs; CTA r holds vectors [v0, v1) of every row it
// visits in shared memory. Buffer (it & 1) receives row `it` of this cluster;
// the copy of row it + 1 is issued before row it is reduced.
template <int kBf16, bool kGrad, int kSlice, int kMinB>
__global__ void __launch_bounds__(kCeThreads, kMinB)
    ce_rows_staged_kernel(const uint8_t* z, int64_t ld_bytes,  // may alias g (in place)
                          const int32_t* __restrict__ labels, int N, int V, int ignore_index,
                          const float* __restrict__ scale_ptr, float* __restrict__ lse_out,
                          float* __restrict__ nll_out, uint8_t* g, int64_t gld_bytes,
                          int32_t* status, int64_t timeout_ns) {
  using VT = Vec16<kBf16>;
  constexpr int E = VT::E;
  constexpr int kElt = kBf16 ? 2 : 4;
  extern __shared__ __align__(128) uint8_t ce_smem[];
  __shared__ __align__(8) uint64_t s_bar[2];
  // per-row exchange: every CTA of the cluster stores its (max, sum exp, target
  // logit if the label is in its slice) into slot [row parity][its rank] of every
  // CTA, counted on that CTA's s_xbar[row parity]
  __shared__ __align__(8) uint64_t s_xbar[2];
  __shared__ __align__(16) float4 s_msg[2][kMaxCeCluster];
  __shared__ float2 s_red[kCeThreads / 32];
  // the row's -max * log2 e, that plus log2 |scale / sum| (bf16 rows), scale / sum and
  // 1 - p of the target
  __shared__ float s_nm2, s_c, s_a, s_q;
  __shared__ float s_zt;  // the target logit, when it lies in this CTA's slice
  __shared__ int s_y;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const float scale = kGrad ? *scale_ptr : 0.f;
  const int nvec = V / E;
  const int crank = static_cast<int>(cta_rank_in_cluster());
  const int csize = static_cast<int>(ctas_in_cluster());
  const int cluster = static_cast<int>(blockIdx.x) / csize;
  const int nclusters = static_cast<int>(gridDim.x) / csize;
  const int per = (nvec + csize - 1) / csize;
  const int v0 = min(nvec, crank * per), v1 = min(nvec, v0 + per);
  const int nv = v1 - v0;                      // vectors in this CTA's slice
  const uint32_t slice_bytes = static_cast<uint32_t>(nv) * 16u;
  const bool last = crank == csize - 1;
  uint8_t* buf[2] = {ce_smem, ce_smem + kSlice};
  const uint32_t bar0 = smem_addr(&s_bar[0]), bar1 = smem_addr(&s_bar[1]);
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar1) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&s_xbar[0])) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&s_xbar[1])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  cluster_barrier();  // every CTA's exchange barriers exist before any peer stores to them

  // thread 0: expect the slice's bytes on the buffer's barrier and copy it
  auto issue = [&](int row, int b) {
    const uint32_t bar = b ? bar1 : bar0;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(slice_bytes)
                 : "memory");
    const uint8_t* src = z + static_cast<int64_t>(row) * ld_bytes + static_cast<int64_t>(v0) * 16;
    const uint32_t dst = smem_addr(buf[b]);
    for (uint32_t off = 0; off < slice_bytes; off += kBulkPiece) {
      const uint32_t n = min(static_cast<uint32_t>(kBulkPiece), slice_bytes - off);
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              dst + off),
          "l"(src + off), "r"(n), "r"(bar)
          : "memory");
    }
  };

  int it = 0;
  int row = cluster;
  if (tid == 0 && row < N && nv > 0) issue(row, 0);
  bool timed_out = false;
  int yl_next = row < N ? labels[row] : 0;  // each row's label is read a row ahead
  for (; row < N; row += nclusters, ++it) {
    const int b = it & 1;
    const uint8_t* zr = z + static_cast<int64_t>(row) * ld_bytes;
    // the next row's slice streams into the other buffer meanwhile (its last
    // reader, the previous row, finished at the end of the previous iteration)
    if (tid == 0 && row + nclusters < N && nv > 0) issue(row + nclusters, b ^ 1);
    if (nv > 0 && !wait_phase_bounded(b ? bar1 : bar0, static_cast<uint32_t>((it >> 1) & 1),
                                      static_cast<uint64_t>(timeout_ns)))
      timed_out = true;
    uint8_t* sl = buf[b];
    const int yl = yl_next;
    if (row + nclusters < N) yl_next = labels[row + nclusters];
    const int yt = (yl != ignore_index && yl >= 0 && yl < V) ? yl : -1;  // target, or -1
    // The target's element, when it lies in this slice, is read by one thread in
    // both loops of pass 1: that thread keeps z_t, counts it in its maximum and
    // sets it to -inf in the staged copy, so that no sum (and no branch in the
    // loops) includes it; the gradient pass writes the target's entry itself.
    const int vt = (yt >= v0 * E && yt < v1 * E) ? yt / E - v0 : -1;  // its vector in the slice
    const bool own = vt >= 0 && vt % kCeThreads == tid;
    uint8_t* const tgt = sl + (own ? static_cast<int64_t>(yt - v0 * E) * kElt : 0);
    // pass 1: max (the target included) and sum of exponentials (the target's
    // term left out) over the staged slice
    float m = -INFINITY, s = 0.f;
    if constexpr (kBf16) {
      // The thread's maximum first, two elements per packed compare (exact on
      // bf16), then the sum of exponentials against that one maximum: a second
      // read of shared memory instead of an fp32 compare and a running rescale
      // per element.
      uint32_t pm0 = kBf16NegInf2, pm1 = kBf16NegInf2;
#pragma unroll 4
      for (int v = tid; v < nv; v += kCeThreads) {
        const uint4 w = *reinterpret_cast<const uint4*>(sl + static_cast<int64_t>(v) * 16);
        pm0 = bf16x2_max(pm0, bf16x2_max(w.x, w.y));
        pm1 = bf16x2_max(pm1, bf16x2_max(w.z, w.w));
      }
      pm0 = bf16x2_max(pm0, pm1);
      m = fmaxf(bf16_lo(pm0), bf16_hi(pm0));
      if (own) {   // after the maximum, before the sum (this thread reads it in both)
        const uint16_t bits = *reinterpret_cast<const uint16_t*>(tgt);
        s_zt = __uint_as_float(static_cast<uint32_t>(bits) << 16);
        *reinterpret_cast<uint16_t*>(tgt) = 0xFF80u;   // -inf
      }
      if (m != -INFINITY) {
        const float ms = m * kLog2e;
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 2
        for (int v = tid; v < nv; v += kCeThreads) {
          const uint4 w = *reinterpret_cast<const uint4*>(sl + static_cast<int64_t>(v) * 16);
          acc0 += ex2a(fmaf(bf16_lo(w.x), kLog2e, -ms)) + ex2a(fmaf(bf16_hi(w.x), kLog2e, -ms));
          acc1 += ex2a(fmaf(bf16_lo(w.y), kLog2e, -ms)) + ex2a(fmaf(bf16_hi(w.y), kLog2e, -ms));
          acc0 += ex2a(fmaf(bf16_lo(w.z), kLog2e, -ms)) + ex2a(fmaf(bf16_hi(w.z), kLog2e, -ms));
          acc1 += ex2a(fmaf(bf16_lo(w.w), kLog2e, -ms)) + ex2a(fmaf(bf16_hi(w.w), kLog2e, -ms));
        }
        s = acc0 + acc1;
      }
    } else {
      if (own) {   // before the online loop: its maximum starts at z_t
        m = *reinterpret_cast<const float*>(tgt);
        s_zt = m;
        *reinterpret_cast<float*>(tgt) = -INFINITY;
      }
      constexpr int kU = 2;
      int v = tid;
      for (; v + (kU - 1) * kCeThreads < nv; v += kU * kCeThreads) {
        float x[kU][E];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const uint4 w = *reinterpret_cast<const uint4*>(sl + static_cast<int64_t>(v + u * kCeThreads) * 16);
          x[u][0] = __uint_as_float(w.x); x[u][1] = __uint_as_float(w.y);
          x[u][2] = __uint_as_float(w.z); x[u][3] = __uint_as_float(w.w);
        }
        float cm = m;
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
          for (int e = 0; e < E; ++e) cm = fmaxf(cm, x[u][e]);
        const float ms = cm * kLog2e;
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
          for (int e = 0; e < E; ++e) acc += ex2a(fmaf(x[u][e], kLog2e, -ms));
        if (cm != -INFINITY) {
          s = s * ex2a((m - cm) * kLog2e) + acc;
          m = cm;
        }
      }
      for (; v < nv; v += kCeThreads) {
        const uint4 w = *reinterpret_cast<const uint4*>(sl + static_cast<int64_t>(v) * 16);
        float x[E];
        x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
        x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
        float cm = m;
#pragma unroll
        for (int e = 0; e < E; ++e) cm = fmaxf(cm, x[e]);
        if (cm == -INFINITY) continue;
        const float ms = cm * kLog2e;
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc += ex2a(fmaf(x[e], kLog2e, -ms));
        s = s * ex2a((m - cm) * kLog2e) + acc;
        m = cm;
      }
    }
    if (last) {
      for (int i = nvec * E + tid; i < V; i += kCeThreads) {
        const float x = VT::load1(zr + static_cast<int64_t>(i) * kElt);
        lse_merge(m, s, x, i == yt ? 0.f : 1.f);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      lse_merge(m, s, m2, s2);
    }
    if (lane == 0) s_red[warp] = make_float2(m, s);
    __syncthreads();
    RowStat rs;
    if (warp == 0) {
      float2 r = lane < kCeThreads / 32 ? s_red[lane] : make_float2(-INFINITY, 0.f);
      m = r.x;
      s = r.y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        lse_merge(m, s, m2, s2);
      }
      if (lane == 0) {  // tid 0: send this CTA's part of the row to every CTA
        const int y = yt;
        const bool valid = yt >= 0;
        // the target logit, from this CTA's staged slice (or its global tail),
        // so that no CTA reads a part of the row a peer may be overwriting
        float zt = 0.f;
        if (vt >= 0)
          zt = s_zt;   // written by its owner before the block barrier above
        else if (valid && last && y >= nvec * E)
          zt = VT::load1(zr + static_cast<int64_t>(y) * kElt);
        const int k = it & 1;
        for (int r = 0; r < csize; ++r)
          st_async_f4(&s_msg[k][crank], &s_xbar[k], static_cast<uint32_t>(r),
                      make_float4(m, s, zt, 0.f));
        const uint32_t xb = smem_addr(&s_xbar[k]);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(xb),
                     "r"(static_cast<uint32_t>(16 * csize))
                     : "memory");
        if (!wait_phase_bounded(xb, static_cast<uint32_t>((it >> 1) & 1),
                                static_cast<uint64_t>(timeout_ns)))
          timed_out = true;
        float M = -INFINITY, S = 0.f, ZT = 0.f;
        for (int r = 0; r < csize; ++r) {
          const float4 pr = s_msg[k][r];
          lse_merge(M, S, pr.x, pr.y);
          ZT += pr.z;
        }
        rs = row_grad(M, S, ZT, valid, scale);
        s_nm2 = -M * kLog2e;
        if constexpr (kBf16) {
          float lg;   // log2 |a|; -inf for a = 0 (an ignored token)
          asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(fabsf(rs.a)));
          s_c = s_nm2 + lg;
        }
        s_a = rs.a;
        s_q = rs.q;
        s_y = yt;
      }
    }
    __syncthreads();
    if (tid == 0 && crank == 0) {  // the loss, off the gradient pass's critical path
      float lse, nll;
      row_loss(rs, lse, nll);
      if (lse_out != nullptr) lse_out[row] = lse;
      nll_out[row] = nll;
    }
    if constexpr (kGrad) {
      // pass 2: dZ = (exp(z - lse) - [v = y]) * scale from the staged slice, as
      // exp(z - M) * a off the target (a = scale / S) and -scale * (1 - p) at it.
      // Off the target the exponent is one FMA, with log2 |a| folded in for bf16
      // rows and a's sign applied to the packed pair: the rounding of those row
      // constants is a common relative error of about 1e-6 per entry, and the
      // target's entry, where a difference would lose it, does not use them.
      const float nm2 = s_nm2, a = s_a;
      const int y = s_y;
      const float gt = y >= 0 ? -scale * s_q : 0.f;
      uint8_t* gr = g + static_cast<int64_t>(row) * gld_bytes;
      if constexpr (kBf16) {
        const float c = s_c;
        const uint32_t sgn = a < 0.f ? 0x80008000u : 0u;
        const float gt_pre = sgn ? -gt : gt;   // the pair's sign flip restores it
        for (int v = tid; v < nv; v += kCeThreads) {
          const uint4 w = *reinterpret_cast<const uint4*>(sl + static_cast<int64_t>(v) * 16);
          float x[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                        bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = ex2a(fmaf(x[e], kLog2e, c));
          const int base = (v0 + v) * 8;
          if (static_cast<unsigned>(y - base) < 8u) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (base + e == y) x[e] = gt_pre;
          }
          *reinterpret_cast<uint4*>(gr + static_cast<int64_t>(v0 + v) * 16) =
              make_uint4(pack_bf16(x[0], x[1]) ^ sgn, pack_bf16(x[2], x[3]) ^ sgn,
                         pack_bf16(x[4], x[5]) ^ sgn, pack_bf16(x[6], x[7]) ^ sgn);
        }
      } else {
        for (int v = tid; v < nv; v += kCeThreads) {
          const uint4 w = *reinterpret_cast<const uint4*>(sl + static_cast<int64_t>(v) * 16);
          float x[4] = {__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                        __uint_as_float(w.w)};
#pragma unroll
          for (int e = 0; e < 4; ++e) x[e] = ex2a(fmaf(x[e], kLog2e, nm2)) * a;
          const int base = (v0 + v) * 4;
          if (static_cast<unsigned>(y - base) < 4u) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (base + e == y) x[e] = gt;
          }
          VT::store(gr + static_cast<int64_t>(v0 + v) * 16, x);
        }
      }
      if (last) {
        for (int i = nvec * E + tid; i < V; i += kCeThreads) {
          float x = ex2a(fmaf(VT::load1(zr + static_cast<int64_t>(i) * kElt), kLog2e, nm2)) * a;
          if (i == y) x = gt;
          VT::store1(gr + static_cast<int64_t>(i) * kElt, x);
        }
      }
    }
    __syncthreads();  // the buffer, s_red and the row's values in shared memory are reused
  }
  if (timed_out && status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, 9);
  cluster_barrier();
}

template <int kBf16, bool kGrad, int kSlice, int kMinB>
cudaError_t launch_rows_staged(int cluster, int grid, const uint8_t* z, int64_t ld_bytes,
                               const int32_t* labels, int N, int V, int ignore_index,
                               const float* scale, float* lse, float* nll, uint8_t* g,
                               int64_t gld_bytes, int32_t* status, int64_t timeout_ns,
                               cudaStream_t stream) {
  auto kern = ce_rows_staged_kernel<kBf16, kGrad, kSlice, kMinB>;
  constexpr int smem = 2 * kSlice;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kCeThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent clusters: launch only as many as can be resident at once (a
  // cluster that had to wait for a free GPC would run its rows after the rest)
  int active = 0;
  if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) == cudaSuccess && active > 0 &&
      active * cluster < grid)
    cfg.gridDim = dim3(static_cast<unsigned>(active * cluster), 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, z, ld_bytes, labels, N, V, ignore_index, scale, lse, nll,
                            g, gld_bytes, status, timeout_ns);
}

template <int kBf16, bool kGrad>
cudaError_t launch_rows(int cluster, int grid, const uint8_t* z, int64_t ld_bytes,
                        const int32_t* labels, int N, int V, int ignore_index, const float* scale,
                        float* lse, float* nll, uint8_t* g, int64_t gld_bytes,
                        cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kCeThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ce_rows_kernel<kBf16, kGrad>, z, ld_bytes, labels, N, V,
                            ignore_index, scale, lse, nll, g, gld_bytes);
}

}  // namespace

cudaError_t launch_ce_count(const int32_t* labels, int N, int V, int ignore_index, int reduction,
                            float grad_scale, float normalizer, float* scale, int32_t* status,
                            cudaStream_t stream) {
  ce_count_kernel<<<1, kCountThreads, 0, stream>>>(labels, N, V, ignore_index, reduction,
                                                   grad_scale, normalizer, scale, status);
  return cudaGetLastError();
}

cudaError_t launch_ce_rows(int bf16, const void* z, int64_t ld_bytes, const int32_t* labels,
                           int N, int V, int ignore_index, const float* scale, float* lse,
                           float* nll, void* g, int64_t gld_bytes, int sms, int32_t* status,
                           int64_t timeout_ns, cudaStream_t stream) {
  // Rows of 64-880 KB: slices staged in shared memory by a cluster of
  // ceil(row / slice) CTAs (at most eight).
  const int64_t vec_bytes = static_cast<int64_t>(V / (bf16 ? 8 : 4)) * 16;
  auto cluster_for = [&](int64_t slice) -> int {
    if (vec_bytes < (64 << 10) || vec_bytes > 8 * slice) return 0;
    int cl = static_cast<int>((vec_bytes + slice - 1) / slice);
    // the slices are whole 16-byte vectors: make sure the rounding up of the
    // per-CTA vector count keeps every slice within one buffer
    while (cl < 8 && ((vec_bytes / 16 + cl - 1) / cl) * 16 > slice) ++cl;
    return ((vec_bytes / 16 + cl - 1) / cl) * 16 <= slice ? cl : 0;
  };
  const uint8_t* zp = static_cast<const uint8_t*>(z);
  uint8_t* gp = static_cast<uint8_t*>(g);
  auto clusters = [&](int cl, int per_sm) {
    int ncl = per_sm * sms / cl;
    if (ncl > N) ncl = N;
    return ncl < 1 ? 1 : ncl;
  };
  if (int cl = bf16 ? cluster_for(kSliceTwo) : 0) {
    const int grid = clusters(cl, 2) * cl;
    return g ? launch_rows_staged<1, true, kSliceTwo, 2>(cl, grid, zp, ld_bytes, labels, N, V,
                                                         ignore_index, scale, lse, nll, gp,
                                                         gld_bytes, status, timeout_ns, stream)
             : launch_rows_staged<1, false, kSliceTwo, 2>(cl, grid, zp, ld_bytes, labels, N, V,
                                                          ignore_index, scale, lse, nll, gp,
                                                          gld_bytes, status, timeout_ns, stream);
  }
  if (int cl = cluster_for(kSliceOne)) {
    const int grid = clusters(cl, 1) * cl;
    if (bf16)
      return g ? launch_rows_staged<1, true, kSliceOne, 1>(cl, grid, zp, ld_bytes, labels, N, V,
                                                           ignore_index, scale, lse, nll, gp,
                                                           gld_bytes, status, timeout_ns, stream)
               : launch_rows_staged<1, false, kSliceOne, 1>(cl, grid, zp, ld_bytes, labels, N,
                                                            V, ignore_index, scale, lse, nll, gp,
                                                            gld_bytes, status, timeout_ns, stream);
    return g ? launch_rows_staged<0, true, kSliceOne, 1>(cl, grid, zp, ld_bytes, labels, N, V,
                                                         ignore_index, scale, lse, nll, gp,
                                                         gld_bytes, status, timeout_ns, stream)
             : launch_rows_staged<0, false, kSliceOne, 1>(cl, grid, zp, ld_bytes, labels, N, V,
                                                          ignore_index, scale, lse, nll, gp,
                                                          gld_bytes, status, timeout_ns, stream);
  }
  // Cluster size: slices of about 256 KB of a row per CTA, at least two CTAs for
  // rows over 128 KB, at most eight; two CTAs per SM (the register budget of a
  // 512-thread CTA), rounded down to whole clusters, no more clusters than rows.
  // Measured on the 8192 x 128256 logits: clusters of 2 beat 1, 3 and 4 for both
  // fp32 and bf16 rows (smaller slices pay the per-row cluster barrier).
  const int64_t row_bytes = static_cast<int64_t>(V) * (bf16 ? 2 : 4);
  int cluster = static_cast<int>((row_bytes + (256 << 10) - 1) / (256 << 10));
  if (row_bytes > (128 << 10) && cluster < 2) cluster = 2;
  cluster = cluster < 1 ? 1 : (cluster > 8 ? 8 : cluster);
  const int grid = clusters(cluster, 2) * cluster;
  cudaError_t e;
  if (bf16) {
    e = g ? launch_rows<1, true>(cluster, grid, zp, ld_bytes, labels, N, V, ignore_index, scale,
                                 lse, nll, gp, gld_bytes, stream)
          : launch_rows<1, false>(cluster, grid, zp, ld_bytes, labels, N, V, ignore_index, scale,
                                  lse, nll, gp, gld_bytes, stream);
  } else {
    e = g ? launch_rows<0, true>(cluster, grid, zp, ld_bytes, labels, N, V, ignore_index, scale,
                                 lse, nll, gp, gld_bytes, stream)
          : launch_rows<0, false>(cluster, grid, zp, ld_bytes, labels, N, V, ignore_index, scale,
                                  lse, nll, gp, gld_bytes, stream);
  }
  return e;
}

}  // namespace flce
