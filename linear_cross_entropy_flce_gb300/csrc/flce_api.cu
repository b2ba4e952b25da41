// C ABI of the fused linear cross-entropy library (declared in include/flce.h):
// argument checks, the workspace plan, tensor-map encoding and the stream-ordered
// launch sequence.
//
// Launch sequence of flce_forward_backward (all on the caller's stream):
//   1. LSE GEMM   Z = H W^T, online max/sum-exp per (token block, vocabulary
//                 range) and the target logit      ("Liger Kernel: Fused Triton
//                 Kernels for LLM Training", The Architecture, 1.)
//   2. merge      per-token lse and NLL from the partials
//   3. reduce     n_valid, label check, loss, gradient scale (one block, fixed order)
//   4. for each token block b, for each vocabulary chunk c:
//        GRAD GEMM  recompute Z_bc, write G_bc = (softmax - onehot) * scale in bf16
//        dH + dW    one launch of both products (same page, 2.):
//                   dH_b  (+)= G_bc W_c     (fp32 accumulator over the chunks)
//                   dW_c  (+)= G_bc^T H_b   (fixed order over token blocks)
//      then, with several chunks, the rounding of the block's dH accumulator to bf16
// Nothing of size N x V is ever written: the largest buffer is one G chunk.
// flce_forward runs steps 1-3. On one vocabulary shard, flce_forward_shard runs
// step 1 with global label ids, a merge into the shard's (m, s, zt) and step 3
// for the label check; flce_backward_shard runs step 3 for the scale and step 4
// from the caller's combined lse, accumulating its dH part in fp32.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/flce.h"
#include "flce_internal.h"

namespace flce {
namespace {

constexpr int64_t kDefaultTimeoutNs = 2000000000LL;
constexpr size_t kGChunkCapBytes = size_t(256) << 20;  // planned bf16 G chunk
constexpr int kMaxDevices = 64;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct DeviceInfo {
  bool init = false;
  int status = FLCE_OK;
  int sms = 0;
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

int device_info(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLCE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FLCE_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0, count = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      return FLCE_ERR_CUDA;
    }
    d.status = (major == 10 && minor == 3) ? FLCE_OK : FLCE_ERR_DEVICE;
    d.sms = count;
    d.init = true;
  }
  *sms = d.sms;
  return d.status;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
  });
  return fn;
}

// bf16 matrix [outer][inner] (inner contiguous, row stride ld elements), read in
// boxes of box_inner x box_outer with 128-byte swizzle; out-of-range elements
// read as zero.
bool encode_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                 uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output map of the GEMM epilogue's TMA stores: [rows][cols] row-major with row
// stride ld elements, boxes of 32 x 32; fp32 boxes use the 128-byte swizzle and
// bf16 boxes the 64-byte one (the layouts the epilogue stages in shared memory).
// Stores outside [rows) x [cols) are dropped, which clips ragged tiles.
bool encode_out(CUtensorMap* m, const void* base, bool bf16, uint64_t cols, uint64_t rows,
                uint64_t ld) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const uint64_t esz = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * esz};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  bf16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The bf16 G chunk is stored chunk-major, [v_chunk/64][rows][64]: the 64 vocabulary
// ids of one K block of the dH product, or one 64-wide MN chunk of the dW product,
// are contiguous for a run of rows, so each copy of a consumer reads whole
// contiguous blocks (8-16 KB) instead of 128-byte pieces of rows v_chunk·2 bytes
// apart. Three views of it: the gradient epilogue's 32 x 32 store boxes, the
// K-major A operand of dH (64 ids x 128 rows per box) and the MN-major A operand of
// dW (64 ids x 64 rows x 2 chunks per box).
bool encode_g_chunked(CUtensorMap* m, void* G, uint64_t rows, uint64_t v_chunk, uint32_t box_x,
                      uint32_t box_y, uint32_t box_z, bool sw64) {
  auto fn = encode_fn();
  if (fn == nullptr || v_chunk % 64 != 0) return false;
  cuuint64_t dims[3] = {64, rows, v_chunk / 64};
  cuuint64_t strides[2] = {128, rows * 128};
  cuuint32_t box[3] = {box_x, box_y, box_z};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, G, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  sw64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  sw64 ? CU_TENSOR_MAP_L2_PROMOTION_NONE : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tiles are computed by cluster pairs (tcgen05 cta_group::2, 256-row tiles).
constexpr int kCtaGroup = 2;
// The dW and dH products (K = the token block / the vocabulary chunk, 8192 and
// 16032 at the Llama-3-8B head) run 256 x 512 tiles: a quarter fewer operand bytes
// per flop and fewer distinct operand rows per wave, for an epilogue that no longer
// overlaps the next tile (about 1% of a tile that long). Requested together they
// share one launch, dH's tiles first, because dH alone has too few wide tiles to
// fill the pairs (256 for 76 pairs at the Llama-3-8B head: a last wave 37% full);
// dH alone keeps 256 x 256 tiles.
constexpr bool kWideDw = true;
constexpr bool kWideDhAlone = false;

// MN-major bf16 operand [rows][mn] (mn contiguous, mn % 64 == 0, row stride ld
// elements) as a 3-D map [mn/64][rows][64] read in boxes of 64 x box_rows x
// box_chunks with 128-byte swizzle. The view covers exactly the 2-D tensor, so
// every address it can form lies inside it; rows past the end read as zero.
bool encode_bf16_mn3(CUtensorMap* m, const void* base, uint64_t mn, uint64_t rows, uint64_t ld,
                     uint32_t box_rows, uint32_t box_chunks) {
  auto fn = encode_fn();
  if (fn == nullptr || mn % 64 != 0) return false;
  cuuint64_t dims[3] = {64, rows, mn / 64};
  cuuint64_t strides[2] = {ld * 2, 128};
  cuuint32_t box[3] = {64, box_rows, box_chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct Plan {
  int64_t N = 0, D = 0, V = 0;
  int cta = kCtaGroup;  // CTAs per tile
  int tile_m = BM * kCtaGroup;
  int m_blocks = 0;     // ceil(N / tile_m): row tiles of the forward pass
  int part_stride = 0;  // 128-row blocks per vocabulary range in the partials
  int v_tiles = 0;    // ceil(V / BN)
  int splits = 0;     // forward vocabulary ranges per token block
  int64_t n_block = 0, v_chunk = 0;
  int n_nblocks = 0, n_chunks = 0;
  bool need_dh_acc = false, need_dw_acc = false;
  size_t off_part = 0, off_zt = 0, off_nll = 0, off_lse = 0, off_scal = 0, off_gstat = 0,
         off_g = 0, off_dhacc = 0, off_dwacc = 0, total = 0;
};

int choose_splits(int m_blocks, int v_tiles, int sms) {
  // Minimise (waves of units) x (tiles per unit); ties go to fewer splits.
  int best = 1;
  int64_t best_cost = INT64_MAX;
  const int max_s = std::min(v_tiles, 128);
  for (int s = 1; s <= max_s; ++s) {
    const int64_t waves = ceil_div(static_cast<int64_t>(m_blocks) * s, sms);
    const int64_t cost = waves * ceil_div(v_tiles, s);
    if (cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// backward = false: only the forward pieces (partials, target logits, NLL, lse,
// scalars); the G chunk and the dH / dW accumulators are left out of the total.
int make_plan(int64_t N, int64_t D, int64_t V, const flce_options& o, int sms, Plan* P,
              bool backward = true) {
  Plan p;
  p.N = N;
  p.D = D;
  p.V = V;
  p.m_blocks = static_cast<int>(ceil_div(N, p.tile_m));
  p.part_stride = p.m_blocks * p.cta;
  p.v_tiles = static_cast<int>(ceil_div(V, BN));
  if (o.v_splits < 0 || o.v_splits > p.v_tiles) return FLCE_ERR_OPTION;
  p.splits = o.v_splits > 0 ? o.v_splits
                            : choose_splits(p.m_blocks, p.v_tiles, std::max(1, sms / p.cta));

  const int64_t v_round = ceil_div(V, BN) * BN;
  if (o.v_chunk < 0 || o.n_block < 0) return FLCE_ERR_OPTION;
  if (o.v_chunk > 0 && o.v_chunk % BN != 0) return FLCE_ERR_OPTION;
  if (o.n_block > 0 && o.n_block % BM != 0) return FLCE_ERR_OPTION;
  // Planned G chunk: vocabulary chunks of at most 16384 ids, balanced in length
  // (a chunk's dH accumulation and launch ramp are paid per chunk, so fewer,
  // longer chunks are faster); the tokens form one block unless one chunk of G
  // would exceed kGChunkCapBytes, in which case they are split into equal
  // blocks of whole 256-row pair tiles. Measured on GB300: long-sequence head
  // 99.7 -> 93.9 ms with half the workspace, Llama-2-like head 1.93 -> 1.40 ms.
  int64_t cv = o.v_chunk, nb = o.n_block;
  if (cv == 0) {
    const int64_t chunks = ceil_div(V, 16384);
    cv = ceil_div(ceil_div(V, chunks), BN) * BN;
  }
  if (nb == 0) {
    const int64_t bytes = ceil_div(N, BM * 2) * (BM * 2) * cv * 2;
    const int64_t blocks = std::max<int64_t>(1, ceil_div(bytes, static_cast<int64_t>(kGChunkCapBytes)));
    nb = blocks == 1 ? N : ceil_div(ceil_div(N, blocks), BM * 2) * (BM * 2);
  }
  cv = std::min(cv, v_round);
  nb = std::min(nb, N);
  p.v_chunk = cv;
  p.n_block = nb;
  p.n_chunks = static_cast<int>(ceil_div(V, cv));
  p.n_nblocks = static_cast<int>(ceil_div(N, nb));
  p.need_dh_acc = p.n_chunks > 1;
  p.need_dw_acc = (o.dw_dtype == FLCE_DTYPE_BF16) && p.n_nblocks > 1;

  const int64_t rows_b = ceil_div(nb, p.tile_m) * p.tile_m;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  p.off_part = take(static_cast<size_t>(p.splits) * p.part_stride * BM * sizeof(float2));
  p.off_zt = take(static_cast<size_t>(N) * 4);
  p.off_nll = take(static_cast<size_t>(N) * 4);
  p.off_lse = take(static_cast<size_t>(N) * 4);
  p.off_scal = take(256);
  if (backward) {
    p.off_gstat = take(static_cast<size_t>(N) * 16);   // float4 per token
    p.off_g = take(static_cast<size_t>(rows_b) * cv * 2);
    p.off_dhacc = p.need_dh_acc ? take(static_cast<size_t>(rows_b) * D * 4) : off;
    p.off_dwacc = p.need_dw_acc ? take(static_cast<size_t>(V) * D * 4) : off;
  } else {
    p.off_gstat = p.off_g = p.off_dhacc = p.off_dwacc = off;
  }
  p.total = off;
  *P = p;
  return FLCE_OK;
}

int check_options(const flce_options& o) {
  if (o.reduction != FLCE_REDUCTION_MEAN && o.reduction != FLCE_REDUCTION_SUM &&
      o.reduction != FLCE_REDUCTION_NONE)
    return FLCE_ERR_OPTION;
  if (o.dw_dtype != FLCE_DTYPE_F32 && o.dw_dtype != FLCE_DTYPE_BF16) return FLCE_ERR_OPTION;
  if (!(o.normalizer >= 0.f) || !(o.grad_scale == o.grad_scale)) return FLCE_ERR_OPTION;
  if (o.timeout_ns < 0) return FLCE_ERR_OPTION;
  if (o.trace_capacity < 0 || (o.trace_capacity > 0 && o.trace_events == nullptr) ||
      o.reserved != 0)
    return FLCE_ERR_OPTION;
  return FLCE_OK;
}

int check_shape(int64_t N, int64_t D, int64_t V) {
  if (N < 1 || D < 1 || V < 1) return FLCE_ERR_SHAPE;
  // int32 coordinates and indices inside the kernels
  if (N > (int64_t(1) << 30) || V > (int64_t(1) << 30) || D > (int64_t(1) << 20))
    return FLCE_ERR_SHAPE;
  if (D % 8 != 0) return FLCE_ERR_ALIGN;
  return FLCE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Fp8 carries the E4M3 operands of the FP8 variant (null for the bf16 path):
// they feed the two logits products; H and W (bf16) feed the gradient products.
struct Fp8Operands {
  const uint8_t* H8 = nullptr;
  const uint8_t* W8 = nullptr;
  const float* scale_h = nullptr;  // device fp32 scalars
  const float* scale_w = nullptr;
};

// A call on one vocabulary shard, rows [v_offset, v_offset + V) of a vocabulary of
// V_total ids (V_total == 0: an ordinary call over the whole vocabulary). The
// forward writes the shard's per-token (m, s, zt); the backward takes the combined
// lse and writes the shard's fp32 part of dH and its rows of dW.
struct Shard {
  int64_t v_offset = 0;
  int64_t V_total = 0;
  float* m = nullptr;
  float* s = nullptr;
  float* zt = nullptr;
  const float* lse_in = nullptr;
  float* dh_f32 = nullptr;
};

// uint8 matrix [outer][inner] read in boxes of box_inner x box_outer bytes with
// 128-byte swizzle; out-of-range elements read as zero.
bool encode_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
               uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int run(const uint16_t* H, const uint16_t* W, const Fp8Operands& f8, const int32_t* labels,
        int64_t N, int64_t D, int64_t V, const flce_options* opt_in, float* loss, float* lse_out,
        uint16_t* dH, void* dW, bool backward, void* workspace, size_t ws_bytes, int32_t* status,
        void* stream_v, const Shard& sh = Shard{}) {
  flce_options o;
  flce_default_options(&o);
  if (opt_in != nullptr) o = *opt_in;
  const bool fp8 = f8.H8 != nullptr || f8.W8 != nullptr;
  if (!backward) {
    dH = nullptr;
    dW = nullptr;
  }
  const bool shard = sh.V_total > 0;
  // the backward of a shard writes fp32 dH parts instead of bf16 dH
  const bool want_dh = dH != nullptr || (shard && backward && sh.dh_f32 != nullptr);
  const bool need_bf16 = !fp8 || want_dh || dW != nullptr;
  if (labels == nullptr || (!shard && loss == nullptr) || workspace == nullptr)
    return FLCE_ERR_NULL;
  if (shard) {
    if (backward ? (sh.lse_in == nullptr || (!want_dh && dW == nullptr))
                 : (sh.m == nullptr || sh.s == nullptr || sh.zt == nullptr))
      return FLCE_ERR_NULL;
    if (sh.v_offset < 0 || sh.V_total > (int64_t(1) << 30) || sh.v_offset + V > sh.V_total)
      return FLCE_ERR_SHAPE;
    const uintptr_t a4 = reinterpret_cast<uintptr_t>(sh.m) | reinterpret_cast<uintptr_t>(sh.s) |
                         reinterpret_cast<uintptr_t>(sh.zt) | reinterpret_cast<uintptr_t>(sh.lse_in);
    if ((a4 & 3u) || (sh.dh_f32 && !aligned16(sh.dh_f32))) return FLCE_ERR_ALIGN;
  }
  // labels are ids of the whole vocabulary
  const int64_t V_lab = shard ? sh.V_total : V;
  const int64_t v_base = shard ? sh.v_offset : 0;   // id of W's row 0
  if (fp8 && (f8.H8 == nullptr || f8.W8 == nullptr)) return FLCE_ERR_NULL;
  if (need_bf16 && (H == nullptr || W == nullptr)) return FLCE_ERR_NULL;
  int rc = check_shape(N, D, V);
  if (rc != FLCE_OK) return rc;
  rc = check_options(o);
  if (rc != FLCE_OK) return rc;
  if (fp8 && (D % 16 != 0 || !aligned16(f8.H8) || !aligned16(f8.W8))) return FLCE_ERR_ALIGN;
  if (fp8 && (f8.scale_h == nullptr || f8.scale_w == nullptr)) return FLCE_ERR_NULL;
  if (fp8 && ((reinterpret_cast<uintptr_t>(f8.scale_h) & 3u) ||
              (reinterpret_cast<uintptr_t>(f8.scale_w) & 3u)))
    return FLCE_ERR_ALIGN;
  if ((H && !aligned16(H)) || (W && !aligned16(W)) || !aligned16(labels) ||
      !aligned16(workspace) ||
      (lse_out && !aligned16(lse_out)) || (dH && !aligned16(dH)) || (dW && !aligned16(dW)) ||
      (reinterpret_cast<uintptr_t>(loss) & 3u) || (reinterpret_cast<uintptr_t>(status) & 3u))
    return FLCE_ERR_ALIGN;
  int sms = 0;
  rc = device_info(&sms);
  if (rc != FLCE_OK) return rc;
  Plan P;
  rc = make_plan(N, D, V, o, sms, &P, backward);
  if (rc != FLCE_OK) return rc;
  if (ws_bytes < P.total) return FLCE_ERR_WORKSPACE;
  if (backward && o.reduction == FLCE_REDUCTION_NONE) {
    return FLCE_ERR_OPTION;  // a per-token loss needs a per-token upstream gradient
  }
  const bool per_token = o.reduction == FLCE_REDUCTION_NONE;

  cudaStream_t st = static_cast<cudaStream_t>(stream_v);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float2* part = reinterpret_cast<float2*>(ws + P.off_part);
  float* zt = reinterpret_cast<float*>(ws + P.off_zt);
  // reduction "none": the merge writes each token's loss straight to the caller
  float* nll = per_token ? loss : reinterpret_cast<float*>(ws + P.off_nll);
  float* loss_scalar =
      (per_token || shard) ? reinterpret_cast<float*>(ws + P.off_scal + 8) : loss;
  float* lse = lse_out ? lse_out : reinterpret_cast<float*>(ws + P.off_lse);
  float* scal = reinterpret_cast<float*>(ws + P.off_scal);  // [0] scale
  int32_t* nvalid = reinterpret_cast<int32_t*>(ws + P.off_scal + 4);
  // per token (max, 1 / sum exp, 1 - p of the target) for the gradient epilogue;
  // a shard's backward has only the caller's combined lse
  float4* gstat = (backward && !shard) ? reinterpret_cast<float4*>(ws + P.off_gstat) : nullptr;
  uint16_t* G = reinterpret_cast<uint16_t*>(ws + P.off_g);
  float* dh_acc = reinterpret_cast<float*>(ws + P.off_dhacc);
  float* dw_acc = reinterpret_cast<float*>(ws + P.off_dwacc);
  const int64_t tmo = o.timeout_ns > 0 ? o.timeout_ns : kDefaultTimeoutNs;

  if (status != nullptr && cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess)
    return FLCE_ERR_CUDA;
  // Optional per-kernel trace: event 0 before the first kernel, event k after kernel k.
  int n_traced = 0;
  auto trace = [&]() -> bool {
    if (o.trace_events == nullptr || n_traced >= o.trace_capacity) return true;
    const bool ok = cudaEventRecord(static_cast<cudaEvent_t>(o.trace_events[n_traced]), st) ==
                    cudaSuccess;
    ++n_traced;
    return ok;
  };
  if (!trace()) return FLCE_ERR_CUDA;

  const int cta = P.cta;
  const int pairs = std::max(1, sms / cta);
  // Operands of the two logits products: bf16 H, W, or E4M3 H8, W8 (128 bytes =
  // 128 elements per stage row).
  CUtensorMap mH_k, mW_k;
  if (fp8) {
    if (!encode_u8(&mH_k, f8.H8, D, N, D, 2 * BK, BM) ||
        !encode_u8(&mW_k, f8.W8, D, V, D, 2 * BK, static_cast<uint32_t>(BN / cta)))
      return FLCE_ERR_CUDA;
  } else if (!encode_bf16(&mH_k, H, D, N, D, BK, BM) ||
             !encode_bf16(&mW_k, W, D, V, D, BK, static_cast<uint32_t>(BN / cta))) {
    return FLCE_ERR_CUDA;
  }
  const int k_blocks_z = static_cast<int>(ceil_div(D, fp8 ? 2 * BK : BK));
  const uint32_t idesc_z = fp8 ? make_idesc_e4m3_f32(P.tile_m, BN) : make_idesc_bf16_f32(P.tile_m, BN, 0, 0);


  // ---- 1. forward LSE GEMM (the backward of a shard starts from the given lse) ----
  if (!(shard && backward)) {
    GemmParams g{};
    g.a_mn_major = 0;
    g.b_mn_major = 0;
    g.m_blocks = P.m_blocks;
    g.n_blocks = P.v_tiles;
    g.k_blocks = k_blocks_z;
    g.acc_scale_h = f8.scale_h;
    g.acc_scale_w = f8.scale_w;
    g.splits = P.splits;
    g.part_stride = P.part_stride;
    g.num_units = P.splits * P.m_blocks;
    g.group_m = std::min(P.m_blocks, 16);
    g.idesc = idesc_z;
    g.timeout_ns = tmo;
    g.status = status;
    g.m_valid = static_cast<int>(N);
    g.n_valid = static_cast<int>(V);
    g.labels = labels;
    g.row_base = 0;
    g.col_base = static_cast<int>(v_base);
    g.ignore_index = o.ignore_index;
    g.part = part;
    g.zt = zt;
    if (launch_gemm_lse(cta, mH_k, mW_k, g, cta * std::min(g.num_units, pairs), st, fp8 ? 1 : 0) !=
            cudaSuccess ||
        !trace())
      return FLCE_ERR_CUDA;

    // ---- 2. merge: lse and NLL, or a shard's (m, s, zt) ----
    const cudaError_t me =
        shard ? launch_shard_merge(part, zt, labels, static_cast<int>(N), static_cast<int>(v_base),
                                   static_cast<int>(v_base + V), P.part_stride, P.splits,
                                   o.ignore_index, sh.m, sh.s, sh.zt, st)
              : launch_lse_merge(part, zt, labels, static_cast<int>(N), static_cast<int>(V),
                                 P.part_stride, P.splits, o.ignore_index, lse, nll, gstat, st);
    if (me != cudaSuccess || !trace()) return FLCE_ERR_CUDA;
  }
  // ---- 3. reduce: label check, n, the gradient scale and (not for shards) the loss ----
  if (launch_loss_reduce(shard ? nullptr : nll, labels, static_cast<int>(N),
                         static_cast<int>(V_lab), o.ignore_index,
                         per_token ? FLCE_REDUCTION_SUM : o.reduction, o.grad_scale,
                         o.normalizer, loss_scalar, scal, nvalid, status,
                         st) != cudaSuccess ||
      !trace())
    return FLCE_ERR_CUDA;
  if (!want_dh && dW == nullptr) return FLCE_OK;
  const float* lse_g = shard ? sh.lse_in : lse;   // the lse the gradient is formed from

  // ---- 4. backward, token block outer, vocabulary chunk inner ----
  const int64_t rows_b = ceil_div(P.n_block, P.tile_m) * P.tile_m;
  // MN-major operands: one 3-D copy per CTA when the MN extent is a multiple of
  // 64 (always for the G chunk), else 64-wide 2-D boxes.
  CUtensorMap mH_mn, mW_mn, mG_mn, mG_k, mG_out;
  const bool d_box3 = D % 64 == 0;
  const uint32_t b_chunks = static_cast<uint32_t>(BN / cta / 64);
  const bool ok_h = d_box3 ? encode_bf16_mn3(&mH_mn, H, D, N, D, BK, b_chunks)
                           : encode_bf16(&mH_mn, H, D, N, D, 64, BK);
  const bool ok_w = d_box3 ? encode_bf16_mn3(&mW_mn, W, D, V, D, BK, b_chunks)
                           : encode_bf16(&mW_mn, W, D, V, D, 64, BK);
  if (!ok_h || !ok_w || !encode_g_chunked(&mG_mn, G, rows_b, P.v_chunk, 64, BK, BM / 64, false) ||
      !encode_g_chunked(&mG_k, G, rows_b, P.v_chunk, 64, BM, 1, false) ||
      !encode_g_chunked(&mG_out, G, rows_b, P.v_chunk, 32, 32, 1, true))
    return FLCE_ERR_CUDA;
  const bool dw_bf16 = o.dw_dtype == FLCE_DTYPE_BF16;
  // dW goes to fp32 dW, to bf16 dW (one token block), or to the fp32 accumulator
  // that bf16 dW is rounded from after the last token block.
  const bool dw_direct_bf16 = dw_bf16 && P.n_nblocks == 1;

  for (int b = 0; b < P.n_nblocks; ++b) {
    const int64_t b0 = static_cast<int64_t>(b) * P.n_block;
    const int nb_len = static_cast<int>(std::min<int64_t>(P.n_block, N - b0));
    for (int c = 0; c < P.n_chunks; ++c) {
      const int64_t c0 = static_cast<int64_t>(c) * P.v_chunk;
      const int c_len = static_cast<int>(std::min<int64_t>(P.v_chunk, V - c0));

      // G chunk: recompute Z_bc and form (softmax - onehot) * scale in bf16.
      GemmParams q{};
      q.a_mn_major = 0;
      q.b_mn_major = 0;
      q.a_mn0 = static_cast<int>(b0);
      q.b_mn0 = static_cast<int>(c0);
      q.m_blocks = static_cast<int>(ceil_div(nb_len, P.tile_m));
      q.n_blocks = static_cast<int>(ceil_div(c_len, BN));
      q.k_blocks = k_blocks_z;
      q.acc_scale_h = f8.scale_h;
      q.acc_scale_w = f8.scale_w;
      q.num_units = q.m_blocks * q.n_blocks;
      q.group_m = std::min(q.m_blocks, 16);
      q.idesc = idesc_z;
      q.timeout_ns = tmo;
      q.status = status;
      q.m_valid = nb_len;
      q.n_valid = c_len;
      q.labels = labels;
      q.row_base = static_cast<int>(b0);
      q.col_base = static_cast<int>(v_base + c0);
      q.ignore_index = o.ignore_index;
      q.lse = lse_g;
      q.gstat = gstat;
      q.scale = scal;
      q.out_row0 = 0;
      if (launch_gemm_grad(cta, mH_k, mW_k, mG_out, q, cta * std::min(q.num_units, pairs), st,
                           fp8 ? 1 : 0) !=
              cudaSuccess ||
          !trace())
        return FLCE_ERR_CUDA;

      const bool both = dW != nullptr && want_dh;
      GemmArgs aw{}, ah{};
      if (dW != nullptr) {
        // dW rows [c0, c0 + c_len) (+)= G_bc^T H_b: M = vocabulary, N = hidden, K = tokens.
        GemmParams& w = aw.p;
        w.a_mn_major = 1;
        w.b_mn_major = 1;
        w.a_box3 = 1;
        w.b_box3 = d_box3 ? 1 : 0;
        w.b_k0 = static_cast<int>(b0);
        w.m_blocks = static_cast<int>(ceil_div(c_len, P.tile_m));
        w.n_blocks = static_cast<int>(ceil_div(D, kWideDw ? 2 * BN : BN));
        w.k_blocks = static_cast<int>(ceil_div(nb_len, BK));
        w.num_units = w.m_blocks * w.n_blocks;
        w.group_m = std::min(w.m_blocks, 8);
        // every second tile of a pair walks K backwards, so a wave starts on the K
        // blocks the previous wave read last (still in L2); on the Llama-3-8B head
        // (N 8192, D 4096, 16128-id chunks) 19% fewer DRAM reads per launch
        w.k_serpentine = 1;
        w.idesc = make_idesc_bf16_f32(P.tile_m, BN, 1, 1);
        w.timeout_ns = tmo;
        w.status = status;
        w.m_valid = c_len;
        w.n_valid = static_cast<int>(D);
        // the map holds exactly the chunk's rows, so ragged tiles are clipped
        const int64_t dw_off = c0 * D;
        void* dw_base = dw_direct_bf16 ? static_cast<void*>(static_cast<uint16_t*>(dW) + dw_off)
                        : dw_bf16      ? static_cast<void*>(dw_acc + dw_off)
                                       : static_cast<void*>(static_cast<float*>(dW) + dw_off);
        if (!encode_out(&aw.c, dw_base, dw_direct_bf16, D, c_len, D)) return FLCE_ERR_CUDA;
        aw.a = mG_mn;
        aw.b = mH_mn;
        w.out_row0 = 0;
        w.out_mode = dw_direct_bf16 ? OUT_STORE_BF16 : (b == 0 ? OUT_STORE_F32 : OUT_ADD_F32);
      }

      const bool wide_dh = both || kWideDhAlone;
      if (want_dh) {
        // dH rows [b0, b0 + nb_len) (+)= G_bc W_c: M = tokens, N = hidden, K = vocabulary.
        GemmParams& h = ah.p;
        h.a_mn_major = 0;
        h.a_kchunk = 1;
        h.b_mn_major = 1;
        h.b_box3 = d_box3 ? 1 : 0;
        h.b_k0 = static_cast<int>(c0);
        h.m_blocks = static_cast<int>(ceil_div(nb_len, P.tile_m));
        h.n_blocks = static_cast<int>(ceil_div(D, wide_dh ? 2 * BN : BN));
        h.k_blocks = static_cast<int>(ceil_div(c_len, BK));
        h.num_units = h.m_blocks * h.n_blocks;
        h.group_m = std::min(h.m_blocks, 8);
        h.k_serpentine = 1;   // as for dW (9% fewer DRAM reads on the same head)
        h.idesc = make_idesc_bf16_f32(P.tile_m, BN, 0, 1);
        h.timeout_ns = tmo;
        h.status = status;
        h.m_valid = nb_len;
        h.n_valid = static_cast<int>(D);
        // one chunk: bf16 dH directly; else an fp32 accumulator of this token
        // block's rows (stored by chunk 0, reduce-added by the others), rounded
        // to bf16 after the last chunk. The map holds exactly the block's rows.
        // A shard accumulates straight into its fp32 dH part.
        const bool dh_direct = P.n_chunks == 1 && !shard;
        const bool ok_dh = shard ? encode_out(&ah.c, sh.dh_f32 + b0 * D, false, D, nb_len, D)
                           : dh_direct ? encode_out(&ah.c, dH + b0 * D, true, D, nb_len, D)
                                       : encode_out(&ah.c, dh_acc, false, D, nb_len, D);
        if (!ok_dh) return FLCE_ERR_CUDA;
        ah.a = mG_k;
        ah.b = mW_mn;
        h.out_row0 = 0;
        h.out_mode = dh_direct ? OUT_STORE_BF16 : (c == 0 ? OUT_STORE_F32 : OUT_ADD_F32);
      }
      // dW and dH both read only G (and H, W), and write different outputs
      cudaError_t ge = cudaSuccess;
      if (both) {
        const int units = ah.p.num_units + aw.p.num_units;
        ge = launch_gemm_f32_pair(cta, ah, aw, cta * std::min(units, pairs), st);
      } else if (dW != nullptr) {
        ge = launch_gemm_f32(cta, aw.a, aw.b, aw.c, aw.p, cta * std::min(aw.p.num_units, pairs),
                             st, kWideDw ? 1 : 0);
      } else if (want_dh) {
        ge = launch_gemm_f32(cta, ah.a, ah.b, ah.c, ah.p, cta * std::min(ah.p.num_units, pairs),
                             st, wide_dh ? 1 : 0);
      }
      if (ge != cudaSuccess || ((dW != nullptr || want_dh) && !trace())) return FLCE_ERR_CUDA;
    }
    if (dH != nullptr && !shard && P.n_chunks > 1 &&
        (launch_f32_to_bf16(dh_acc, dH + b0 * D, static_cast<int64_t>(nb_len) * D, sms, st) !=
             cudaSuccess ||
         !trace()))
      return FLCE_ERR_CUDA;
  }
  if (dW != nullptr && dw_bf16 && !dw_direct_bf16 &&
      (launch_f32_to_bf16(dw_acc, static_cast<uint16_t*>(dW), V * D, sms, st) != cudaSuccess ||
       !trace()))
    return FLCE_ERR_CUDA;
  return FLCE_OK;
}

int workspace_bytes(int64_t N, int64_t D, int64_t V, const flce_options* opt, bool backward,
                    size_t* bytes) {
  if (bytes == nullptr) return FLCE_ERR_NULL;
  flce_options o;
  flce_default_options(&o);
  if (opt != nullptr) o = *opt;
  int rc = flce::check_shape(N, D, V);
  if (rc != FLCE_OK) return rc;
  rc = flce::check_options(o);
  if (rc != FLCE_OK) return rc;
  // The vocabulary-range split count depends on the SM count; plan for the
  // largest split count that choose_splits can return so that the size does not
  // depend on the device (and can be asked for without one).
  flce_options big = o;
  if (big.v_splits == 0) big.v_splits = static_cast<int32_t>(std::min<int64_t>(
                                            flce::ceil_div(V, flce::BN), 128));
  flce::Plan P;
  rc = flce::make_plan(N, D, V, big, 1, &P, backward);
  if (rc != FLCE_OK) return rc;
  *bytes = P.total;
  return FLCE_OK;
}

}  // namespace
}  // namespace flce

extern "C" {

void flce_default_options(flce_options* opt) {
  if (opt == nullptr) return;
  std::memset(opt, 0, sizeof(*opt));
  opt->ignore_index = -100;
  opt->reduction = FLCE_REDUCTION_MEAN;
  opt->grad_scale = 1.0f;
  opt->normalizer = 0.0f;
  opt->dw_dtype = FLCE_DTYPE_F32;
  opt->timeout_ns = 0;
}

int flce_workspace_size(int64_t N, int64_t D, int64_t V, const flce_options* opt, size_t* bytes) {
  return flce::workspace_bytes(N, D, V, opt, true, bytes);
}

int flce_forward_workspace_size(int64_t N, int64_t D, int64_t V, const flce_options* opt,
                                size_t* bytes) {
  return flce::workspace_bytes(N, D, V, opt, false, bytes);
}

int flce_get_plan(int64_t N, int64_t D, int64_t V, const flce_options* opt, int32_t want_dh,
                  int32_t want_dw, flce_plan_info* info) {
  if (info == nullptr) return FLCE_ERR_NULL;
  flce_options o;
  flce_default_options(&o);
  if (opt != nullptr) o = *opt;
  int rc = flce::check_shape(N, D, V);
  if (rc != FLCE_OK) return rc;
  rc = flce::check_options(o);
  if (rc != FLCE_OK) return rc;
  size_t ws = 0;
  rc = flce_workspace_size(N, D, V, &o, &ws);
  if (rc != FLCE_OK) return rc;
  int sms = 0;
  rc = flce::device_info(&sms);
  if (rc != FLCE_OK) return rc;
  flce::Plan P;
  rc = flce::make_plan(N, D, V, o, sms, &P, want_dh != 0 || want_dw != 0);
  if (rc != FLCE_OK) return rc;
  info->n_block = P.n_block;
  info->v_chunk = P.v_chunk;
  info->n_blocks = P.n_nblocks;
  info->n_chunks = P.n_chunks;
  info->v_splits = P.splits;
  // LSE GEMM, merge, reduce; per token block: per chunk the gradient GEMM and
  // one launch of the dW and / or dH products asked for, then (several chunks) the
  // bf16 rounding of dH; bf16 dW over several token blocks: one rounding of its
  // accumulator at the end.
  const int per_chunk = 1 + ((want_dh || want_dw) ? 1 : 0);
  const int per_block = P.n_chunks * per_chunk + ((want_dh && P.n_chunks > 1) ? 1 : 0);
  const bool dw_round = want_dw && o.dw_dtype == FLCE_DTYPE_BF16 && P.n_nblocks > 1;
  info->kernel_launches =
      3 + ((want_dh || want_dw) ? P.n_nblocks * per_block + (dw_round ? 1 : 0) : 0);
  info->workspace_bytes = ws;
  info->plan_bytes = P.total;
  return FLCE_OK;
}

int flce_ce_workspace_size(int64_t N, int64_t V, const flce_options* opt, size_t* bytes) {
  if (bytes == nullptr) return FLCE_ERR_NULL;
  flce_options o;
  flce_default_options(&o);
  if (opt != nullptr) o = *opt;
  if (N < 1 || V < 1 || N > (int64_t(1) << 30) || V > (int64_t(1) << 30)) return FLCE_ERR_SHAPE;
  const int rc = flce::check_options(o);
  if (rc != FLCE_OK) return rc;
  *bytes = 2 * flce::align_up(static_cast<size_t>(N) * 4, 256) + 256;
  return FLCE_OK;
}

int flce_ce_logits(const void* logits, int32_t dtype, int64_t ld, const int32_t* labels,
                   int64_t N, int64_t V, const flce_options* opt, float* loss, float* lse,
                   void* dlogits, int64_t dld, void* workspace, size_t ws_bytes, int32_t* status,
                   void* stream) {
  flce_options o;
  flce_default_options(&o);
  if (opt != nullptr) o = *opt;
  if (logits == nullptr || labels == nullptr || loss == nullptr || workspace == nullptr)
    return FLCE_ERR_NULL;
  if (N < 1 || V < 1 || N > (int64_t(1) << 30) || V > (int64_t(1) << 30)) return FLCE_ERR_SHAPE;
  int rc = flce::check_options(o);
  if (rc != FLCE_OK) return rc;
  if (dtype != FLCE_DTYPE_F32 && dtype != FLCE_DTYPE_BF16) return FLCE_ERR_OPTION;
  const int64_t elt = dtype == FLCE_DTYPE_BF16 ? 2 : 4;
  if (ld < V || (dlogits != nullptr && dld < V)) return FLCE_ERR_SHAPE;
  if ((ld * elt) % 16 != 0 || (dlogits != nullptr && (dld * elt) % 16 != 0)) return FLCE_ERR_ALIGN;
  if (!flce::aligned16(logits) || !flce::aligned16(labels) || !flce::aligned16(workspace) ||
      (dlogits && !flce::aligned16(dlogits)) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) ||
      (reinterpret_cast<uintptr_t>(loss) & 3u) || (reinterpret_cast<uintptr_t>(status) & 3u))
    return FLCE_ERR_ALIGN;
  if (dlogits == logits && dld != ld) return FLCE_ERR_OPTION;
  if (dlogits != nullptr && o.reduction == FLCE_REDUCTION_NONE) return FLCE_ERR_OPTION;
  size_t need = 0;
  rc = flce_ce_workspace_size(N, V, &o, &need);
  if (rc != FLCE_OK) return rc;
  if (ws_bytes < need) return FLCE_ERR_WORKSPACE;
  int sms = 0;
  rc = flce::device_info(&sms);
  if (rc != FLCE_OK) return rc;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t nb = flce::align_up(static_cast<size_t>(N) * 4, 256);
  const bool per_token = o.reduction == FLCE_REDUCTION_NONE;
  float* nll = per_token ? loss : reinterpret_cast<float*>(ws);
  float* lse_ws = reinterpret_cast<float*>(ws + nb);
  float* scal = reinterpret_cast<float*>(ws + 2 * nb);
  int32_t* nvalid = reinterpret_cast<int32_t*>(ws + 2 * nb + 4);
  float* loss_scalar = per_token ? reinterpret_cast<float*>(ws + 2 * nb + 8) : loss;
  if (status != nullptr && cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess)
    return FLCE_ERR_CUDA;
  int n_traced = 0;
  auto trace = [&]() -> bool {
    if (o.trace_events == nullptr || n_traced >= o.trace_capacity) return true;
    const bool ok = cudaEventRecord(static_cast<cudaEvent_t>(o.trace_events[n_traced]), st) ==
                    cudaSuccess;
    ++n_traced;
    return ok;
  };
  if (!trace()) return FLCE_ERR_CUDA;
  const int Ni = static_cast<int>(N), Vi = static_cast<int>(V);
  if (dlogits != nullptr &&
      (flce::launch_ce_count(labels, Ni, Vi, o.ignore_index, o.reduction, o.grad_scale,
                             o.normalizer, scal, status, st) != cudaSuccess ||
       !trace()))
    return FLCE_ERR_CUDA;
  if (flce::launch_ce_rows(dtype == FLCE_DTYPE_BF16 ? 1 : 0, logits, ld * elt, labels, Ni, Vi,
                           o.ignore_index, scal, lse ? lse : lse_ws, nll, dlogits, dld * elt, sms,
                           status, o.timeout_ns > 0 ? o.timeout_ns : flce::kDefaultTimeoutNs,
                           st) != cudaSuccess ||
      !trace())
    return FLCE_ERR_CUDA;
  if (flce::launch_loss_reduce(nll, labels, Ni, Vi, o.ignore_index,
                               per_token ? FLCE_REDUCTION_SUM : o.reduction, o.grad_scale,
                               o.normalizer, loss_scalar, scal + 3, nvalid, status,
                               st) != cudaSuccess ||
      !trace())
    return FLCE_ERR_CUDA;
  return FLCE_OK;
}

int flce_forward_backward(const uint16_t* H, const uint16_t* W, const int32_t* labels, int64_t N,
                          int64_t D, int64_t V, const flce_options* opt, float* loss, float* lse,
                          uint16_t* dH, void* dW, void* workspace, size_t ws_bytes,
                          int32_t* status, void* stream) {
  return flce::run(H, W, flce::Fp8Operands{}, labels, N, D, V, opt, loss, lse, dH, dW, true,
                   workspace, ws_bytes, status, stream);
}

int flce_forward(const uint16_t* H, const uint16_t* W, const int32_t* labels, int64_t N, int64_t D,
                 int64_t V, const flce_options* opt, float* loss, float* lse, void* workspace,
                 size_t ws_bytes, int32_t* status, void* stream) {
  return flce::run(H, W, flce::Fp8Operands{}, labels, N, D, V, opt, loss, lse, nullptr, nullptr,
                   false, workspace, ws_bytes, status, stream);
}

int flce_forward_shard(const uint16_t* H, const uint16_t* W_shard, const int32_t* labels,
                       int64_t N, int64_t D, int64_t V_shard, int64_t v_offset, int64_t V_total,
                       const flce_options* opt, float* m, float* s, float* zt, void* workspace,
                       size_t ws_bytes, int32_t* status, void* stream) {
  if (V_total < 1) return FLCE_ERR_SHAPE;
  flce::Shard sh;
  sh.v_offset = v_offset;
  sh.V_total = V_total;
  sh.m = m;
  sh.s = s;
  sh.zt = zt;
  return flce::run(H, W_shard, flce::Fp8Operands{}, labels, N, D, V_shard, opt, nullptr, nullptr,
                   nullptr, nullptr, false, workspace, ws_bytes, status, stream, sh);
}

int flce_backward_shard(const uint16_t* H, const uint16_t* W_shard, const int32_t* labels,
                        int64_t N, int64_t D, int64_t V_shard, int64_t v_offset, int64_t V_total,
                        const flce_options* opt, const float* lse, float* dH_part, void* dW_shard,
                        void* workspace, size_t ws_bytes, int32_t* status, void* stream) {
  if (V_total < 1) return FLCE_ERR_SHAPE;
  flce::Shard sh;
  sh.v_offset = v_offset;
  sh.V_total = V_total;
  sh.lse_in = lse;
  sh.dh_f32 = dH_part;
  return flce::run(H, W_shard, flce::Fp8Operands{}, labels, N, D, V_shard, opt, nullptr, nullptr,
                   nullptr, dW_shard, true, workspace, ws_bytes, status, stream, sh);
}

int flce_forward_fp8(const uint8_t* H8, const float* scale_h, const uint8_t* W8,
                     const float* scale_w,
                     const int32_t* labels, int64_t N, int64_t D, int64_t V,
                     const flce_options* opt, float* loss, float* lse, void* workspace,
                     size_t ws_bytes, int32_t* status, void* stream) {
  flce::Fp8Operands f8;
  f8.H8 = H8;
  f8.W8 = W8;
  f8.scale_h = scale_h;
  f8.scale_w = scale_w;
  return flce::run(nullptr, nullptr, f8, labels, N, D, V, opt, loss, lse, nullptr, nullptr, false,
                   workspace, ws_bytes, status, stream);
}

int flce_forward_backward_fp8(const uint8_t* H8, const float* scale_h, const uint8_t* W8,
                              const float* scale_w,
                              const uint16_t* H, const uint16_t* W, const int32_t* labels,
                              int64_t N, int64_t D, int64_t V, const flce_options* opt,
                              float* loss, float* lse, uint16_t* dH, void* dW, void* workspace,
                              size_t ws_bytes, int32_t* status, void* stream) {
  flce::Fp8Operands f8;
  f8.H8 = H8;
  f8.W8 = W8;
  f8.scale_h = scale_h;
  f8.scale_w = scale_w;
  return flce::run(H, W, f8, labels, N, D, V, opt, loss, lse, dH, dW, true, workspace, ws_bytes,
                   status, stream);
}

int flce_quantize_e4m3(const uint16_t* x, int64_t n, uint8_t* q, float* out, void* stream) {
  if (x == nullptr || q == nullptr || out == nullptr) return FLCE_ERR_NULL;
  if (n < 1) return FLCE_ERR_SHAPE;
  if (n % 8 != 0 || !flce::aligned16(x) || !flce::aligned16(q) ||
      (reinterpret_cast<uintptr_t>(out) & 7u))
    return FLCE_ERR_ALIGN;
  int sms = 0;
  const int rc = flce::device_info(&sms);
  if (rc != FLCE_OK) return rc;
  return flce::launch_quantize_e4m3(x, n, q, out, sms, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FLCE_OK
             : FLCE_ERR_CUDA;
}

int flce_scale_grads(uint16_t* dH, int64_t dh_elems, void* dW, int64_t dw_elems,
                     int32_t dw_dtype, const float* scale, void* stream) {
  if (scale == nullptr) return FLCE_ERR_NULL;
  if (dh_elems < 0 || dw_elems < 0) return FLCE_ERR_SHAPE;
  if ((dH == nullptr && dh_elems > 0) || (dW == nullptr && dw_elems > 0)) return FLCE_ERR_NULL;
  if (dw_dtype != FLCE_DTYPE_F32 && dw_dtype != FLCE_DTYPE_BF16) return FLCE_ERR_OPTION;
  const int64_t dw_bytes = dw_elems * (dw_dtype == FLCE_DTYPE_BF16 ? 2 : 4);
  if ((dh_elems * 2) % 16 != 0 || dw_bytes % 16 != 0) return FLCE_ERR_ALIGN;
  if ((dH && !flce::aligned16(dH)) || (dW && !flce::aligned16(dW)) ||
      (reinterpret_cast<uintptr_t>(scale) & 3u))
    return FLCE_ERR_ALIGN;
  int sms = 0;
  const int rc = flce::device_info(&sms);
  if (rc != FLCE_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dh_elems > 0 && flce::launch_scale(dH, dh_elems * 2, 1, scale, sms, st) != cudaSuccess)
    return FLCE_ERR_CUDA;
  if (dw_elems > 0 &&
      flce::launch_scale(dW, dw_bytes, dw_dtype == FLCE_DTYPE_BF16 ? 1 : 0, scale, sms, st) !=
          cudaSuccess)
    return FLCE_ERR_CUDA;
  return FLCE_OK;
}

int flce_check_status(const int32_t* status, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FLCE_ERR_CUDA;
  if (status == nullptr) return FLCE_OK;
  int32_t h = 0;
  if (cudaMemcpy(&h, status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FLCE_ERR_CUDA;
  return h;
}

const char* flce_status_string(int code) {
  switch (code) {
    case FLCE_OK: return "ok";
    case FLCE_ERR_NULL: return "a required pointer is NULL";
    case FLCE_ERR_SHAPE: return "N, D or V out of range";
    case FLCE_ERR_ALIGN: return "pointer not 16-byte aligned or D not a multiple of 8";
    case FLCE_ERR_WORKSPACE: return "workspace too small";
    case FLCE_ERR_OPTION: return "option out of range";
    case FLCE_ERR_CUDA: return "CUDA call failed";
    case FLCE_ERR_DEVICE: return "device is not an sm_103 GPU";
    case FLCE_ERR_LABEL_RANGE: return "a label is outside [0, V) and is not ignore_index";
    case FLCE_ERR_TIMEOUT: return "a device pipeline wait timed out";
    default: return "unknown status";
  }
}

}  // extern "C"
