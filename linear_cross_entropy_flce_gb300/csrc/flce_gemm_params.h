// Tile constants and launch parameters of the tcgen05 GEMM (flce_gemm.cuh),
// shared with the host code that plans and launches it.
#pragma once

#include <cuda.h>

#include <cstddef>
#include <cstdint>

#include <vector_types.h>

namespace flce {

constexpr int BM = 128;  // tile rows held by one CTA (tokens, or vocabulary ids for dW)
constexpr int BN = 256;  // tile columns
constexpr int BK = 64;   // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int UK = 16;   // K per tcgen05.mma for 16-bit inputs
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 2 * BN;         // two accumulators of BN fp32 columns
constexpr uint32_t kMnBoxBytes = 64 * BK * 2;  // one 64(MN) x 64(K) MN-major box

// Tile configuration. kCta = 1: one CTA computes a 128 x 256 tile. kCta = 2: a
// cluster pair computes a 256 x 256 tile with tcgen05 cta_group::2; each CTA holds
// its 128 rows of A and half (128 rows) of B, so each SM stages 32 KB per 64-deep K
// block instead of 48 KB.
// A ring stage holds kSub consecutive K blocks under one full/empty barrier pair.
// The MMA thread's wait and commit per stage cost about as much as one MMA, and the
// tensor pipe queues little work ahead, so with cta_group::2 two K blocks (eight
// MMAs) share each wait and commit; three 64 KB stages keep as many bytes in flight
// as six 32 KB ones.
// kWide = 1 (pair only): a 256 x 512 tile, two N = 256 MMAs per K step sharing the A
// block, one accumulator of all 512 TMEM columns. Each SM stages 48 KB per K block
// for twice the MMAs of a 32 KB block (a quarter fewer operand bytes per flop, and
// each wave of tiles touches fewer distinct operand rows), four stages of one K
// block (eight MMAs each); the epilogue no longer overlaps the next tile's MMAs,
// which only long-K products (dW, dH) can afford.
template <int kCta, int kWide = 0>
struct TileCfg {
  static_assert(kWide == 0 || kCta == 2, "the wide tile is a cluster-pair tile");
  static constexpr int kSub = kWide ? 1 : (kCta == 2 ? 2 : 1);   // K blocks per ring stage
  static constexpr int kStages = kWide ? 4 : (kCta == 2 ? 3 : 4);
  static constexpr int kTileM = BM * kCta;         // rows of the tile (both CTAs)
  static constexpr int kTileN = kWide ? 2 * BN : BN;  // columns of the tile
  static constexpr int kBHalves = kWide ? 2 : 1;   // N = 256 MMAs per K step
  static constexpr int kAccs = kWide ? 1 : 2;      // TMEM accumulators of kTileN columns
  static constexpr int kBRows = BN / kCta;         // rows of B (tile columns) per CTA and MMA
  static constexpr uint32_t kABytes = BM * BK * 2;
  static constexpr uint32_t kBHalfBytes = kBRows * BK * 2;
  static constexpr uint32_t kBBytes = kBHalves * kBHalfBytes;
  static constexpr uint32_t kSubBytes = kABytes + kBBytes;    // one K block, per CTA
  static constexpr uint32_t kStageBytes = kSub * kSubBytes;   // one ring stage, per CTA
  // Epilogue staging for TMA stores: two 4 KB boxes (32 rows x 128 bytes) per
  // epilogue warp, after the ring.
  static constexpr uint32_t kStgBytes = 4096;
  static constexpr uint32_t kRingBytes = kStages * kStageBytes;
  static constexpr size_t kSmemBytes = 1024 + kRingBytes + 4 * 2 * kStgBytes + 256;
  static_assert(kSmemBytes <= 232448, "more dynamic shared memory than a CTA may have");
};

constexpr float kLog2e = 1.4426950408889634f;

enum EpiKind { EPI_LSE = 0, EPI_GRAD = 1, EPI_F32 = 2 };
// Output of the fp32 epilogue through the output tensor map: store fp32, add fp32
// to what is there (TMA reduce-add), or store rounded to bf16.
enum OutMode { OUT_STORE_F32 = 0, OUT_ADD_F32 = 1, OUT_STORE_BF16 = 2 };

constexpr int kStatusTimeout = 9;  // FLCE_ERR_TIMEOUT

// Instruction descriptor for kind::f16 with bf16 A/B and an fp32 accumulator.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format (1 = bf16),
//   bit 15 A major (1 = MN-major), bit 16 B major, bits 17-22 N >> 3, bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t make_idesc_bf16_f32(int M, int N, int a_mn_major,
                                                           int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn_major & 1) << 15) |
         (static_cast<uint32_t>(b_mn_major & 1) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor for kind::f8f6f4 with E4M3 A/B (format code 0) and an
// fp32 accumulator: the same field positions as kind::f16.
__host__ __device__ constexpr uint32_t make_idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

struct GemmParams {
  // operand geometry: coordinates of tile (m, n, k) in the tensor maps are
  //   K-major  operand: x = k*BK + k0,         y = mn*BLOCK + mn0
  //   MN-major operand: x = mn*BLOCK + 64j + mn0, y = k*BK + k0
  int a_mn_major, b_mn_major;
  // MN-major operand given as a 3-D map [MN/64][K][64] (MN extent a multiple of 64):
  // one copy per CTA fills all of its 64-wide chunks; coordinate z = mn / 64.
  int a_box3, b_box3;
  // K-major A stored chunk-major, [K/64][rows][64] (the G chunk): one 3-D copy with
  // coordinates (0, row, k / 64) per K block.
  int a_kchunk;
  int a_mn0, a_k0, b_mn0, b_k0;
  int m_blocks, n_blocks, k_blocks;  // m_blocks counts tiles of TileCfg::kTileM rows
  int num_units;
  int splits;   // EPI_LSE: vocabulary ranges per row block
  int part_stride;  // EPI_LSE: 128-row blocks per vocabulary range in `part`
  int k_serpentine;  // 1: each CTA pair walks K backwards on every second tile it runs
  int group_m;  // tile raster: groups of group_m row blocks (EPI_LSE: units of a group
                // walk the vocabulary ranges together)
  int a_hint, b_hint;  // L2 policy of the A / B loads: 0 none, 1 evict_first, 2 evict_last
  uint32_t idesc;
  // FP8 operands: z = scale_h * scale_w * accumulator, the two scales read from
  // device memory once per epilogue thread
  const float* acc_scale_h;
  const float* acc_scale_w;
  int64_t timeout_ns;
  int32_t* status;
  int m_valid;  // rows of the product that exist
  int n_valid;  // columns of the product that exist
  // EPI_LSE / EPI_GRAD
  const int32_t* labels;  // labels[row_base + row]
  int row_base;
  int col_base;           // vocabulary id of product column 0
  int ignore_index;
  float2* part;           // EPI_LSE: [splits][part_stride][BM] (max, sum exp)
  float* zt;              // EPI_LSE: target logit per token
  const float* lse;       // EPI_GRAD: lse[row_base + row] (used when gstat is null)
  // EPI_GRAD: per token (max of z, 1 / sum exp(z - max), 1 - p of the target, 0):
  // G = exp(z - max) / sum * scale, and the target entry -scale * (1 - p) taken as
  // it is, with no difference of nearly equal numbers when p is close to 1
  const float4* gstat;
  const float* scale;     // EPI_GRAD: device scalar grad_scale / n
  // EPI_F32: the output map (third tensor map) holds product row r at map row
  // out_row0 + r, product column c at map column c; boxes of 32 x 32. EPI_GRAD: the
  // map is the chunk-major G, [columns/64][rows][64], boxes of 32 x 32 x 1.
  int out_row0;
  int out_mode;           // EPI_F32: OutMode (EPI_GRAD always stores bf16)
};

// Everything one product of a launch needs: the operand maps (A, B), the output
// map of the epilogue's TMA stores (C; unused by the LSE epilogue) and the
// parameters. A launch carries one or two of them (flce_gemm_kernel kProducts).
struct GemmArgs {  // aligned as CUtensorMap (128 bytes)
  CUtensorMap a, b, c;
  GemmParams p;
};

}  // namespace flce
