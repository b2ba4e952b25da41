// Persistent, warp-specialised tcgen05 GEMM for sm_103a with three fused
// epilogues. Every product of fused linear cross-entropy runs through it:
//
//   LSE  : Z = H W^T tile by tile, accumulated in TMEM; the epilogue keeps a
//          per-token running max and sum of exponentials (the target's own term
//          left out) across the vocabulary tiles of a work unit and extracts the
//          target logit ("Liger Kernel: Fused Triton Kernels for LLM Training",
//          The Architecture, 1. steps 2-5: in-SRAM tile product, online
//          LogSumExp, immediate target extraction, no logits written).
//   GRAD : Z recomputed tile by tile; the epilogue forms
//          G = (exp(z - lse) - [v = y]) * scale in bf16, as exp(z - max) * scale /
//          sum off the target and -scale * (1 - p) at it, and writes one chunk of
//          G, stored chunk-major (same page, 2. In-Kernel Gradient Computation:
//          recompute the tile logits from the saved LSE, derive dL/dz in the kernel).
//   F32  : plain product whose tile is stored as fp32, added to fp32 already in
//          memory, or stored as bf16 — used for dW = G^T H and dH = G W (same
//          page, 2.).
//
// CTA layout (192 threads, one CTA per SM). kCta = 1: each CTA computes a
// 128 x 256 tile. kCta = 2: a cluster pair computes a 256 x 256 tile with
// tcgen05 cta_group::2 MMAs; each CTA holds its 128 rows of A and 128 of the 256
// rows of B, and its own 128 x 256 fp32 accumulator rows in TMEM.
//   warp 0     : TMA producer (each CTA; all lanes wait, one elected lane issues)
//                — streams the CTA's A rows and B half, K-slice by K-slice, into a
//                ring of shared-memory stages; the copies of both CTAs complete on
//                the even CTA's stage barrier. With k_serpentine, every second tile
//                of a pair walks K from the end, so that it starts on the K slices
//                the tiles before it read last, which are the ones still in L2.
//   warp 1     : TMEM allocator (both CTAs) and MMA issuer (the even CTA's warp:
//                all lanes wait on the barriers, one elected lane issues the
//                tcgen05.mma M x 256 x 16 steps into one of two TMEM accumulators
//                and the commits).
//   warps 2..5 : epilogue — warp w reads TMEM lanes 32*(w%4) .. +31, so each
//                thread owns one output row of its CTA's 128 rows; tiles that
//                leave the SM go through per-warp 32 x 32 staging boxes in shared
//                memory and TMA stores (or reduce-adds).
// Every wait is bounded (see mbar_wait_bounded); on a timeout the CTA records
// FLCE_ERR_TIMEOUT, the producer drains the copies it issued, the MMA warp
// drains its MMAs, and both CTAs free TMEM and exit.
#pragma once

#include <cmath>
#include <cstdint>

#include "flce_gemm_params.h"
#include "ptx.cuh"

namespace flce {

// Units are ordered in groups of group_m row tiles; inside a group the column
// index (EPI_LSE: the vocabulary range) is the outer loop, so the tiles running at
// the same time share both their A row blocks and their B column blocks.
// Returns the column index (EPI_LSE: the vocabulary range) of unit u.
template <int kEpi>
__device__ __forceinline__ int unit_tiles(const GemmParams& p, int u, int& m_blk, int& n_begin,
                                          int& n_end) {
  const int n_units_per_row = (kEpi == EPI_LSE) ? p.splits : p.n_blocks;
  const int per_group = p.group_m * n_units_per_row;
  const int g = u / per_group;
  const int first_m = g * p.group_m;
  const int gm = min(p.m_blocks - first_m, p.group_m);
  const int r = u - g * per_group;
  const int col = r / gm;
  m_blk = first_m + (r - col * gm);
  if constexpr (kEpi == EPI_LSE) {
    n_begin = static_cast<int>((static_cast<int64_t>(col) * p.n_blocks) / p.splits);
    n_end = static_cast<int>((static_cast<int64_t>(col + 1) * p.n_blocks) / p.splits);
  } else {
    n_begin = col;
    n_end = col + 1;
  }
  return col;
}

__device__ __forceinline__ void record_status(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

// ---- epilogue bodies ---------------------------------------------------------------

struct LseState {
  float m;   // running max of z (the target's logit included)
  float s;   // running sum of exp(z - m) over every column but the target's
  float zt;  // target logit
  bool found;
};

// One 32-column chunk of the logits tile for this thread's row. The target's own
// term is left out of the sum (the merge adds it back), so that 1 - p of the
// target, the sum of the other terms over the whole sum, is known without a
// difference of nearly equal numbers.
__device__ __forceinline__ void lse_chunk(const float (&v)[32], int col_local, int n_valid,
                                          int rel_target, LseState& st) {
  float x[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) x[k] = v[k];
  if (col_local + 32 > n_valid) {
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (col_local + k >= n_valid) x[k] = -INFINITY;
  }
  float c0 = fmaxf(x[0], x[1]), c1 = fmaxf(x[2], x[3]);
#pragma unroll
  for (int k = 4; k < 32; k += 4) {
    c0 = fmaxf(c0, fmaxf(x[k], x[k + 1]));
    c1 = fmaxf(c1, fmaxf(x[k + 2], x[k + 3]));
  }
  const float mn = fmaxf(st.m, fmaxf(c0, c1));
  if (static_cast<unsigned>(rel_target) < 32u) {
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (k == rel_target) {
        st.zt = v[k];
        x[k] = -INFINITY;   // in the max above, not in the sum below
      }
    st.found = true;
  }
  if (mn == -INFINITY) return;
  const float ms = mn * kLog2e;
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int k = 0; k < 32; k += 4) {
    s0 += ex2_approx(fmaf(x[k + 0], kLog2e, -ms));
    s1 += ex2_approx(fmaf(x[k + 1], kLog2e, -ms));
    s2 += ex2_approx(fmaf(x[k + 2], kLog2e, -ms));
    s3 += ex2_approx(fmaf(x[k + 3], kLog2e, -ms));
  }
  st.s = st.s * ex2_approx((st.m - mn) * kLog2e) + ((s0 + s1) + (s2 + s3));
  st.m = mn;
}

// Epilogue staging. Each epilogue warp writes its 32 rows x 32 columns into a
// shared-memory box in the layout the output map's swizzle expects, then one lane
// hands the box to a TMA store: the global writes leave the SM as whole lines
// instead of one 16-byte piece of 32 different rows per store instruction.
//   fp32 box: rows of 128 bytes, 128-byte swizzle: 16-byte chunk q of row r sits
//             at chunk q ^ (r % 8);
//   bf16 box: rows of 64 bytes, 64-byte swizzle: chunk q of row r at q ^ ((r / 2) % 4).
__device__ __forceinline__ void stage_f32_row(uint32_t box, int r, const float (&v)[32]) {
  const uint32_t row = box + static_cast<uint32_t>(r) * 128u;
#pragma unroll
  for (int q = 0; q < 8; ++q)
    st_shared_v4(row + ((static_cast<uint32_t>(q ^ (r & 7))) << 4), __float_as_uint(v[4 * q]),
                 __float_as_uint(v[4 * q + 1]), __float_as_uint(v[4 * q + 2]),
                 __float_as_uint(v[4 * q + 3]));
}

__device__ __forceinline__ void stage_bf16_row(uint32_t box, int r, const float (&v)[32]) {
  const uint32_t row = box + static_cast<uint32_t>(r) * 64u;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    st_shared_v4(row + ((static_cast<uint32_t>(q ^ ((r >> 1) & 3))) << 4),
                 pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                 pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
}

// G for one 32-column chunk: (exp(z - zmax) * a - [v = y] * sc, 0 past n_valid,
// with a = sc / sum exp(z - zmax) (or zmax = lse and a = sc). The exponent's
// difference is taken first, exact when z is close to zmax. The target entry is
// -sc * q with q = 1 - p as the merge formed it, when q >= 0 is given; else
// (a vocabulary shard, which has only lse) exp(z - lse) * sc - sc.
__device__ __forceinline__ void grad_chunk(const float (&v)[32], int col_local, int n_valid,
                                           int rel_target, float zmax, float a, float sc,
                                           float q, float (&g)[32]) {
#pragma unroll
  for (int k = 0; k < 32; ++k) g[k] = ex2_approx((v[k] - zmax) * kLog2e) * a;
  if (static_cast<unsigned>(rel_target) < 32u) {
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (k == rel_target) g[k] = q >= 0.f ? -sc * q : g[k] - sc;
  }
  if (col_local + 32 > n_valid) {
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (col_local + k >= n_valid) g[k] = 0.f;
  }
}

// ---- the kernel --------------------------------------------------------------------

// kFp8 = 1: A and B are E4M3 bytes (K-major only), 128 of them per 128-byte
// stage row, multiplied with tcgen05 kind::f8f6f4; the epilogue scales z by
// the product of the two device scales. The shared-memory image of a stage is
// the same as for bf16.
// kWide = 1: 256 x 512 tiles (TileCfg): each CTA stages two 128-row halves of B
// per K block, the MMA thread issues one N = 256 MMA per half into columns
// [256 h, 256 h + 256) of the single accumulator, and tile column c is product
// column n_blk * 512 + c.
// kProducts = 2: one launch computes two independent products of the same tile
// shape and epilogue, g0's units first, then g1's (the dH and dW products of a
// vocabulary chunk, which both only read G). Units are dealt to the pairs in that
// fixed order, each unit taking its maps and parameters from its own product, so
// every output element still has one writer per launch.
template <int kEpi, int kCta, int kFp8 = 0, int kWide = 0, int kProducts = 1>
__global__ void __launch_bounds__(kThreads, 1)
    flce_gemm_kernel(const __grid_constant__ GemmArgs g0, const __grid_constant__ GemmArgs g1) {
  using Cfg = TileCfg<kCta, kWide>;
  static_assert(kWide == 0 || kEpi == EPI_F32, "wide tiles carry the fp32 epilogue only");
  static_assert(kProducts == 1 || kEpi == EPI_F32, "two products per launch: fp32 epilogue only");
  constexpr int kStages = Cfg::kStages;
  constexpr int kSub = Cfg::kSub;
  // settings shared by every unit of the launch come from the first product
  const GemmParams& p0 = g0.p;
  const int units0 = p0.num_units;
  const int total_units = units0 + (kProducts == 2 ? g1.p.num_units : 0);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kRingBytes + 8 * Cfg::kStgBytes);
  // bars: full[kStages] | empty[kStages] | tfull[2] | tempty[2] | drain
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = (kCta == 2) ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int pair = static_cast<int>(blockIdx.x) / kCta;
  const int num_pairs = static_cast<int>(gridDim.x) / kCta;
  const uint32_t stage0 = smem_u32(smem);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + kStages + s); };
  auto tfull_bar = [&](int a) { return smem_u32(bars + 2 * kStages + a); };
  auto tempty_bar = [&](int a) { return smem_u32(bars + 2 * kStages + 2 + a); };
  const uint32_t drain_bar = smem_u32(bars + 2 * kStages + 4);
  constexpr bool kCl = kCta == 2;  // waits acquire at cluster scope in pair mode

  if (threadIdx.x == 0) {
    // full[s] of the even CTA counts the copies of both CTAs of a pair (the odd
    // CTA's copies complete on it remotely); the odd CTA's full[s] is unused.
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4 * kCta);  // four epilogue warps per CTA
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&g0.a);
    tma_prefetch_desc(&g0.b);
    if constexpr (kEpi != EPI_LSE) tma_prefetch_desc(&g0.c);
    if constexpr (kProducts == 2) {
      tma_prefetch_desc(&g1.a);
      tma_prefetch_desc(&g1.b);
      tma_prefetch_desc(&g1.c);
    }
  }
  // Barriers of both CTAs are initialised before either CTA touches the other's.
  if constexpr (kCta == 2) cluster_sync();
  else __syncthreads();
  if (warp == 1) {
    tmem_alloc_cg<kCta>(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish_cg<kCta>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_holder);
  const uint64_t tmo = p0.timeout_ns;

  if (warp == 0) {
    // ---------------- TMA producer (each CTA loads its own A rows and B half) -----
    {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_par = 0;
      bool ok = true;
      const uint64_t pol_a = make_l2_policy(p0.a_hint);
      const uint64_t pol_b = make_l2_policy(p0.b_hint);
      int tile_it = 0;
      for (int u = pair; ok && u < total_units; u += num_pairs) {
        const bool second = kProducts == 2 && u >= units0;
        const GemmArgs& G = second ? g1 : g0;
        const GemmParams& p = G.p;
        const int k_stages = (p.k_blocks + kSub - 1) / kSub;  // ring stages per tile
        int m_blk, n_begin, n_end;
        unit_tiles<kEpi>(p, second ? u - units0 : u, m_blk, n_begin, n_end);
        for (int n_blk = n_begin; ok && n_blk < n_end; ++n_blk, ++tile_it) {
          const bool k_rev = p.k_serpentine && (tile_it & 1);
          for (int kq = 0; kq < k_stages; ++kq) {
            const int ks = k_rev ? k_stages - 1 - kq : kq;   // K block group this stage holds
            const bool empty_ok = mbar_wait_bounded<kCl>(empty_bar(stage), phase ^ 1u, tmo, abort_flag);
            if (!__all_sync(0xffffffffu, empty_ok)) {  // one decision for the whole warp
              ok = false;
              break;
            }
            if (elect_one()) {
            const int nsub = min(kSub, p.k_blocks - ks * kSub);
            const uint32_t fb_local = full_bar(stage);
            if (leader)
              mbar_arrive_expect_tx(fb_local, static_cast<uint32_t>(kCta * nsub) * Cfg::kSubBytes);
            // copies complete on the even CTA's barrier
            const uint32_t fb = (kCta == 2) ? mapa_shared(fb_local, 0) : fb_local;
            const int am = m_blk * Cfg::kTileM + static_cast<int>(rank) * BM;   // A rows
            auto load = [&](uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t pol) {
              if constexpr (kCta == 2) tma_load_2d_pair(dst, map, x, y, fb, pol);
              else tma_load_2d_hint(dst, map, x, y, fb, pol);
            };
            auto load3 = [&](uint32_t dst, const CUtensorMap* map, int y, int z, uint64_t pol) {
              if constexpr (kCta == 2) tma_load_3d_pair(dst, map, 0, y, z, fb, pol);
              else tma_load_3d_hint(dst, map, 0, y, z, fb, pol);
            };
#pragma unroll
            for (int sub = 0; sub < kSub; ++sub) {
              if (sub >= nsub) break;
              const int kx = (ks * kSub + sub) * (kFp8 ? 2 * BK : BK);  // elements per 128-byte row
              const uint32_t sa = stage0 + stage * Cfg::kStageBytes + sub * Cfg::kSubBytes;
              const uint32_t sb = sa + Cfg::kABytes;
              if (!p.a_mn_major && p.a_kchunk) {
                load3(sa, &G.a, am + p.a_mn0, (kx + p.a_k0) >> 6, pol_a);
              } else if (!p.a_mn_major) {
                load(sa, &G.a, kx + p.a_k0, am + p.a_mn0, pol_a);
              } else if (p.a_box3) {
                load3(sa, &G.a, kx + p.a_k0, (am + p.a_mn0) >> 6, pol_a);
              } else {
#pragma unroll
                for (int j = 0; j < BM / 64; ++j)
                  load(sa + j * kMnBoxBytes, &G.a, am + 64 * j + p.a_mn0, kx + p.a_k0, pol_a);
              }
#pragma unroll
              for (int h = 0; h < Cfg::kBHalves; ++h) {
                // B rows of this CTA for the MMA of tile columns [256 h, 256 h + 256)
                const int bn = n_blk * Cfg::kTileN + h * BN + static_cast<int>(rank) * Cfg::kBRows;
                const uint32_t sbh = sb + h * Cfg::kBHalfBytes;
                if (!p.b_mn_major) {
                  load(sbh, &G.b, kx + p.b_k0, bn + p.b_mn0, pol_b);
                } else if (p.b_box3) {
                  load3(sbh, &G.b, kx + p.b_k0, (bn + p.b_mn0) >> 6, pol_b);
                } else {
#pragma unroll
                  for (int j = 0; j < Cfg::kBRows / 64; ++j)
                    load(sbh + j * kMnBoxBytes, &G.b, bn + 64 * j + p.b_mn0, kx + p.b_k0, pol_b);
                }
              }
            }
            }
            __syncwarp();
            issued_mask |= 1u << stage;
            issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        if (lane == 0) record_status(p0.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // Drain before the final barrier. The even CTA waits for every stage phase it
      // armed; those phases count the odd CTA's copies too, and in a normal run the
      // odd CTA issues exactly those phases. After an abort the odd CTA may have
      // issued a phase the even CTA never armed, which it cannot observe: it then
      // waits a bounded grace period (far longer than a copy takes) so that its
      // copies land while both CTAs are still resident.
      const volatile int no_abort = 0;
      if (leader) {
        for (int s = 0; s < kStages; ++s)
          if (issued_mask & (1u << s))
            mbar_wait_bounded<kCl>(full_bar(s), (issued_par >> s) & 1u, 1000000000ull, &no_abort);
      } else if (!ok || *abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 200000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (even CTA) ----------------
    if (leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool issued_any = false;
      int tile_it = 0;
      for (int u = pair; ok && u < total_units; u += num_pairs) {
        const bool second = kProducts == 2 && u >= units0;
        const GemmParams& p = second ? g1.p : g0.p;
        const int k_stages = (p.k_blocks + kSub - 1) / kSub;  // ring stages per tile
        const int k_blocks = p.k_blocks;
        const bool a_mn = p.a_mn_major != 0, b_mn = p.b_mn_major != 0;
        const uint32_t idesc = p.idesc;
        const bool serp = p.k_serpentine != 0;
        int m_blk, n_begin, n_end;
        unit_tiles<kEpi>(p, second ? u - units0 : u, m_blk, n_begin, n_end);
        for (int n_blk = n_begin; ok && n_blk < n_end; ++n_blk, ++tile_it) {
          const bool k_rev = serp && (tile_it & 1);
          // both CTAs' epilogues must have drained this accumulator
          bool got;
          if constexpr (kCta == 2) {
            got = mbar_try_wait_cluster(tempty_bar(acc), acc_phase ^ 1u);
            if (!got) {
              const uint64_t t0 = global_timer_ns();
              while (!(got = mbar_try_wait_cluster(tempty_bar(acc), acc_phase ^ 1u))) {
                if (*abort_flag || global_timer_ns() - t0 > tmo) break;
              }
            }
          } else {
            got = mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, tmo, abort_flag);
          }
          if (!__all_sync(0xffffffffu, got)) {  // one decision for the whole warp
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Cfg::kTileN);
          for (int kq = 0; kq < k_stages; ++kq) {
            const bool full_ok = mbar_wait_bounded<kCl>(full_bar(stage), phase, tmo, abort_flag);
            if (!__all_sync(0xffffffffu, full_ok)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const int ks = k_rev ? k_stages - 1 - kq : kq;   // as the producer loaded it
            const int nsub = min(kSub, k_blocks - ks * kSub);
            if (elect_one()) {
#pragma unroll
            for (int sub = 0; sub < kSub; ++sub) {
              if (sub >= nsub) break;
              const uint32_t sa = stage0 + stage * Cfg::kStageBytes + sub * Cfg::kSubBytes;
              const uint32_t sb = sa + Cfg::kABytes;
#pragma unroll
              for (int k = 0; k < BK / UK; ++k) {
                const uint64_t da = a_mn ? make_sw128_desc(sa + k * (UK * 128), kMnBoxBytes, 1024)
                                         : make_sw128_desc(sa + k * (UK * 2), 16, 1024);
                const uint32_t accum = (kq | sub | k) != 0 ? 1u : 0u;   // first MMA of the tile overwrites
#pragma unroll
                for (int h = 0; h < Cfg::kBHalves; ++h) {
                  const uint32_t sbh = sb + h * Cfg::kBHalfBytes;
                  const uint64_t db = b_mn ? make_sw128_desc(sbh + k * (UK * 128), kMnBoxBytes, 1024)
                                           : make_sw128_desc(sbh + k * (UK * 2), 16, 1024);
                  const uint32_t dh = d_tmem + static_cast<uint32_t>(h * BN);
                  if constexpr (kFp8) umma_f8_cg<kCta>(dh, da, db, idesc, accum);
                  else umma_bf16_cg<kCta>(dh, da, db, idesc, accum);
                }
              }
            }
            umma_commit_pair<kCta>(empty_bar(stage));  // frees the stage in both CTAs
            }
            __syncwarp();
            issued_any = true;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if (elect_one()) umma_commit_pair<kCta>(tfull_bar(acc));
          __syncwarp();
          if (++acc == Cfg::kAccs) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
      }
      if (!ok) {
        if (lane == 0) record_status(p0.status, kStatusTimeout);
        *abort_flag = 1;
      }
      if (issued_any) {
        // Drain: all MMAs of this warp complete before TMEM is freed.
        const volatile int no_abort = 0;
        if (lane == 0) umma_commit_cg<kCta>(drain_bar);
        __syncwarp();
        mbar_wait_bounded(drain_bar, 0, 1000000000ull, &no_abort);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps (both CTAs) ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // row within this CTA's 128 rows
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tempty_leader0 = (kCta == 2) ? mapa_shared(tempty_bar(0), 0) : tempty_bar(0);
    const uint32_t tempty_leader1 = (kCta == 2) ? mapa_shared(tempty_bar(1), 0) : tempty_bar(1);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    float scale_v = 0.f;
    if constexpr (kEpi == EPI_GRAD) scale_v = *p0.scale;
    float acc_scale = 1.f;  // FP8 operands: product of the two per-tensor scales
    if constexpr (kFp8) acc_scale = *p0.acc_scale_h * *p0.acc_scale_w;
    // this warp's two staging boxes, used alternately
    const uint32_t stg = stage0 + Cfg::kRingBytes + static_cast<uint32_t>(quarter) * 2u * Cfg::kStgBytes;
    uint32_t nbox = 0;
    for (int u = pair; ok && u < total_units; u += num_pairs) {
      const bool second = kProducts == 2 && u >= units0;
      const GemmArgs& G = second ? g1 : g0;
      const GemmParams& p = G.p;
      int m_blk, n_begin, n_end;
      const int col_unit = unit_tiles<kEpi>(p, second ? u - units0 : u, m_blk, n_begin, n_end);
      const int prow = m_blk * Cfg::kTileM + static_cast<int>(rank) * BM + row;  // product row
      const bool row_ok = prow < p.m_valid;
      int y = -1;
      if constexpr (kEpi != EPI_F32) {
        if (row_ok) {
          const int lab = p.labels[p.row_base + prow];
          y = (lab == p.ignore_index) ? -1 : lab;
        }
      }
      LseState st{-INFINITY, 0.f, 0.f, false};
      // Rows past the product (or of another token block) take zmax = +inf, so
      // their G is exactly 0 whatever logits the tile holds for them.
      float zmax = INFINITY, a = 0.f, sc = 0.f, q = -1.f;
      if constexpr (kEpi == EPI_GRAD) {
        if (row_ok) {
          sc = (y >= 0) ? scale_v : 0.f;
          if (p.gstat != nullptr) {
            const float4 gs = p.gstat[p.row_base + prow];
            zmax = gs.x;
            a = sc * gs.y;
            q = gs.z;
          } else {
            zmax = p.lse[p.row_base + prow];
            a = sc;
          }
        }
      }
      for (int n_blk = n_begin; n_blk < n_end; ++n_blk) {
        int got = 0;
        if (lane == 0) {
          if constexpr (kCta == 2) {
            got = mbar_try_wait_cluster(tfull_bar(acc), acc_phase);
            if (!got) {
              const uint64_t t0 = global_timer_ns();
              while (!(got = mbar_try_wait_cluster(tfull_bar(acc), acc_phase))) {
                if (*abort_flag || global_timer_ns() - t0 > tmo) break;
              }
            }
          } else {
            got = mbar_wait_bounded(tfull_bar(acc), acc_phase, tmo, abort_flag) ? 1 : 0;
          }
        }
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + lane_addr + static_cast<uint32_t>(acc * Cfg::kTileN);
#pragma unroll 1
        for (int c = 0; c < Cfg::kTileN / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c * 32, r);
          tmem_wait_ld();
          float v[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
          if constexpr (kFp8) {
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] *= acc_scale;
          }
          const int col = n_blk * Cfg::kTileN + c * 32;  // product column
          if constexpr (kEpi == EPI_LSE) {
            lse_chunk(v, col, p.n_valid, y - (p.col_base + col), st);
          } else {
            const uint32_t box = stg + (nbox & 1u) * Cfg::kStgBytes;
            // the store issued two boxes ago from this buffer has read it
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            if constexpr (kEpi == EPI_GRAD) {
              float g[32];
              grad_chunk(v, col, p.n_valid, y - (p.col_base + col), zmax, a, sc, q, g);
              stage_bf16_row(box, lane, g);
            } else if (p.out_mode == OUT_STORE_BF16) {
              stage_bf16_row(box, lane, v);
            } else {
              stage_f32_row(box, lane, v);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              // rows and columns outside the map are dropped by the store
              const int oy = p.out_row0 + m_blk * Cfg::kTileM + static_cast<int>(rank) * BM +
                             quarter * 32;
              if constexpr (kEpi == EPI_GRAD) tma_store_3d(&G.c, box, col & 63, oy, col >> 6);
              else if (p.out_mode == OUT_ADD_F32) tma_reduce_add_2d(&G.c, box, col, oy);
              else tma_store_2d(&G.c, box, col, oy);
              bulk_commit_group();
            }
            ++nbox;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (kCta == 2) mbar_arrive_cluster(acc == 0 ? tempty_leader0 : tempty_leader1);
          else mbar_arrive(tempty_bar(acc));
        }
        if (++acc == Cfg::kAccs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if constexpr (kEpi == EPI_LSE) {
        if (ok) {
          // partial slot of (vocabulary range, 128-row block), independent of the raster
          const int blk128 = m_blk * kCta + static_cast<int>(rank);
          p.part[(static_cast<int64_t>(col_unit) * p.part_stride + blk128) * BM + row] =
              make_float2(st.m, st.s);
          if (row_ok && st.found) p.zt[p.row_base + prow] = st.zt;
        }
      }
    }
    if (!ok) {
      if (lane == 0) record_status(p0.status, kStatusTimeout);
      *abort_flag = 1;
    }
    // every store of this warp has landed before the CTA can exit
    if constexpr (kEpi != EPI_LSE) {
      if (lane == 0) bulk_wait_group_all();
      __syncwarp();
    }
  }

  tc_fence_before();
  if constexpr (kCta == 2) cluster_sync();  // the pair's copies and MMAs have drained
  else __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_cg<kCta>(tmem_base, kTmemCols);
}

// Host-side launch of one instantiation: grid/kCta clusters of kCta CTAs, the tile
// configuration's dynamic shared memory, the products' maps and parameters passed
// by value (g1 is ignored unless kProducts == 2).
template <int kEpi, int kCta, int kFp8, int kWide, int kProducts = 1>
cudaError_t launch_gemm(const GemmArgs& g0, const GemmArgs& g1, int grid, cudaStream_t stream) {
  auto kern = flce_gemm_kernel<kEpi, kCta, kFp8, kWide, kProducts>;
  constexpr size_t smem = TileCfg<kCta, kWide>::kSmemBytes;
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
  return cudaLaunchKernelEx(&cfg, kern, g0, g1);
}

}  // namespace flce
