// flce_forward_noalloc: the forward pass (loss and per-token lse) for callers
// that cannot give the library a device workspace.
//
// Who needs it: code that has no way to obtain device memory at call time. For
// example, a plugin inside a host application that owns every byte of device
// memory through its own pool and gives its plugins no allocator, or a serving
// process that reserved all of its memory at start-up so that nothing can fail
// with out-of-memory in the middle of a run. Such callers can pass inputs and
// outputs they already own, but not a workspace.
//
// How: the scratch that flce_forward would take from the caller's workspace
// lives here in one file-scope __device__ array of kNoAllocScratchBytes. Every
// GPU that loads this part of the library keeps that array until the process
// exits. Nothing here calls cudaMalloc, cudaFree or any allocating routine, but
// the array itself comes into being when the CUDA runtime loads this file's
// device code on a device; with lazy module loading (the default) that happens
// at the first cudaGetSymbolAddress below, i.e. during the first call on that
// device, which is therefore the set-up call.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/flce.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

// In host code this name is only a host-side stand-in for the device array, not
// a device address: the address each device uses comes from
// cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device; looked up once per
// device, on the first call made with that device current.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLCE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FLCE_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return FLCE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FLCE_OK;
}

}  // namespace

extern "C" int flce_forward_noalloc(const uint16_t* H, const uint16_t* W, const int32_t* labels,
                                    int64_t N, int64_t D, int64_t V, const flce_options* opt,
                                    float* loss, float* lse, int32_t* status, void* stream) {
  void* scratch = nullptr;
  // The set-up form: no problem, only the array's creation and address lookup on
  // the current device.
  if (H == nullptr && W == nullptr && labels == nullptr && loss == nullptr && lse == nullptr &&
      status == nullptr && N == 0 && D == 0 && V == 0)
    return scratch_address(&scratch);
  flce_options o;
  flce_default_options(&o);
  if (opt != nullptr) o = *opt;
  const bool planned = o.v_splits == 0;
  if (planned) {
    flce_plan_info info;
    const int rc = flce_get_plan(N, D, V, &o, 0, 0, &info);
    if (rc != FLCE_OK) return rc;
    o.v_splits = info.v_splits;
  }
  size_t need = 0;
  int rc = flce_forward_workspace_size(N, D, V, &o, &need);
  if (rc != FLCE_OK) return rc;
  // A planned split count may be lowered until the partials fit (fewer
  // vocabulary ranges need fewer partials); a caller's explicit one is kept.
  while (planned && need > kNoAllocScratchBytes && o.v_splits > 1) {
    o.v_splits = (o.v_splits + 1) / 2;
    rc = flce_forward_workspace_size(N, D, V, &o, &need);
    if (rc != FLCE_OK) return rc;
  }
  if (need > kNoAllocScratchBytes) return FLCE_ERR_WORKSPACE;
  rc = scratch_address(&scratch);
  if (rc != FLCE_OK) return rc;
  // Every scratch word the forward pass reads is written earlier in the same
  // call, so nothing has to be cleared between calls.
  return flce_forward(H, W, labels, N, D, V, &o, loss, lse, scratch, kNoAllocScratchBytes, status,
                      stream);
}
