// liger_moe_dispatch_noalloc: the dispatch entry point for callers that
// cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: code running under a
// memory planner that hands out no extra buffers, plug-ins that may only use
// the tensors they are given, or host code that must not allocate in the
// middle of a step.  This entry point takes the same inputs and outputs as
// liger_moe_dispatch but keeps its scratch (the per-chunk expert histograms)
// in a fixed array compiled into this library, so it calls no cudaMalloc,
// cudaFree or allocating routine of any library.
//
// The array lives in device memory of every GPU that loads the library, for
// as long as the process runs (kDispatchScratchBytes per device).  All calls
// on a device share it, so two calls that overlap on the GPU (different
// streams without ordering between them) race on it and give wrong results.
// The array keeps whatever the last call left there; the dispatch kernels
// overwrite every histogram entry they later read, so nothing needs clearing.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

#define LIGER_MOE_API extern "C" __attribute__((visibility("default")))

namespace lmoe {
namespace {

// 1 MiB: histograms of ceil(T*k / 256) slot chunks x E experts, int32 each,
// so T*k up to 131072 with E = 512, or up to 65536 with E = 1024.  The array
// is 256-byte aligned, which is all the dispatch kernels ask of their scratch.
constexpr size_t kDispatchScratchBytes = size_t(1) << 20;

static __device__ __align__(256) int32_t g_dispatch_scratch[kDispatchScratchBytes / sizeof(int32_t)];

constexpr int kMaxDev = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDev] = {};

// Device address of the scratch array on the current device (looked up once
// per device; in host code the array's name is not a device address).
int scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDev) return LIGER_MOE_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[device] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess || p == nullptr) {
      set_cuda_error(e, "cudaGetSymbolAddress(dispatch scratch)");
      return LIGER_MOE_ERR_LAUNCH;
    }
    g_scratch_ptr[device] = p;
  }
  *out = g_scratch_ptr[device];
  return LIGER_MOE_OK;
}

}  // namespace
}  // namespace lmoe

using namespace lmoe;

LIGER_MOE_API int liger_moe_dispatch_noalloc(const int32_t* topk_ids, const float* topk_w, const void* x, int T,
                                             int H, int E, int k, int32_t* counts, int32_t* m_indptr,
                                             int32_t* row_to_slot, int32_t* slot_to_row, float* w_perm,
                                             void* x_perm, void* stream) {
  if (int rc = check_topk(T, E, k)) return rc;
  const long long R = static_cast<long long>(T) * k;
  if (counts == nullptr || m_indptr == nullptr) return LIGER_MOE_ERR_INVALID_ARG;
  if (R > 0 && (topk_ids == nullptr || row_to_slot == nullptr || slot_to_row == nullptr))
    return LIGER_MOE_ERR_INVALID_ARG;
  if (w_perm != nullptr && R > 0 && topk_w == nullptr) return LIGER_MOE_ERR_INVALID_ARG;
  if (x_perm != nullptr && R > 0) {
    if (x == nullptr) return LIGER_MOE_ERR_INVALID_ARG;
    if (H < 64 || H % 64 != 0 || (reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(x_perm) & 15u))
      return LIGER_MOE_ERR_MISALIGNED;
  }
  // the stated limit: the histograms, ceil(T*k / 256) * E * 4 bytes, fit in the array
  if (dispatch_scratch_bytes(R, E) > kDispatchScratchBytes) return LIGER_MOE_ERR_CAPACITY;
  PdlScope pdl(R);
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  void* scratch = nullptr;
  if (int rc = scratch_address(dev.device, &scratch)) return rc;
  return launch_dispatch(topk_ids, topk_w, static_cast<const uint16_t*>(x), T, H, E, k, counts, m_indptr, row_to_slot,
                         slot_to_row, w_perm, static_cast<uint16_t*>(x_perm), scratch, dev,
                         static_cast<cudaStream_t>(stream));
}
