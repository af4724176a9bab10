// The C ABI of the routed MoE layer (see include/liger_moe.h): argument
// validation, workspace layout and the launch sequence of each entry point.
// No entry point allocates, frees or synchronises (except
// liger_moe_device_error, whose job is to synchronise and read the flag).
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"

#define LIGER_MOE_API extern "C" __attribute__((visibility("default")))

namespace lmoe {

namespace {
thread_local char g_last_error[256] = "";
__device__ int g_device_error = 0;  // device-side error word, one per device
__device__ int g_device_error_taken = 0;  // what the last read-and-clear took out of it

// Reads and clears the error word in one atomic exchange, so that a bit a kernel on another
// stream sets at the same moment is either taken now or left for the next read, never lost.
__global__ void take_device_error_kernel() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  g_device_error_taken = atomicExch(&g_device_error, 0);
}

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceInfo g_dev_cache[kMaxDevices];
bool g_dev_known[kMaxDevices] = {};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by the expert entry points.
int check_shapes(long long R, int H, int I, int E) {
  if (R < 0 || E < 1 || H < 1 || I < 1) return LIGER_MOE_ERR_INVALID_ARG;
  if (E > kMaxExperts) return LIGER_MOE_ERR_CAPACITY;
  if (H % 64 != 0 || I % 64 != 0) return LIGER_MOE_ERR_MISALIGNED;
  if (R > kIndexLimit || 2LL * I * E > kIndexLimit || 1LL * H * E > kIndexLimit) return LIGER_MOE_ERR_CAPACITY;
  return LIGER_MOE_OK;
}

// activation id and clamp (enum liger_moe_activation)
int check_activation(int act, float clamp) {
  if (act < LIGER_MOE_ACT_SWIGLU || act > LIGER_MOE_ACT_RELU2) return LIGER_MOE_ERR_INVALID_ARG;
  if ((act == LIGER_MOE_ACT_SWIGLU_BOUNDED || act == LIGER_MOE_ACT_SWIGLU_OAI) && !(clamp > 0.f && clamp < 3.0e38f))
    return LIGER_MOE_ERR_INVALID_ARG;
  return LIGER_MOE_OK;
}

template <class T>
T* carve(uint8_t*& cursor, size_t bytes) {
  T* p = reinterpret_cast<T*>(cursor);
  cursor += align_up(bytes, 256);
  return p;
}

}  // namespace

int check_topk(long long T, int E, int k) {
  if (T < 0 || E < 1 || k < 1 || k > E) return LIGER_MOE_ERR_INVALID_ARG;
  if (E > kMaxExperts || k > kMaxTopK) return LIGER_MOE_ERR_CAPACITY;
  if (T * k > kIndexLimit) return LIGER_MOE_ERR_CAPACITY;
  return LIGER_MOE_OK;
}

// ---------------------------------------------------------------- kernel trace
namespace {
struct TraceRecord {
  const char* name;
  cudaEvent_t start, stop;
  int launches;  // kernels launched inside the interval
};
std::atomic<int> g_trace_on{0};
std::mutex g_trace_mu;
std::vector<TraceRecord> g_trace;
std::vector<cudaEvent_t> g_event_pool;

// Records `e` on `s`; inside a stream capture the record becomes an external event node, so
// the event still marks the time when the captured graph is replayed.
void trace_record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) == cudaSuccess && st == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

cudaEvent_t trace_event() {
  // caller holds g_trace_mu
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
}  // namespace

KernelScope::KernelScope(const char* name, cudaStream_t s) : name_(name), stream_(s) {
  if (name == nullptr || !g_trace_on.load(std::memory_order_relaxed)) return;  // nullptr: not traced
  std::lock_guard<std::mutex> lock(g_trace_mu);
  start_ = trace_event();
  if (start_ != nullptr) trace_record(start_, stream_);
  launches0_ = t_kernel_launches;
}

KernelScope::~KernelScope() {
  if (start_ == nullptr) return;
  std::lock_guard<std::mutex> lock(g_trace_mu);
  cudaEvent_t stop = trace_event();
  if (stop == nullptr) {
    g_event_pool.push_back(start_);
    return;
  }
  trace_record(stop, stream_);
  g_trace.push_back(TraceRecord{name_, start_, stop, static_cast<int>(t_kernel_launches - launches0_)});
}

void set_cuda_error(cudaError_t e, const char* where) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where, cudaGetErrorString(e));
}

bool pdl_enabled() {
  static const int mode = [] {  // 0 never, 1 always, 2 small calls
    const char* v = std::getenv("LIGER_MOE_PDL");
    if (v == nullptr || v[0] == '\0') return 2;
    return std::strcmp(v, "0") == 0 ? 0 : 1;
  }();
  return mode == 1 || (mode == 2 && t_pdl_small);
}

int check_launch(const char* where) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_cuda_error(e, where);
    return LIGER_MOE_ERR_LAUNCH;
  }
  return LIGER_MOE_OK;
}

int current_device(DeviceInfo* info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_cuda_error(e, "cudaGetDevice");
    return LIGER_MOE_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (dev >= 0 && dev < kMaxDevices && g_dev_known[dev]) {
    *info = g_dev_cache[dev];
    return LIGER_MOE_OK;
  }
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3) return LIGER_MOE_ERR_UNSUPPORTED_DEVICE;
  void* flag = nullptr;
  e = cudaGetSymbolAddress(&flag, g_device_error);
  if (e != cudaSuccess) {
    set_cuda_error(e, "cudaGetSymbolAddress(device error flag)");
    return LIGER_MOE_ERR_LAUNCH;
  }
  DeviceInfo d{dev, sms, static_cast<int*>(flag)};
  if (dev >= 0 && dev < kMaxDevices) {
    g_dev_cache[dev] = d;
    g_dev_known[dev] = true;
  }
  *info = d;
  return LIGER_MOE_OK;
}

namespace {

// Rows of each half of the padded weight-gradient operands: every expert's rows rounded up to 16.
long long padded_rows(long long R, int E) { return R + 15LL * E; }

// The backward may use fp16 weight-gradient operands (f16 rows, expert-major inputs, gated experts):
// the workspace then holds the fp16 words and the fp16 copies of the x and dY rows.
bool bwd_f16_possible(long long R, bool gated, bool gather) { return gated && !gather && R >= kF16MinR; }

size_t bwd_workspace_bytes(long long R, int H, int I, int E, bool recompute_gu, bool gather, bool f16) {
  const long long Rp = padded_rows(R, E);
  // tile prefix, padded row prefix, 256-row pair block prefix, light tile and heavy pair prefixes,
  // expert order and its [E][4] table, claim counters
  size_t b = 10 * schedule_bytes(E) + kClaimBytes;
  if (!gather) b += align_up(static_cast<size_t>(R) * H * 2, 256);  // dy_perm
  b += align_up(static_cast<size_t>(Rp) * 2 * I * 2 * 2, 256);        // dgu (hi, lo), padded rows
  b += align_up(static_cast<size_t>(R) * H * 2, 256);                 // dx_perm
  b += align_up(static_cast<size_t>(Rp) * I * 2 * 2, 256);            // hw_perm (hi, lo), padded rows
  b += align_up(static_cast<size_t>(R) * gdot_tiles(I) * 4, 256);     // gdot
  if (recompute_gu) b += align_up(static_cast<size_t>(R) * 2 * I * 4, 256);
  if (f16) b += f16_words_bytes(E) + 2 * align_up(static_cast<size_t>(R) * H * 2, 256);  // words, x16, dy16
  return b;
}

std::atomic<int> g_dw_fp16{1};

}  // namespace
}  // namespace lmoe

using namespace lmoe;

LIGER_MOE_API int liger_moe_abi_version(void) { return 100; }

LIGER_MOE_API const char* liger_moe_last_cuda_error(void) { return g_last_error; }

LIGER_MOE_API const char* liger_moe_status_string(int status) {
  switch (status) {
    case LIGER_MOE_OK: return "LIGER_MOE_OK";
    case LIGER_MOE_ERR_INVALID_ARG: return "LIGER_MOE_ERR_INVALID_ARG";
    case LIGER_MOE_ERR_MISALIGNED: return "LIGER_MOE_ERR_MISALIGNED";
    case LIGER_MOE_ERR_CAPACITY: return "LIGER_MOE_ERR_CAPACITY";
    case LIGER_MOE_ERR_UNSUPPORTED_DEVICE: return "LIGER_MOE_ERR_UNSUPPORTED_DEVICE";
    case LIGER_MOE_ERR_LAUNCH: return "LIGER_MOE_ERR_LAUNCH";
    case LIGER_MOE_ERR_DEVICE: return "LIGER_MOE_ERR_DEVICE";
    default: return "unknown liger_moe status";
  }
}

LIGER_MOE_API int liger_moe_route_topk(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                                       void* stream) {
  if (int rc = check_topk(T, E, k)) return rc;
  if (T > 0 && (logits == nullptr || topk_ids == nullptr || topk_w == nullptr)) return LIGER_MOE_ERR_INVALID_ARG;
  PdlScope pdl(static_cast<long long>(T) * k);
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  if (T == 0) return LIGER_MOE_OK;
  return launch_route_topk(logits, T, E, k, topk_ids, topk_w, static_cast<cudaStream_t>(stream));
}

LIGER_MOE_API int liger_moe_dispatch(const int32_t* topk_ids, const float* topk_w, const void* x, int T, int H, int E,
                                     int k, int32_t* counts, int32_t* m_indptr, int32_t* row_to_slot,
                                     int32_t* slot_to_row, float* w_perm, void* x_perm, void* workspace,
                                     size_t* workspace_bytes, void* stream) {
  if (int rc = check_topk(T, E, k)) return rc;
  const long long R = static_cast<long long>(T) * k;
  if (workspace_bytes == nullptr || counts == nullptr || m_indptr == nullptr) return LIGER_MOE_ERR_INVALID_ARG;
  if (R > 0 && (topk_ids == nullptr || row_to_slot == nullptr || slot_to_row == nullptr))
    return LIGER_MOE_ERR_INVALID_ARG;
  if (w_perm != nullptr && R > 0 && topk_w == nullptr) return LIGER_MOE_ERR_INVALID_ARG;
  if (x_perm != nullptr && R > 0) {
    if (x == nullptr) return LIGER_MOE_ERR_INVALID_ARG;
    if (H < 64 || H % 64 != 0 || !aligned16(x) || !aligned16(x_perm)) return LIGER_MOE_ERR_MISALIGNED;
  }
  const size_t need = dispatch_workspace_bytes(R, E);
  if (workspace == nullptr) {
    *workspace_bytes = need;
    return LIGER_MOE_OK;
  }
  if (*workspace_bytes < need) return LIGER_MOE_ERR_CAPACITY;
  if (!aligned16(workspace)) return LIGER_MOE_ERR_MISALIGNED;
  PdlScope pdl(R);
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  return launch_dispatch(topk_ids, topk_w, static_cast<const uint16_t*>(x), T, H, E, k, counts, m_indptr, row_to_slot,
                         slot_to_row, w_perm, static_cast<uint16_t*>(x_perm), workspace, dev,
                         static_cast<cudaStream_t>(stream));
}

namespace {

// Forward expert MLP.  A rows come from x_perm [R, H] or, when x != NULL, are gathered from
// x [T, H] by token (row_to_slot[r] / k).
int grouped_swiglu_fwd_impl(const void* x_perm, const void* x, const int32_t* row_to_slot, int T, int k,
                            const int32_t* m_indptr, const void* w_gate_up, const void* w_down, const float* w_perm,
                            long long R, int H, int I, int E, void* h_perm, float* gu_perm, void* y_perm,
                            void* workspace, size_t* workspace_bytes, void* stream, int act = LIGER_MOE_ACT_SWIGLU,
                            float clamp = 0.f) {
  if (int rc = check_shapes(R, H, I, E)) return rc;
  if (int rc = check_activation(act, clamp)) return rc;
  if (workspace_bytes == nullptr || m_indptr == nullptr) return LIGER_MOE_ERR_INVALID_ARG;
  const void* a_src = x != nullptr ? x : x_perm;
  if (R > 0 && (a_src == nullptr || w_gate_up == nullptr || w_down == nullptr || w_perm == nullptr ||
                h_perm == nullptr || y_perm == nullptr))
    return LIGER_MOE_ERR_INVALID_ARG;
  if (R > 0 && x != nullptr && row_to_slot == nullptr) return LIGER_MOE_ERR_INVALID_ARG;
  if (!aligned16(a_src) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(h_perm) ||
      !aligned16(gu_perm) || !aligned16(y_perm))
    return LIGER_MOE_ERR_MISALIGNED;
  // tile prefixes of 128-row tiles and of 256-row pair tiles, and the two of the heavy / light split
  const size_t need = 4 * schedule_bytes(E);
  if (workspace == nullptr) {
    *workspace_bytes = need;
    return LIGER_MOE_OK;
  }
  if (*workspace_bytes < need) return LIGER_MOE_ERR_CAPACITY;
  if (!aligned16(workspace)) return LIGER_MOE_ERR_MISALIGNED;
  PdlScope pdl(R);
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  if (R == 0) return LIGER_MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* cur = static_cast<uint8_t*>(workspace);
  ScheduleBufs sb;
  sb.tile_prefix = carve<int32_t>(cur, schedule_bytes(E));
  sb.pair_prefix = carve<int32_t>(cur, schedule_bytes(E));
  int32_t* light = carve<int32_t>(cur, schedule_bytes(E));
  int32_t* heavy = carve<int32_t>(cur, schedule_bytes(E));
  if (split_schedule(R, E)) {  // the heavy / light split may run: the schedule builds its prefixes
    sb.light_prefix = light;
    sb.heavy_pair_prefix = heavy;
  }
  if (int rc = launch_tile_schedule(m_indptr, E, R, sb, dev, s)) return rc;
  int32_t* tile_prefix = sb.tile_prefix;
  int32_t* pair_prefix = sb.pair_prefix;
  FwdGemmArgs a{};
  a.x_perm = static_cast<const uint16_t*>(x_perm);
  a.x = static_cast<const uint16_t*>(x);
  a.row_to_slot = row_to_slot;
  a.T = T;
  a.k = k;
  a.m_indptr = m_indptr;
  a.tile_prefix = tile_prefix;
  a.pair_prefix = pair_prefix;
  a.light_prefix = sb.light_prefix;
  a.heavy_pair_prefix = sb.heavy_pair_prefix;
  a.w_gate_up = static_cast<const uint16_t*>(w_gate_up);
  a.w_down = static_cast<const uint16_t*>(w_down);
  a.w_perm = w_perm;
  a.R = R;
  a.H = H;
  a.I = I;
  a.E = E;
  a.h_perm = static_cast<uint16_t*>(h_perm);
  a.gu_perm = gu_perm;
  a.y_perm = static_cast<uint16_t*>(y_perm);
  a.act = act;
  a.act_clamp = clamp;
  if (int rc = launch_gate_up(a, dev, s)) return rc;
  return launch_down(a, dev, s);
}

}  // namespace

LIGER_MOE_API int liger_moe_grouped_swiglu_fwd(const void* x_perm, const int32_t* m_indptr, const void* w_gate_up,
                                               const void* w_down, const float* w_perm, int R, int H, int I, int E,
                                               void* h_perm, float* gu_perm, void* y_perm, void* workspace,
                                               size_t* workspace_bytes, void* stream) {
  return grouped_swiglu_fwd_impl(x_perm, nullptr, nullptr, 0, 1, m_indptr, w_gate_up, w_down, w_perm, R, H, I, E,
                                 h_perm, gu_perm, y_perm, workspace, workspace_bytes, stream);
}

LIGER_MOE_API int liger_moe_grouped_glu_fwd(const void* x_perm, const int32_t* m_indptr, const void* w_gate_up,
                                            const void* w_down, const float* w_perm, int R, int H, int I, int E,
                                            int activation, float clamp, void* h_perm, float* gu_perm, void* y_perm,
                                            void* workspace, size_t* workspace_bytes, void* stream) {
  return grouped_swiglu_fwd_impl(x_perm, nullptr, nullptr, 0, 1, m_indptr, w_gate_up, w_down, w_perm, R, H, I, E,
                                 h_perm, gu_perm, y_perm, workspace, workspace_bytes, stream, activation, clamp);
}

LIGER_MOE_API int liger_moe_grouped_swiglu_fwd_gather(const void* x, const int32_t* row_to_slot, int T, int k,
                                                      const int32_t* m_indptr, const void* w_gate_up,
                                                      const void* w_down, const float* w_perm, int H, int I, int E,
                                                      void* h_perm, float* gu_perm, void* y_perm, void* workspace,
                                                      size_t* workspace_bytes, void* stream) {
  if (T < 0 || k < 1) return LIGER_MOE_ERR_INVALID_ARG;
  if (k > kMaxTopK) return LIGER_MOE_ERR_CAPACITY;
  const long long R = static_cast<long long>(T) * k;
  if (R > 0 && x == nullptr) return LIGER_MOE_ERR_INVALID_ARG;
  return grouped_swiglu_fwd_impl(nullptr, R > 0 ? x : nullptr, row_to_slot, T, k, m_indptr, w_gate_up, w_down,
                                 w_perm, R, H, I, E, h_perm, gu_perm, y_perm, workspace, workspace_bytes, stream);
}

LIGER_MOE_API int liger_moe_combine(const void* y_perm, const int32_t* slot_to_row, int T, int H, int k, void* y,
                                    void* stream) {
  if (T < 0 || k < 1 || H < 1) return LIGER_MOE_ERR_INVALID_ARG;
  if (k > kMaxTopK || static_cast<long long>(T) * k > kIndexLimit) return LIGER_MOE_ERR_CAPACITY;
  if (H % 64 != 0) return LIGER_MOE_ERR_MISALIGNED;
  if (T > 0 && (y_perm == nullptr || slot_to_row == nullptr || y == nullptr)) return LIGER_MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(y)) return LIGER_MOE_ERR_MISALIGNED;
  PdlScope pdl(static_cast<long long>(T) * k);
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  return launch_combine(static_cast<const uint16_t*>(y_perm), slot_to_row, T, H, k, static_cast<uint16_t*>(y), dev,
                        static_cast<cudaStream_t>(stream));
}

namespace {

// A second stream of the calling thread on one device, with a fork and a join event, for work
// that may run beside the caller's stream.  Created on first use, never while the caller's
// stream is being captured (it is then retried on a later call); nullptr when unavailable, in
// which case the caller runs everything in order on its own stream.  Per thread, so that two
// threads capturing graphs never share it.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr;
  cudaEvent_t join = nullptr;
  bool failed = false;
};

SideStream* side_stream(int device, cudaStream_t caller) {
  thread_local SideStream per_device[kMaxDevices];
  if (device < 0 || device >= kMaxDevices) return nullptr;
  SideStream& ss = per_device[device];
  if (ss.stream != nullptr) return &ss;
  if (ss.failed) return nullptr;
  cudaStreamCaptureStatus status = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(caller, &status) != cudaSuccess || status != cudaStreamCaptureStatusNone) {
    cudaGetLastError();  // a refused query is not a launch error of this call
    return nullptr;
  }
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  if (cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) {
    if (join != nullptr) cudaEventDestroy(join);
    if (fork != nullptr) cudaEventDestroy(fork);
    if (stream != nullptr) cudaStreamDestroy(stream);
    cudaGetLastError();
    ss.failed = true;
    return nullptr;
  }
  ss.stream = stream;
  ss.fork = fork;
  ss.join = join;
  return &ss;
}

// Backward of the layer.  With x_perm: dY is copied to expert-major order (dy_perm, in the
// workspace) and both are read as dense tiles.  With x (x_perm NULL): x and dY rows are
// gathered by token inside the GEMMs and no expert-major copy is made.
int bwd_dx_dw_impl(const void* dy, const void* x_perm, const void* x, const void* h_perm, const float* gu_perm,
                   const int32_t* topk_ids, const float* topk_w, const int32_t* m_indptr, const int32_t* row_to_slot,
                   const int32_t* slot_to_row, const float* w_perm, const void* w_gate_up, const void* w_down, int T,
                   int H, int I, int E, int k, void* dx, void* dw_gate_up, void* dw_down, float* d_logits,
                   void* workspace, size_t* workspace_bytes, void* stream, int act = LIGER_MOE_ACT_SWIGLU,
                   float clamp = 0.f) {
  if (int rc = check_topk(T, E, k)) return rc;
  if (int rc = check_activation(act, clamp)) return rc;
  const long long R = static_cast<long long>(T) * k;
  if (int rc = check_shapes(R, H, I, E)) return rc;
  if (2 * padded_rows(R, E) > kIndexLimit) return LIGER_MOE_ERR_CAPACITY;  // the padded dW operands' rows
  if (workspace_bytes == nullptr || m_indptr == nullptr || w_gate_up == nullptr || w_down == nullptr ||
      dw_gate_up == nullptr || dw_down == nullptr)
    return LIGER_MOE_ERR_INVALID_ARG;
  const void* x_src = x != nullptr ? x : x_perm;
  if (R > 0 && (dy == nullptr || x_src == nullptr || h_perm == nullptr || topk_ids == nullptr ||
                topk_w == nullptr || row_to_slot == nullptr || slot_to_row == nullptr || w_perm == nullptr ||
                dx == nullptr || d_logits == nullptr))
    return LIGER_MOE_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(x_src) || !aligned16(h_perm) || !aligned16(gu_perm) || !aligned16(w_gate_up) ||
      !aligned16(w_down) || !aligned16(dx) || !aligned16(dw_gate_up) || !aligned16(dw_down))
    return LIGER_MOE_ERR_MISALIGNED;
  const bool recompute = (gu_perm == nullptr);
  const bool gather = (x != nullptr);  // token-major inputs: x and dY rows gathered inside the GEMMs
  const bool f16_ws = bwd_f16_possible(R, act != LIGER_MOE_ACT_RELU2, gather);
  const size_t need = bwd_workspace_bytes(R, H, I, E, recompute, gather, f16_ws);
  if (workspace == nullptr) {
    *workspace_bytes = need;
    return LIGER_MOE_OK;
  }
  if (*workspace_bytes < need) return LIGER_MOE_ERR_CAPACITY;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LIGER_MOE_ERR_MISALIGNED;
  PdlScope pdl(R);
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  uint8_t* cur = static_cast<uint8_t*>(workspace);
  const long long Rp = padded_rows(R, E);
  ScheduleBufs sb;
  sb.tile_prefix = carve<int32_t>(cur, schedule_bytes(E));
  sb.pad_indptr = carve<int32_t>(cur, schedule_bytes(E));
  sb.pair_prefix = carve<int32_t>(cur, schedule_bytes(E));
  int32_t* light = carve<int32_t>(cur, schedule_bytes(E));
  int32_t* heavy = carve<int32_t>(cur, schedule_bytes(E));
  if (split_schedule(R, E)) {
    sb.light_prefix = light;
    sb.heavy_pair_prefix = heavy;
  }
  sb.order = carve<int32_t>(cur, schedule_bytes(E));
  sb.order_info = carve<int32_t>(cur, 4 * schedule_bytes(E));
  sb.claims = carve<int>(cur, kClaimBytes);
  int32_t* tile_prefix = sb.tile_prefix;
  int32_t* pad_indptr = sb.pad_indptr;
  int32_t* pair_prefix = sb.pair_prefix;
  uint16_t* dy_perm = gather ? nullptr : carve<uint16_t>(cur, static_cast<size_t>(R) * H * 2);
  uint16_t* dgu = carve<uint16_t>(cur, static_cast<size_t>(Rp) * 2 * I * 2 * 2);
  uint16_t* dx_perm = carve<uint16_t>(cur, static_cast<size_t>(R) * H * 2);
  uint16_t* hw_perm = carve<uint16_t>(cur, static_cast<size_t>(Rp) * I * 2 * 2);
  float* gdot = carve<float>(cur, static_cast<size_t>(R) * gdot_tiles(I) * 4);
  float* gu_ws = recompute ? carve<float>(cur, static_cast<size_t>(R) * 2 * I * 4) : nullptr;
  unsigned* f16_words = f16_ws ? carve<unsigned>(cur, f16_words_bytes(E)) : nullptr;
  uint16_t* x16 = f16_ws ? carve<uint16_t>(cur, static_cast<size_t>(R) * H * 2) : nullptr;
  uint16_t* dy16 = f16_ws ? carve<uint16_t>(cur, static_cast<size_t>(R) * H * 2) : nullptr;
  const bool f16 = f16_ws && g_dw_fp16.load() != 0;
  if (f16) sb.f16_words = f16_words;  // zeroed (and the any-heavy word set) by the schedule kernel

  BwdGemmArgs a{};
  a.m_indptr = m_indptr;
  a.tile_prefix = tile_prefix;
  a.pair_prefix = pair_prefix;
  a.light_prefix = sb.light_prefix;
  a.heavy_pair_prefix = sb.heavy_pair_prefix;
  a.sched_order = sb.order;
  a.sched_info = sb.order_info;
  a.claims = sb.claims;
  a.w_gate_up = static_cast<const uint16_t*>(w_gate_up);
  a.w_down = static_cast<const uint16_t*>(w_down);
  a.x_perm = static_cast<const uint16_t*>(x_perm);
  a.x = static_cast<const uint16_t*>(x);
  a.dy = static_cast<const uint16_t*>(dy);
  a.dy_perm = dy_perm;
  a.row_to_slot = row_to_slot;
  a.T = T;
  a.k = k;
  a.h_perm = static_cast<const uint16_t*>(h_perm);
  a.gu = recompute ? gu_ws : gu_perm;
  a.w_perm = w_perm;
  a.pad_indptr = pad_indptr;
  a.R_pad = Rp;
  a.hw_perm = hw_perm;
  a.dgu = dgu;
  a.dx_perm = dx_perm;
  a.gdot = gdot;
  a.dw_gate_up = static_cast<uint16_t*>(dw_gate_up);
  a.dw_down = static_cast<uint16_t*>(dw_down);
  a.R = R;
  a.H = H;
  a.I = I;
  a.E = E;
  a.nin = act == LIGER_MOE_ACT_RELU2 ? I : 2 * I;  // ReLU²: one up weight, one factor, da [.., I]
  if (f16) {
    a.x16 = x16;
    a.dy16 = dy16;
    a.f16_words = f16_words;
    a.f16_rows = kF16Rows;
  }

  if (R > 0) {
    if (int rc = launch_tile_schedule(m_indptr, E, R, sb, dev, s)) return rc;
    if (f16) {
      // the largest |dY| and |x|, then dy_perm with the fp16 copies of the dY and x rows
      if (int rc = launch_f16_prep(static_cast<const uint16_t*>(dy), a.x_perm, slot_to_row, T, H, k, f16_words, dev,
                                   s))
        return rc;
      if (int rc = launch_scatter_rows_f16(static_cast<const uint16_t*>(dy), a.x_perm, slot_to_row, T, H, k, m_indptr,
                                           E, dy_perm, dy16, x16, f16_words, dev, s))
        return rc;
    } else if (!gather) {  // dy_perm[r] = dY[token of r]: the dH and dW_down GEMMs read it as dense tiles
      if (int rc = launch_scatter_rows(static_cast<const uint16_t*>(dy), slot_to_row, T, H, k, dy_perm, dev, s))
        return rc;
    }
    if (recompute) {
      FwdGemmArgs f{};
      f.x_perm = a.x_perm;
      f.x = a.x;
      f.row_to_slot = row_to_slot;
      f.T = T;
      f.k = k;
      f.m_indptr = m_indptr;
      f.tile_prefix = tile_prefix;
      f.w_gate_up = a.w_gate_up;
      f.w_down = a.w_down;
      f.w_perm = w_perm;
      f.R = R;
      f.H = H;
      f.I = I;
      f.E = E;
      f.gu_perm = gu_ws;
      f.act = act;
      f.act_clamp = clamp;
      if (int rc = launch_gate_up(f, dev, s)) return rc;
    }
    if (int rc = launch_bwd_dh(a, dev, s)) return rc;
    if (int rc = launch_bwd_dx(a, dev, s)) return rc;
    // The weight-gradient GEMMs, the per-token sum of dX_perm and d_logits all depend only on
    // what is done by now.  The two small kernels go to a side stream, where their CTAs share
    // the SMs (and the spare bandwidth) with the GEMMs' one CTA per SM; the GEMMs are enqueued
    // first so that they take their SMs first.  Measured on GB300: 1.864 -> 1.844 ms per layer
    // step at T=8192, H=2048, I=512, E=256, k=8 (in order, or with the side work first: 1.869).
    if (SideStream* side = side_stream(dev.device, s)) {
      if (cudaEventRecord(side->fork, s) != cudaSuccess) {
        set_cuda_error(cudaGetLastError(), "cudaEventRecord");
        return LIGER_MOE_ERR_LAUNCH;
      }
      int rc = launch_bwd_dw(a, dev, s);
      cudaStreamWaitEvent(side->stream, side->fork, 0);
      if (rc == LIGER_MOE_OK)
        rc = launch_combine(dx_perm, slot_to_row, T, H, k, static_cast<uint16_t*>(dx), dev, side->stream);
      if (rc == LIGER_MOE_OK)
        rc = launch_router_grad(gdot, gdot_tiles(I), topk_ids, topk_w, slot_to_row, T, E, k, d_logits, dev,
                                side->stream);
      // joined on every path, so that a capture of the caller's stream stays well formed
      cudaEventRecord(side->join, side->stream);
      cudaStreamWaitEvent(s, side->join, 0);
      if (rc == LIGER_MOE_OK) rc = check_launch("side stream join");
      return rc;
    }
    if (int rc = launch_combine(dx_perm, slot_to_row, T, H, k, static_cast<uint16_t*>(dx), dev, s)) return rc;
  }
  if (int rc = launch_bwd_dw(a, dev, s)) return rc;
  if (R > 0)
    return launch_router_grad(gdot, gdot_tiles(I), topk_ids, topk_w, slot_to_row, T, E, k, d_logits, dev, s);
  return LIGER_MOE_OK;
}

}  // namespace

LIGER_MOE_API int liger_moe_bwd_dx_dw(const void* dy, const void* x_perm, const void* h_perm, const float* gu_perm,
                                      const int32_t* topk_ids, const float* topk_w, const int32_t* m_indptr,
                                      const int32_t* row_to_slot, const int32_t* slot_to_row, const float* w_perm,
                                      const void* w_gate_up, const void* w_down, int T, int H, int I, int E, int k,
                                      void* dx, void* dw_gate_up, void* dw_down, float* d_logits, void* workspace,
                                      size_t* workspace_bytes, void* stream) {
  return bwd_dx_dw_impl(dy, x_perm, nullptr, h_perm, gu_perm, topk_ids, topk_w, m_indptr, row_to_slot, slot_to_row,
                        w_perm, w_gate_up, w_down, T, H, I, E, k, dx, dw_gate_up, dw_down, d_logits, workspace,
                        workspace_bytes, stream);
}

LIGER_MOE_API int liger_moe_bwd_dx_dw_glu(const void* dy, const void* x_perm, const void* h_perm,
                                          const float* gu_perm, const int32_t* topk_ids, const float* topk_w,
                                          const int32_t* m_indptr, const int32_t* row_to_slot,
                                          const int32_t* slot_to_row, const float* w_perm, const void* w_gate_up,
                                          const void* w_down, int T, int H, int I, int E, int k, int activation,
                                          float clamp, void* dx, void* dw_gate_up, void* dw_down, float* d_logits,
                                          void* workspace, size_t* workspace_bytes, void* stream) {
  return bwd_dx_dw_impl(dy, x_perm, nullptr, h_perm, gu_perm, topk_ids, topk_w, m_indptr, row_to_slot, slot_to_row,
                        w_perm, w_gate_up, w_down, T, H, I, E, k, dx, dw_gate_up, dw_down, d_logits, workspace,
                        workspace_bytes, stream, activation, clamp);
}

LIGER_MOE_API int liger_moe_bwd_dx_dw_gather(const void* dy, const void* x, const void* h_perm, const float* gu_perm,
                                             const int32_t* topk_ids, const float* topk_w, const int32_t* m_indptr,
                                             const int32_t* row_to_slot, const int32_t* slot_to_row,
                                             const float* w_perm, const void* w_gate_up, const void* w_down, int T,
                                             int H, int I, int E, int k, void* dx, void* dw_gate_up, void* dw_down,
                                             float* d_logits, void* workspace, size_t* workspace_bytes,
                                             void* stream) {
  if (static_cast<long long>(T) * k > 0 && x == nullptr) return LIGER_MOE_ERR_INVALID_ARG;
  return bwd_dx_dw_impl(dy, nullptr, x, h_perm, gu_perm, topk_ids, topk_w, m_indptr, row_to_slot, slot_to_row, w_perm,
                        w_gate_up, w_down, T, H, I, E, k, dx, dw_gate_up, dw_down, d_logits, workspace,
                        workspace_bytes, stream);
}

LIGER_MOE_API int liger_moe_router_logits(const void* x, const void* w_router, const float* bias, int T, int H,
                                          int E, float* logits, void* stream) {
  if (T < 0 || H < 1 || E < 1) return LIGER_MOE_ERR_INVALID_ARG;
  if (E > kMaxExperts || 1LL * T * E > kIndexLimit * 4LL) return LIGER_MOE_ERR_CAPACITY;
  if (H % 64 != 0) return LIGER_MOE_ERR_MISALIGNED;
  if (w_router == nullptr || (T > 0 && (x == nullptr || logits == nullptr))) return LIGER_MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(logits)) return LIGER_MOE_ERR_MISALIGNED;
  PdlScope pdl(T);
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  return launch_router_logits(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(w_router), bias, T, H,
                              E, logits, dev, static_cast<cudaStream_t>(stream));
}

LIGER_MOE_API int liger_moe_router_bwd(const float* d_logits, const int32_t* topk_ids, const int32_t* m_indptr,
                                       const int32_t* row_to_slot, const void* x, const void* w_router, int T, int H,
                                       int E, int k, void* dx, void* dw_router, float* d_bias, void* stream) {
  if (int rc = check_topk(T, E, k)) return rc;
  if (H < 1) return LIGER_MOE_ERR_INVALID_ARG;
  if (H % 64 != 0) return LIGER_MOE_ERR_MISALIGNED;
  if (m_indptr == nullptr || w_router == nullptr || dw_router == nullptr) return LIGER_MOE_ERR_INVALID_ARG;
  if (T > 0 && (d_logits == nullptr || topk_ids == nullptr || row_to_slot == nullptr || x == nullptr ||
                dx == nullptr))
    return LIGER_MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(dx)) return LIGER_MOE_ERR_MISALIGNED;
  PdlScope pdl(static_cast<long long>(T) * k);
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  return launch_router_bwd(d_logits, topk_ids, m_indptr, row_to_slot, static_cast<const uint16_t*>(x),
                           static_cast<const uint16_t*>(w_router), T, H, E, k, static_cast<uint16_t*>(dx),
                           static_cast<uint16_t*>(dw_router), d_bias, dev, static_cast<cudaStream_t>(stream));
}

LIGER_MOE_API int liger_moe_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return LIGER_MOE_ERR_INVALID_ARG;
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  return launch_bounded_wait_selftest(static_cast<uint64_t>(limit_us) * 1000ull, dev, static_cast<cudaStream_t>(stream));
}

LIGER_MOE_API int liger_moe_set_dw_fp16(int on) {
  if (on != 0 && on != 1) return LIGER_MOE_ERR_INVALID_ARG;
  g_dw_fp16.store(on);
  return LIGER_MOE_OK;
}

LIGER_MOE_API int liger_moe_trace_enable(int on) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  for (const TraceRecord& r : g_trace) {
    g_event_pool.push_back(r.start);
    g_event_pool.push_back(r.stop);
  }
  g_trace.clear();
  g_trace_on.store(on ? 1 : 0);
  return LIGER_MOE_OK;
}

LIGER_MOE_API int liger_moe_trace_count(void) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  return static_cast<int>(g_trace.size());
}

LIGER_MOE_API int liger_moe_trace_get(int i, const char** name, float* ms) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  if (i < 0 || i >= static_cast<int>(g_trace.size()) || name == nullptr || ms == nullptr)
    return LIGER_MOE_ERR_INVALID_ARG;
  const TraceRecord& r = g_trace[i];
  *name = r.name;
  cudaError_t e = cudaEventSynchronize(r.stop);
  if (e == cudaSuccess) e = cudaEventElapsedTime(ms, r.start, r.stop);
  if (e != cudaSuccess) {
    set_cuda_error(e, "trace event");
    return LIGER_MOE_ERR_LAUNCH;
  }
  return LIGER_MOE_OK;
}

LIGER_MOE_API int liger_moe_trace_launches(int i, int* launches) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  if (i < 0 || i >= static_cast<int>(g_trace.size()) || launches == nullptr) return LIGER_MOE_ERR_INVALID_ARG;
  *launches = g_trace[i].launches;
  return LIGER_MOE_OK;
}

LIGER_MOE_API int liger_moe_device_error(void* stream, int* flags) {
  if (flags == nullptr) return LIGER_MOE_ERR_INVALID_ARG;
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* taken = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&taken, g_device_error_taken);
  if (e == cudaSuccess) e = launch_kernel(take_device_error_kernel, dim3(1), dim3(1), 0, s, "take_device_error", 1);
  int v = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&v, taken, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    set_cuda_error(e, "reading the device error flag");
    return LIGER_MOE_ERR_LAUNCH;
  }
  *flags = v;
  return v ? LIGER_MOE_ERR_DEVICE : LIGER_MOE_OK;
}
