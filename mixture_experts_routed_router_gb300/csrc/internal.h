// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>

#include "../../include/liger_moe.h"

namespace lmoe {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr long long kIndexLimit = 2147483647LL;  // int32 row / slot indices and TMA coordinates

// Validates T, E and k of an entry point that takes top-k routing (a liger_moe_status).
int check_topk(long long T, int E, int k);

// Records a CUDA error message for liger_moe_last_cuda_error().
void set_cuda_error(cudaError_t e, const char* where);
// Returns LIGER_MOE_OK or LIGER_MOE_ERR_LAUNCH (recording the error).
int check_launch(const char* where);

// Per-device state: SM count and the device error flag's address.
struct DeviceInfo {
  int device;
  int sm_count;
  int* err_flag;  // device address of the library's error word for this device
};
// Fills `info` for the current device; returns a liger_moe_status.
int current_device(DeviceInfo* info);

// ---- launchers (each enqueues on `s`; return a liger_moe_status)
int launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s);

// Bytes of scratch the dispatch kernels use for R slots and E experts (per-chunk histograms),
// and the workspace size the dispatch entry point asks for (that, plus alignment slack).
size_t dispatch_scratch_bytes(long long R, int E);
size_t dispatch_workspace_bytes(long long R, int E);
int launch_dispatch(const int32_t* ids, const float* w, const uint16_t* x, int T, int H, int E, int k,
                    int32_t* counts, int32_t* m_indptr, int32_t* row_to_slot, int32_t* slot_to_row, float* w_perm,
                    uint16_t* x_perm, void* workspace, const DeviceInfo& dev, cudaStream_t s);

// The expert-major row copy dst[r, :] = src[row_to_slot[r] / k, :], written by token:
// dst[slot_to_row[t*k + j], :] = src[t, :] for j < k (each token row read once).
int launch_scatter_rows(const uint16_t* src, const int32_t* slot_to_row, int T, int H, int k, uint16_t* dst,
                        const DeviceInfo& dev, cudaStream_t s);

// ---------------------------------------------------------------- fp16 weight-gradient operands
// Experts with at least f16 rows (kF16Rows) take their weight gradients in one fp16 MMA per K step
// instead of two bf16 ones (the hi and lo parts): x and dY rows as fp16(v 2^s) with s from the
// tensor's largest magnitude, and the dH epilogue's dgu and w h as fp16 with fixed offsets from
// those scales.  An expert whose fp16 parts fall outside their window (f16_in_range) falls back
// to the hi / lo parts, which a second dH pass then writes.  Words in the backward's workspace:
//   [kF16MaxX]  largest |x| (float bits),  [kF16MaxDy] largest |dY|,  [kF16Any] 1 when some
//   expert has at least f16 rows,  [kF16Range + e] / [kF16Range + E + e] largest |scaled dgu| /
//   |scaled w h| of expert e (float bits; atomicMax of the dH epilogue).
constexpr int kF16Rows = 384;
// Routed rows below which the backward never takes the fp16 pass: at fewer rows its fixed costs (four
// launches, which leave at once when no expert reaches kF16Rows) were measured at 1.3 % of a step
// (8192 and 16384 rows, 64-128 per expert) and even a skewed batch has few heavy rows to gain on.
constexpr long long kF16MinR = 32768;
constexpr int kF16MaxX = 0, kF16MaxDy = 1, kF16Any = 2, kF16Range = 4;
constexpr int kF16DguShift = -6;  // dgu scaled by 2^(s_dY - 6)
constexpr int kF16HwShift = 4;    // w h scaled by 2^4
inline size_t f16_words_bytes(int E) { return ((static_cast<size_t>(kF16Range) + 2 * E) * 4 + 255) / 256 * 256; }
// The largest |dY| and |x| (x read as x_perm[slot_to_row[t k]]) into words zeroed, and [kF16Any]
// set, by the schedule kernel (ScheduleBufs::f16_words).
int launch_f16_prep(const uint16_t* dy, const uint16_t* x_perm, const int32_t* slot_to_row, int T, int H, int k,
                    unsigned* words, const DeviceInfo& dev, cudaStream_t s);
// The backward's row copies in one launch: dy_perm[r, :] = dY[token of r, :] (bf16) with dy16[r, :]
// = fp16(dY[token of r, :] 2^s_dY), and x16[r, :] = fp16(x_perm[r, :] 2^s_x) (x_perm read once per
// token); the fp16 copies only when words[kF16Any] is set and the scales exist, and only for the rows
// the fp16 weight-gradient tiles read (experts with kF16Rows rows and the 15 rows after each).
int launch_scatter_rows_f16(const uint16_t* dy, const uint16_t* x_perm, const int32_t* slot_to_row, int T, int H,
                            int k, const int32_t* m_indptr, int E, uint16_t* dy_perm, uint16_t* dy16, uint16_t* x16,
                            const unsigned* words, const DeviceInfo& dev, cudaStream_t s);

#ifdef __CUDACC__
// 2^s as a float (s in [-126, 127]).
__device__ __forceinline__ float f16_pow2(int s) { return __uint_as_float(static_cast<unsigned>(127 + s) << 23); }
// The scale exponent s of a tensor whose largest magnitude has the float bits m: m 2^s in
// [2^14, 2^15), so every value within 2^28 of m keeps its full precision in fp16.  false when m is
// not finite or outside [2^-40, 2^41) (the fp16 operands are then not used); m = 0 gives s = 0.
__device__ __forceinline__ bool f16_scale_exp(unsigned m, int& s) {
  s = 0;
  if (m == 0u) return true;
  const int ex = static_cast<int>(m >> 23) - 127;  // m >= 0: no sign bit
  if (ex < -40 || ex > 40) return false;
  s = 14 - ex;
  return true;
}
// The window of an fp16 part's largest scaled magnitude: below 65504 (no overflow) and at least
// 2^-6, so that values down to 2^-8 of it are normal fp16 numbers.
__device__ __forceinline__ bool f16_in_range(unsigned m) {
  const float f = __uint_as_float(m);
  return f >= 0.015625f && f < 65504.f;
}
#endif

// y[t, :] = bf16(sum_j y_perm[slot_to_row[t*k+j], :]).
int launch_combine(const uint16_t* y_perm, const int32_t* slot_to_row, int T, int H, int k, uint16_t* y,
                   const DeviceInfo& dev, cudaStream_t s);

// d_logits from the per-row router-gradient partials (see grouped_gemm.cu).
int launch_router_grad(const float* gdot, int gdot_tiles, const int32_t* ids, const float* w,
                       const int32_t* slot_to_row, int T, int E, int k, float* d_logits, const DeviceInfo& dev,
                       cudaStream_t s);

// Router projection backward (router.cu): dx[t] = bf16(dx[t] + sum_j d_logits[t, id_j] Wr[id_j]),
// dw_router[e] = bf16(sum over e's rows of d_logits[t, e] x[t]), d_bias[e] (nullable).
int launch_router_bwd(const float* d_logits, const int32_t* topk_ids, const int32_t* m_indptr,
                      const int32_t* row_to_slot, const uint16_t* x, const uint16_t* w_router, int T, int H, int E,
                      int k, uint16_t* dx, uint16_t* dw_router, float* d_bias, const DeviceInfo& dev,
                      cudaStream_t s);

// Failure-detection self-test (selftest.cu): a bounded wait on a phase nothing completes.
int launch_bounded_wait_selftest(uint64_t limit_ns, const DeviceInfo& dev, cudaStream_t s);

// ---- grouped GEMMs (grouped_gemm.cu)
// Router projection logits[T, E] = x Wr^T (+ bias), fp32, as one dense tcgen05 GEMM.
int launch_router_logits(const uint16_t* x, const uint16_t* w_router, const float* bias, int T, int H, int E,
                         float* logits, const DeviceInfo& dev, cudaStream_t s);
// The device-built schedule of one layer call, carved from the caller's workspace:
//   tile_prefix[e]   sum over e' < e of ceil(rows_e' / 128) ([E] = total M tiles)
//   pad_indptr[e]    the padded row prefix (row counts rounded up to 16), or nullptr
//   pair_prefix[e]   the prefix of 256-row blocks (the 2-SM pair GEMMs' tiles), or nullptr
//   light_prefix[e], heavy_pair_prefix[e]   (both or neither) the 128-row tile prefix counting only
//                    experts below the forward / dX pair threshold, and the 256-row block prefix
//                    counting only those at or above it (the heavy / light split of those GEMMs)
//   order[i]         experts by rows, most first, equal rows in id order, or nullptr
//   order_info[4i..] the expert at order[i], its first row, its rows and its first padded row (the
//                    first row when there is no padded row prefix); with order, or nullptr
//   claims           kClaimSlots claim counters, zeroed by the schedule kernel (one per GEMM launch
//                    that may take its tiles in that order), then the skew flag, the count of
//                    experts at or above the dW_down pair threshold and the count at or above
//                    kF16Rows (the fp16 weight-gradient experts); or nullptr
struct ScheduleBufs {
  int32_t* tile_prefix = nullptr;
  int32_t* pad_indptr = nullptr;
  int32_t* pair_prefix = nullptr;
  int32_t* light_prefix = nullptr;
  int32_t* heavy_pair_prefix = nullptr;
  int32_t* order = nullptr;
  int32_t* order_info = nullptr;
  int* claims = nullptr;
  // the backward's fp16 operand words (kF16Range + 2E of them), or NULL: zeroed, and [kF16Any] set
  // when some expert has at least kF16Rows rows
  unsigned* f16_words = nullptr;
};
constexpr int kClaimSlots = 8;
// Claim counters of the launches that may use the dynamic order: the weight-gradient GEMMs.
enum ClaimSlot : int { kClaimDwGateUp = 0, kClaimDwDown = 1, kClaimDwGateUpF16 = 2, kClaimDwDownF16 = 3 };
size_t schedule_bytes(int E);                  // one [E+1] int32 array, 256-byte aligned
constexpr size_t kClaimBytes = 256;            // kClaimSlots counters and the skew flag, 256-byte aligned
int launch_tile_schedule(const int32_t* m_indptr, int E, long long R, const ScheduleBufs& b, const DeviceInfo& dev,
                         cudaStream_t s);
// True when R routed rows over E experts may take the heavy / light split of the forward and dX
// GEMMs (then the schedule needs light_prefix and heavy_pair_prefix).
bool split_schedule(long long R, int E);

struct FwdGemmArgs {
  const uint16_t* x_perm;       // [R, H]; used when x is NULL
  const uint16_t* x;            // [T, H] or NULL: A rows gathered by token (row_to_slot / k)
  const int32_t* row_to_slot;   // [R] (gather only)
  int T, k;                     // (gather only)
  const int32_t* m_indptr;
  const int32_t* tile_prefix;
  const int32_t* pair_prefix = nullptr;  // 256-row block prefix: the pair GEMMs run when set
  // heavy / light split (both set): 2-SM pairs over the experts with many rows, one CTA per tile
  // over the others (ScheduleBufs)
  const int32_t* light_prefix = nullptr;
  const int32_t* heavy_pair_prefix = nullptr;
  const uint16_t* w_gate_up;
  const uint16_t* w_down;
  const float* w_perm;
  long long R;
  int H, I, E;
  uint16_t* h_perm;  // nullable (then only gu is stored)
  float* gu_perm;     // [R, 2I] fp32, nullable
  uint16_t* y_perm;
  int act = LIGER_MOE_ACT_SWIGLU;  // gated activation of the gate/up epilogue
  float act_clamp = 0.f;
};
// gate/up GEMM + SwiGLU epilogue (h_perm may be NULL: only gu is stored).
int launch_gate_up(const FwdGemmArgs& a, const DeviceInfo& dev, cudaStream_t s);
// down GEMM + routing-weight epilogue.
int launch_down(const FwdGemmArgs& a, const DeviceInfo& dev, cudaStream_t s);

struct BwdGemmArgs {
  const int32_t* m_indptr;
  const int32_t* tile_prefix;
  const int32_t* pair_prefix = nullptr;  // 256-row block prefix: the pair GEMMs run when set
  const int32_t* light_prefix = nullptr;  // heavy / light split of the dX GEMM (ScheduleBufs)
  const int32_t* heavy_pair_prefix = nullptr;
  const int32_t* sched_order = nullptr;   // experts by rows (the weight gradients' dynamic order and split)
  const int32_t* sched_info = nullptr;    // [E][4]: each sorted expert's id, first row, rows, first padded row
  int* claims = nullptr;                  // the schedule's claim counters, skew flag and heavy counts
  const uint16_t* w_gate_up;
  const uint16_t* w_down;
  const uint16_t* x_perm;   // [R, H]; used when x is NULL
  const uint16_t* x;        // [T, H] or NULL: dW_gate_up's B rows gathered by token
  const uint16_t* dy;       // [T, H]: rows gathered by token when dy_perm is NULL
  const uint16_t* dy_perm;  // [R, H] dY[token of row] (read as dense tiles), or NULL
  const int32_t* row_to_slot;  // [R]; token of row r = row_to_slot[r] / k
  int T, k;
  const uint16_t* h_perm;
  const float* gu;       // [R, nin] fp32 [dh/dg | dh/du] (saved or recomputed); ReLU²: dh/da
  const float* w_perm;   // [R]
  // Weight-gradient operands in the padded row space: expert e's rows start at pad_indptr[e]
  // and are followed by zero rows up to a multiple of 16; R_pad (>= pad_indptr[E]) is the
  // row count of each half.
  const int32_t* pad_indptr;  // [E+1]
  long long R_pad;
  uint16_t* hw_perm;     // [2 R_pad, I]: hi rows bf16(w h), then lo rows bf16(w h - hi)
  uint16_t* dgu;         // [2 R_pad, 2I]: hi rows bf16(dgu), then lo rows bf16(dgu - hi)
  // fp16 weight-gradient operands (f16_words != NULL): x16 / dy16 [R, H] fp16 copies of x_perm and
  // dy_perm; an expert with at least f16_rows rows gets fp16(dgu 2^sg) and fp16(w h 2^sh) in the
  // lo rows of dgu and hw_perm instead of lo parts (the hi rows stay bf16 for the dX GEMM).
  const uint16_t* x16 = nullptr;
  const uint16_t* dy16 = nullptr;
  unsigned* f16_words = nullptr;
  int f16_rows = 0;
  uint16_t* dx_perm;     // [R, H]
  float* gdot;           // [R, ceil(I / 256)]
  uint16_t* dw_gate_up;  // [E, 2I, H]
  uint16_t* dw_down;     // [E, H, I]
  long long R;
  int H, I, E;
  // rows of the first weight per expert: 2I (gated: W_gu, factors [dh/dg | dh/du], dgu [.., 2I],
  // dW_gu [E, 2I, H]) or I (ReLU²: W_up, one factor dh/da, da [.., I], dW_up [E, I, H])
  int nin = 0;
};
int gdot_tiles(int I);
int launch_bwd_dh(const BwdGemmArgs& a, const DeviceInfo& dev, cudaStream_t s);
int launch_bwd_dx(const BwdGemmArgs& a, const DeviceInfo& dev, cudaStream_t s);
int launch_bwd_dw(const BwdGemmArgs& a, const DeviceInfo& dev, cudaStream_t s);

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Programmatic dependent launch: kernels launched with programmatic stream serialization, so each
// one's launch and prologue overlap the end of the kernel before it (every kernel waits on its
// predecessor before touching memory).  LIGER_MOE_PDL (read once): "0" never, any other non-empty
// value always, unset or empty for the calls with fewer than kPdlMaxRows routed rows only.  On
// GB300 it shortened a launch-bound step (256 tokens) by about 7 % but lengthened a 65536-row step
// by 1.5-4 %, wherever the GEMMs signalled their dependents.
constexpr long long kPdlMaxRows = 4096;
inline thread_local bool t_pdl_small = false;  // this thread is inside a call below kPdlMaxRows rows
// Marks the launches of one entry-point call as small (rows < kPdlMaxRows) or not.
struct PdlScope {
  bool prev;
  explicit PdlScope(long long rows) : prev(t_pdl_small) { t_pdl_small = rows < kPdlMaxRows; }
  ~PdlScope() { t_pdl_small = prev; }
  PdlScope(const PdlScope&) = delete;
  PdlScope& operator=(const PdlScope&) = delete;
};
bool pdl_enabled();  // for a launch made now by this thread

// Launches `kern` on `s` with programmatic stream serialization (when enabled) and, for
// cluster > 1, that cluster size; records and returns the launch error.
// Kernels launched by this thread (the trace's per-interval launch counts).
inline thread_local unsigned long long t_kernel_launches = 0;

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          const char* name, int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  if (e != cudaSuccess) set_cuda_error(e, name);
  ++t_kernel_launches;
  return e;
}

// Kernel trace (off by default): while enabled, each KernelScope brackets the launches made
// inside it with two CUDA events recorded on its stream and counts them (a scope named nullptr
// records nothing; traced scopes do not nest).
class KernelScope {
 public:
  KernelScope(const char* name, cudaStream_t s);
  ~KernelScope();
  KernelScope(const KernelScope&) = delete;
  KernelScope& operator=(const KernelScope&) = delete;

 private:
  const char* name_;
  cudaStream_t stream_;
  cudaEvent_t start_ = nullptr;
  unsigned long long launches0_ = 0;
};

}  // namespace lmoe
