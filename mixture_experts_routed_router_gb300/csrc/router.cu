// Backward of the router projection logits = x Wr^T + b, for the routed layer's own logit
// gradient (LightMoE README, "MoE training": the router-gradient kernels produce d_logits; the
// router itself belongs to the host framework, whose plainest form is one linear layer).
//
// The layer's d_logits are zero off each token's top-k selection (the renormalised softmax
// depends only on the selected logits), so both products reduce to k-term row sums in fp32:
//   dX[t, :]  = bf16( dX[t, :] + sum_j d_logits[t, id_j] * Wr[id_j, :] )   (j = 0..k-1, in order)
//   dWr[e, :] = bf16( sum over expert e's routed rows r of d_logits[t(r), e] * x[t(r), :] )
//   dbias[e]  = sum over the same rows of d_logits[t(r), e]
// That is 2 R H multiply-adds instead of the 4 T E H of two dense GEMMs, exact fp32
// accumulation and no bf16 rounding of d_logits.  Entries of d_logits off the selection are
// not read.
//
// router_dx_kernel: one warp per (token, 512-column segment), 16-byte vectors (like the combine).
// router_dw_kernel: one CTA per (expert, 256-column block); its 8 warps split each pass of the
// expert's rows into 8 contiguous ranges (rows in token order), then the partial sums are added
// in warp order, so the result does not depend on timing.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace lmoe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kDwWarps = 8;
constexpr int kDwCols = 256;  // columns per CTA: 32 lanes x 8

__device__ __forceinline__ void fma8(float (&acc)[8], float d, const uint4& v) {
  acc[0] += d * bf16_lo(v.x);
  acc[1] += d * bf16_hi(v.x);
  acc[2] += d * bf16_lo(v.y);
  acc[3] += d * bf16_hi(v.y);
  acc[4] += d * bf16_lo(v.z);
  acc[5] += d * bf16_hi(v.z);
  acc[6] += d * bf16_lo(v.w);
  acc[7] += d * bf16_hi(v.w);
}

// Work item = (token, segment of 64 16-byte chunks = 512 columns), one warp per item, as in the
// combine: a small batch still spreads over many warps.  Each lane owns two chunks; the k rows of
// Wr are read four at a time (eight independent 16-byte loads in flight), and the lane's dX chunks
// are loaded before them.
constexpr int kDxLaneChunks = 2;
constexpr int kDxSeg = 32 * kDxLaneChunks;

__global__ void __launch_bounds__(256) router_dx_kernel(const float* __restrict__ d_logits,
                                                        const int32_t* __restrict__ ids,
                                                        const uint16_t* __restrict__ w_router, int T, int H, int E,
                                                        int k, uint16_t* __restrict__ dx, int* err) {
  griddep_wait();  // earlier kernels on the stream are complete
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int chunks = H >> 3;  // 16-byte chunks of a row
  const int nseg = (chunks + kDxSeg - 1) / kDxSeg;
  const long long items = static_cast<long long>(T) * nseg;
  for (long long it = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; it < items;
       it += nwarps) {
    const long long t = it / nseg;
    const int seg = static_cast<int>(it - t * nseg);
    int id = 0;
    float d = 0.f;
    bool bad = false;
    if (lane < k) {
      id = __ldg(ids + t * k + lane);
      bad = static_cast<unsigned>(id) >= static_cast<unsigned>(E);
      if (!bad) d = __ldg(d_logits + t * E + id);
    }
    if (__any_sync(kFull, bad)) {
      if (lane == 0 && seg == 0) atomicOr(err, LIGER_MOE_DEVERR_BAD_EXPERT_ID);
      continue;
    }
    uint4* row = reinterpret_cast<uint4*>(dx + static_cast<size_t>(t) * H);
    const int c0 = seg * kDxSeg + lane;  // this lane's chunks: c0, c0 + 32
    uint4 base[kDxLaneChunks];
#pragma unroll
    for (int q = 0; q < kDxLaneChunks; ++q)
      if (c0 + 32 * q < chunks) base[q] = __ldcs(row + c0 + 32 * q);  // read once, overwritten below
    float acc[kDxLaneChunks][8];
#pragma unroll
    for (int q = 0; q < kDxLaneChunks; ++q)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[q][i] = 0.f;
    for (int j0 = 0; j0 < k; j0 += 4) {
      uint4 v[4][kDxLaneChunks];
      float dj[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int e = __shfl_sync(kFull, id, (j0 + jj) & 31);
        dj[jj] = __shfl_sync(kFull, d, (j0 + jj) & 31);
        if (j0 + jj < k) {
          const uint4* w = reinterpret_cast<const uint4*>(w_router + static_cast<size_t>(e) * H);
#pragma unroll
          for (int q = 0; q < kDxLaneChunks; ++q)
            if (c0 + 32 * q < chunks) v[jj][q] = __ldg(w + c0 + 32 * q);
        }
      }
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        if (j0 + jj >= k) break;
#pragma unroll
        for (int q = 0; q < kDxLaneChunks; ++q)
          if (c0 + 32 * q < chunks) fma8(acc[q], dj[jj], v[jj][q]);
      }
    }
#pragma unroll
    for (int q = 0; q < kDxLaneChunks; ++q) {
      const int c = c0 + 32 * q;
      if (c >= chunks) continue;
      const uint4 b = base[q];
      uint4 o;
      o.x = pack_bf16x2(bf16_lo(b.x) + acc[q][0], bf16_hi(b.x) + acc[q][1]);
      o.y = pack_bf16x2(bf16_lo(b.y) + acc[q][2], bf16_hi(b.y) + acc[q][3]);
      o.z = pack_bf16x2(bf16_lo(b.z) + acc[q][4], bf16_hi(b.z) + acc[q][5]);
      o.w = pack_bf16x2(bf16_lo(b.w) + acc[q][6], bf16_hi(b.w) + acc[q][7]);
      row[c] = o;
    }
  }
}

// grid (E, ceil(H / 256)), block kDwWarps warps.  m_indptr / row_to_slot: the dispatch of the same
// routing (expert e's rows in token order); the token of row r is row_to_slot[r] / k.  The
// expert's rows are taken in passes of up to kDwStage: the whole CTA first stages their tokens
// and d_logits entries in shared memory (every load independent), then each warp streams the x
// rows of its contiguous share of the pass, eight rows in flight.
constexpr int kDwStage = 2048;
constexpr int kDwUnroll = 8;

__global__ void __launch_bounds__(kDwWarps * 32) router_dw_kernel(const float* __restrict__ d_logits,
                                                                  const int32_t* __restrict__ m_indptr,
                                                                  const int32_t* __restrict__ row_to_slot,
                                                                  const uint16_t* __restrict__ x, int H, int E,
                                                                  int k, long long R, uint16_t* __restrict__ dw,
                                                                  float* __restrict__ d_bias, int* err) {
  griddep_wait();  // earlier kernels on the stream are complete
  griddep_launch_dependents();
  __shared__ float part[kDwWarps][kDwCols];
  __shared__ float part_b[kDwWarps];
  __shared__ int s_tok[kDwStage];
  __shared__ float s_d[kDwStage];
  const int e = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = blockIdx.y * kDwCols + lane * 8;
  const bool col_ok = col < H;
  const int r0 = __ldg(m_indptr + e), r1 = __ldg(m_indptr + e + 1);
  const bool indptr_ok = r1 >= r0 && r0 >= 0 && r1 <= R;
  if (threadIdx.x == 0 && !indptr_ok) atomicOr(err, LIGER_MOE_DEVERR_BAD_INDPTR);
  const int n_all = indptr_ok ? r1 - r0 : 0;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  float db = 0.f;
  bool bad = false;
  for (int base = 0; base < n_all; base += kDwStage) {
    const int n = min(kDwStage, n_all - base);
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const int sl = __ldg(row_to_slot + r0 + base + i);
      const bool ok = static_cast<unsigned long long>(sl) < static_cast<unsigned long long>(R);
      bad |= !ok;
      const int t = ok ? sl / k : 0;
      s_tok[i] = t;
      s_d[i] = __ldg(d_logits + static_cast<size_t>(t) * E + e);
    }
    __syncthreads();
    const int a = n * warp / kDwWarps, b = n * (warp + 1) / kDwWarps;
    int i = a;
    for (; i + kDwUnroll <= b; i += kDwUnroll) {
      uint4 v[kDwUnroll];
#pragma unroll
      for (int q = 0; q < kDwUnroll; ++q)
        if (col_ok) v[q] = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(s_tok[i + q]) * H + col));
#pragma unroll
      for (int q = 0; q < kDwUnroll; ++q) {
        const float d = s_d[i + q];
        if (col_ok) fma8(acc, d, v[q]);
        db += d;
      }
    }
    for (; i < b; ++i) {
      const float d = s_d[i];
      if (col_ok) fma8(acc, d, __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(s_tok[i]) * H + col)));
      db += d;
    }
    __syncthreads();  // the staged rows are consumed before the next pass overwrites them
  }
  if (bad) atomicOr(err, LIGER_MOE_DEVERR_BAD_ROW);
#pragma unroll
  for (int q = 0; q < 8; ++q) part[warp][lane * 8 + q] = acc[q];
  if (lane == 0) part_b[warp] = db;
  __syncthreads();
  // thread c adds column c of the kDwWarps partials in warp order
  for (int c = threadIdx.x; c < kDwCols; c += blockDim.x) {
    const int gc = blockIdx.y * kDwCols + c;
    if (gc >= H) continue;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kDwWarps; ++w) sum += part[w][c];
    dw[static_cast<size_t>(e) * H + gc] = static_cast<uint16_t>(pack_bf16x2(sum, 0.f) & 0xFFFFu);
  }
  if (d_bias != nullptr && blockIdx.y == 0 && threadIdx.x == 0) {
    float sum = 0.f;
    for (int w = 0; w < kDwWarps; ++w) sum += part_b[w];
    d_bias[e] = sum;
  }
}

int grid_warps(long long nwarps_needed, int warps_per_block, const DeviceInfo& dev) {
  long long blocks = (nwarps_needed + warps_per_block - 1) / warps_per_block;
  const long long cap = static_cast<long long>(dev.sm_count) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<int>(blocks);
}

}  // namespace

int launch_router_bwd(const float* d_logits, const int32_t* topk_ids, const int32_t* m_indptr,
                      const int32_t* row_to_slot, const uint16_t* x, const uint16_t* w_router, int T, int H, int E,
                      int k, uint16_t* dx, uint16_t* dw_router, float* d_bias, const DeviceInfo& dev,
                      cudaStream_t s) {
  const long long R = static_cast<long long>(T) * k;
  if (T > 0) {
    {
      KernelScope trace("router_dx", s);
      const long long items = static_cast<long long>(T) * ((H / 8 + kDxSeg - 1) / kDxSeg);
      launch_kernel(router_dx_kernel, dim3(grid_warps(items, 8, dev)), dim3(256), 0, s, "router_dx", 1, d_logits,
                    topk_ids, w_router, T, H, E, k, dx, dev.err_flag);
    }
    if (int rc = check_launch("router_dx")) return rc;
  }
  {
    // every expert's block is written, zero for an expert with no rows
    KernelScope trace("router_dw", s);
    const dim3 grid(static_cast<unsigned>(E), static_cast<unsigned>((H + kDwCols - 1) / kDwCols));
    launch_kernel(router_dw_kernel, dim3(grid), dim3(kDwWarps * 32), 0, s, "router_dw", 1, d_logits, m_indptr,
                  row_to_slot, x, H, E, k, R, dw_router, d_bias, dev.err_flag);
  }
  return check_launch("router_dw");
}

}  // namespace lmoe
