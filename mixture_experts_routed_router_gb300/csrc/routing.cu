// Bandwidth-bound kernels of the routed MoE layer: router top-k, the
// deterministic expert-major dispatch, row gathers, the combine back to token
// order, and the router-logit gradient.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace lmoe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

// ============================================================================
// Router: top-k + renormalised softmax.  LightMoE README, "MoE inference"
// (top_k_ids distinct per token, top_k_weights float32) and "MoE training"
// (differentiable_probs).  One warp per token; lane i holds experts
// i, i+32, ... as the order-preserving bits of their logits (NaN lowest,
// -0.0 as +0.0).  Each round takes the warp-wide maximum of those bits with one
// reduction, then the smallest expert id among the lanes that hold it with a
// second: the largest logit wins, ties go to the smallest id.
// ============================================================================
__device__ __forceinline__ uint32_t route_ord(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN: below every number
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The logit back from its order bits: the map above is one-to-one on non-NaN floats (with -0.0
// folded into +0.0); a NaN comes back as a NaN.
__device__ __forceinline__ float ord_value(uint32_t ord) {
  if (ord == 0u) return __uint_as_float(0x7FFFFFFFu);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}

template <int EPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int32_t* __restrict__ ids, float* __restrict__ w) {
  griddep_wait();  // earlier kernels on the stream are complete
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long t = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const float* row = logits + t * E;
  // order bits + 1 of the lane's experts; 0 = no expert there, or already selected
  uint32_t ord1[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = i * 32 + lane;
    ord1[i] = (e < E) ? route_ord(__ldg(row + e)) + 1u : 0u;  // +inf gives 0xFF800001: no overflow
  }
  // the lane's best: largest value, then smallest slot i (= smallest id within the lane)
  uint32_t bv = 0u;
  int bi = 0;
  auto lane_best = [&]() {
    bv = 0u;
    bi = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (ord1[i] > bv) {
        bv = ord1[i];
        bi = i;
      }
  };
  lane_best();
  float my_val = 0.f, top = 0.f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    const uint32_t m = __reduce_max_sync(kFull, bv);
    const uint32_t cand = (bv == m) ? static_cast<uint32_t>(bi * 32 + lane) : 0xFFFFFFFFu;
    const int id = static_cast<int>(__reduce_min_sync(kFull, cand));
    if ((id & 31) == lane) {  // the winner's lane takes it out and finds its next best
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (i == (id >> 5)) ord1[i] = 0u;
      lane_best();
    }
    const float v = ord_value(m - 1u);  // the winner's logit, without another load
    if (j == 0) top = v;
    if (lane == j) {
      my_val = v;
      my_id = id;
    }
  }
  // w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0), sum in j order.
  const float ex = (lane < k) ? expf(my_val - top) : 0.f;
  float s = 0.f;
  for (int j = 0; j < k; ++j) s += __shfl_sync(kFull, ex, j);
  if (lane < k) {
    ids[t * k + lane] = my_id;
    w[t * k + lane] = ex / s;
  }
}

// ============================================================================
// Dispatch.  LightMoE README, "MoE training" / "Grouped GEMM"; LigerCute
// README, "Forward pass".  The R = T*k slots are cut into units of kUnit
// consecutive slots.
//   1. hist:    per unit, a histogram of its expert ids  -> hist[e][unit]
//   2. scan:    per expert, exclusive scan over units     -> base[e][unit], counts[e]
//   3. scatter: per unit, walking its slots in order, the row of slot s is
//               m_indptr[e] + base[e][unit] + (earlier slots of e in this unit)
// The rank inside a 32-slot group comes from __match_any_sync; groups are
// walked in order, so rows of one expert follow slot order (stable).
// ============================================================================
constexpr int kUnit = 256;
constexpr int kWarpsPerBlock = 8;
constexpr int kGroups = kUnit / 32;  // 32-slot groups of a unit (one per lane round)
constexpr int kNoSlot = -1;          // register placeholder past the last slot

__global__ void __launch_bounds__(kWarpsPerBlock * 32) dispatch_hist_kernel(const int32_t* __restrict__ ids,
                                                                           long long R, int E, int nunits,
                                                                           int32_t* __restrict__ hist, int* err) {
  griddep_wait();  // earlier kernels on the stream are complete
  griddep_launch_dependents();
  extern __shared__ int s_hist[];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x * kWarpsPerBlock + wib;
  int* h = s_hist + wib * E;
  for (int e = lane; e < E; e += 32) h[e] = 0;
  __syncwarp();
  if (unit >= nunits) return;
  const long long s0 = static_cast<long long>(unit) * kUnit;
  // all of the unit's ids are loaded first, so their latencies overlap
  int ev[kGroups];
#pragma unroll
  for (int g = 0; g < kGroups; ++g) {
    const long long s = s0 + g * 32 + lane;
    ev[g] = (s < R) ? __ldg(ids + s) : kNoSlot;
  }
  int bad = 0;
#pragma unroll
  for (int g = 0; g < kGroups; ++g) {
    if (s0 + g * 32 + lane >= R) continue;  // past the last slot
    const int e = ev[g];
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E))
      atomicAdd(&h[e], 1);
    else
      bad = 1;
  }
  if (__any_sync(kFull, bad) && lane == 0) atomicOr(err, LIGER_MOE_DEVERR_BAD_EXPERT_ID);
  __syncwarp();
  for (int e = lane; e < E; e += 32) hist[static_cast<size_t>(e) * nunits + unit] = h[e];
}

// One warp per expert: exclusive scan of hist[e][*] in place, counts[e] = total.
__global__ void __launch_bounds__(256) dispatch_scan_kernel(int32_t* __restrict__ hist, int nunits, int E,
                                                            int32_t* __restrict__ counts) {
  griddep_wait();  // earlier kernels on the stream are complete
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int e = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (e >= E) return;
  int32_t* row = hist + static_cast<size_t>(e) * nunits;
  int run = 0;
  for (int u0 = 0; u0 < nunits; u0 += 32) {
    const int u = u0 + lane;
    const int v = (u < nunits) ? row[u] : 0;
    int incl = v;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const int o = __shfl_up_sync(kFull, incl, m);
      if (lane >= m) incl += o;
    }
    if (u < nunits) row[u] = run + incl - v;
    run += __shfl_sync(kFull, incl, 31);
  }
  if (lane == 0) counts[e] = run;
}

// Exclusive scan of counts[0..E) into s_off[0..E] by one block (E <= 1024).
__device__ void block_exclusive_scan(const int32_t* __restrict__ counts, int E, int* s_off, int* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  for (int base = 0; base < E; base += blockDim.x) {
    const int carry = (base == 0) ? 0 : s_off[base];  // total of the earlier passes
    const int e = base + tid;
    const int v = (e < E) ? counts[e] : 0;
    int incl = v;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const int o = __shfl_up_sync(kFull, incl, m);
      if (lane >= m) incl += o;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int x = (lane < nwarps) ? s_warp[lane] : 0;
      int xi = x;
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const int o = __shfl_up_sync(kFull, xi, m);
        if (lane >= m) xi += o;
      }
      if (lane < nwarps) s_warp[lane] = xi - x;
    }
    __syncthreads();
    if (e < E) s_off[e] = carry + s_warp[warp] + incl - v;
    if (tid == blockDim.x - 1) s_off[min(base + static_cast<int>(blockDim.x), E)] = carry + s_warp[warp] + incl;
    __syncthreads();
  }
  if (E == 0 && tid == 0) s_off[0] = 0;
  __syncthreads();
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32) dispatch_scatter_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ w, long long R, int E, int nunits,
    const int32_t* __restrict__ base, const int32_t* __restrict__ counts, int32_t* __restrict__ m_indptr,
    int32_t* __restrict__ row_to_slot, int32_t* __restrict__ slot_to_row, float* __restrict__ w_perm) {
  griddep_wait();  // earlier kernels on the stream are complete
  griddep_launch_dependents();
  extern __shared__ int smem[];
  int* s_off = smem;                       // [E + 1]
  int* s_warp = s_off + (E + 1);           // [32]
  int* s_cnt = s_warp + 32;                // [kWarpsPerBlock][E]
  block_exclusive_scan(counts, E, s_off, s_warp);
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) m_indptr[e] = s_off[e];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x * kWarpsPerBlock + wib;
  if (unit >= nunits) return;
  int* cnt = s_cnt + wib * E;
  for (int e = lane; e < E; e += 32) cnt[e] = s_off[e] + __ldg(base + static_cast<size_t>(e) * nunits + unit);
  __syncwarp();
  const long long s0 = static_cast<long long>(unit) * kUnit;
  // the unit's ids and weights are loaded first, so their latencies overlap; the rounds below
  // then only wait on shared memory
  int ev[kGroups];
  float wv[kGroups];
#pragma unroll
  for (int g = 0; g < kGroups; ++g) {
    const long long s = s0 + g * 32 + lane;
    ev[g] = (s < R) ? __ldg(ids + s) : kNoSlot;
    wv[g] = (w_perm != nullptr && s < R) ? __ldg(w + s) : 0.f;
  }
#pragma unroll
  for (int g = 0; g < kGroups; ++g) {
    const long long s = s0 + g * 32 + lane;
    int e = ev[g];
    const bool ok = s < R && static_cast<unsigned>(e) < static_cast<unsigned>(E);
    if (!ok) e = E + lane;  // unique per lane: never matches a real expert
    const unsigned peers = __match_any_sync(kFull, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int leader = __ffs(peers) - 1;
    int pos = 0;
    if (ok) pos = cnt[e];
    __syncwarp();
    if (ok && lane == leader) cnt[e] = pos + __popc(peers);
    __syncwarp();
    if (ok) {
      const int r = pos + rank;
      slot_to_row[s] = r;
      row_to_slot[r] = static_cast<int32_t>(s);
      if (w_perm) w_perm[r] = wv[g];
    }
  }
}

// The three steps in one block for small batches: one warp per unit, kSmallUnits units at most
// (R <= 8192 slots) and at most kSmallExperts experts, so that every unit's histogram fits in
// shared memory.  The units, their order and the ranks inside a unit are those of the three
// kernels above, so the outputs are identical; two launches fewer matter when a whole layer
// step takes tens of microseconds.
constexpr int kSmallUnits = 32;
constexpr int kSmallExperts = 256;

__global__ void __launch_bounds__(kSmallUnits * 32) dispatch_small_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ w, long long R, int E, int nunits,
    int32_t* __restrict__ counts, int32_t* __restrict__ m_indptr, int32_t* __restrict__ row_to_slot,
    int32_t* __restrict__ slot_to_row, float* __restrict__ w_perm, int* err) {
  griddep_wait();  // earlier kernels on the stream are complete
  griddep_launch_dependents();
  __shared__ int s_hist[kSmallUnits * kSmallExperts];  // [unit][e]: counts, then the unit's base
  __shared__ int s_cnt[kSmallExperts];
  __shared__ int s_off[kSmallExperts + 1];
  __shared__ int s_warp[32];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = wib;
  int* h = s_hist + wib * E;
  for (int e = lane; e < E; e += 32) h[e] = 0;
  __syncwarp();
  const long long s0 = static_cast<long long>(unit) * kUnit;
  int ev[kGroups];
  float wv[kGroups];
#pragma unroll
  for (int g = 0; g < kGroups; ++g) {
    const long long s = s0 + g * 32 + lane;
    const bool in = unit < nunits && s < R;
    ev[g] = in ? __ldg(ids + s) : kNoSlot;
    wv[g] = (in && w_perm != nullptr) ? __ldg(w + s) : 0.f;
  }
  // 1. the unit's histogram
  int bad = 0;
#pragma unroll
  for (int g = 0; g < kGroups; ++g) {
    if (unit >= nunits || s0 + g * 32 + lane >= R) continue;
    const int e = ev[g];
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E))
      atomicAdd(&h[e], 1);
    else
      bad = 1;
  }
  if (__any_sync(kFull, bad) && lane == 0) atomicOr(err, LIGER_MOE_DEVERR_BAD_EXPERT_ID);
  __syncthreads();
  // 2. per expert, the exclusive scan over units in place, and the expert's count
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int u = 0; u < nunits; ++u) {
      const int v = s_hist[u * E + e];
      s_hist[u * E + e] = run;
      run += v;
    }
    s_cnt[e] = run;
    counts[e] = run;
  }
  __syncthreads();
  block_exclusive_scan(s_cnt, E, s_off, s_warp);
  for (int e = threadIdx.x; e <= E; e += blockDim.x) m_indptr[e] = s_off[e];
  if (unit >= nunits) return;
  // 3. the unit's slots in order, as the scatter kernel
  for (int e = lane; e < E; e += 32) h[e] += s_off[e];
  __syncwarp();
#pragma unroll
  for (int g = 0; g < kGroups; ++g) {
    const long long s = s0 + g * 32 + lane;
    int e = ev[g];
    const bool ok = s < R && static_cast<unsigned>(e) < static_cast<unsigned>(E);
    if (!ok) e = E + lane;  // unique per lane: never matches a real expert
    const unsigned peers = __match_any_sync(kFull, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int leader = __ffs(peers) - 1;
    int pos = 0;
    if (ok) pos = h[e];
    __syncwarp();
    if (ok && lane == leader) h[e] = pos + __popc(peers);
    __syncwarp();
    if (ok) {
      const int r = pos + rank;
      slot_to_row[s] = r;
      row_to_slot[r] = static_cast<int32_t>(s);
      if (w_perm) w_perm[r] = wv[g];
    }
  }
}

// ============================================================================
// Row copy to expert-major order: dst[r] = src[row_to_slot[r] / k], written by token as
// dst[slot_to_row[t*k + j]] = src[t] for j < k, 16-byte vectors.
// ============================================================================
// Each token row is read once and written to its k rows, so the source comes from DRAM once even
// though the copy's writes push its lines out of L2 (a gather by row reads a token row k times:
// measured 0.32 GB of x reads against 67 MB at T=8192, H=4096, k=10).  Work item = (token,
// segment of kScatterSeg 16-byte chunks), one warp per item, two chunks per lane; lane j < k
// fetches the row of slot j once.
constexpr int kScatterLaneChunks = 2;
constexpr int kScatterSeg = 32 * kScatterLaneChunks;  // 16-byte chunks (512 columns) per item

__global__ void __launch_bounds__(256) scatter_rows_kernel(const uint16_t* __restrict__ src,
                                                           const int32_t* __restrict__ slot_to_row, int T, int H,
                                                           int k, long long R, uint16_t* __restrict__ dst, int* err) {
  griddep_wait();  // earlier kernels on the stream are complete
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int chunks = H >> 3;
  const int nseg = (chunks + kScatterSeg - 1) / kScatterSeg;
  const long long items = static_cast<long long>(T) * nseg;
  for (long long it = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; it < items;
       it += nwarps) {
    const long long t = it / nseg;
    const int seg = static_cast<int>(it - t * nseg);
    const int my_row = (lane < k) ? __ldg(slot_to_row + t * k + lane) : 0;
    const bool bad = lane < k && static_cast<unsigned long long>(my_row) >= static_cast<unsigned long long>(R);
    if (__any_sync(kFull, bad)) {
      if (lane == 0 && seg == 0) atomicOr(err, LIGER_MOE_DEVERR_BAD_ROW);
      continue;
    }
    const int c0 = seg * kScatterSeg + lane;  // this lane's chunks: c0, c0 + 32
    const uint4* a = reinterpret_cast<const uint4*>(src + static_cast<size_t>(t) * H);
    uint4 v[kScatterLaneChunks];
#pragma unroll
    for (int q = 0; q < kScatterLaneChunks; ++q)
      if (c0 + 32 * q < chunks) v[q] = __ldg(a + c0 + 32 * q);
    for (int j = 0; j < k; ++j) {
      const int r = __shfl_sync(kFull, my_row, j & 31);
      uint4* b = reinterpret_cast<uint4*>(dst + static_cast<size_t>(r) * H);
#pragma unroll
      for (int q = 0; q < kScatterLaneChunks; ++q)
        if (c0 + 32 * q < chunks) __stcs(b + c0 + 32 * q, v[q]);  // the GEMMs read the copy only after the whole copy
    }
  }
}

// ============================================================================
// fp16 operands of the weight gradients (experts with many rows): the largest |dY| and |x| of the
// step, then fp16 copies of the token rows scaled by a power of two from them.
// ============================================================================
// |v| of the eight bf16 values of a 16-byte chunk, as the largest bf16 magnitude bits.
__device__ __forceinline__ unsigned absmax_bf16x8(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  unsigned m = 0u;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
  return m;
}

// Largest |dY| and |x| (token t's x row read as x_perm[slot_to_row[t k]]) into words[kF16MaxDy],
// words[kF16MaxX] (float bits; a bf16 NaN gives NaN bits, which disable the fp16 operands).  The
// words were zeroed by the schedule kernel, which also set words[kF16Any]; without an expert of
// f16 rows nothing is done.  Work item = (token, segment), as in the row copy.
__global__ void __launch_bounds__(256) f16_prep_kernel(const uint16_t* __restrict__ dy,
                                                       const uint16_t* __restrict__ x_perm,
                                                       const int32_t* __restrict__ slot_to_row, int T, int H, int k,
                                                       long long R, unsigned* words, int* err) {
  __shared__ unsigned s_max[2];
  griddep_wait();
  griddep_launch_dependents();
  if (words[kF16Any] == 0u) return;
  if (threadIdx.x < 2) s_max[threadIdx.x] = 0u;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int chunks = H >> 3;
  const int nseg = (chunks + kScatterSeg - 1) / kScatterSeg;
  const long long items = static_cast<long long>(T) * nseg;
  unsigned md = 0u, mx = 0u;
  for (long long it = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; it < items;
       it += nwarps) {
    const long long t = it / nseg;
    const int seg = static_cast<int>(it - t * nseg);
    const int row = __ldg(slot_to_row + t * k);
    if (static_cast<unsigned long long>(row) >= static_cast<unsigned long long>(R)) {
      if (lane == 0 && seg == 0) atomicOr(err, LIGER_MOE_DEVERR_BAD_ROW);
      continue;
    }
    const int c0 = seg * kScatterSeg + lane;
    const uint4* a = reinterpret_cast<const uint4*>(dy + static_cast<size_t>(t) * H);
    const uint4* b = reinterpret_cast<const uint4*>(x_perm + static_cast<size_t>(row) * H);
#pragma unroll
    for (int q = 0; q < kScatterLaneChunks; ++q)
      if (c0 + 32 * q < chunks) {
        md = max(md, absmax_bf16x8(__ldg(a + c0 + 32 * q)));
        mx = max(mx, absmax_bf16x8(__ldg(b + c0 + 32 * q)));
      }
  }
  md = __reduce_max_sync(kFull, md);
  mx = __reduce_max_sync(kFull, mx);
  if (lane == 0) {
    atomicMax(&s_max[0], md);
    atomicMax(&s_max[1], mx);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    atomicMax(words + kF16MaxDy, s_max[0] << 16);  // bf16 magnitude bits -> float bits
    atomicMax(words + kF16MaxX, s_max[1] << 16);
  }
}

// Two row copies in one launch (blockIdx.y picks the job): dst16[slot_to_row[t k + j], :] =
// fp16(row_t 2^s) for j < k, and the plain bf16 copy into dst when dst is set; row_t = src[t, :]
// or, with src_rows, src_rows[slot_to_row[t k], :].  The fp16 copy is written only when
// words[kF16Any] is set and words[max_word] gives a scale (f16_scale_exp), and only for the rows
// the fp16 weight-gradient tiles read: those of experts with at least f16_rows rows, and the 15
// rows after each of them (the last 16-row K step of such an expert reaches up to 15 rows into the
// next experts; its padded operand is zero there, so those rows must hold finite values).
// Scaling by a power of two is exact.
struct RowCopyF16 {
  const uint16_t* src;
  const uint16_t* src_rows;
  uint16_t* dst;
  uint16_t* dst16;
  int max_word;
};

// Expert holding row r: the largest e with m_indptr[e] <= r (empty experts repeat a value).
__device__ __forceinline__ int expert_of_row(const int32_t* __restrict__ m_indptr, int E, int r) {
  int lo = 0, hi = E;  // m_indptr[lo] <= r < m_indptr[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(m_indptr + mid) <= r)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(256) scatter_rows_f16_kernel(RowCopyF16 j0, RowCopyF16 j1,
                                                               const int32_t* __restrict__ slot_to_row, int T, int H,
                                                               int k, long long R, const int32_t* __restrict__ m_indptr,
                                                               int E, int f16_rows, const unsigned* words, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  const RowCopyF16 job = blockIdx.y == 0 ? j0 : j1;
  int sexp = 0;
  const bool f16 = job.dst16 != nullptr && words[kF16Any] != 0u && f16_scale_exp(words[job.max_word], sexp);
  if (!f16 && job.dst == nullptr) return;
  const float sc = f16_pow2(sexp);
  const int lane = threadIdx.x & 31;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int chunks = H >> 3;
  const int nseg = (chunks + kScatterSeg - 1) / kScatterSeg;
  const long long items = static_cast<long long>(T) * nseg;
  for (long long it = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; it < items;
       it += nwarps) {
    const long long t = it / nseg;
    const int seg = static_cast<int>(it - t * nseg);
    const int my_row = (lane < k) ? __ldg(slot_to_row + t * k + lane) : 0;
    const bool bad = lane < k && static_cast<unsigned long long>(my_row) >= static_cast<unsigned long long>(R);
    if (__any_sync(kFull, bad)) {
      if (lane == 0 && seg == 0) atomicOr(err, LIGER_MOE_DEVERR_BAD_ROW);
      continue;
    }
    const int c0 = seg * kScatterSeg + lane;
    const int first = __shfl_sync(kFull, my_row, 0);
    bool need = false;  // lane j < k: row my_row is read by an fp16 tile
    if (f16 && lane < k) {
      const auto heavy = [&](int e) { return __ldg(m_indptr + e + 1) - __ldg(m_indptr + e) >= f16_rows; };
      need = heavy(expert_of_row(m_indptr, E, my_row)) ||
             (my_row >= 15 && heavy(expert_of_row(m_indptr, E, my_row - 15)));
    }
    const unsigned need_mask = __ballot_sync(kFull, need);
    const uint4* a = reinterpret_cast<const uint4*>(
        job.src_rows != nullptr ? job.src_rows + static_cast<size_t>(first) * H : job.src + static_cast<size_t>(t) * H);
    uint4 v[kScatterLaneChunks], h[kScatterLaneChunks];
#pragma unroll
    for (int q = 0; q < kScatterLaneChunks; ++q)
      if (c0 + 32 * q < chunks) {
        v[q] = __ldg(a + c0 + 32 * q);
        uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = pack_f16x2(bf16_lo(w[i]) * sc, bf16_hi(w[i]) * sc);
        h[q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    for (int j = 0; j < k; ++j) {
      const size_t r = static_cast<size_t>(__shfl_sync(kFull, my_row, j & 31));
#pragma unroll
      for (int q = 0; q < kScatterLaneChunks; ++q)
        if (c0 + 32 * q < chunks) {
          if (job.dst != nullptr) __stcs(reinterpret_cast<uint4*>(job.dst + r * H) + c0 + 32 * q, v[q]);
          if ((need_mask >> j) & 1u) __stcs(reinterpret_cast<uint4*>(job.dst16 + r * H) + c0 + 32 * q, h[q]);
        }
    }
  }
}

// ============================================================================
// Combine.  LigerCute README, "Forward pass" (final local combine);
// LightMoE README, "Highlights" (deterministic combine).
//   y[t, :] = bf16( sum_{j=0..k-1} y_perm[slot_to_row[t*k + j], :] )  (fp32, j ascending)
// One warp per token; lane j fetches the row index of slot j once.
// ============================================================================
// Work item = (token, segment of kCombineSeg 16-byte chunks); one warp per item, so that a small
// batch (decode) still spreads over many warps.  Each lane owns two chunks of the segment and
// reads the k rows four at a time: eight independent 16-byte loads in flight.  The sum over j
// still runs in j order for every element.
constexpr int kCombineLaneChunks = 2;
constexpr int kCombineSeg = 32 * kCombineLaneChunks;  // 16-byte chunks (512 columns) per item

__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ y_perm,
                                                      const int32_t* __restrict__ slot_to_row, int T, int H, int k,
                                                      long long R, uint16_t* __restrict__ y, int* err) {
  griddep_wait();  // earlier kernels on the stream are complete
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int chunks = H >> 3;
  const int nseg = (chunks + kCombineSeg - 1) / kCombineSeg;
  const long long items = static_cast<long long>(T) * nseg;
  for (long long it = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; it < items;
       it += nwarps) {
    const long long t = it / nseg;
    const int seg = static_cast<int>(it - t * nseg);
    int my_row = (lane < k) ? __ldg(slot_to_row + t * k + lane) : 0;
    const bool bad = static_cast<unsigned long long>(my_row) >= static_cast<unsigned long long>(R);
    if (__any_sync(kFull, bad)) {
      if (lane == 0 && seg == 0) atomicOr(err, LIGER_MOE_DEVERR_BAD_ROW);
      continue;
    }
    const int c0 = seg * kCombineSeg + lane;  // this lane's chunks: c0, c0 + 32
    float acc[kCombineLaneChunks][8];
#pragma unroll
    for (int q = 0; q < kCombineLaneChunks; ++q)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[q][i] = 0.f;
    for (int j0 = 0; j0 < k; j0 += 4) {
      uint4 v[4][kCombineLaneChunks];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int r = __shfl_sync(kFull, my_row, (j0 + jj) & 31);
        if (j0 + jj < k) {
          const uint4* src = reinterpret_cast<const uint4*>(y_perm + static_cast<size_t>(r) * H);
#pragma unroll
          for (int q = 0; q < kCombineLaneChunks; ++q)
            if (c0 + 32 * q < chunks) v[jj][q] = __ldcs(src + c0 + 32 * q);  // each row is read once
        }
      }
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        if (j0 + jj >= k) break;
#pragma unroll
        for (int q = 0; q < kCombineLaneChunks; ++q) {
          if (c0 + 32 * q >= chunks) continue;
          const uint4 u = v[jj][q];
          acc[q][0] += bf16_lo(u.x);
          acc[q][1] += bf16_hi(u.x);
          acc[q][2] += bf16_lo(u.y);
          acc[q][3] += bf16_hi(u.y);
          acc[q][4] += bf16_lo(u.z);
          acc[q][5] += bf16_hi(u.z);
          acc[q][6] += bf16_lo(u.w);
          acc[q][7] += bf16_hi(u.w);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kCombineLaneChunks; ++q) {
      const int c = c0 + 32 * q;
      if (c >= chunks) continue;
      uint4 o;
      o.x = pack_bf16x2(acc[q][0], acc[q][1]);
      o.y = pack_bf16x2(acc[q][2], acc[q][3]);
      o.z = pack_bf16x2(acc[q][4], acc[q][5]);
      o.w = pack_bf16x2(acc[q][6], acc[q][7]);
      reinterpret_cast<uint4*>(y + static_cast<size_t>(t) * H)[c] = o;
    }
  }
}

// ============================================================================
// Router-logit gradient.  LightMoE README, "MoE training" (router-gradient
// kernel, differentiable_probs).  With gamma'_j = w_j * <dY, o_j> (computed
// per row by the dH GEMM epilogue as partial sums over its column tiles):
//   d_logits[t, ids_j] = gamma'_j - w_j * sum_i gamma'_i,  0 elsewhere,
// which equals w_j (gamma_j - sum_i w_i gamma_i).  One warp per token.
// ============================================================================
__global__ void __launch_bounds__(256) router_grad_kernel(const float* __restrict__ gdot, int ntiles,
                                                          const int32_t* __restrict__ ids,
                                                          const float* __restrict__ w,
                                                          const int32_t* __restrict__ slot_to_row, int T, int E,
                                                          int k, long long R, float* __restrict__ d_logits,
                                                          int* err) {
  griddep_wait();  // earlier kernels on the stream are complete
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long t = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
    float* out = d_logits + t * E;
    for (int e = lane; e < E; e += 32) out[e] = 0.f;
    float gp = 0.f, wj = 0.f;
    int id = 0;
    bool bad = false;
    if (lane < k) {
      const int r = __ldg(slot_to_row + t * k + lane);
      id = __ldg(ids + t * k + lane);
      wj = __ldg(w + t * k + lane);
      bad = static_cast<unsigned long long>(r) >= static_cast<unsigned long long>(R) ||
            static_cast<unsigned>(id) >= static_cast<unsigned>(E);
      if (!bad)
        for (int q = 0; q < ntiles; ++q) gp += __ldg(gdot + static_cast<size_t>(r) * ntiles + q);
    }
    if (__any_sync(kFull, bad)) {
      if (lane == 0) atomicOr(err, LIGER_MOE_DEVERR_BAD_ROW);
      continue;
    }
    float S = 0.f;
    for (int j = 0; j < k; ++j) S += __shfl_sync(kFull, gp, j);
    __syncwarp();
    if (lane < k) out[id] = gp - wj * S;
  }
}

int grid_for_warps(long long nwarps_needed, int warps_per_block, const DeviceInfo& dev, int waves = 16) {
  long long blocks = (nwarps_needed + warps_per_block - 1) / warps_per_block;
  const long long cap = static_cast<long long>(dev.sm_count) * waves;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<int>(blocks);
}

}  // namespace

int launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s) {
  if (T == 0) return LIGER_MOE_OK;
  const int blocks = static_cast<int>((static_cast<long long>(T) * 32 + 255) / 256);
  const int epl = (E + 31) / 32;
  KernelScope trace("route_topk", s);
  if (epl <= 1)
    launch_kernel(route_topk_kernel<1>, dim3(blocks), dim3(256), 0, s, "route_topk", 1, logits, T, E, k, ids, w);
  else if (epl <= 2)
    launch_kernel(route_topk_kernel<2>, dim3(blocks), dim3(256), 0, s, "route_topk", 1, logits, T, E, k, ids, w);
  else if (epl <= 4)
    launch_kernel(route_topk_kernel<4>, dim3(blocks), dim3(256), 0, s, "route_topk", 1, logits, T, E, k, ids, w);
  else if (epl <= 8)
    launch_kernel(route_topk_kernel<8>, dim3(blocks), dim3(256), 0, s, "route_topk", 1, logits, T, E, k, ids, w);
  else if (epl <= 16)
    launch_kernel(route_topk_kernel<16>, dim3(blocks), dim3(256), 0, s, "route_topk", 1, logits, T, E, k, ids, w);
  else
    launch_kernel(route_topk_kernel<32>, dim3(blocks), dim3(256), 0, s, "route_topk", 1, logits, T, E, k, ids, w);
  return check_launch("route_topk");
}

size_t dispatch_scratch_bytes(long long R, int E) {
  const long long nunits = (R + kUnit - 1) / kUnit;
  return static_cast<size_t>(nunits) * E * sizeof(int32_t);
}

size_t dispatch_workspace_bytes(long long R, int E) { return align_up(dispatch_scratch_bytes(R, E), 256) + 256; }

int launch_dispatch(const int32_t* ids, const float* w, const uint16_t* x, int T, int H, int E, int k,
                    int32_t* counts, int32_t* m_indptr, int32_t* row_to_slot, int32_t* slot_to_row, float* w_perm,
                    uint16_t* x_perm, void* workspace, const DeviceInfo& dev, cudaStream_t s) {
  const long long R = static_cast<long long>(T) * k;
  const int nunits = static_cast<int>((R + kUnit - 1) / kUnit);
  int32_t* hist = static_cast<int32_t*>(workspace);
  const int blocks = (nunits + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (nunits > 0 && nunits <= kSmallUnits && E <= kSmallExperts) {  // one launch instead of three
    {
      KernelScope trace("dispatch_small", s);
      launch_kernel(dispatch_small_kernel, dim3(1), dim3(kSmallUnits * 32), 0, s, "dispatch_small", 1, ids, w, R, E,
                    nunits, counts, m_indptr, row_to_slot, slot_to_row, w_perm, dev.err_flag);
    }
    if (int rc = check_launch("dispatch_small")) return rc;
    if (x_perm != nullptr) return launch_scatter_rows(x, slot_to_row, T, H, k, x_perm, dev, s);
    return LIGER_MOE_OK;
  }
  if (nunits > 0) {
    {
      KernelScope trace("dispatch_hist", s);
      launch_kernel(dispatch_hist_kernel, dim3(blocks), dim3(kWarpsPerBlock * 32), kWarpsPerBlock * E * sizeof(int), s,
                    "dispatch_hist", 1, ids, R, E, nunits, hist, dev.err_flag);
    }
    if (int rc = check_launch("dispatch_hist")) return rc;
    {
      KernelScope trace("dispatch_scan", s);
      launch_kernel(dispatch_scan_kernel, dim3((E * 32 + 255) / 256), dim3(256), 0, s, "dispatch_scan", 1, hist,
                    nunits, E, counts);
    }
    if (int rc = check_launch("dispatch_scan")) return rc;
  } else {
    cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
  }
  const size_t smem = (E + 1 + 32 + kWarpsPerBlock * E) * sizeof(int);
  {
    KernelScope trace("dispatch_scatter", s);
    launch_kernel(dispatch_scatter_kernel, dim3(blocks > 0 ? blocks : 1), dim3(kWarpsPerBlock * 32), smem, s,
                  "dispatch_scatter", 1, ids, w, R, E, nunits, hist, counts, m_indptr, row_to_slot, slot_to_row,
                  w_perm);
  }
  if (int rc = check_launch("dispatch_scatter")) return rc;
  if (x_perm != nullptr && R > 0) return launch_scatter_rows(x, slot_to_row, T, H, k, x_perm, dev, s);
  return LIGER_MOE_OK;
}

int launch_scatter_rows(const uint16_t* src, const int32_t* slot_to_row, int T, int H, int k, uint16_t* dst,
                        const DeviceInfo& dev, cudaStream_t s) {
  if (T == 0) return LIGER_MOE_OK;
  {
    KernelScope trace("gather_rows", s);
    const long long items = static_cast<long long>(T) * ((H / 8 + kScatterSeg - 1) / kScatterSeg);
    launch_kernel(scatter_rows_kernel, dim3(grid_for_warps(items, 8, dev)), dim3(256), 0, s, "gather_rows", 1, src,
                  slot_to_row, T, H, k, static_cast<long long>(T) * k, dst, dev.err_flag);
  }
  return check_launch("gather_rows");
}

int launch_f16_prep(const uint16_t* dy, const uint16_t* x_perm, const int32_t* slot_to_row, int T, int H, int k,
                    unsigned* words, const DeviceInfo& dev, cudaStream_t s) {
  if (T == 0) return LIGER_MOE_OK;
  {
    KernelScope trace("f16_prep", s);
    const long long items = static_cast<long long>(T) * ((H / 8 + kScatterSeg - 1) / kScatterSeg);
    launch_kernel(f16_prep_kernel, dim3(grid_for_warps(items, 8, dev)), dim3(256), 0, s, "f16_prep", 1, dy, x_perm,
                  slot_to_row, T, H, k, static_cast<long long>(T) * k, words, dev.err_flag);
  }
  return check_launch("f16_prep");
}

int launch_scatter_rows_f16(const uint16_t* dy, const uint16_t* x_perm, const int32_t* slot_to_row, int T, int H,
                            int k, const int32_t* m_indptr, int E, uint16_t* dy_perm, uint16_t* dy16, uint16_t* x16,
                            const unsigned* words, const DeviceInfo& dev, cudaStream_t s) {
  if (T == 0) return LIGER_MOE_OK;
  const RowCopyF16 j0{dy, nullptr, dy_perm, dy16, kF16MaxDy};
  const RowCopyF16 j1{nullptr, x_perm, nullptr, x16, kF16MaxX};
  {
    KernelScope trace("gather_rows_f16", s);
    const long long items = static_cast<long long>(T) * ((H / 8 + kScatterSeg - 1) / kScatterSeg);
    launch_kernel(scatter_rows_f16_kernel, dim3(grid_for_warps(items, 8, dev), 2), dim3(256), 0, s,
                  "gather_rows_f16", 1, j0, j1, slot_to_row, T, H, k, static_cast<long long>(T) * k, m_indptr, E,
                  kF16Rows, words, dev.err_flag);
  }
  return check_launch("gather_rows_f16");
}

int launch_combine(const uint16_t* y_perm, const int32_t* slot_to_row, int T, int H, int k, uint16_t* y,
                   const DeviceInfo& dev, cudaStream_t s) {
  if (T == 0) return LIGER_MOE_OK;
  {
    KernelScope trace("combine", s);
    const long long items = static_cast<long long>(T) * ((H / 8 + kCombineSeg - 1) / kCombineSeg);
    launch_kernel(combine_kernel, dim3(grid_for_warps(items, 8, dev)), dim3(256), 0, s, "combine", 1, y_perm,
                  slot_to_row, T, H, k, static_cast<long long>(T) * k, y, dev.err_flag);
  }
  return check_launch("combine");
}

int launch_router_grad(const float* gdot, int gdot_tiles_, const int32_t* ids, const float* w,
                       const int32_t* slot_to_row, int T, int E, int k, float* d_logits, const DeviceInfo& dev,
                       cudaStream_t s) {
  if (T == 0) return LIGER_MOE_OK;
  {
    KernelScope trace("router_grad", s);
    launch_kernel(router_grad_kernel, dim3(grid_for_warps(T, 8, dev)), dim3(256), 0, s, "router_grad", 1, gdot,
                  gdot_tiles_, ids, w, slot_to_row, T, E, k, static_cast<long long>(T) * k, d_logits, dev.err_flag);
  }
  return check_launch("router_grad");
}

}  // namespace lmoe
