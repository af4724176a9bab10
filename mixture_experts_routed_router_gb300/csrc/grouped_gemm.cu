// Grouped GEMMs of the routed MoE layer on the 5th-generation tensor cores.
//
// One persistent, warp-specialised kernel template serves every contraction
// of the layer (LightMoE README, "Grouped GEMM": expert-major rows, m_indptr,
// b laid out [num_experts, N, K]; LigerCute README, "LigerMoE design":
// persistent warp-specialised TMA / MMA pipeline):
//   warp 0      TMA producer: one elected lane streams A and B tiles into a
//               shared-memory ring of 2-6 stages (128-byte swizzle), mbarrier-tracked.
//               In the memory-lean variant an operand whose rows are token rows picked
//               by the routing (x or dY in expert-major order) is instead gathered by
//               the whole warp with TMA gather4 (four rows per copy) straight from the
//               token-major tensor, so no permuted copy of it is ever written.
//   warp 1      MMA issuer: allocates 512 TMEM columns, one elected lane issues
//               tcgen05.mma (M=128, N=256, K=16, bf16 x bf16 -> fp32, or fp16 x fp16 in
//               the weight gradients' fp16 launch; M=256 across a 2-SM CTA pair) and
//               commits stage releases and accumulator-ready events to mbarriers
//   warps 2..9  epilogue: tcgen05.ld of the fp32 accumulator, fused math, TMA bulk
//               stores.  Two warps per 32-lane TMEM quadrant (the quadrant's 32 rows),
//               each owning half of the tile's columns.
// The two 128x256 fp32 accumulators in TMEM are double-buffered, so the
// epilogue of tile i overlaps the MMAs of tile i+1.
//
// Schedules:
//   RowsM  rows of an expert are the GEMM's M (forward gate/up and down,
//          backward dH and dX): tiles (expert, 128-row block, N block), K fixed.
//          The per-expert M-tile prefix is built on the device from m_indptr.
//   RowsK  rows of an expert are the GEMM's K (weight gradients): tiles
//          (expert, M block, N block), K = rows of that expert, walked in row
//          order by one CTA (deterministic, no split-K atomics).  The operand the
//          dH epilogue writes (dgu, w h) sits in a padded row space: each expert's
//          rows are followed by zero rows up to a multiple of 16, so the last
//          16-row K step adds nothing from the next expert's rows of the other operand.
//          A launch may take one part of the experts, a range of their sorted order
//          (the experts of the fp16 pass, the 2-SM pair experts of dW_down).
//   Dense  one plain GEMM over R rows (the router projection).
// Epilogues: SwiGLU (h = silu(g)*u, optional fp32 derivative factors), ScaleRows
// (y = w_r * acc), DH (SwiGLU backward from the saved factors, hi/lo operands for
// the weight gradients or, for experts with many rows, fp16 ones, per-row partial
// <dh, h> for the router gradient), Store (the weight gradients: scaled back from
// the fp16 operands' powers of two where they were used).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace lmoe {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB

constexpr int MN_BOX_BYTES = 64 * BK * 2;  // one 64 (MN) x 64 (K) box of an MN-major operand
constexpr int kEpiWarps = 8;  // two per TMEM lane quadrant, each owning half of the tile's columns
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTmemCols = 2 * BN;
// Epilogue staging: per epilogue warp one 32-row x 128-byte box (128-byte swizzle) that
// feeds TMA bulk stores, so output rows leave the SM as whole lines.
constexpr int STG_BYTES = 32 * 128;
constexpr int STG_PER_WARP = 1;
constexpr int kBarrierBytes = 1024;  // barriers, the tile ring, and (at kZeroOffset) a zero row for zero tiles
constexpr int kZeroOffset = 768;
constexpr int kZeroBytes = 256;     // one warp row of a zero tile: BN / 2 bf16 columns
// Per-expert 2-SM pair thresholds (rows of one expert): the forward and dX GEMMs (256-row pair tiles)
// and the two weight-gradient GEMMs.  An expert with fewer rows runs one CTA per tile.
constexpr int kPairRowsM = 512, kPairRowsDwGu = 192, kPairRowsDwD = 128;  // dW_gate_up: on the mean rows

// The tile ring: slots of the ring that passes decoded tiles from the producer to the MMA and
// epilogue warps (kRingInts ints each), and the index of its first barrier in the barrier area
// (after the pipeline barriers).
constexpr int kSchedSlots = 8;
constexpr int kSchedBarIndex = 24;
constexpr int kRingInts = 11;
constexpr int kDhBoxBytes = 32 * 32;            // dH epilogue: 32 rows x 16 bf16 columns
constexpr int kDhSetBytes = 6 * kDhBoxBytes;    // six output boxes per 16 columns

// Shared memory of one CTA: operand stages | epilogue staging | barriers.
//   SPLIT = 0: one A and one B tile per stage (48 KB), 4 stages (also the weight gradients'
//              fp16 launch, whose tiles take one part of each operand);
//   SPLIT = 1: A as two bf16 parts (hi, lo) + B (64 KB), 3 stages: two MMAs per K step share B;
//   SPLIT = 2: A + B as two parts (80 KB), 2 stages: two MMAs per K step share A.
//   PAIR: a CTA of a 2-SM pair holds its 128 rows (RowsM) or columns (RowsK) of A and half of B's
//         256 rows or columns: 32 KB and 6 stages, or 48 KB and 4 stages with hi/lo parts.
// Epilogue staging per warp: one 4 KB box, or for the dH kernel one set of six 1 KB boxes
// (3 operand stages there: its MMAs are a small part of its time).
template <int kDh, int SPLIT, int PAIR = 0>
struct Layout {
  static constexpr int kABytes = A_BYTES * (SPLIT == 1 ? 2 : 1);
  static constexpr int kBBytes = B_BYTES * (SPLIT == 2 ? 2 : 1) / (PAIR ? 2 : 1);
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages =
      PAIR ? (kDh ? 4 : (SPLIT == 0 ? 6 : 4)) : (kDh ? 3 : (SPLIT == 0 ? 4 : (SPLIT == 1 ? 3 : 2)));
  static constexpr int kStgWarpBytes = kDh ? kDhSetBytes : STG_PER_WARP * STG_BYTES;
  static constexpr int kStgOffset = kStages * kStageBytes;
  static constexpr int kBarOffset = kStgOffset + kEpiWarps * kStgWarpBytes;
  static constexpr int kSmemBytes = kBarOffset + kBarrierBytes + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned");
};

// Dense: one plain GEMM over p.R rows (no experts): the router projection.
enum class Sched : int { RowsM = 0, RowsK = 1, Dense = 2 };
// SwiGLU: the gate/up GEMM with SwiGLU; GLU: the same with the activation chosen at run time
// (Params::act), kept apart so that the default SwiGLU kernel carries none of the variants' code.
// ReLU2: the up GEMM of a two-weight (non-gated) expert, h = max(a, 0)^2.  DH1: the dH epilogue
// of such an expert (one derivative factor, one output instead of [dg | du]).  Logits: fp32
// output plus a per-column bias (the router projection).
// DH16: the DH epilogue that writes fp16 parts for the experts with many rows (the first dH pass of a
// backward with the fp16 weight-gradient pass), kept apart so that the plain DH kernel carries none of
// that code (with it, DH measured 7 % slower where no expert takes the pass).
enum class Epi : int { SwiGLU = 0, ScaleRows = 1, DH = 2, Store = 3, GLU = 4, ReLU2 = 5, DH1 = 6, Logits = 7, DH16 = 8 };
constexpr bool gate_up_epi(Epi e) { return e == Epi::SwiGLU || e == Epi::GLU; }
constexpr bool dh_epi(Epi e) { return e == Epi::DH || e == Epi::DH1 || e == Epi::DH16; }
template <Epi EP, int SPLIT, int PAIR = 0>
using LayoutOf = Layout<dh_epi(EP) ? 1 : 0, SPLIT, PAIR>;

struct Params {
  const int32_t* m_indptr;     // [E+1]
  const int32_t* tile_prefix;  // RowsM: [E+1] M-tile prefix
  int E;
  int n_tiles;            // tiles along N
  int m_tiles;            // RowsK: M tiles per expert
  int num_kb;             // RowsM: K / BK
  int b_rows_per_expert;  // rows of B's tensor map per expert
  int b_split;            // SwiGLU: row offset of the up half of W_gu (= I)
  int M_out;              // RowsK: output rows per expert
  int a_split_rows;       // RowsK, SPLIT = 1: row offset of A's lo part (A stored as bf16 hi, lo)
  int b_split_rows;       // RowsK, SPLIT = 2: row offset of B's lo part
  int N_out;              // valid output columns
  int I;
  uint16_t* out;
  long long ld_out;
  long long out_expert_stride;
  uint16_t* out2;         // DH: dgu [2R, 2I] (hi rows, then lo rows); DH1: da [2R, I]
  float* gu_out;          // SwiGLU: derivative factors [a | b] fp32 [R, 2I] (nullable)
  int act;                // SwiGLU epilogue: gated activation (LIGER_MOE_ACT_*)
  float act_clamp;        // its clamp (bounded SwiGLU) or limit (SwiGLU-OAI)
  const float* row_scale; // ScaleRows, DH: w_perm
  const float* gu_in;     // DH: derivative factors [a | b] fp32 [R, 2I]
  const uint16_t* h_in;   // DH: h [R, I]
  uint16_t* hw_out;       // DH: bf16(w * h) [R, I]
  float* gdot;            // DH: [R, 2 n_tiles] partial <dh, h> (per N tile and column half)
  long long R;            // routed rows
  // Row-padded operands of the weight-gradient GEMMs: the dH epilogue writes dgu and w h with
  // each expert's rows starting at pad_indptr[e] (exclusive scan of the row counts rounded up
  // to 16) and zero rows up to the next multiple of 16, so a weight-gradient K step never reads
  // another expert's rows in that operand.  lo_rows: row offset of the lo halves.
  const int32_t* pad_indptr;  // [E+1] or NULL (no padding)
  long long lo_rows;
  int pad_a, pad_b;           // A / B rows are padded rows (RowsM: A only)
  const int32_t* row_slot;  // gathered operand: row_to_slot [R]; token of row r = row_slot[r] / topk
  int topk;
  // Dynamic tile order of the weight-gradient GEMMs (claims != NULL): when the schedule found the
  // load skewed (*sched_skewed != 0), the tiles are queued expert by expert with the experts
  // sorted by rows, most first (sched_order, and sched_info for each sorted expert), and each CTA's
  // producer claims the next positions through one counter (zeroed by the schedule kernel).
  // Otherwise the static order.
  const int32_t* sched_order;   // [E]
  const int32_t* sched_info;    // [E][4]: expert, first row, rows, first padded row of each sorted expert
  const int* sched_skewed;
  int* claims;
  // Weight gradients in parts (parted != 0): this launch takes the experts at positions
  // [*part_begin, *part_end) of the sorted order (NULL: 0 / E), counts the schedule kernel wrote
  // (experts with at least the fp16 or the pair threshold's rows, which lead the order); else
  // every expert, in id order (static) or sorted (dynamic).
  int parted;
  const int* part_begin;
  const int* part_end;
  // Logits: fp32 output [R, N_out] (row stride ld_out), optional bias [N_out]; out_tma: 32-column
  // chunks leave through TMA boxes (N_out a multiple of 32), else by masked direct stores
  float* out_f32;
  const float* col_bias;
  int out_tma;
  // fp16 weight-gradient operands (f16_role != 0), for the experts with at least f16_rows rows;
  // f16_words: the backward's words (kF16MaxX, kF16MaxDy, kF16Any, per-expert range maxima).
  //   DH16, role 1: those experts' tiles write fp16(dgu 2^sg) and fp16(w h 2^sh) into the lo rows
  //     (and no hi rows of w h), and the largest magnitudes into the range words; the launch leaves
  //     at once when no expert has f16_rows rows;
  //   DH, role 2: then only those experts whose fp16 parts are unusable (f16_usable), with hi / lo
  //     parts (the refill); or, when no expert has f16_rows rows, the whole dH GEMM;
  //   RowsK, role 3 (dW_gate_up) / 4 (dW_down), in the launch of those experts (f16_part, one
  //     operand part per stage): an expert with usable fp16 parts takes one fp16 MMA per K step,
  //     the lo rows of the padded operand against the fp16 token rows (tensor map tmF), and
  //     scales the result back by the inverse powers of two; an expert without takes its hi and lo
  //     parts as two passes over its K blocks (bf16).
  int f16_role;
  int f16_rows;
  int f16_part;
  unsigned* f16_words;
  int* err;
};

struct Tile {
  int e;
  int m0;        // RowsM: first global row of the tile; RowsK: first output row inside the expert
  int rows;      // RowsM: valid rows in the tile; RowsK: rows of the expert (K extent)
  int nt;        // N tile
  int row0;      // RowsK: first global row of the expert
  int am0;       // RowsM: first row of the tile in the padded row space (= m0 without padding)
  int prow0;     // RowsK: first padded row of the expert (= row0 without padding)
  int kb_count;  // K blocks
  int f16;       // RowsK: one fp16 MMA per K step; DH: write the fp16 parts
};

// Expert e's fp16 weight-gradient operands are usable: both token-row scales exist and both of
// its fp16 parts (written by the dH epilogue) lie within their window.
__device__ __forceinline__ bool f16_usable(int e, const Params& p) {
  int s;
  return p.f16_words[kF16Any] != 0u && f16_scale_exp(p.f16_words[kF16MaxX], s) &&
         f16_scale_exp(p.f16_words[kF16MaxDy], s) && f16_in_range(p.f16_words[kF16Range + e]) &&
         f16_in_range(p.f16_words[kF16Range + p.E + e]);
}

// K blocks and precision of a weight-gradient tile of expert tl.e with tl.rows rows: in the fp16
// experts' launch, one fp16 pass (usable parts) or the hi and lo parts as two passes over the K
// blocks; elsewhere the template's own operand parts.
__device__ __forceinline__ void rows_k_finish(Tile& tl, const Params& p) {
  tl.kb_count = tl.rows > 0 ? (tl.rows + BK - 1) / BK : 0;
  tl.f16 = 0;
  if (p.f16_part) {
    tl.f16 = f16_usable(tl.e, p) ? 1 : 0;
    if (!tl.f16) tl.kb_count *= 2;
  }
}

// The experts of a parted launch: positions [part_lo, part_hi) of the sorted order.
__device__ __forceinline__ int part_lo(const Params& p) { return p.part_begin != nullptr ? __ldg(p.part_begin) : 0; }
__device__ __forceinline__ int part_hi(const Params& p) { return p.part_end != nullptr ? __ldg(p.part_end) : p.E; }
// Expert of position i of a launch's static order: the sorted order inside a part that leaves some
// experts out, else the id order (a part holding every expert keeps it: measured faster for the
// uniform loads, where the sorted order only shuffles equal experts).
__device__ __forceinline__ int static_expert(int i, const Params& p) {
  if (!p.parted) return i;
  const int lo = part_lo(p);
  return (lo == 0 && part_hi(p) == p.E) ? i : __ldg(p.sched_order + lo + i);
}

// The factor that undoes the fp16 operands' scales in a weight gradient: 2^-(s_x + s_g) for
// dW_gate_up (x 2^s_x against dgu 2^s_g, s_g = s_dY + kF16DguShift), 2^-(s_dY + kF16HwShift) for
// dW_down.  Exact: a power of two.
__device__ __forceinline__ float f16_unscale(const Params& p) {
  int sx = 0, sd = 0;
  f16_scale_exp(p.f16_words[kF16MaxX], sx);
  f16_scale_exp(p.f16_words[kF16MaxDy], sd);
  return p.f16_role == 3 ? f16_pow2(-(sx + sd + kF16DguShift)) : f16_pow2(-(sd + kF16HwShift));
}

// RowsM tile of expert e: its local M tile lm (128 rows) and N tile nt.
__device__ __forceinline__ Tile rows_m_tile(int e, int lm, int nt, const Params& p) {
  Tile tl;
  tl.e = e;
  tl.nt = nt;
  const int end = __ldg(p.m_indptr + e + 1);
  const int start = __ldg(p.m_indptr + e);
  tl.m0 = start + lm * BM;
  tl.rows = min(BM, end - tl.m0);
  tl.row0 = 0;
  tl.am0 = p.pad_indptr != nullptr ? __ldg(p.pad_indptr + e) + (tl.m0 - start) : tl.m0;
  tl.prow0 = 0;
  tl.kb_count = p.num_kb;
  tl.f16 = 0;
  if (p.f16_role != 0) {  // the dH passes
    const bool heavy = end - start >= p.f16_rows;
    if (p.f16_role == 1)
      tl.f16 = heavy ? 1 : 0;
    else if (p.f16_words[kF16Any] != 0u && (!heavy || f16_usable(e, p)))
      tl.kb_count = 0;  // refill: only the experts whose fp16 parts are unusable
  }
  return tl;
}

// RowsK tile r (of m_tiles * n_tiles) of expert e, M blocks fastest: neighbouring tiles share the
// expert and the N block, so they read the same B tile (through L2).
__device__ __forceinline__ Tile rows_k_tile(int e, int r, const Params& p) {
  Tile tl;
  tl.e = e;
  tl.nt = r / p.m_tiles;
  const int mt = r - tl.nt * p.m_tiles;
  tl.m0 = mt * BM;
  tl.row0 = __ldg(p.m_indptr + e);
  tl.rows = __ldg(p.m_indptr + e + 1) - tl.row0;
  tl.am0 = tl.m0;
  tl.prow0 = p.pad_indptr != nullptr ? __ldg(p.pad_indptr + e) : tl.row0;
  rows_k_finish(tl, p);
  return tl;
}

// The same tile from the schedule's table entry of its expert (id, first row, rows, first padded
// row): one 16-byte load instead of the order and then the expert's row offsets.
__device__ __forceinline__ Tile rows_k_tile_info(int4 q, int r, const Params& p) {
  Tile tl;
  tl.e = q.x;
  tl.nt = r / p.m_tiles;
  tl.m0 = (r - tl.nt * p.m_tiles) * BM;
  tl.row0 = q.y;
  tl.rows = q.z;
  tl.am0 = tl.m0;
  tl.prow0 = q.w;
  rows_k_finish(tl, p);
  return tl;
}

// Largest i in [0, n) with prefix[i] <= v (prefix non-decreasing, prefix[0] = 0 <= v).
__device__ __forceinline__ int prefix_search(const int32_t* prefix, int n, int v) {
  int lo = 0, hi = n;  // prefix[lo] <= v < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(prefix + mid) <= v)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

// Tile t of the launch in the static order, experts in id order (RowsK parts of a heavy / light
// split: in the sorted order).  The dynamic order decodes its tiles from the schedule's table
// (rows_k_tile_info).
template <Sched S>
__device__ __forceinline__ Tile decode_tile(int t, const Params& p) {
  if constexpr (S == Sched::RowsM) {
    const int mt = t / p.n_tiles;
    const int nt = t - mt * p.n_tiles;
    const int i = prefix_search(p.tile_prefix, p.E, mt);
    return rows_m_tile(i, mt - __ldg(p.tile_prefix + i), nt, p);
  } else if constexpr (S == Sched::Dense) {
    Tile tl;
    const int mt = t / p.n_tiles;
    tl.nt = t - mt * p.n_tiles;
    tl.e = 0;
    tl.m0 = mt * BM;
    tl.rows = static_cast<int>(min(static_cast<long long>(BM), p.R - tl.m0));
    tl.row0 = 0;
    tl.am0 = tl.m0;
    tl.prow0 = 0;
    tl.kb_count = p.num_kb;
    tl.f16 = 0;
    return tl;
  } else {
    const int per_e = p.m_tiles * p.n_tiles;
    const int i = t / per_e;
    return rows_k_tile(static_expert(i, p), t - i * per_e, p);
  }
}

// Tile of a 2-SM pair.  RowsM: tile_prefix counts 256-row blocks per expert; CTA `rank` of the
// pair owns rows [m0, m0 + 128) of the block (none when the expert ends before them).  RowsK:
// CTA `rank` owns output rows [m0, m0 + 128) of the expert's weight gradient.
template <Sched S>
__device__ __forceinline__ Tile decode_tile_pair(int t, const Params& p, uint32_t rank) {
  Tile tl;
  if constexpr (S == Sched::RowsK) {
    // weight gradients: the pair covers M blocks 2 mp and 2 mp + 1 of the expert's output; pair
    // blocks fastest, so neighbouring pairs share the expert and the N block
    const int mpt = p.m_tiles / 2;
    const int per_e = mpt * p.n_tiles;
    const int i = t / per_e;
    tl.e = static_expert(i, p);
    const int r = t - i * per_e;
    tl.nt = r / mpt;
    const int mp = r - tl.nt * mpt;
    tl.m0 = mp * (2 * BM) + static_cast<int>(rank) * BM;
    tl.row0 = __ldg(p.m_indptr + tl.e);
    tl.rows = __ldg(p.m_indptr + tl.e + 1) - tl.row0;
    tl.am0 = tl.m0;
    tl.prow0 = p.pad_indptr != nullptr ? __ldg(p.pad_indptr + tl.e) : tl.row0;
    rows_k_finish(tl, p);
    return tl;
  }
  const int mt = t / p.n_tiles;
  tl.nt = t - mt * p.n_tiles;
  int lo = 0, hi = p.E;  // tile_prefix[lo] <= mt < tile_prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(p.tile_prefix + mid) <= mt)
      lo = mid;
    else
      hi = mid;
  }
  tl.e = lo;
  const int end = __ldg(p.m_indptr + lo + 1);
  const int start = __ldg(p.m_indptr + lo);
  tl.m0 = start + (mt - __ldg(p.tile_prefix + lo)) * (2 * BM) + static_cast<int>(rank) * BM;
  tl.rows = max(0, min(BM, end - tl.m0));
  tl.row0 = 0;
  tl.am0 = p.pad_indptr != nullptr ? __ldg(p.pad_indptr + lo) + (tl.m0 - start) : tl.m0;
  tl.prow0 = 0;
  tl.kb_count = p.num_kb;
  tl.f16 = 0;
  return tl;
}

__device__ __forceinline__ void raise_abort(int* err, volatile int* abort_flag) {
  if (!*abort_flag) {
    atomicOr(err, LIGER_MOE_DEVERR_WAIT_TIMEOUT);
    *abort_flag = 1;
  }
}

__device__ __forceinline__ void load16_f32(const float* src, float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 q = __ldg(reinterpret_cast<const float4*>(src) + i);
    v[4 * i] = q.x;
    v[4 * i + 1] = q.y;
    v[4 * i + 2] = q.z;
    v[4 * i + 3] = q.w;
  }
}

__device__ __forceinline__ void load16_bf16(const uint16_t* src, float (&v)[16]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
  const uint4 b = __ldg(reinterpret_cast<const uint4*>(src) + 1);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16_lo(w[i]);
    v[2 * i + 1] = bf16_hi(w[i]);
  }
}

// ---------------------------------------------------------------- gated activations
// h = act(g, u) from the fp32 gate/up accumulators, with the backward's derivative factors
// a = dh/dg and b = dh/du (LightMoE README, "Compatibility" / "Highlights" name the variants):
//   SwiGLU          h = silu(g) u
//   bounded SwiGLU  h = silu(gc) uc,  gc = min(g, c), uc = clamp(u, -c, c)
//   SwiGLU-OAI      h = gc sigmoid(1.702 gc) (uc + 1), same clamps, c the limit
//   GeGLU           h = gelu(g) u, gelu with the tanh form
//   ReGLU           h = max(g, 0) u
// A clamp passes the gradient on its closed interval and blocks it outside.
template <int ACT>
__device__ __forceinline__ void gated_act(float g, float u, float c, float& h, float& a, float& b) {
  if constexpr (ACT == LIGER_MOE_ACT_SWIGLU) {
    const float sg = 1.0f / (1.0f + expf(-g));
    const float sl = g * sg;
    h = sl * u;
    a = u * sg * (1.0f + g * (1.0f - sg));
    b = sl;
  } else if constexpr (ACT == LIGER_MOE_ACT_SWIGLU_BOUNDED || ACT == LIGER_MOE_ACT_SWIGLU_OAI) {
    constexpr float kAlpha = ACT == LIGER_MOE_ACT_SWIGLU_OAI ? 1.702f : 1.0f;
    const float gc = fminf(g, c), uc = fminf(fmaxf(u, -c), c);
    const float sg = 1.0f / (1.0f + expf(-kAlpha * gc));
    const float glu = gc * sg;
    const float lin = ACT == LIGER_MOE_ACT_SWIGLU_OAI ? uc + 1.0f : uc;
    h = glu * lin;
    a = (g <= c) ? lin * sg * (1.0f + kAlpha * gc * (1.0f - sg)) : 0.0f;
    b = (u >= -c && u <= c) ? glu : 0.0f;
  } else if constexpr (ACT == LIGER_MOE_ACT_GEGLU) {
    constexpr float k0 = 0.7978845608028654f, k1 = 0.044715f;  // sqrt(2/pi), cubic coefficient
    const float t = tanhf(k0 * (g + k1 * g * g * g));
    const float gelu = 0.5f * g * (1.0f + t);
    h = gelu * u;
    a = u * (0.5f * (1.0f + t) + 0.5f * g * (1.0f - t * t) * k0 * (1.0f + 3.0f * k1 * g * g));
    b = gelu;
  } else {  // ReGLU
    const float r = fmaxf(g, 0.0f);
    h = r * u;
    a = g > 0.0f ? u : 0.0f;
    b = r;
  }
}

template <int ACT>
__device__ __forceinline__ void gated_act32(const float (&g)[32], const float (&u)[32], float c, float (&hv)[32],
                                            uint32_t (&aw)[32], uint32_t (&bw)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float a, b;
    gated_act<ACT>(g[i], u[i], c, hv[i], a, b);
    aw[i] = __float_as_uint(a);
    bw[i] = __float_as_uint(b);
  }
}

// ---------------------------------------------------------------- epilogue output path
// An epilogue warp owns 32 accumulator rows.  Each output box is 32 rows x 128 bytes
// (64 bf16 or 32 fp32 columns): every lane writes its row into a swizzled staging buffer,
// then lane 0 issues one TMA store.  Where only part of the warp's 32 rows belong to the
// tile (the last tile of an expert), the valid rows are stored directly instead.
enum class Rows : int { Full = 0, Partial = 1, None = 2 };

struct Stager {
  uint32_t base;  // this warp's staging buffers (shared address, 1024-aligned)
  int idx;        // buffer to fill next
};

template <int RANK>
__device__ __forceinline__ void emit_box(const CUtensorMap* tm, Stager& st, int lane, const uint32_t (&w)[32], int x,
                                         int y, int z) {
  if (lane == 0) bulk_wait_group_read<STG_PER_WARP - 1>();  // the buffer's previous store has read it
  __syncwarp();
  const uint32_t row = st.base + st.idx * STG_BYTES + lane * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    st_shared_v4(row + ((c ^ (lane & 7)) << 4), make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]));
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if constexpr (RANK == 3)
      tma_store_3d(tm, st.base + st.idx * STG_BYTES, x, y, z);
    else
      tma_store_2d(tm, st.base + st.idx * STG_BYTES, x, y);
    bulk_commit_group();
  }
  st.idx = (st.idx + 1) % STG_PER_WARP;
}

// One 128-byte output row segment: a TMA box for full slices, direct stores otherwise.
__device__ __forceinline__ void emit_row(Rows mode, bool row_ok, const CUtensorMap* tm, Stager& st, int lane,
                                         const uint32_t (&w)[32], int x, int y, void* direct) {
  if (mode == Rows::Full) {
    emit_box<2>(tm, st, lane, w, x, y, 0);
  } else if (row_ok) {
    uint4* d = reinterpret_cast<uint4*>(direct);
#pragma unroll
    for (int c = 0; c < 8; ++c) d[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  }
}

template <Sched S>
__device__ __forceinline__ Rows slice_mode(const Tile& tl, int sub) {
  if constexpr (S == Sched::RowsK) return Rows::Full;  // 3D output maps clip the M tail
  const int n = tl.rows - sub * 32;
  return n >= 32 ? Rows::Full : (n > 0 ? Rows::Partial : Rows::None);
}

// Epilogue of one tile for one warp: each lane is one accumulator row; the warp covers the
// rows of TMEM quadrant `sub` and the tile's output columns of half `colhalf`.
template <Sched S, Epi EP>
__device__ __forceinline__ void epilogue_tile(uint32_t t_row, const Tile& tl, int sub, int colhalf, int lane,
                                              const Params& p, const CUtensorMap* tmC0, const CUtensorMap* tmC1,
                                              Stager& st) {
  const int row_local = sub * 32 + lane;
  const Rows mode = slice_mode<S>(tl, sub);
  const bool row_ok = (S == Sched::RowsK) ? true : row_local < tl.rows;
  if constexpr (gate_up_epi(EP)) {
    if (mode == Rows::None) return;
    // accumulator columns [0, BN/2) = g, [BN/2, BN) = u for output columns nt*BN/2 + c;
    // this warp's output columns: [64 colhalf, 64 colhalf + 64)
    const long long r = tl.m0 + row_local;
    const int y = tl.m0 + sub * 32;
    const int j0 = tl.nt * (BN / 2);
#pragma unroll 1
    for (int q = colhalf; q < colhalf + 1; ++q) {
      const int col = j0 + q * 64;
      if (col >= p.I) break;
      uint32_t hw[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float g[32], u[32];
        tmem_ld32(t_row + q * 64 + half * 32, g);
        tmem_ld32(t_row + BN / 2 + q * 64 + half * 32, u);
        tmem_ld_wait();
        // h = act(g, u); the backward's derivative factors dh/dg, dh/du are saved in fp32
        // (GLU: the activation is the same for the whole launch, so the switch is warp-uniform)
        uint32_t aw[32], bw[32];
        float hv[32];
        if constexpr (EP == Epi::SwiGLU) {
          gated_act32<LIGER_MOE_ACT_SWIGLU>(g, u, 0.f, hv, aw, bw);
        } else {
          switch (p.act) {
            case LIGER_MOE_ACT_SWIGLU_BOUNDED:
              gated_act32<LIGER_MOE_ACT_SWIGLU_BOUNDED>(g, u, p.act_clamp, hv, aw, bw);
              break;
            case LIGER_MOE_ACT_SWIGLU_OAI:
              gated_act32<LIGER_MOE_ACT_SWIGLU_OAI>(g, u, p.act_clamp, hv, aw, bw);
              break;
            case LIGER_MOE_ACT_GEGLU:
              gated_act32<LIGER_MOE_ACT_GEGLU>(g, u, p.act_clamp, hv, aw, bw);
              break;
            case LIGER_MOE_ACT_REGLU:
              gated_act32<LIGER_MOE_ACT_REGLU>(g, u, p.act_clamp, hv, aw, bw);
              break;
            default:
              gated_act32<LIGER_MOE_ACT_SWIGLU>(g, u, p.act_clamp, hv, aw, bw);
          }
        }
        if (p.gu_out != nullptr) {
          const int xg = col + half * 32;
          emit_row(mode, row_ok, tmC1, st, lane, aw, xg, y, p.gu_out + r * (2LL * p.I) + xg);
          emit_row(mode, row_ok, tmC1, st, lane, bw, p.I + xg, y, p.gu_out + r * (2LL * p.I) + p.I + xg);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) hw[half * 16 + i] = pack_bf16x2(hv[2 * i], hv[2 * i + 1]);
      }
      if (p.out != nullptr) emit_row(mode, row_ok, tmC0, st, lane, hw, col, y, p.out + r * p.ld_out + col);
    }
  } else if constexpr (EP == Epi::ReLU2) {
    // acc = a = x W_up[e]^T (the expert's one projection); h = r^2 with r = max(a, 0), and the
    // backward's derivative factor dh/da = 2 r in fp32 ([R, I]).  This warp's output columns:
    // [128 colhalf, 128 colhalf + 128) of the tile's BN.
    if (mode == Rows::None) return;
    const long long r = tl.m0 + row_local;
    const int y = tl.m0 + sub * 32;
#pragma unroll 1
    for (int q = 2 * colhalf; q < 2 * colhalf + 2; ++q) {
      const int col = tl.nt * BN + q * 64;
      if (col >= p.I) break;
      uint32_t hw[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float a[32];
        tmem_ld32(t_row + q * 64 + half * 32, a);
        tmem_ld_wait();
        uint32_t fw[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float rr = fmaxf(a[i], 0.0f);
          fw[i] = __float_as_uint(2.0f * rr);
          a[i] = rr * rr;
        }
        if (p.gu_out != nullptr) {
          const int xg = col + half * 32;
          emit_row(mode, row_ok, tmC1, st, lane, fw, xg, y, p.gu_out + r * p.I + xg);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) hw[half * 16 + i] = pack_bf16x2(a[2 * i], a[2 * i + 1]);
      }
      if (p.out != nullptr) emit_row(mode, row_ok, tmC0, st, lane, hw, col, y, p.out + r * p.ld_out + col);
    }
  } else if constexpr (EP == Epi::Logits) {
    // acc = x[r] Wr^T over this tile's columns; out = acc + bias (fp32).  This warp's columns:
    // [128 colhalf, 128 colhalf + 128) of the tile, in chunks of 32.  Chunks that lie wholly
    // inside N_out leave as 32 x 32 fp32 boxes (or 32-float row stores in a partial slice);
    // a chunk that crosses N_out, or any chunk when the row stride is not a multiple of 32,
    // is stored element by element.
    if (mode == Rows::None) return;
    const long long r = tl.m0 + row_local;
    const int y = tl.m0 + sub * 32;
#pragma unroll 1
    for (int q = 4 * colhalf; q < 4 * colhalf + 4; ++q) {
      const int col = tl.nt * BN + q * 32;
      if (col >= p.N_out) break;
      const int ncol = min(32, p.N_out - col);
      float v[32];
      tmem_ld32(t_row + q * 32, v);
      tmem_ld_wait();
      if (p.col_bias != nullptr) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i < ncol) v[i] += __ldg(p.col_bias + col + i);
      }
      if (p.out_tma && ncol == 32) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i]);
        emit_row(mode, row_ok, tmC0, st, lane, w, col, y, p.out_f32 + r * p.ld_out + col);
      } else if (row_ok) {
        float* dst = p.out_f32 + r * p.ld_out + col;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i < ncol) dst[i] = v[i];
      }
    }
  } else if constexpr (dh_epi(EP)) {
    // acc = dHu = dY[token] W_d[e] for this row; d = w_r * dHu in fp32.  The saved forward
    // state gives the SwiGLU derivative factors a = dh/dg, b = dh/du (fp32) and h (bf16):
    //   dg = d a,  du = d b,  <d, h> (router-gradient partial),  w_r h (the dW_down operand).
    // Every bf16 operand of the weight-gradient GEMMs is written as two bf16 parts,
    // hi = bf16(v) in rows [0, R) and lo = bf16(v - hi) in rows [R, 2R), so that hi + lo
    // carries v to about 2^-17 relative:  dgu = [dg | du] ([2R, 2I]; the dX GEMM reads only
    // the hi rows) and hw = w_r h ([2R, I]).  Outputs leave through 32-row x 16-column boxes
    // (32-byte swizzle), six per 16 columns, double-buffered; the loads of the next 16
    // columns are issued before the current ones are processed.
    // This warp's columns: [n0 + c_lo, n0 + c_hi), half of the tile's N columns.
    // Input rows are routed rows r; outputs go to padded rows ro (their expert's padded range).
    // In an expert's last tile the lanes past its rows, up to the next multiple of 16, write
    // zero rows (all inside the slice that holds the expert's last row, since 16 divides 32).
    // DH1 (two-weight experts, h = max(a, 0)^2): one factor a = dh/da per element ([R, I]) and one
    // gradient da = d a, written as hi/lo into [2R, I]; four output boxes per 16 columns.
    // fp16 tiles (tl.f16, experts with many rows): the lo rows receive fp16(dg 2^sg), fp16(du 2^sg)
    // and fp16(w h 2^sh) instead, the hi rows of w h are not written (five boxes per 16 columns),
    // and the largest scaled magnitudes go to the expert's range words.
    constexpr bool kGated = EP != Epi::DH1;
    const bool f16 = EP == Epi::DH16 && tl.f16 != 0;
    float sg = 1.f;
    if (f16) {
      int sd = 0;
      f16_scale_exp(p.f16_words[kF16MaxDy], sd);
      sg = f16_pow2(sd + kF16DguShift);
    }
    const float sh = f16_pow2(kF16HwShift);
    float mg = 0.f, mh = 0.f;  // largest |scaled dgu| and |scaled w h| of this thread's row
    const long long r = tl.m0 + row_local;
    const long long ro = tl.am0 + row_local;
    const bool pad_row = !row_ok && row_local < ((tl.rows + 15) & ~15);
    const long long two_i = (kGated ? 2LL : 1LL) * p.I;  // row length of the factors and of dgu
    const int y = tl.am0 + sub * 32;
    const int n0 = tl.nt * BN;
    const int ncols = min(BN, p.I - n0);  // a positive multiple of 64
    const int c_lo = colhalf * (BN / 2);
    const int c_hi = min(c_lo + BN / 2, ncols);
    const float wr = row_ok ? __ldg(p.row_scale + r) : 0.f;
    const float* arow = p.gu_in + r * two_i;
    const uint16_t* hrow = p.h_in + r * p.I;
    float part = 0.f;
    auto load_ops = [&](int n, float (&a)[16], float (&b)[16], float (&h)[16]) {
      if (row_ok) {
        load16_f32(arow + n, a);
        if constexpr (kGated) load16_f32(arow + p.I + n, b);
        load16_bf16(hrow + n, h);
      }
    };
    auto process = [&](int c, const float (&a)[16], const float (&b)[16], const float (&h)[16]) {
      float dh[16];
      tmem_ld16(t_row + c, dh);
      tmem_ld_wait();
      uint32_t o[6][8];  // dg hi, dg lo, du hi, du lo, hw hi, hw lo (8 bf16 pairs each)
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        float v[3][2];
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int q = i + e2;
          const float d = wr * dh[q];
          part += d * h[q];
          v[0][e2] = d * a[q];
          v[1][e2] = kGated ? d * b[q] : 0.f;
          v[2][e2] = wr * h[q];
        }
#pragma unroll
        for (int f = 0; f < 3; ++f) {
          if (!kGated && f == 1) continue;
          const uint32_t hi = pack_bf16x2(v[f][0], v[f][1]);
          o[2 * f][i / 2] = hi;
          if (f16) {
            const float sc = f == 2 ? sh : sg;
            const float x0 = v[f][0] * sc, x1 = v[f][1] * sc;
            o[2 * f + 1][i / 2] = pack_f16x2(x0, x1);
            const float m = row_ok ? fmaxf(fabsf(x0), fabsf(x1)) : 0.f;
            if (f == 2)
              mh = fmaxf(mh, m);
            else
              mg = fmaxf(mg, m);
          } else {
            o[2 * f + 1][i / 2] = pack_bf16x2(v[f][0] - bf16_lo(hi), v[f][1] - bf16_hi(hi));
          }
        }
      }
      const int n = n0 + c;
      if (mode == Rows::Full) {
        if (lane == 0) bulk_wait_group_read<0>();  // the boxes' previous stores have read them
        __syncwarp();
        const uint32_t base = st.base;
        const uint32_t sw = (lane >> 2) & 1;  // 32-byte swizzle: chunk ^= (row >> 2) & 1
#pragma unroll
        for (int f = 0; f < 6; ++f) {
          if ((!kGated && (f == 2 || f == 3)) || (f16 && f == 4)) continue;
          const uint32_t row_addr = base + f * kDhBoxBytes + lane * 32;
          st_shared_v4(row_addr + ((0 ^ sw) << 4), make_uint4(o[f][0], o[f][1], o[f][2], o[f][3]));
          st_shared_v4(row_addr + ((1 ^ sw) << 4), make_uint4(o[f][4], o[f][5], o[f][6], o[f][7]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int yl = y + static_cast<int>(p.lo_rows);
          tma_store_2d(tmC0, base + 0 * kDhBoxBytes, n, y);
          tma_store_2d(tmC0, base + 1 * kDhBoxBytes, n, yl);
          if constexpr (kGated) {
            tma_store_2d(tmC0, base + 2 * kDhBoxBytes, p.I + n, y);
            tma_store_2d(tmC0, base + 3 * kDhBoxBytes, p.I + n, yl);
          }
          if (!f16) tma_store_2d(tmC1, base + 4 * kDhBoxBytes, n, y);
          tma_store_2d(tmC1, base + 5 * kDhBoxBytes, n, yl);
          bulk_commit_group();
        }
      } else if (row_ok || pad_row) {
        if (pad_row) {
#pragma unroll
          for (int f = 0; f < 6; ++f)
#pragma unroll
            for (int q = 0; q < 8; ++q) o[f][q] = 0u;
        }
        const long long rl = p.lo_rows + ro;
        uint16_t* dst[6] = {p.out2 + ro * two_i + n, p.out2 + rl * two_i + n, p.out2 + ro * two_i + p.I + n,
                            p.out2 + rl * two_i + p.I + n, p.hw_out + ro * p.I + n, p.hw_out + rl * p.I + n};
#pragma unroll
        for (int f = 0; f < 6; ++f) {
          if ((!kGated && (f == 2 || f == 3)) || (f16 && f == 4)) continue;
          reinterpret_cast<uint4*>(dst[f])[0] = make_uint4(o[f][0], o[f][1], o[f][2], o[f][3]);
          reinterpret_cast<uint4*>(dst[f])[1] = make_uint4(o[f][4], o[f][5], o[f][6], o[f][7]);
        }
      }
    };
    if (mode != Rows::None) {
      float a0[16], b0[16], h0[16], a1[16], b1[16], h1[16];
      if (c_lo < c_hi) load_ops(n0 + c_lo, a0, b0, h0);
#pragma unroll 1
      for (int c = c_lo; c < c_hi; c += 32) {
        load_ops(n0 + c + 16, a1, b1, h1);
        process(c, a0, b0, h0);
        if (c + 32 < c_hi) load_ops(n0 + c + 32, a0, b0, h0);
        process(c + 16, a1, b1, h1);
      }
    }
    if (row_ok) p.gdot[r * (2LL * p.n_tiles) + 2 * tl.nt + colhalf] = part;
    if (f16 && mode != Rows::None) {
      // non-negative floats order as their bits
      const unsigned bg = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(mg));
      const unsigned bh = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(mh));
      if (lane == 0) {
        atomicMax(p.f16_words + kF16Range + tl.e, bg);
        atomicMax(p.f16_words + kF16Range + p.E + tl.e, bh);
      }
    }
  } else {  // ScaleRows, Store: this warp's columns [128 colhalf, 128 colhalf + 128)
    if (mode == Rows::None) return;
    float sc = 1.f;
    if constexpr (EP == Epi::ScaleRows) sc = row_ok ? __ldg(p.row_scale + tl.m0 + row_local) : 0.f;
    if constexpr (S == Sched::RowsK)
      if (tl.f16) sc = f16_unscale(p);  // fp16 operands: undo their scales
#pragma unroll 1
    for (int q = 2 * colhalf; q < 2 * colhalf + 2; ++q) {
      const int col = tl.nt * BN + q * 64;
      if (col >= p.N_out) break;
      float a[32], b[32];
      tmem_ld32(t_row + q * 64, a);
      tmem_ld32(t_row + q * 64 + 32, b);
      tmem_ld_wait();
      uint32_t w[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        w[i] = pack_bf16x2(sc * a[2 * i], sc * a[2 * i + 1]);
        w[16 + i] = pack_bf16x2(sc * b[2 * i], sc * b[2 * i + 1]);
      }
      if constexpr (S == Sched::RowsK) {
        emit_box<3>(tmC0, st, lane, w, col, tl.m0 + sub * 32, tl.e);
      } else {
        const long long r = tl.m0 + row_local;
        emit_row(mode, row_ok, tmC0, st, lane, w, col, tl.m0 + sub * 32, p.out + r * p.ld_out + col);
      }
    }
  }
}

// RowsK tile of an expert with no rows: the gradient block is exactly zero.  Each lane copies its
// output row's part of the tile (128 columns, 256 bytes) from a zero row in shared memory that no
// one ever writes again, so zero tiles need no staging and no wait between them.
__device__ __forceinline__ void store_zero_tile(const Tile& tl, int sub, int colhalf, int lane, const Params& p,
                                                uint32_t zero_row) {
  const int row = tl.m0 + sub * 32 + lane;
  const int c0 = tl.nt * BN + colhalf * (BN / 2);
  const int n = min(BN / 2, p.N_out - c0);  // a multiple of 64 (N_out is)
  if (row < p.M_out && n > 0) {
    bulk_store_s2g(p.out + tl.e * p.out_expert_stride + static_cast<long long>(row) * p.ld_out + c0, zero_row,
                   static_cast<uint32_t>(n) * 2u);
    bulk_commit_group();
  }
}

// DH epilogue operands of one tile row (the fp32 derivative factors and bf16 h) are pulled into
// L2 when the epilogue warp reaches the tile (before waiting for its accumulator).  One tile
// earlier proved too early: in the epilogue-bound dH kernel a tile takes tens of microseconds,
// and the prefetched lines were evicted before use.
template <Sched S, Epi EP>
__device__ __forceinline__ void prefetch_epilogue_operands(const Tile& tl, int row_local, int colhalf,
                                                           const Params& p) {
  if constexpr (dh_epi(EP)) {
    constexpr int kFactors = EP != Epi::DH1 ? 2 : 1;  // [a | b] or a alone per row
    if (row_local >= tl.rows) return;
    const long long r = tl.m0 + row_local;
    const int n0 = tl.nt * BN + colhalf * (BN / 2);
    const int ncols = min(BN / 2, p.I - n0);
    if (ncols <= 0) return;
    prefetch_l2_bulk(p.gu_in + r * kFactors * p.I + n0, ncols * 4);
    if constexpr (kFactors == 2) prefetch_l2_bulk(p.gu_in + r * 2LL * p.I + p.I + n0, ncols * 4);
    prefetch_l2_bulk(p.h_in + r * p.I + n0, ncols * 2);
  }
}

// Operand sources.  Gather::None: both operands through tiled TMA boxes.  Gather::A / B: that
// operand's rows are token rows of a token-major [T, cols] bf16 matrix, fetched with TMA
// gather4 through a tensor map whose box is one row high; RowsM gathers a K-major A (rows =
// M), RowsK an MN-major operand (rows = K).
enum class Gather : int { None = 0, A = 1, B = 2 };

// Where K block kb of a weight-gradient tile comes from.  In the fp16 experts' launch (f16_part,
// one operand part per stage): an fp16 tile reads the lo rows of the padded operand (its fp16 part,
// row offset a_split_rows for dW_gate_up's A, b_split_rows for dW_down's B) and the other operand
// from tmF (the fp16 token rows); a two-pass tile reads K block kbe = kb of the hi rows, then
// kbe = kb - n of the lo rows, against the bf16 token rows.  Elsewhere: block kb, tmA and tmB.
struct KbSource {
  int kbe;           // K block within the expert's rows
  int off_a, off_b;  // row offsets of A and B
  bool a_f16, b_f16; // A / B from tmF
};
__device__ __forceinline__ KbSource kb_source(const Tile& tl, int kb, const Params& p) {
  KbSource q{kb, 0, 0, false, false};
  if (!p.f16_part) return q;
  const bool gu = p.f16_role == 3;  // the padded operand: A (dW_gate_up) or B (dW_down)
  bool lo = tl.f16 != 0;
  if (!lo) {
    const int n = tl.kb_count / 2;
    lo = kb >= n;
    if (lo) q.kbe = kb - n;
  } else if (gu) {
    q.b_f16 = true;
  } else {
    q.a_f16 = true;
  }
  if (lo) (gu ? q.off_a : q.off_b) = gu ? p.a_split_rows : p.b_split_rows;
  return q;
}

// Tiled loads of one stage for the operands that are not gathered (lane 0 of the producer).
// Every box lands in this CTA's own shared memory and completes on its own full barrier.
template <Sched S, Epi EP, bool A_MN, bool B_MN, int SPLIT, bool kLoadA, bool kLoadB>
__device__ __forceinline__ void load_stage_tiled(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmF,
                                                 const Params& p, const Tile& tl, int kb, uint32_t sa, uint32_t sb,
                                                 uint32_t fb) {
  const KbSource q = S == Sched::RowsK ? kb_source(tl, kb, p) : KbSource{kb, 0, 0, false, false};
  if constexpr (kLoadA) {
    if constexpr (!A_MN) {  // RowsM: the tile's rows, in the padded row space when A is a padded operand
      tma_load_2d(sa, tmA, fb, kb * BK, p.pad_a ? tl.am0 : tl.m0);
    } else {
      const int krow = (p.pad_a ? tl.prow0 : tl.row0) + q.kbe * BK + q.off_a;
      const CUtensorMap* src = q.a_f16 ? tmF : tmA;
#pragma unroll
      for (int part = 0; part < (SPLIT == 1 ? 2 : 1); ++part)
#pragma unroll
        for (int i = 0; i < BM / 64; ++i)
          tma_load_2d(sa + part * A_BYTES + i * MN_BOX_BYTES, src, fb, tl.m0 + 64 * i,
                      krow + part * p.a_split_rows);
    }
  }
  if constexpr (kLoadB) {
    if constexpr (!B_MN) {
      if constexpr (gate_up_epi(EP)) {
        const int r = tl.e * p.b_rows_per_expert + tl.nt * (BN / 2);
        tma_load_2d(sb, tmB, fb, kb * BK, r);
        tma_load_2d(sb + B_BYTES / 2, tmB, fb, kb * BK, r + p.b_split);
      } else {
        tma_load_2d(sb, tmB, fb, kb * BK, tl.e * p.b_rows_per_expert + tl.nt * BN);
      }
    } else {
      const int krow = (S == Sched::RowsM) ? tl.e * p.b_rows_per_expert + kb * BK
                                           : (p.pad_b ? tl.prow0 : tl.row0) + q.kbe * BK + q.off_b;
      const CUtensorMap* src = q.b_f16 ? tmF : tmB;
#pragma unroll
      for (int part = 0; part < (SPLIT == 2 ? 2 : 1); ++part)
#pragma unroll
        for (int i = 0; i < BN / 64; ++i)
          tma_load_2d(sb + part * B_BYTES + i * MN_BOX_BYTES, src, fb, tl.nt * BN + 64 * i,
                      krow + part * p.b_split_rows);
    }
  }
}

// Loads of one stage in a 2-SM pair (RowsM, K-major A): this CTA's 128 rows of A and its half of
// B's 256 rows, both completing on the even CTA's full barrier (`bar`, a shared::cluster
// address), which expects the bytes of both CTAs.  Gate/up tiles put the gate rows in the even
// CTA and the up rows in the odd one, so the accumulator columns stay [g | u].
template <Sched S, Epi EP, bool B_MN, int SPLIT>
__device__ __forceinline__ void load_stage_pair(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmF,
                                                const Params& p, const Tile& tl, int kb, uint32_t sa, uint32_t sb,
                                                uint32_t bar, uint32_t rank) {
  if constexpr (S == Sched::RowsK) {
    // weight gradients, both operands MN-major with the expert's rows as K: this CTA's 128 M
    // columns of A (two 64-column boxes, hi and lo parts for SPLIT 1) and its 128 of the N
    // block's 256 columns of B (hi and lo parts for SPLIT 2).  The fp16 experts' launch: as
    // kb_source says.
    const KbSource q = kb_source(tl, kb, p);
    const int krow_a = (p.pad_a ? tl.prow0 : tl.row0) + q.kbe * BK + q.off_a;
    const int krow_b = (p.pad_b ? tl.prow0 : tl.row0) + q.kbe * BK + q.off_b;
    const CUtensorMap* src_a = q.a_f16 ? tmF : tmA;
    const CUtensorMap* src_b = q.b_f16 ? tmF : tmB;
#pragma unroll
    for (int part = 0; part < (SPLIT == 1 ? 2 : 1); ++part)
#pragma unroll
      for (int i = 0; i < 2; ++i)
        tma_load_2d_pair(sa + part * A_BYTES + i * MN_BOX_BYTES, src_a, bar, tl.m0 + 64 * i,
                         krow_a + part * p.a_split_rows);
#pragma unroll
    for (int part = 0; part < (SPLIT == 2 ? 2 : 1); ++part)
#pragma unroll
      for (int i = 0; i < 2; ++i)
        tma_load_2d_pair(sb + part * (B_BYTES / 2) + i * MN_BOX_BYTES, src_b, bar,
                         tl.nt * BN + static_cast<int>(rank) * (BN / 2) + 64 * i, krow_b + part * p.b_split_rows);
    return;
  }
  tma_load_2d_pair(sa, tmA, bar, kb * BK, p.pad_a ? tl.am0 : tl.m0);  // A box: 128 rows (past the end: zeros)
  if constexpr (!B_MN) {
    const int r = gate_up_epi(EP) ? tl.e * p.b_rows_per_expert + tl.nt * (BN / 2) + (rank ? p.b_split : 0)
                                  : tl.e * p.b_rows_per_expert + tl.nt * BN + static_cast<int>(rank) * (BN / 2);
    tma_load_2d_pair(sb, tmB, bar, kb * BK, r);  // B box: 128 rows
  } else {
    const int krow = tl.e * p.b_rows_per_expert + kb * BK;
#pragma unroll
    for (int i = 0; i < BN / 128; ++i)  // this CTA's two 64-column boxes of the tile's N columns
      tma_load_2d_pair(sb + i * MN_BOX_BYTES, tmB, bar, tl.nt * BN + static_cast<int>(rank) * (BN / 2) + 64 * i,
                       krow);
  }
}

// Tokens of the four rows a producer lane gathers for (tile, K block): RowsM, rows 4 lane ..
// 4 lane + 3 of the tile; RowsK, rows 4 (lane & 15) .. + 3 of the K block.  Rows outside the
// tile or expert take token 0 (their products are discarded, or their shared-memory rows are
// zeroed before the MMA); a slot outside [0, R) raises BAD_ROW and also reads token 0.
template <Sched S>
__device__ __forceinline__ void gather_tokens(const Tile& tl, int kb, int lane, const Params& p, int (&tk)[4]) {
  int first;
  long long base;
  if constexpr (S == Sched::RowsM) {
    first = 4 * lane;
    base = tl.m0;
  } else {
    first = kb * BK + 4 * (lane & 15);
    base = tl.row0;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int tok = 0;
    if (first + j < tl.rows) {
      const int slot = __ldg(p.row_slot + base + first + j);
      if (slot >= 0 && slot < p.R)
        tok = slot / p.topk;
      else
        atomicOr(p.err, LIGER_MOE_DEVERR_BAD_ROW);
    }
    tk[j] = tok;
  }
}

// PAIR (launched as clusters of two CTAs): the two CTAs work on one 256-row tile with 2-SM MMAs
// (cta_group::2): each loads its own halves of the operands into its own shared memory, the even
// CTA's MMA warp issues every MMA and commits to both CTAs' barriers, and both CTAs' epilogues
// release the accumulator to the even CTA.  Without PAIR every CTA works alone (CL = 1).
template <Sched S, Epi EP, bool A_MN, bool B_MN, int SPLIT, Gather G, int CL, int PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC0, const __grid_constant__ CUtensorMap tmC1,
                        const __grid_constant__ CUtensorMap tmF, const Params p) {
  using L = LayoutOf<EP, SPLIT, PAIR>;
  constexpr bool kPair = PAIR != 0;
  static_assert(CL == (kPair ? 2 : 1), "clusters exist only as the 2-SM pairs");
  static_assert(!kPair || (CL == 2 && G == Gather::None &&
                            ((S == Sched::RowsM && !A_MN && SPLIT == 0) || (S == Sched::RowsK && A_MN && B_MN))),
                "2-SM pairs: RowsM tiles with K-major A and one operand part, or RowsK tiles, no gather");
  constexpr int STAGES = L::kStages;
  constexpr int STAGE_BYTES = L::kStageBytes;
  constexpr uint16_t kClusterMask = static_cast<uint16_t>((1u << CL) - 1u);
  const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;
  const bool leader = !kPair || rank == 0;  // the CTA that issues the MMAs
  // pairs walk the tiles together: tile t of cluster c is t = c, c + clusters, ...
  const int tile0 = kPair ? static_cast<int>(blockIdx.x) / 2 : static_cast<int>(blockIdx.x);
  const int tstride = kPair ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);
  // dynamic order: weight gradients of one-CTA tiles with tiled operands, when the load is skewed
  // (every role reads the same flag, written by the schedule kernel before this launch)
  bool dyn = false;
  auto decode = [&](int t) -> Tile {
    if constexpr (kPair)
      return decode_tile_pair<S>(t, p, rank);
    else
      return decode_tile<S>(t, p);
  };
  static_assert(SPLIT == 0 || (S == Sched::RowsK && A_MN && B_MN), "hi/lo operands only in the dW GEMMs");
  static_assert(G == Gather::None || (S == Sched::RowsM ? (G == Gather::A && !A_MN)
                                                         : (G == Gather::A ? (A_MN && SPLIT != 1)
                                                                           : (B_MN && SPLIT != 2))),
                "RowsM gathers a K-major A; RowsK gathers an MN-major operand held as one part");
  if (p.f16_role == 1) {
    // the fp16 dH pass: leave at once when no expert has f16 rows (the next launch is then the whole dH)
    griddep_wait();
    if (p.f16_words[kF16Any] == 0u) return;
  }
  if (p.f16_role == 2 && p.f16_words[kF16Any] != 0u) {
    // dH refill: leave at once (before any set-up) when no expert with f16 rows has unusable fp16
    // parts, which is the usual case; the range words are the previous kernel's output
    griddep_wait();
    bool need = false;
    for (int e = threadIdx.x; e < p.E; e += blockDim.x)
      need = need || (__ldg(p.m_indptr + e + 1) - __ldg(p.m_indptr + e) >= p.f16_rows && !f16_usable(e, p));
    if (!__syncthreads_or(need ? 1 : 0)) return;
  }
  if (p.parted) {
    // an empty part of the experts (e.g. no expert reaches the fp16 pass's rows): leave before any
    // set-up; every CTA of a pair reads the same counts, so both leave
    griddep_wait();
    if (part_hi(p) <= part_lo(p)) return;
  }
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (sbase - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + L::kBarOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // the tile ring (dynamic order): decoded tiles from the producer to the MMA and epilogue warps
  // (full: written; empty: read by all of them), so that only the producer reads the schedule from
  // global memory
  static_assert(2 * 6 + 5 + 1 <= kSchedBarIndex &&
                    (kSchedBarIndex + 2 * kSchedSlots) * 8 + 4 * kRingInts * kSchedSlots <= kBarrierBytes,
                "barrier area layout");
  volatile int* sched_ring = reinterpret_cast<volatile int*>(bars + kSchedBarIndex + 2 * kSchedSlots);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + STAGES);
  const uint32_t tfull0 = smem_u32(bars + 2 * STAGES);
  const uint32_t tempty0 = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t drain = smem_u32(bars + 2 * STAGES + 4);
  const uint32_t sfull0 = smem_u32(bars + kSchedBarIndex);
  const uint32_t sempty0 = smem_u32(bars + kSchedBarIndex + kSchedSlots);
  const uint32_t zero_row = smem_u32(base_ptr + L::kBarOffset + kZeroOffset);  // kZeroBytes of zeros
  static_assert(kSchedBarIndex * 8 + 2 * kSchedSlots * 8 + 4 * kRingInts * kSchedSlots <= kZeroOffset &&
                    kZeroOffset + kZeroBytes <= kBarrierBytes,
                "barrier area: barriers, tile ring, zero row");

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);  // released by this CTA's MMA commit (pair: the even CTA's)
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, kPair ? 2 * kEpiWarps : kEpiWarps);  // pair: both CTAs' epilogue warps
    }
    mbar_init(drain, 1);
    for (int q = 0; q < kSchedSlots; ++q) {
      mbar_init(sfull0 + 8 * q, 1);
      mbar_init(sempty0 + 8 * q, (leader ? 1 : 0) + kEpiWarps);  // the MMA warp (if it issues) and every epilogue warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < kZeroBytes / 16) {  // the zero row that zero tiles copy out (async proxy reads it)
    st_shared_v4(zero_row + 16 * threadIdx.x, make_uint4(0u, 0u, 0u, 0u));
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC0);
    tma_prefetch_desc(&tmC1);
    if (p.f16_role >= 3) tma_prefetch_desc(&tmF);
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  if constexpr (CL > 1)
    cluster_sync();  // both CTAs' barriers exist before a pair load or commit reaches them
  else
    __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // barriers, TMEM and descriptors are ready: from here on the kernel reads what earlier kernels wrote
  griddep_wait();
  griddep_launch_dependents();
  if constexpr (S == Sched::RowsK && !kPair && G == Gather::None)
    dyn = p.claims != nullptr && __ldg(p.sched_skewed) != 0;

  int total;
  if constexpr (S == Sched::RowsM)
    total = __ldg(p.tile_prefix + p.E) * p.n_tiles;
  else if constexpr (S == Sched::Dense)
    total = static_cast<int>((p.R + BM - 1) / BM) * p.n_tiles;
  else
    total = (p.parted ? part_hi(p) - part_lo(p) : p.E) * (kPair ? p.m_tiles / 2 : p.m_tiles) *
            p.n_tiles;  // experts of the part x tiles (pair: M blocks two at a time)

  // The tile sequence of the MMA warp and the epilogue warps: the tile at queue position t (t < 0 or
  // past the launch's tiles ends it) and its accumulator.  In the static order every warp walks
  // tile0, tile0 + tstride, ... and decodes the tiles itself, the accumulators alternating over
  // tiles with K blocks; in the dynamic order the producer decodes every tile and passes it, with
  // its accumulator, through the ring.  (slot, sphase: this warp's position in the ring; the
  // producer writes through its own copy.)  false: a wait gave up.
  int slot = 0;
  uint32_t sphase = 0;
  int acc_walk = 1;
  auto next_tile = [&](int& t, Tile& tl, int& acc, bool first) -> bool {
    if (G != Gather::None || !dyn) {
      t = first ? tile0 : t + tstride;
      if (t < total) {
        tl = decode(t);
        if (tl.kb_count > 0) acc_walk ^= 1;
        acc = acc_walk;
      }
      return true;
    } else {
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(sfull0 + 8 * slot, sphase, abort_flag))) return false;
      const volatile int* r = sched_ring + kRingInts * slot;
      t = r[0];
      acc = r[1];
      tl.e = r[2];
      tl.m0 = r[3];
      tl.rows = r[4];
      tl.nt = r[5];
      tl.row0 = r[6];
      tl.am0 = r[7];
      tl.prow0 = r[8];
      tl.kb_count = r[9];
      tl.f16 = r[10];
      __syncwarp();
      if (lane == 0) mbar_arrive(sempty0 + 8 * slot);
      if (++slot == kSchedSlots) {
        slot = 0;
        sphase ^= 1u;
      }
      return true;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if constexpr (G == Gather::None) {
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        bool failed = false;
        // the K blocks of a tile into the stage ring, in order.  false: a wait gave up.
        auto load_tile = [&](const Tile& tl) -> bool {
          for (int kb = 0; kb < tl.kb_count; ++kb) {
            if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag)) return false;
            const uint32_t sa = sbase + stage * STAGE_BYTES;
            const uint32_t fb = full0 + 8 * stage;
            if constexpr (kPair) {
              // the even CTA's full barrier counts both CTAs' bytes of this stage
              if (leader) mbar_arrive_expect_tx(fb, 2 * STAGE_BYTES);
              load_stage_pair<S, EP, B_MN, SPLIT>(&tmA, &tmB, &tmF, p, tl, kb, sa, sa + L::kABytes,
                                                  mapa_shared(fb, 0), rank);
            } else {
              mbar_arrive_expect_tx(fb, STAGE_BYTES);
              load_stage_tiled<S, EP, A_MN, B_MN, SPLIT, true, true>(&tmA, &tmB, &tmF, p, tl, kb, sa,
                                                                     sa + L::kABytes, fb);
            }
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          return true;
        };
        // a tile's position, accumulator and decoded fields into the ring (before its loads)
        auto publish = [&](int t, const Tile& tl, int acc) -> bool {
          if (!mbar_wait(sempty0 + 8 * slot, sphase ^ 1u, abort_flag)) return false;
          volatile int* r = sched_ring + kRingInts * slot;
          r[0] = t;
          r[1] = acc;
          r[2] = tl.e;
          r[3] = tl.m0;
          r[4] = tl.rows;
          r[5] = tl.nt;
          r[6] = tl.row0;
          r[7] = tl.am0;
          r[8] = tl.prow0;
          r[9] = tl.kb_count;
          r[10] = tl.f16;
          mbar_arrive(sfull0 + 8 * slot);
          if (++slot == kSchedSlots) {
            slot = 0;
            sphase ^= 1u;
          }
          return true;
        };
        if (!dyn) {
          for (int t = tile0; t < total; t += tstride) {
            const Tile tl = decode(t);
            if (!load_tile(tl)) {
              failed = true;
              break;
            }
          }
        } else {
          // Dynamic order: the queue positions (experts sorted by rows, most first, their tiles
          // expert by expert) are claimed through one counter, two claims ahead, and the next
          // tile's table entry is loaded one tile ahead, so that the atomics' and the loads'
          // latency passes during the loads of earlier tiles.  A claimed position is always
          // processed by its claimer.  Every tile is published to the ring before its loads, the
          // accumulators alternating over tiles with K blocks; a -1 position ends the sequence.
          const int per_e = p.m_tiles * p.n_tiles;
          const int4* info = reinterpret_cast<const int4*>(p.sched_info) + (p.parted ? part_lo(p) : 0);
          auto claim = [&]() -> int {
            const int c = atomicAdd(p.claims, 1);
            return c < total ? c : -1;
          };
          auto info_of = [&](int t) -> int4 { return t >= 0 ? __ldg(info + t / per_e) : make_int4(0, 0, 0, 0); };
          int next = claim();
          int next2 = claim();
          int4 next_info = info_of(next);
          int acc = 1;
          for (;;) {
            const int t = next;
            Tile tl{};
            if (t >= 0) {
              tl = rows_k_tile_info(next_info, t - (t / per_e) * per_e, p);
              next = next2;
              next2 = claim();
              next_info = info_of(next);
              if (tl.kb_count > 0) acc ^= 1;
            }
            if (!publish(t, tl, acc) || (t >= 0 && !load_tile(tl))) {
              failed = true;
              break;
            }
            if (t < 0) break;
          }
        }
        if (failed) raise_abort(p.err, abort_flag);
        if constexpr (kPair) {
          // the even CTA has released the last fill of each stage: no release from the peer is
          // still on its way to this CTA's barriers when it exits
          for (int i = 0; i < STAGES && !failed; ++i) {
            if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag)) {
              raise_abort(p.err, abort_flag);
              failed = true;
            }
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (failed) {
          // let loads already in flight land before the CTA's shared memory goes away
          for (int i = 0; i < 200; ++i) __nanosleep(1000);
        }
      }
    } else {
      // The whole warp: lane 0 arms the stage's barrier and loads the tiled operand, then every
      // lane gathers four rows per 64-column box.  The tokens of the next (tile, K block) are read
      // before the stage wait, so their latency overlaps it.
      constexpr bool kGA = (G == Gather::A);
      const CUtensorMap* tmG = kGA ? &tmA : &tmB;
      int stage = 0;
      uint32_t phase = 0;
      bool failed = false;
      int t = blockIdx.x, kb = 0;
      Tile tl{};
      auto seek = [&](int from) {  // first tile at or after `from` (stride gridDim.x) with K blocks
        for (t = from; t < total; t += gridDim.x) {
          tl = decode_tile<S>(t, p);
          if (tl.kb_count > 0) return;
        }
      };
      seek(blockIdx.x);
      int tok[4] = {0, 0, 0, 0};
      if (t < total) gather_tokens<S>(tl, kb, lane, p, tok);
      while (t < total) {
        const Tile ct = tl;
        const int ckb = kb;
        const int c0 = tok[0], c1 = tok[1], c2 = tok[2], c3 = tok[3];
        if (++kb == tl.kb_count) {
          kb = 0;
          seek(t + gridDim.x);
        }
        if (t < total && (S == Sched::RowsK || kb == 0)) gather_tokens<S>(tl, kb, lane, p, tok);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag))) {
          if (lane == 0) raise_abort(p.err, abort_flag);
          failed = true;
          break;
        }
        const uint32_t sa = sbase + stage * STAGE_BYTES;
        const uint32_t sb = sa + L::kABytes;
        const uint32_t fb = full0 + 8 * stage;
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          load_stage_tiled<S, EP, A_MN, B_MN, SPLIT, !kGA, kGA>(&tmA, &tmB, &tmF, p, ct, ckb, sa, sb, fb);
        }
        __syncwarp();
        if constexpr (S == Sched::RowsM) {
          // K-major A: four consecutive tile rows, one K block wide (4 x 128 bytes)
          tma_gather4(sa + lane * 512, tmG, fb, ckb * BK, c0, c1, c2, c3);
        } else {
          // MN-major: four K rows of each 64-column box; half of the boxes per half-warp
          constexpr int kBoxes = (kGA ? BM : BN) / 64;
          const uint32_t dst = (kGA ? sa : sb) + (lane & 15) * 512;
          const int col0 = kGA ? ct.m0 : ct.nt * BN;
#pragma unroll
          for (int i = 0; i < kBoxes / 2; ++i) {
            const int box = (lane >> 4) * (kBoxes / 2) + i;
            tma_gather4(dst + box * MN_BOX_BYTES, tmG, fb, col0 + 64 * box, c0, c1, c2, c3);
          }
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (failed && lane == 0) {
        for (int i = 0; i < 200; ++i) __nanosleep(1000);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // pair: M = 256 across the two CTAs (the odd CTA's MMA warp issues nothing)
    constexpr uint32_t idesc = idesc_bf16_f32(kPair ? 2 * BM : BM, BN, A_MN, B_MN);
    constexpr uint32_t idesc16 = idesc_f16_f32(kPair ? 2 * BM : BM, BN, A_MN, B_MN);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t acc_phase = 0;  // bit a: the phase of accumulator a
    bool failed = false;
    int t = 0, acc = 0;
    Tile tl{};
    for (bool first = true; leader && !failed; first = false) {
      if (!next_tile(t, tl, acc, first)) {
        raise_abort(p.err, abort_flag);
        break;
      }
      if (t < 0 || t >= total) break;
      if (tl.kb_count == 0) continue;
      // every lane waits (so every lane acquires the phase); the outcome is made warp-uniform.
      // Pair: the accumulator is free once both CTAs' epilogues have read it (cluster scope).
      const uint32_t par = ((acc_phase >> acc) & 1u) ^ 1u;
      const bool freed = kPair ? mbar_wait_cluster(tempty0 + 8 * acc, par, abort_flag)
                               : mbar_wait(tempty0 + 8 * acc, par, abort_flag);
      if (!__all_sync(0xFFFFFFFFu, freed)) {
        raise_abort(p.err, abort_flag);
        break;
      }
      tc_fence_after_sync();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
      // fp16 operands: a weight-gradient tile of the fp16 experts' launch (in the dH GEMM the flag
      // marks the tiles that write fp16 parts; its operands are bf16)
      const uint32_t id = (S == Sched::RowsK && tl.f16) ? idesc16 : idesc;
      for (int kb = 0; kb < tl.kb_count; ++kb) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8 * stage, phase, abort_flag))) {
          raise_abort(p.err, abort_flag);
          failed = true;
          break;
        }
        tc_fence_after_sync();
        const uint32_t sa = sbase + stage * STAGE_BYTES;
        const uint32_t sb = sa + L::kABytes;
        // K steps of 16 rows to issue: all of them, except in a weight-gradient tile's last
        // block, which ends at the 16-row step holding the expert's last row.  That step's rows
        // past the expert are zero in the padded operand (dgu for dW_gate_up, w h for dW_down),
        // so the other operand's rows there (the next expert's) add nothing.
        int ksteps = BK / 16;
        if constexpr (S == Sched::RowsK) {
          const int valid = tl.rows - kb_source(tl, kb, p).kbe * BK;
          if (valid < BK) ksteps = (valid + 15) / 16;
        }
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (kk >= ksteps) break;
            const uint64_t ad = A_MN ? smem_desc_sw128(sa + kk * 2048, MN_BOX_BYTES, 1024)
                                     : smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(sb + kk * 2048, MN_BOX_BYTES, 1024)
                                     : smem_desc_sw128(sb + kk * 32, 16, 1024);
            if constexpr (kPair)
              umma_bf16_f32_pair(d_tmem, ad, bd, id, (kb | kk) != 0 ? 1u : 0u);
            else
              umma_bf16_f32(d_tmem, ad, bd, id, (kb | kk) != 0 ? 1u : 0u);
            if constexpr (SPLIT == 1) {  // lo part of A against the same B
              const uint64_t lo = smem_desc_sw128(sa + A_BYTES + kk * 2048, MN_BOX_BYTES, 1024);
              if constexpr (kPair)
                umma_bf16_f32_pair(d_tmem, lo, bd, idesc, 1u);
              else
                umma_bf16_f32(d_tmem, lo, bd, idesc, 1u);
            }
            if constexpr (SPLIT == 2) {  // the same A against the lo part of B (half of it per CTA in a pair)
              const uint64_t lo = smem_desc_sw128(sb + L::kBBytes / 2 + kk * 2048, MN_BOX_BYTES, 1024);
              if constexpr (kPair)
                umma_bf16_f32_pair(d_tmem, ad, lo, idesc, 1u);
              else
                umma_bf16_f32(d_tmem, ad, lo, idesc, 1u);
            }
          }
          if constexpr (kPair)
            umma_commit_pair_mc(empty0 + 8 * stage, kClusterMask);  // both CTAs' stage is free
          else
            umma_commit(empty0 + 8 * stage);
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (failed) break;
      if (lane == 0) {
        if constexpr (kPair)
          umma_commit_pair_mc(tfull0 + 8 * acc, kClusterMask);  // both CTAs' accumulators are ready
        else
          umma_commit(tfull0 + 8 * acc);
      }
      __syncwarp();
      acc_phase ^= 1u << acc;
    }
    // every MMA issued by this CTA has completed before TMEM is released
    if (lane == 0 && leader) {
      if constexpr (kPair)
        umma_commit_pair(drain);
      else
        umma_commit(drain);
      const int never = 0;
      mbar_wait(drain, 0, &never);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int sub = warp & 3;      // TMEM lane quadrant this warp may access
    const int colhalf = ew >> 2;   // which half of the tile's columns
    const int row_local = sub * 32 + lane;
    Stager st{sbase + L::kStgOffset + static_cast<uint32_t>(ew * L::kStgWarpBytes), 0};
    uint32_t acc_phase = 0;
    int t = 0, acc = 0;
    Tile tl{};
    for (bool first = true;; first = false) {
      if (!next_tile(t, tl, acc, first)) {
        raise_abort(p.err, abort_flag);
        break;
      }
      if (t < 0 || t >= total) break;
      if (tl.kb_count == 0) {
        if constexpr (S == Sched::RowsK) store_zero_tile(tl, sub, colhalf, lane, p, zero_row);
        continue;
      }
      // the tile's epilogue operands (DH) start moving into L2 now, a tile's MMA time ahead of use
      // when the MMAs lead, and at least ahead of the later column chunks when the epilogue does
      prefetch_epilogue_operands<S, EP>(tl, row_local, colhalf, p);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(tfull0 + 8 * acc, (acc_phase >> acc) & 1u, abort_flag))) {
        raise_abort(p.err, abort_flag);
        break;
      }
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + static_cast<uint32_t>(acc * BN);
      epilogue_tile<S, EP>(t_row, tl, sub, colhalf, lane, p, &tmC0, &tmC1, st);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kPair)
          mbar_arrive_cluster(mapa_shared(tempty0 + 8 * acc, 0));  // the even CTA issues the next MMAs
        else
          mbar_arrive(tempty0 + 8 * acc);
      }
      acc_phase ^= 1u << acc;
    }
    // outputs are in global memory (and the staging buffers free) before the CTA exits; every lane
    // waits for its own bulk copies (zero tiles)
    bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if constexpr (kPair) {
    // neither CTA of the pair leaves while the other may still arrive on its barriers, and the
    // odd CTA's TMEM (written by the even CTA's MMAs) is released by both together
    cluster_sync();
  }
  tc_fence_after_sync();
  if (warp == 1) {
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ============================================================================
// Tile schedule: tile_prefix[e] = sum_{e' < e} ceil(rows_e' / BM), tile_prefix[E]
// = total; and, when pad_indptr != NULL, pad_indptr[e] = sum_{e' < e} of rows_e' rounded up
// to 16 (the padded row space of the weight-gradient operands).  m_indptr is validated
// (0 = m[0] <= ... <= m[E] = R); if it is not, the schedule is empty and the device error
// flag is set.
// ============================================================================
__device__ __forceinline__ int block_exclusive_scan_1024(int v, int* s_warp, int lane, int warp, int* total) {
  int incl = v;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, m);
    if (lane >= m) incl += o;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int x = s_warp[lane];
    int xi = x;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, xi, m);
      if (lane >= m) xi += o;
    }
    s_warp[lane] = xi - x;
    if (lane == 31) *total = xi;
  }
  __syncthreads();
  const int excl = s_warp[warp] + incl - v;
  __syncthreads();  // s_warp is reused by the next scan
  return excl;
}

__global__ void __launch_bounds__(1024) tile_schedule_kernel(const int32_t* __restrict__ m_indptr, int E,
                                                             long long R, ScheduleBufs sb, int* err) {
  __shared__ int s_warp[32];
  __shared__ int s_bad;
  __shared__ int s_max;
  __shared__ int s_heavy;
  __shared__ int s_f16;
  __shared__ int s_total[5];
  __shared__ int s_rows[1024];
  griddep_wait();
  griddep_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_bad = (m_indptr[0] != 0 || static_cast<long long>(m_indptr[E]) != R) ? 1 : 0;
    s_max = 0;
    s_heavy = 0;
    s_f16 = 0;
  }
  if (sb.claims != nullptr && tid < kClaimSlots) sb.claims[tid] = 0;
  __syncthreads();
  int rows = 0;
  if (tid < E) {
    const int a = m_indptr[tid], b = m_indptr[tid + 1];
    if (b < a) atomicOr(&s_bad, 1);
    rows = max(b - a, 0);
    atomicMax(&s_max, rows);
    if (rows >= kPairRowsDwD) atomicAdd(&s_heavy, 1);
    if (rows >= kF16Rows) atomicAdd(&s_f16, 1);
  }
  s_rows[tid] = rows;
  const bool heavy_m = rows >= kPairRowsM;
  const int tiles = (rows + BM - 1) / BM;
  const int padded = (rows + 15) & ~15;
  const int pairs = (rows + 2 * BM - 1) / (2 * BM);
  const int t_excl = block_exclusive_scan_1024(tiles, s_warp, lane, warp, &s_total[0]);  // (syncs s_rows too)
  const int p_excl = sb.pad_indptr != nullptr ? block_exclusive_scan_1024(padded, s_warp, lane, warp, &s_total[1]) : 0;
  const int q_excl = sb.pair_prefix != nullptr ? block_exclusive_scan_1024(pairs, s_warp, lane, warp, &s_total[2]) : 0;
  int l_excl = 0, h_excl = 0;
  if (sb.light_prefix != nullptr) {
    l_excl = block_exclusive_scan_1024(heavy_m ? 0 : tiles, s_warp, lane, warp, &s_total[3]);
    h_excl = block_exclusive_scan_1024(heavy_m ? pairs : 0, s_warp, lane, warp, &s_total[4]);
  }
  const bool bad = s_bad != 0;
  if (sb.f16_words != nullptr) {  // s_max is final here (the scans synchronise)
    for (int i = tid; i < kF16Range + 2 * E; i += blockDim.x)
      sb.f16_words[i] = (i == kF16Any && !bad && s_max >= kF16Rows) ? 1u : 0u;
  }
  if (tid < E) {
    sb.tile_prefix[tid] = bad ? 0 : t_excl;
    if (sb.pad_indptr != nullptr) sb.pad_indptr[tid] = bad ? 0 : p_excl;
    if (sb.pair_prefix != nullptr) sb.pair_prefix[tid] = bad ? 0 : q_excl;
    if (sb.light_prefix != nullptr) {
      sb.light_prefix[tid] = bad ? 0 : l_excl;
      sb.heavy_pair_prefix[tid] = bad ? 0 : h_excl;
    }
  }
  if (tid == 0) {
    sb.tile_prefix[E] = bad ? 0 : s_total[0];
    if (sb.pad_indptr != nullptr) sb.pad_indptr[E] = bad ? 0 : s_total[1];
    if (sb.pair_prefix != nullptr) sb.pair_prefix[E] = bad ? 0 : s_total[2];
    if (sb.light_prefix != nullptr) {
      sb.light_prefix[E] = bad ? 0 : s_total[3];
      sb.heavy_pair_prefix[E] = bad ? 0 : s_total[4];
    }
  }
  if (sb.order != nullptr) {
    // experts by rows, most first; equal rows in id order (the rank of expert tid)
    if (tid < E) {
      int rank = 0;
      for (int e = 0; e < E; ++e) {
        const int r = s_rows[e];
        rank += (r > rows || (r == rows && e < tid)) ? 1 : 0;
      }
      sb.order[rank] = tid;
      if (sb.order_info != nullptr) {
        const int a0 = bad ? 0 : m_indptr[tid];
        int4 q;
        q.x = tid;
        q.y = a0;
        q.z = bad ? 0 : rows;
        q.w = sb.pad_indptr != nullptr ? (bad ? 0 : p_excl) : a0;
        reinterpret_cast<int4*>(sb.order_info)[rank] = q;
      }
    }
    if (tid == 0 && sb.claims != nullptr) {
      // skewed load: the largest expert holds at least 512 rows and 4x the mean (the one-CTA
      // weight-gradient tiles are then claimed heaviest first)
      const long long mean = (R + E - 1) / E;
      sb.claims[kClaimSlots] = (!bad && s_max >= 512 && s_max >= 4 * mean) ? 1 : 0;
      // the experts at the head of that order with enough rows for the 2-SM pair dW_down
      sb.claims[kClaimSlots + 1] = bad ? 0 : s_heavy;
      // and those with enough rows for the fp16 weight-gradient pass (kF16Rows >= kPairRowsDwD)
      sb.claims[kClaimSlots + 2] = bad ? 0 : s_f16;
    }
  }
  if (bad && tid == 0) atomicOr(err, LIGER_MOE_DEVERR_BAD_INDPTR);
}

// ============================================================================
// Host side
// ============================================================================
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Row-major tensor (dims[0] innermost) -> tensor map with the given box, 128-byte swizzle,
// zero fill outside the tensor on loads, clipping outside it on stores.
int make_tmap_nd(CUtensorMap* m, const void* ptr, CUtensorMapDataType dtype, int elem_bytes, int rank,
                 const uint64_t* dims, const uint32_t* box,
                 CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return LIGER_MOE_ERR_LAUNCH;
  cuuint64_t d[3], strides[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  uint64_t stride = static_cast<uint64_t>(elem_bytes);
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    if (i > 0) strides[i - 1] = stride;
    stride *= dims[i];
  }
  const CUresult r = enc(m, dtype, rank, const_cast<void*>(ptr), d, strides, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LIGER_MOE_OK : LIGER_MOE_ERR_LAUNCH;
}

// bf16 matrix [outer, inner] with a {box_inner, box_outer} box.
int make_tmap(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer) {
  const uint64_t dims[2] = {inner, outer};
  const uint32_t box[2] = {box_inner, box_outer};
  return make_tmap_nd(m, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 2, dims, box);
}

// Output maps: one epilogue box is 32 rows x 128 bytes.
int make_out_bf16(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows) {
  return make_tmap(m, ptr, cols, rows, 64, 32);
}
int make_out_f32(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint32_t box[2] = {32, 32};
  return make_tmap_nd(m, ptr, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 2, dims, box);
}
// 32-row x 16-column bf16 boxes with a 32-byte swizzle (the dH epilogue's outputs).
int make_out_bf16_narrow(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint32_t box[2] = {16, 32};
  return make_tmap_nd(m, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 2, dims, box, CU_TENSOR_MAP_SWIZZLE_32B);
}
// [E, rows, cols] bf16 weight gradient: the 3D map clips each expert's block at its own row count.
int make_out_bf16_3d(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint64_t experts) {
  const uint64_t dims[3] = {cols, rows, experts};
  const uint32_t box[3] = {64, 32, 1};
  return make_tmap_nd(m, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 3, dims, box);
}

// Launches one grouped GEMM.  `tiles` is the number of tiles the persistent grid walks (for
// RowsM an upper bound: the device schedule decides); the grid is at most one CTA per SM.
// PAIR (CL = 2): the grid is made of CTA pairs, as many as can be resident at once, and `tiles`
// counts 256-row (RowsM) or 256-column (RowsK) pair tiles, one per pair.
template <Sched S, Epi EP, bool A_MN, bool B_MN, int SPLIT = 0, Gather G = Gather::None, int CL = 1,
          int PAIR = 0>
int launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc0, const CUtensorMap& tc1,
                const Params& p, long long tiles, const DeviceInfo& dev, cudaStream_t s, const char* name,
                bool traced = true, const CUtensorMap* tf = nullptr) {
  auto kern = grouped_gemm_kernel<S, EP, A_MN, B_MN, SPLIT, G, CL, PAIR>;
  constexpr int kSmem = LayoutOf<EP, SPLIT, PAIR>::kSmemBytes;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_clusters = 0;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (attr_err == cudaSuccess && CL > 1) {
      cudaLaunchConfig_t cfg{};
      cudaLaunchAttribute attr{};
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = CL;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.gridDim = dim3(static_cast<unsigned>(dev.sm_count / CL * CL));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = kSmem;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      attr_err = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
      if (attr_err == cudaSuccess && max_clusters < 1) attr_err = cudaErrorInvalidConfiguration;
    }
  });
  if (attr_err != cudaSuccess) {
    set_cuda_error(attr_err, name);
    return LIGER_MOE_ERR_LAUNCH;
  }
  if (tiles < 1) return LIGER_MOE_OK;
  int grid;
  if constexpr (CL == 1) {
    grid = static_cast<int>(tiles < dev.sm_count ? tiles : dev.sm_count);
  } else {
    const long long groups = PAIR ? tiles : tiles / CL;  // pair: one tile per cluster
    grid = static_cast<int>(groups < max_clusters ? groups : max_clusters) * CL;
  }
  KernelScope trace(traced ? name : nullptr, s);  // untraced: one scope of the caller spans both parts of a split
  if (launch_kernel(kern, dim3(grid), dim3(kThreads), kSmem, s, name, CL, ta, tb, tc0, tc1, tf != nullptr ? *tf : ta,
                    p) != cudaSuccess)
    return LIGER_MOE_ERR_LAUNCH;
  return check_launch(name);
}

Params base_params(const int32_t* m_indptr, const int32_t* tile_prefix, int E, int* err) {
  Params p{};
  p.m_indptr = m_indptr;
  p.tile_prefix = tile_prefix;
  p.E = E;
  p.err = err;
  return p;
}

// Weight gradients in the dynamic order when the schedule finds the load skewed (claim counter
// `slot` of the schedule's counters; the skew flag follows the counters).
void set_dynamic(Params& p, const int32_t* order, const int32_t* info, int* claims, int slot) {
  if (order == nullptr || info == nullptr || claims == nullptr) return;
  p.sched_order = order;
  p.sched_info = info;
  p.claims = claims + slot;
  p.sched_skewed = claims + kClaimSlots;
}

// Token-major bf16 matrix [rows, cols] as a gather source: box 64 columns x 1 row.
int make_gather_map(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows) {
  return make_tmap(m, ptr, cols, rows, 64, 1);
}

// Gathered operand: row r of the GEMM is row row_to_slot[r] / k of the source matrix.
void set_gather(Params& p, const int32_t* row_to_slot, long long R, int k) {
  p.row_slot = row_to_slot;
  p.R = R;
  p.topk = k;
}

// Upper bound on the RowsM tile count: sum over experts of ceil(rows_e / BM) N tiles.
long long rows_m_tiles(long long R, int E, int n_tiles) { return ((R + BM - 1) / BM + E) * n_tiles; }
// the same bound for 256-row pair tiles
long long pair_m_tiles(long long R, int E, int n_tiles) { return ((R + 2 * BM - 1) / (2 * BM) + E) * n_tiles; }

// The forward GEMMs run as 2-SM pairs when experts hold at least 512 rows on average.  A pair
// tile spans 256 rows of one expert, so below that the rows wasted in each expert's last tile
// (up to 255 instead of 127) cost more than the pairs gain (measured on GB300: about even at
// 512 rows per expert, slower at 256).
bool use_pairs(const FwdGemmArgs& a) { return a.pair_prefix != nullptr && a.R >= 512LL * a.E; }
// The same rule for the backward's dX GEMM (gated experts, expert-major dY rows).
bool use_pairs(const BwdGemmArgs& a) {
  return a.pair_prefix != nullptr && a.R >= 512LL * a.E && a.dy_perm != nullptr && a.nin == 2 * a.I;
}

// Heavy / light split: the experts with at least the pair threshold's rows run as 2-SM pairs and the
// others one CTA per tile, in two launches over the schedule's filtered prefixes (forward and dX
// GEMMs) or the two parts of the sorted expert order (dW_down).  Pairs halve the operand tiles each
// SM streams through L2 for a heavy expert's rows; a light expert's rows would leave most of a
// 256-row pair tile empty.  Taken for skewed batches: experts average fewer than kSplitMeanRows rows
// (with more, every expert runs as pairs or a uniform load gains nothing from a second launch),
// and the batch is large enough for one expert to reach the threshold (R rows in all, T per expert
// at most).  Measured on GB300 (Zipf 4096/1024 workload, 160 rows per expert on average):
// dW_down 1587-1608 -> 1397-1418 us, down 840-846 -> 809-816, dX 1545-1559 -> 1529-1545; on
// uniform loads an empty second launch cost 3-10 us per GEMM.
constexpr long long kSplitMeanRows = 192;
constexpr long long kSplitMinRows = 8 * kPairRowsM;  // forward: R rows in the batch (T is not known)
}  // namespace

bool split_schedule(long long R, int E) { return R >= kSplitMinRows && R < kSplitMeanRows * E; }

namespace {

bool use_split(const FwdGemmArgs& a) {
  return a.light_prefix != nullptr && !use_pairs(a) && a.x == nullptr && a.R >= kSplitMinRows &&
         a.R < kSplitMeanRows * a.E;
}
bool use_split(const BwdGemmArgs& a) {
  return a.light_prefix != nullptr && !use_pairs(a) && a.T >= kPairRowsM && a.dy_perm != nullptr &&
         a.nin == 2 * a.I && a.R < kSplitMeanRows * a.E;
}

int cdiv(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

}  // namespace

size_t schedule_bytes(int E) { return align_up(sizeof(int32_t) * (E + 1), 256); }

int launch_tile_schedule(const int32_t* m_indptr, int E, long long R, const ScheduleBufs& b, const DeviceInfo& dev,
                         cudaStream_t s) {
  {
    KernelScope trace("tile_schedule", s);
    if (launch_kernel(tile_schedule_kernel, dim3(1), dim3(1024), 0, s, "tile_schedule", 1, m_indptr, E, R, b,
                      dev.err_flag) != cudaSuccess)
      return LIGER_MOE_ERR_LAUNCH;
  }
  return check_launch("tile_schedule");
}

int gdot_tiles(int I) { return 2 * cdiv(I, BN); }

// Up GEMM of a two-weight expert (ReLU²): a = x W_up[e]^T over N = I columns in full BN tiles,
// h = max(a, 0)^2 and the factor dh/da (fp32 [R, I]).
int launch_up_relu2(const FwdGemmArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  if (a.x != nullptr) return LIGER_MOE_ERR_INVALID_ARG;  // reads x_perm
  CUtensorMap ta, tb;
  if (make_tmap(&ta, a.x_perm, a.H, a.R, BK, BM) || make_tmap(&tb, a.w_gate_up, a.H, 1ULL * a.I * a.E, BK, BN))
    return LIGER_MOE_ERR_LAUNCH;
  Params p = base_params(a.m_indptr, a.tile_prefix, a.E, dev.err_flag);
  p.n_tiles = cdiv(a.I, BN);
  p.num_kb = a.H / BK;
  p.b_rows_per_expert = a.I;
  p.N_out = a.I;
  p.I = a.I;
  p.out = a.h_perm;
  p.ld_out = a.I;
  p.gu_out = a.gu_perm;
  CUtensorMap tc0, tc1;  // h (bf16) and dh/da (fp32); an absent output reuses the other's map
  if (a.h_perm != nullptr && make_out_bf16(&tc0, a.h_perm, a.I, a.R)) return LIGER_MOE_ERR_LAUNCH;
  if (a.gu_perm != nullptr && make_out_f32(&tc1, a.gu_perm, a.I, a.R)) return LIGER_MOE_ERR_LAUNCH;
  if (a.h_perm == nullptr) tc0 = tc1;
  if (a.gu_perm == nullptr) tc1 = tc0;
  if (a.h_perm == nullptr && a.gu_perm == nullptr) return LIGER_MOE_OK;
  return launch_gemm<Sched::RowsM, Epi::ReLU2, false, false>(ta, tb, tc0, tc1, p, rows_m_tiles(a.R, a.E, p.n_tiles),
                                                              dev, s, "gemm_up_relu2");
}

int launch_gate_up(const FwdGemmArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  if (a.R == 0) return LIGER_MOE_OK;
  if (a.act == LIGER_MOE_ACT_RELU2) return launch_up_relu2(a, dev, s);
  const bool gather = a.x != nullptr;  // A rows gathered from x [T, H]; else read from x_perm [R, H]
  CUtensorMap ta, tb;
  if ((gather ? make_gather_map(&ta, a.x, a.H, a.T) : make_tmap(&ta, a.x_perm, a.H, a.R, BK, BM)) ||
      make_tmap(&tb, a.w_gate_up, a.H, 2ULL * a.I * a.E, BK, BN / 2))
    return LIGER_MOE_ERR_LAUNCH;
  Params p = base_params(a.m_indptr, a.tile_prefix, a.E, dev.err_flag);
  if (gather) set_gather(p, a.row_to_slot, a.R, a.k);
  p.n_tiles = cdiv(a.I, BN / 2);
  p.num_kb = a.H / BK;
  p.b_rows_per_expert = 2 * a.I;
  p.b_split = a.I;
  p.N_out = a.I;
  p.I = a.I;
  p.out = a.h_perm;
  p.ld_out = a.I;
  p.gu_out = a.gu_perm;
  p.act = a.act;
  p.act_clamp = a.act_clamp;
  CUtensorMap tc0, tc1;  // h (bf16) and [g|u] (fp32); an absent output reuses the other's map
  if (a.h_perm != nullptr && make_out_bf16(&tc0, a.h_perm, a.I, a.R)) return LIGER_MOE_ERR_LAUNCH;
  if (a.gu_perm != nullptr && make_out_f32(&tc1, a.gu_perm, 2ULL * a.I, a.R)) return LIGER_MOE_ERR_LAUNCH;
  if (a.h_perm == nullptr) tc0 = tc1;
  if (a.gu_perm == nullptr) tc1 = tc0;
  if (a.h_perm == nullptr && a.gu_perm == nullptr) return LIGER_MOE_OK;
  const long long tiles = rows_m_tiles(a.R, a.E, p.n_tiles);
  if (use_pairs(a) && !gather && a.act == LIGER_MOE_ACT_SWIGLU) {
    // 2-SM pairs over 256-row blocks: the even CTA loads the gate rows of B, the odd one the up rows
    p.tile_prefix = a.pair_prefix;
    return launch_gemm<Sched::RowsM, Epi::SwiGLU, false, false, 0, Gather::None, 2, 1>(
        ta, tb, tc0, tc1, p, pair_m_tiles(a.R, a.E, p.n_tiles), dev, s, "gemm_gate_up_swiglu");
  }
  if (use_split(a) && a.act == LIGER_MOE_ACT_SWIGLU) {  // heavy experts as pairs, then the light ones
    KernelScope trace("gemm_gate_up_swiglu", s);
    Params ph = p;
    ph.tile_prefix = a.heavy_pair_prefix;
    if (int rc = launch_gemm<Sched::RowsM, Epi::SwiGLU, false, false, 0, Gather::None, 2, 1>(
            ta, tb, tc0, tc1, ph, pair_m_tiles(a.R, a.E, p.n_tiles), dev, s, "gemm_gate_up_swiglu", false))
      return rc;
    p.tile_prefix = a.light_prefix;
    return launch_gemm<Sched::RowsM, Epi::SwiGLU, false, false>(ta, tb, tc0, tc1, p, tiles, dev, s,
                                                                 "gemm_gate_up_swiglu", false);
  }
  if (a.act != LIGER_MOE_ACT_SWIGLU) {  // the other gated activations read x_perm
    if (gather) return LIGER_MOE_ERR_INVALID_ARG;
    return launch_gemm<Sched::RowsM, Epi::GLU, false, false>(ta, tb, tc0, tc1, p, tiles, dev, s, "gemm_gate_up_glu");
  }
  if (gather)
    return launch_gemm<Sched::RowsM, Epi::SwiGLU, false, false, 0, Gather::A>(ta, tb, tc0, tc1, p, tiles, dev, s,
                                                                              "gemm_gate_up_swiglu");
  return launch_gemm<Sched::RowsM, Epi::SwiGLU, false, false>(ta, tb, tc0, tc1, p, tiles, dev, s,
                                                               "gemm_gate_up_swiglu");
}

// Router projection logits[T, E] = x[T, H] Wr[E, H]^T (+ bias[E]), fp32: one dense GEMM over T
// rows, N = E in 256-column tiles (Wr rows past E read as zeros), K = H.
int launch_router_logits(const uint16_t* x, const uint16_t* w_router, const float* bias, int T, int H, int E,
                         float* logits, const DeviceInfo& dev, cudaStream_t s) {
  if (T == 0) return LIGER_MOE_OK;
  CUtensorMap ta, tb, tc;
  if (make_tmap(&ta, x, H, T, BK, BM) || make_tmap(&tb, w_router, H, E, BK, BN)) return LIGER_MOE_ERR_LAUNCH;
  Params p = base_params(nullptr, nullptr, 1, dev.err_flag);
  p.R = T;
  p.n_tiles = cdiv(E, BN);
  p.num_kb = H / BK;
  p.b_rows_per_expert = 0;
  p.N_out = E;
  p.ld_out = E;
  p.out_f32 = logits;
  p.col_bias = bias;
  p.out_tma = (E % 32 == 0) ? 1 : 0;  // the fp32 output map needs rows of whole 128-byte boxes
  if (p.out_tma) {
    if (make_out_f32(&tc, logits, E, T)) return LIGER_MOE_ERR_LAUNCH;
  } else {
    tc = ta;  // never used for stores
  }
  const long long tiles = static_cast<long long>(cdiv(T, BM)) * p.n_tiles;
  return launch_gemm<Sched::Dense, Epi::Logits, false, false>(ta, tb, tc, tc, p, tiles, dev, s, "gemm_router_logits");
}

int launch_down(const FwdGemmArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  if (a.R == 0) return LIGER_MOE_OK;
  CUtensorMap ta, tb, tb_half;
  const bool pair = use_pairs(a);  // 2-SM pairs: each CTA loads 128 of a tile's 256 B rows
  const bool split = use_split(a);  // pairs for the heavy experts only
  if (make_tmap(&ta, a.h_perm, a.I, a.R, BK, BM) ||
      make_tmap(&tb, a.w_down, a.I, 1ULL * a.H * a.E, BK, pair ? BN / 2 : BN) ||
      (split && make_tmap(&tb_half, a.w_down, a.I, 1ULL * a.H * a.E, BK, BN / 2)))
    return LIGER_MOE_ERR_LAUNCH;
  Params p = base_params(a.m_indptr, a.tile_prefix, a.E, dev.err_flag);
  p.n_tiles = cdiv(a.H, BN);
  p.num_kb = a.I / BK;
  p.b_rows_per_expert = a.H;
  p.N_out = a.H;
  p.I = a.I;
  p.out = a.y_perm;
  p.ld_out = a.H;
  p.row_scale = a.w_perm;
  CUtensorMap tc0;
  if (make_out_bf16(&tc0, a.y_perm, a.H, a.R)) return LIGER_MOE_ERR_LAUNCH;
  if (pair) {
    p.tile_prefix = a.pair_prefix;
    return launch_gemm<Sched::RowsM, Epi::ScaleRows, false, false, 0, Gather::None, 2, 1>(
        ta, tb, tc0, tc0, p, pair_m_tiles(a.R, a.E, p.n_tiles), dev, s, "gemm_down_scale");
  }
  if (split) {  // heavy experts as pairs, then the light ones
    KernelScope trace("gemm_down_scale", s);
    Params ph = p;
    ph.tile_prefix = a.heavy_pair_prefix;
    if (int rc = launch_gemm<Sched::RowsM, Epi::ScaleRows, false, false, 0, Gather::None, 2, 1>(
            ta, tb_half, tc0, tc0, ph, pair_m_tiles(a.R, a.E, p.n_tiles), dev, s, "gemm_down_scale", false))
      return rc;
    p.tile_prefix = a.light_prefix;
    return launch_gemm<Sched::RowsM, Epi::ScaleRows, false, false>(ta, tb, tc0, tc0, p,
                                                                    rows_m_tiles(a.R, a.E, p.n_tiles), dev, s,
                                                                    "gemm_down_scale", false);
  }
  return launch_gemm<Sched::RowsM, Epi::ScaleRows, false, false>(ta, tb, tc0, tc0, p,
                                                                  rows_m_tiles(a.R, a.E, p.n_tiles), dev, s,
                                                                  "gemm_down_scale");
}

int launch_bwd_dh(const BwdGemmArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  if (a.R == 0) return LIGER_MOE_OK;
  // A: dY rows of the routed rows, from dy_perm [R, H] as dense tiles, or gathered by token from
  // dY [T, H] when dy_perm is NULL
  const bool gather = a.dy_perm == nullptr;
  CUtensorMap ta, tb;
  if ((gather ? make_gather_map(&ta, a.dy, a.H, a.T) : make_tmap(&ta, a.dy_perm, a.H, a.R, BK, BM)) ||
      make_tmap(&tb, a.w_down, a.I, 1ULL * a.H * a.E, 64, BK))
    return LIGER_MOE_ERR_LAUNCH;
  Params p = base_params(a.m_indptr, a.tile_prefix, a.E, dev.err_flag);
  if (gather) set_gather(p, a.row_to_slot, a.R, a.k);
  p.R = a.R;
  p.pad_indptr = a.pad_indptr;  // dgu and hw rows go to the padded row space
  p.lo_rows = a.R_pad;          // row offset of their lo halves
  p.n_tiles = cdiv(a.I, BN);
  p.num_kb = a.H / BK;
  p.b_rows_per_expert = a.H;
  p.N_out = a.I;
  p.I = a.I;
  p.out2 = a.dgu;
  p.gu_in = a.gu;
  p.h_in = a.h_perm;
  p.hw_out = a.hw_perm;
  p.row_scale = a.w_perm;
  p.gdot = a.gdot;
  CUtensorMap tc0, tc1;  // dgu [2R, nin] and hw [2R, I]: hi rows then lo rows
  if (make_out_bf16_narrow(&tc0, a.dgu, static_cast<uint64_t>(a.nin), 2ULL * a.R_pad) ||
      make_out_bf16_narrow(&tc1, a.hw_perm, a.I, 2ULL * a.R_pad))
    return LIGER_MOE_ERR_LAUNCH;
  const long long tiles = rows_m_tiles(a.R, a.E, p.n_tiles);
  if (a.nin == a.I) {  // two-weight experts (ReLU²): one factor, one gradient
    if (gather) return LIGER_MOE_ERR_INVALID_ARG;
    return launch_gemm<Sched::RowsM, Epi::DH1, false, true>(ta, tb, tc0, tc1, p, tiles, dev, s, "gemm_bwd_dh");
  }
  if (gather)
    return launch_gemm<Sched::RowsM, Epi::DH, false, true, 0, Gather::A>(ta, tb, tc0, tc1, p, tiles, dev, s,
                                                                        "gemm_bwd_dh");
  // dH stays one CTA per tile at every load: its epilogue, not its operand pipeline, bounds it.
  // 2-SM pairs measured 5 % slower at 512 rows per expert (their 256-row tiles waste rows), and
  // pairs for the heavy experts of a skewed batch (the split of the forward and dX GEMMs) changed
  // nothing (1161-1165 against 1163-1172 us on the Zipf 4096/1024 workload)
  if (a.f16_words == nullptr)
    return launch_gemm<Sched::RowsM, Epi::DH, false, true>(ta, tb, tc0, tc1, p, tiles, dev, s, "gemm_bwd_dh");
  // fp16 weight-gradient operands: when some expert has f16_rows rows (a device flag), the fp16 pass
  // writes their fp16 parts and the hi / lo parts of the rest; the second launch then rewrites hi /
  // lo parts for those whose fp16 parts are unusable (usually none: it leaves at once).  When no
  // expert has them the first launch leaves at once and the second is the plain dH GEMM, whose
  // kernel carries none of the fp16 code (with it, dH measured 7-9 % slower).  One traced interval.
  KernelScope trace("gemm_bwd_dh", s);
  p.f16_rows = a.f16_rows;
  p.f16_words = a.f16_words;
  p.f16_role = 1;
  if (int rc = launch_gemm<Sched::RowsM, Epi::DH16, false, true>(ta, tb, tc0, tc1, p, tiles, dev, s, "gemm_bwd_dh",
                                                                 false))
    return rc;
  p.f16_role = 2;
  return launch_gemm<Sched::RowsM, Epi::DH, false, true>(ta, tb, tc0, tc1, p, tiles, dev, s, "gemm_bwd_dh", false);
}

int launch_bwd_dx(const BwdGemmArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  if (a.R == 0) return LIGER_MOE_OK;
  CUtensorMap ta, tb;
  if (make_tmap(&ta, a.dgu, static_cast<uint64_t>(a.nin), a.R_pad, BK, BM) ||  // hi rows of dgu, padded row space
      make_tmap(&tb, a.w_gate_up, a.H, 1ULL * a.nin * a.E, 64, BK))
    return LIGER_MOE_ERR_LAUNCH;
  Params p = base_params(a.m_indptr, a.tile_prefix, a.E, dev.err_flag);
  p.pad_indptr = a.pad_indptr;
  p.pad_a = 1;  // A = dgu hi rows in the padded row space
  p.n_tiles = cdiv(a.H, BN);
  p.num_kb = a.nin / BK;
  p.b_rows_per_expert = a.nin;
  p.N_out = a.H;
  p.I = a.I;
  p.out = a.dx_perm;
  p.ld_out = a.H;
  CUtensorMap tc0;
  if (make_out_bf16(&tc0, a.dx_perm, a.H, a.R)) return LIGER_MOE_ERR_LAUNCH;
  if (use_pairs(a)) {  // 2-SM pairs over 256-row blocks: each CTA loads half of the W_gu columns
    p.tile_prefix = a.pair_prefix;
    return launch_gemm<Sched::RowsM, Epi::Store, false, true, 0, Gather::None, 2, 1>(
        ta, tb, tc0, tc0, p, pair_m_tiles(a.R, a.E, p.n_tiles), dev, s, "gemm_bwd_dx");
  }
  if (use_split(a)) {  // heavy experts as pairs, then the light ones
    KernelScope trace("gemm_bwd_dx", s);
    Params ph = p;
    ph.tile_prefix = a.heavy_pair_prefix;
    if (int rc = launch_gemm<Sched::RowsM, Epi::Store, false, true, 0, Gather::None, 2, 1>(
            ta, tb, tc0, tc0, ph, pair_m_tiles(a.R, a.E, p.n_tiles), dev, s, "gemm_bwd_dx", false))
      return rc;
    p.tile_prefix = a.light_prefix;
    return launch_gemm<Sched::RowsM, Epi::Store, false, true>(ta, tb, tc0, tc0, p, rows_m_tiles(a.R, a.E, p.n_tiles),
                                                               dev, s, "gemm_bwd_dx", false);
  }
  return launch_gemm<Sched::RowsM, Epi::Store, false, true>(ta, tb, tc0, tc0, p, rows_m_tiles(a.R, a.E, p.n_tiles),
                                                             dev, s, "gemm_bwd_dx");
}

int launch_bwd_dw(const BwdGemmArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  // dW_gu[e] = dgu_e^T x_e  ([nin, H]),  dW_d[e] = dY_e^T (w h)_e  ([H, I]); K = rows of e.
  // The token-row operands x_e and dY_e are read as dense tiles of x_perm / dy_perm [R, H], or
  // gathered by token from x / dY [T, H] where those copies are absent.  With no rows at all
  // (R = 0) every expert's gradient is zero: the kernel still runs to write the zeros, over
  // 1-row dummy tensor maps that it never reads.
  CUtensorMap ta, tb, tc0;
  const bool empty = a.R == 0;
  const uint64_t rows = empty ? 1 : static_cast<uint64_t>(a.R);
  Params p = base_params(a.m_indptr, nullptr, a.E, dev.err_flag);
  const bool gather_x = a.x != nullptr || empty;
  // dW_gu[e] = dgu_hi_e^T x_e + dgu_lo_e^T x_e: each stage holds both parts of A (rows r and
  // R + r of dgu [2R, 2I]) and one B tile; two MMAs per K step.
  const uint64_t prows = empty ? 1 : static_cast<uint64_t>(a.R_pad);
  p.pad_indptr = a.pad_indptr;
  const uint64_t nin = static_cast<uint64_t>(a.nin);
  if (make_tmap(&ta, empty ? a.dw_gate_up : a.dgu, nin, 2 * prows, 64, BK)) return LIGER_MOE_ERR_LAUNCH;
  if (gather_x) {
    set_gather(p, a.row_to_slot, a.R, a.k);
    if (empty ? make_gather_map(&tb, a.dw_gate_up, a.H, 1) : make_gather_map(&tb, a.x, a.H, a.T))
      return LIGER_MOE_ERR_LAUNCH;
  } else if (make_tmap(&tb, a.x_perm, a.H, rows, 64, BK)) {
    return LIGER_MOE_ERR_LAUNCH;
  }
  p.m_tiles = cdiv(a.nin, BM);
  p.n_tiles = cdiv(a.H, BN);
  p.a_split_rows = static_cast<int>(a.R_pad);
  p.b_split_rows = 0;
  p.pad_a = 1;  // dgu rows: padded row space (zero rows past each expert)
  p.pad_b = 0;
  if (!empty) set_dynamic(p, a.sched_order, a.sched_info, a.claims, kClaimDwGateUp);  // R = 0: no schedule
  p.M_out = a.nin;
  p.N_out = a.H;
  p.out = a.dw_gate_up;
  p.ld_out = a.H;
  p.out_expert_stride = static_cast<long long>(a.nin) * a.H;
  if (make_out_bf16_3d(&tc0, a.dw_gate_up, a.H, nin, a.E)) return LIGER_MOE_ERR_LAUNCH;
  // The fp16 pass (f16): the experts with at least kF16Rows rows lead the sorted order; their
  // count is *f16_count.  They run in a launch of their own with one operand part per stage (more
  // stages in flight), taking one fp16 MMA per K step (lo rows of dgu: fp16(dgu 2^sg); x16: the x
  // rows), or their hi / lo parts as two passes where their fp16 parts are unusable.  The two
  // launches are one traced interval.  The fp16 launch goes first when the experts average
  // kF16Rows rows (then it holds most of the work); else after the two-part launch of the other
  // experts, so that an empty fp16 launch cannot hand the SMs to the side stream's kernels before
  // the GEMM takes them.  Measured, ms per step (fp16 first / last / no fp16 pass): training shape
  // 2.04-2.05 / 2.09-2.10 / 2.19-2.22; 2048/512 workload (no expert of kF16Rows) 1.909 / 1.900 /
  // 1.885-1.891; Zipf 4096/1024 the same either way.
  const bool f16 = a.f16_words != nullptr && !gather_x && !empty;
  const bool f16_first = a.R >= static_cast<long long>(kF16Rows) * a.E;
  const int* f16_count = a.claims + kClaimSlots + 2;
  const int* pair_count = a.claims + kClaimSlots + 1;
  static_assert(kF16Rows >= kPairRowsDwD, "the fp16 experts lead the pair experts of dW_down");
  CUtensorMap tf;
  auto f16_params = [&](Params& pf, int role, int slot) {
    pf.parted = 1;
    pf.part_begin = nullptr;
    pf.part_end = f16_count;
    pf.f16_role = role;
    pf.f16_part = 1;
    pf.f16_rows = a.f16_rows;
    pf.f16_words = a.f16_words;
    set_dynamic(pf, a.sched_order, a.sched_info, a.claims, slot);
  };
  // CTA pairs over neighbouring M blocks (2-SM MMAs, each CTA holding half of the x tile) when the M
  // blocks pair up and experts hold at least kPairRowsDwGu rows on average; below that every CTA
  // works alone on its tile (with few rows per expert the tiles are mostly gradient writes, and a
  // 2-SM pair ties the two CTAs' epilogues to each other).  A heavy / light split measured slower
  // here than one-CTA tiles in the heavy-first dynamic order (2687-2719 against 2647-2688 us on the
  // Zipf 4096/1024 workload).
  const long long tiles_gu = static_cast<long long>(a.E) * p.m_tiles * p.n_tiles;
  const bool pairs_gu = p.m_tiles % 2 == 0 && a.R >= kPairRowsDwGu * a.E;
  {
    KernelScope trace("gemm_bwd_dw_gate_up", s);
    if (gather_x) {
      if (int rc = launch_gemm<Sched::RowsK, Epi::Store, true, true, 1, Gather::B>(ta, tb, tc0, tc0, p, tiles_gu, dev,
                                                                                 s, "gemm_bwd_dw_gate_up", false))
        return rc;
    } else {
      Params pr = p;  // the experts of the two-part launch
      if (f16) {
        pr.parted = 1;
        pr.part_begin = f16_count;
      }
      auto two_part = [&]() {
        return pairs_gu ? launch_gemm<Sched::RowsK, Epi::Store, true, true, 1, Gather::None, 2, 1>(
                              ta, tb, tc0, tc0, pr, tiles_gu / 2, dev, s, "gemm_bwd_dw_gate_up", false)
                        : launch_gemm<Sched::RowsK, Epi::Store, true, true, 1>(ta, tb, tc0, tc0, pr, tiles_gu, dev, s,
                                                                               "gemm_bwd_dw_gate_up", false);
      };
      auto fp16_part = [&]() {
        if (make_tmap(&tf, a.x16, a.H, rows, 64, BK)) return static_cast<int>(LIGER_MOE_ERR_LAUNCH);
        Params pf = p;
        f16_params(pf, 3, kClaimDwGateUpF16);
        // 2-SM pairs whenever the M blocks pair up: every expert here has kF16Rows rows (Zipf
        // 4096/1024: dW_gate_up 2228-2249 -> 2167-2178 us against one CTA per tile)
        if (p.m_tiles % 2 == 0)
          return launch_gemm<Sched::RowsK, Epi::Store, true, true, 0, Gather::None, 2, 1>(
              ta, tb, tc0, tc0, pf, tiles_gu / 2, dev, s, "gemm_bwd_dw_gate_up", false, &tf);
        return launch_gemm<Sched::RowsK, Epi::Store, true, true, 0>(ta, tb, tc0, tc0, pf, tiles_gu, dev, s,
                                                                    "gemm_bwd_dw_gate_up", false, &tf);
      };
      int rc = (f16 && f16_first) ? fp16_part() : LIGER_MOE_OK;
      if (rc == LIGER_MOE_OK) rc = two_part();
      if (rc == LIGER_MOE_OK && f16 && !f16_first) rc = fp16_part();
      if (rc) return rc;
    }
  }
  // dW_d[e] = dY_e^T hw_hi_e + dY_e^T hw_lo_e: each stage holds one A tile (dY rows gathered by
  // token) and both parts of B (rows r and R + r of hw [2R, I]); two MMAs per K step.
  const bool gather_dy = a.dy_perm == nullptr || empty;
  if (make_tmap(&tb, empty ? a.dw_down : a.hw_perm, a.I, 2 * prows, 64, BK)) return LIGER_MOE_ERR_LAUNCH;
  if (gather_dy) {
    set_gather(p, a.row_to_slot, a.R, a.k);
    if (empty ? make_gather_map(&ta, a.dw_down, a.H, 1) : make_gather_map(&ta, a.dy, a.H, a.T))
      return LIGER_MOE_ERR_LAUNCH;
  } else if (make_tmap(&ta, a.dy_perm, a.H, rows, 64, BK)) {
    return LIGER_MOE_ERR_LAUNCH;
  }
  p.m_tiles = cdiv(a.H, BM);
  p.n_tiles = cdiv(a.I, BN);
  p.a_split_rows = 0;
  p.b_split_rows = static_cast<int>(a.R_pad);
  p.pad_a = 0;
  p.pad_b = 1;  // w h rows: padded row space
  if (!empty) set_dynamic(p, a.sched_order, a.sched_info, a.claims, kClaimDwDown);
  p.M_out = a.H;
  p.N_out = a.I;
  p.out = a.dw_down;
  p.ld_out = a.I;
  p.out_expert_stride = 1LL * a.H * a.I;
  if (make_out_bf16_3d(&tc0, a.dw_down, a.I, a.H, a.E)) return LIGER_MOE_ERR_LAUNCH;
  // CTA pairs over neighbouring M blocks (2-SM MMAs, each CTA holding half of the w h tile, 4 stages
  // instead of 2): for every expert when they hold at least kSplitMeanRows rows on average; for the
  // experts with at least kPairRowsDwD rows (the head of the sorted order) when fewer, the others one
  // CTA per tile (the heavy / light split); one CTA per tile for all when no expert can reach it.
  // With the fp16 pass its experts (fp16(w h 2^sh) in the lo rows of hw; dy16: the dY rows) run
  // last, as pairs where the pair experts do.
  const long long tiles_d = static_cast<long long>(a.E) * p.m_tiles * p.n_tiles;
  const bool pairs_all = p.m_tiles % 2 == 0 && a.R >= kSplitMeanRows * a.E;
  const bool split = !pairs_all && p.m_tiles % 2 == 0 && a.T >= kPairRowsDwD;
  KernelScope trace("gemm_bwd_dw_down", s);
  if (gather_dy)
    return launch_gemm<Sched::RowsK, Epi::Store, true, true, 2, Gather::A>(ta, tb, tc0, tc0, p, tiles_d, dev, s,
                                                                           "gemm_bwd_dw_down", false);
  const bool f16_d = f16 && !gather_dy;
  Params pr = p;
  if (f16_d) {  // the two-part launches start after the fp16 experts
    pr.parted = 1;
    pr.part_begin = f16_count;
  }
  auto fp16_part = [&]() {
    if (make_tmap(&tf, a.dy16, a.H, rows, 64, BK)) return static_cast<int>(LIGER_MOE_ERR_LAUNCH);
    Params pf = p;
    f16_params(pf, 4, kClaimDwDownF16);
    return (pairs_all || split) ? launch_gemm<Sched::RowsK, Epi::Store, true, true, 0, Gather::None, 2, 1>(
                                      ta, tb, tc0, tc0, pf, tiles_d / 2, dev, s, "gemm_bwd_dw_down", false, &tf)
                                : launch_gemm<Sched::RowsK, Epi::Store, true, true, 0>(ta, tb, tc0, tc0, pf, tiles_d,
                                                                                       dev, s, "gemm_bwd_dw_down", false,
                                                                                       &tf);
  };
  int rc = (f16_d && f16_first) ? fp16_part() : LIGER_MOE_OK;
  if (rc != LIGER_MOE_OK) return rc;
  if (pairs_all) {
    rc = launch_gemm<Sched::RowsK, Epi::Store, true, true, 2, Gather::None, 2, 1>(ta, tb, tc0, tc0, pr, tiles_d / 2,
                                                                                  dev, s, "gemm_bwd_dw_down", false);
  } else if (split) {
    Params ph = pr;  // [begin, pair_count): pairs; [pair_count, E): one CTA per tile
    ph.parted = 1;
    ph.part_end = pair_count;
    rc = launch_gemm<Sched::RowsK, Epi::Store, true, true, 2, Gather::None, 2, 1>(ta, tb, tc0, tc0, ph, tiles_d / 2,
                                                                                  dev, s, "gemm_bwd_dw_down", false);
    Params pl = p;
    pl.parted = 1;
    pl.part_begin = pair_count;
    if (rc == LIGER_MOE_OK)
      rc = launch_gemm<Sched::RowsK, Epi::Store, true, true, 2>(ta, tb, tc0, tc0, pl, tiles_d, dev, s,
                                                                "gemm_bwd_dw_down", false);
  } else {
    rc = launch_gemm<Sched::RowsK, Epi::Store, true, true, 2>(ta, tb, tc0, tc0, pr, tiles_d, dev, s,
                                                              "gemm_bwd_dw_down", false);
  }
  if (rc == LIGER_MOE_OK && f16_d && !f16_first) rc = fp16_part();
  return rc;
}

}  // namespace lmoe
