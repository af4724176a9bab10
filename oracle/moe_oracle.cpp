// CPU oracle for the routed Mixture-of-Experts layer, forward and backward.
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
// benchmark's CPU-baseline leg may load this library.  The product path
// (the CUDA library and its Python binding) never calls it and shares no
// code, header, table or helper with it.
//
// What it computes, and where that comes from:
//   * LightMoE README, "MoE inference": one layer call is dispatch, gate/up
//     projection, gated activation, down projection, routing-weight
//     application, deterministic combine.
//   * LightMoE README, "MoE training": MoEDispatch turns (top_k_ids,
//     top_k_weights) into expert-major gather indices, m_indptr, permuted
//     routing weights and inverse slots; the expert layer has deterministic
//     input-, weight- and router-gradient kernels.
//   * LightMoE README, "Grouped GEMM": contiguous expert-major rows, m_indptr
//     int32 of length E+1, zero-row experts valid.
//   * LigerCute README, "LigerMoE design": forward sorts routed tokens,
//     applies router weights in a final local combine; backward produces
//     expert-output gradients, recomputes activations, computes dX and dW and
//     reduces routed dX back to tokens.
//   * LigerCute PR summary, "Testing Done": the reference is an fp32 CPU
//     computation on identically bf16-rounded inputs.
//   * Liger Kernel README, "High-level APIs" (LigerSwiGLUMLP): the SwiGLU MLP
//     down(silu(gate(x)) * up(x)).
//   * LightMoE README, "Compatibility" and "Highlights": the gated
//     activations bounded SwiGLU (with an activation clamp), SwiGLU-OAI and
//     GeGLU, plus ReGLU; the pages name them without formulas, so each is
//     written out below in its plainest published form (see act_forward).
//     ReLU² is the one non-gated form: its experts hold two weights (up
//     and down, LightMoE README, "MoE inference"), h = max(a, 0)^2.
//   * The router projection that produces the logits, and its backward
//     (oracle_router_logits, oracle_router_backward).  LightMoE README, "MoE
//     training", leaves the routing policy to the host framework; its
//     plainest form is one linear layer, logits = x Wr^T + b, whose input
//     gradient adds to the layer's dX.
// Readings where the pages are silent (tie order, gate/up row order,
// rounding points, softmax over the selected k) are spelled out at each
// function.  Arithmetic is float (fp32) with bf16 inputs widened exactly;
// sums run in the stated index order; build with -ffp-contract=off so no
// multiply-add is fused.
//
// Parity pins for every function here live in tests/test_oracle_*.py
// (brute force, fp64 dense evaluation, autograd, finite differences,
// closed forms and degenerate cases).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <thread>
#include <vector>

namespace {

inline float bf16_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// float -> bf16, round to nearest, ties to even (the standard conversion).
inline uint16_t float_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return static_cast<uint16_t>((u >> 16) | 0x0040u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

inline float round_to_bf16(float f) { return bf16_to_float(float_to_bf16(f)); }

// silu(a) = a / (1 + exp(-a))   (SwiGLU's gate activation)
inline float silu(float a) { return a / (1.0f + std::exp(-a)); }

// Gated activations h = act(g, u) of the expert MLP, and their partial derivatives.
//   0 SwiGLU          h = silu(g) u
//   1 bounded SwiGLU  h = silu(gc) uc,         gc = min(g, c), uc = clamp(u, -c, c)
//   2 SwiGLU-OAI      h = gc sigmoid(a gc) (uc + 1),  a = 1.702, same clamps with c the limit
//   3 GeGLU           h = gelu(g) u,  gelu(g) = g/2 (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3)))
//   4 ReGLU           h = max(g, 0) u
//   5 ReLU²           h = r r,  r = max(g, 0)   (not gated: there is no u, see gated())
// A clamp passes the gradient where its input lies inside the closed interval and blocks it
// outside.  SwiGLU keeps its own operation order (silu, then the product) everywhere below.
constexpr int kActSwiGLU = 0, kActBounded = 1, kActOAI = 2, kActGeGLU = 3, kActReGLU = 4, kActReLU2 = 5;
constexpr float kOaiAlpha = 1.702f;
constexpr float kGeluK0 = 0.7978845608028654f;  // sqrt(2 / pi)
constexpr float kGeluK1 = 0.044715f;

inline float sigmoid(float a) { return 1.0f / (1.0f + std::exp(-a)); }

// Gated activations read two projections of x (rows [0, I) and [I, 2I) of the expert's first
// weight, [2I, H]); ReLU² reads one (its up weight, [I, H]).
inline bool gated(int act) { return act != kActReLU2; }
inline int first_rows(int act, int I) { return gated(act) ? 2 * I : I; }

inline float act_forward(int act, float c, float g, float u) {
  switch (act) {
    case kActBounded: {
      const float gc = std::min(g, c), uc = std::min(std::max(u, -c), c);
      return silu(gc) * uc;
    }
    case kActOAI: {
      const float gc = std::min(g, c), uc = std::min(std::max(u, -c), c);
      return (gc * sigmoid(kOaiAlpha * gc)) * (uc + 1.0f);
    }
    case kActGeGLU: {
      const float t = std::tanh(kGeluK0 * (g + kGeluK1 * g * g * g));
      return (0.5f * g * (1.0f + t)) * u;
    }
    case kActReGLU:
      return std::max(g, 0.0f) * u;
    case kActReLU2: {
      const float r = std::max(g, 0.0f);
      return r * r;
    }
    default:
      return silu(g) * u;
  }
}

// dh/dg and dh/du of act_forward (every activation other than SwiGLU).
inline void act_partials(int act, float c, float g, float u, float* dhdg, float* dhdu) {
  switch (act) {
    case kActBounded: {
      const float gc = std::min(g, c), uc = std::min(std::max(u, -c), c);
      const float s = sigmoid(gc);
      *dhdg = (g <= c) ? uc * s * (1.0f + gc * (1.0f - s)) : 0.0f;
      *dhdu = (u >= -c && u <= c) ? gc * s : 0.0f;
      return;
    }
    case kActOAI: {
      const float gc = std::min(g, c), uc = std::min(std::max(u, -c), c);
      const float s = sigmoid(kOaiAlpha * gc);
      *dhdg = (g <= c) ? (uc + 1.0f) * s * (1.0f + kOaiAlpha * gc * (1.0f - s)) : 0.0f;
      *dhdu = (u >= -c && u <= c) ? gc * s : 0.0f;
      return;
    }
    case kActGeGLU: {
      const float t = std::tanh(kGeluK0 * (g + kGeluK1 * g * g * g));
      const float dgelu = 0.5f * (1.0f + t) + 0.5f * g * (1.0f - t * t) * kGeluK0 * (1.0f + 3.0f * kGeluK1 * g * g);
      *dhdg = u * dgelu;
      *dhdu = 0.5f * g * (1.0f + t);
      return;
    }
    case kActReGLU:
      *dhdg = (g > 0.0f) ? u : 0.0f;
      *dhdu = std::max(g, 0.0f);
      return;
    case kActReLU2:
      *dhdg = 2.0f * std::max(g, 0.0f);
      *dhdu = 0.0f;
      return;
    default:
      return;
  }
}

// Runs f(i) for i in [0, n) on up to `threads` threads, each owning a
// contiguous block of i.  Each i is computed wholly by one thread, so the
// result does not depend on the thread count.
template <class F>
void parallel_for(int n, int threads, F f) {
  if (threads < 1) threads = 1;
  if (threads > n) threads = n;
  if (threads <= 1) {
    for (int i = 0; i < n; ++i) f(i);
    return;
  }
  std::vector<std::thread> pool;
  for (int w = 0; w < threads; ++w) {
    int b = static_cast<int>(static_cast<long long>(n) * w / threads);
    int e = static_cast<int>(static_cast<long long>(n) * (w + 1) / threads);
    pool.emplace_back([=] {
      for (int i = b; i < e; ++i) f(i);
    });
  }
  for (auto& t : pool) t.join();
}

// Expert order used by the router: larger logit first; equal logits ->
// smaller expert id first; NaN after every number (NaNs by id).  The pages
// only say "top_k_ids ... distinct expert indices per token" (LightMoE
// README, "MoE inference"); the tie rule is this implementation's reading.
inline bool ranks_before(float a, int ia, float b, int ib) {
  bool na = std::isnan(a), nb = std::isnan(b);
  if (na != nb) return nb;
  if (!na && a != b) return a > b;
  return ia < ib;
}

// One expert applied to one token row (SwiGLU MLP).
//   g[n] = sum_h x[h] * Wgu[n, h]          n < I   (rows [0, I) are the gate)
//   u[n] = sum_h x[h] * Wgu[I + n, h]              (rows [I, 2I) are the up)
//   hq[n] = bf16( act(g[n], u[n]) )                 (rounded: h is stored bf16; SwiGLU:
//                                                   silu(g[n]) * u[n])
// Sums in float, h ascending.  ReLU²: Wgu is the up weight [I, H], g[n] = sum_h x[h] * Wup[n, h],
// u[n] = 0.
void gate_up_row(const uint16_t* xrow, const uint16_t* wgu_e, int H, int I, float* g, float* u,
                 float* hq, int act = kActSwiGLU, float clamp = 0.0f) {
  for (int n = 0; n < I; ++n) {
    const uint16_t* wg = wgu_e + static_cast<size_t>(n) * H;
    const uint16_t* wu = gated(act) ? wgu_e + static_cast<size_t>(I + n) * H : nullptr;
    float ag = 0.0f, au = 0.0f;
    for (int h = 0; h < H; ++h) {
      float xv = bf16_to_float(xrow[h]);
      ag += xv * bf16_to_float(wg[h]);
      if (wu) au += xv * bf16_to_float(wu[h]);
    }
    g[n] = ag;
    u[n] = au;
    hq[n] = round_to_bf16(act_forward(act, clamp, ag, au));
  }
}

//   o[c] = sum_n hq[n] * Wd[c, n]      (c < H; sum n ascending)
void down_row(const float* hq, const uint16_t* wd_e, int H, int I, float* o) {
  for (int c = 0; c < H; ++c) {
    const uint16_t* wr = wd_e + static_cast<size_t>(c) * I;
    float a = 0.0f;
    for (int n = 0; n < I; ++n) a += hq[n] * bf16_to_float(wr[n]);
    o[c] = a;
  }
}

// Backward through one routed row (token t, slot j, expert e, weight wj):
//   dHu[n] = sum_c dY[c] * Wd[c, n]                      (c ascending)
//   gamma  = sum_n dHu[n] * hq[n]                        (n ascending)
//   dh[n]  = wj * dHu[n]
//   s      = 1 / (1 + exp(-g[n]))
//   dg[n]  = ((dh[n] * u[n]) * s) * (1 + g[n] * (1 - s))  d/dg of silu(g)*u
//   du[n]  = dh[n] * silu(g[n])                           d/du of silu(g)*u
// (other activations: dg[n] = dh[n] * dh/dg, du[n] = dh[n] * dh/du from act_partials;
//  ReLU²: dg[n] = dh[n] * 2 max(g[n], 0), du[n] = 0)
// g and u are the unrounded float values (recomputed, as LigerCute's
// backward recomputes activations: LigerCute README, "Backward pass").
float swiglu_row_backward(const uint16_t* dyrow, const uint16_t* wd_e, int H, int I, float wj,
                          const float* g, const float* u, const float* hq, float* dHu, float* dg,
                          float* du, int act = kActSwiGLU, float clamp = 0.0f) {
  for (int n = 0; n < I; ++n) dHu[n] = 0.0f;
  for (int c = 0; c < H; ++c) {
    float dyc = bf16_to_float(dyrow[c]);
    const uint16_t* wr = wd_e + static_cast<size_t>(c) * I;
    for (int n = 0; n < I; ++n) dHu[n] += dyc * bf16_to_float(wr[n]);
  }
  float gamma = 0.0f;
  for (int n = 0; n < I; ++n) gamma += dHu[n] * hq[n];
  for (int n = 0; n < I; ++n) {
    float dh = wj * dHu[n];
    if (act == kActSwiGLU) {
      float s = 1.0f / (1.0f + std::exp(-g[n]));
      dg[n] = ((dh * u[n]) * s) * (1.0f + g[n] * (1.0f - s));
      du[n] = dh * silu(g[n]);
    } else {
      float dhdg, dhdu;
      act_partials(act, clamp, g[n], u[n], &dhdg, &dhdu);
      dg[n] = dh * dhdg;
      du[n] = dh * dhdu;
    }
  }
  return gamma;
}

int expert_of_row(const int32_t* m_indptr, int E, int r) {
  // m_indptr[e] <= r < m_indptr[e+1]; empty experts are skipped naturally.
  for (int e = 0; e < E; ++e)
    if (r >= m_indptr[e] && r < m_indptr[e + 1]) return e;
  return -1;
}

}  // namespace

extern "C" {

// Status codes of the oracle (its own; unrelated to the CUDA library's).
enum { ORACLE_OK = 0, ORACLE_BAD_ARG = -1, ORACLE_BAD_ID = -2 };

// ---------------------------------------------------------------------------
// Route: top-k experts per token and their gate weights.
// LightMoE README, "MoE inference" (top_k_ids int32, distinct per token;
// top_k_weights float32) and "MoE training" (routing weights renormalised
// per token: differentiable_probs).
//   ids[t, 0..k-1] = the first k experts in ranks_before order
//   m  = logits[t, ids[t,0]]                      (the largest selected logit)
//   e_j = exp(logits[t, ids[t,j]] - m)
//   w[t, j] = e_j / (e_0 + ... + e_{k-1})         (sum j ascending)
// This is softmax over all E followed by top-k and renormalisation, computed
// on the selected k only (exp is monotone, so the selection is the same).
int oracle_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w) {
  if (T < 0 || E < 1 || k < 1 || k > E) return ORACLE_BAD_ARG;
  std::vector<int> order(E);
  std::vector<float> ex(k);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + static_cast<size_t>(t) * E;
    std::iota(order.begin(), order.end(), 0);
    std::sort(order.begin(), order.end(),
              [&](int a, int b) { return ranks_before(l[a], a, l[b], b); });
    float m = l[order[0]];
    float s = 0.0f;
    for (int j = 0; j < k; ++j) {
      ex[j] = std::exp(l[order[j]] - m);
      s += ex[j];
    }
    for (int j = 0; j < k; ++j) {
      ids[static_cast<size_t>(t) * k + j] = order[j];
      w[static_cast<size_t>(t) * k + j] = ex[j] / s;
    }
  }
  return ORACLE_OK;
}

// ---------------------------------------------------------------------------
// Dispatch: deterministic expert-major order of the T*k routed slots.
// LightMoE README, "MoE training" (gather_indices, m_indptr, routing_weights,
// inverse_slots) and "Grouped GEMM" (contiguous expert-major rows, m_indptr
// of length E+1, empty experts valid); LigerCute README, "Forward pass"
// (routed tokens are sorted before the expert loop).
// Slot s = t*k + j.  Walking s ascending, s is appended to its expert's list;
// the lists concatenated in expert order are the rows.  So within an expert
// rows follow slot order (token ascending): a stable counting sort.
//   counts[e], m_indptr[0]=0, m_indptr[e+1]=m_indptr[e]+counts[e]
//   row_to_slot[r] = slot of row r;  slot_to_row[row_to_slot[r]] = r
//   w_perm[r] = w[row_to_slot[r]]            (optional, may be null)
//   x_perm[r, :] = x[row_to_slot[r] / k, :]  (optional, may be null)
int oracle_dispatch(const int32_t* ids, const float* w, const uint16_t* x, int T, int H, int E, int k,
                    int32_t* counts, int32_t* m_indptr, int32_t* row_to_slot, int32_t* slot_to_row,
                    float* w_perm, uint16_t* x_perm) {
  if (T < 0 || E < 1 || k < 1) return ORACLE_BAD_ARG;
  const long long R = static_cast<long long>(T) * k;
  std::vector<std::vector<int32_t>> lists(E);
  for (long long s = 0; s < R; ++s) {
    int e = ids[s];
    if (e < 0 || e >= E) return ORACLE_BAD_ID;
    lists[e].push_back(static_cast<int32_t>(s));
  }
  m_indptr[0] = 0;
  for (int e = 0; e < E; ++e) {
    counts[e] = static_cast<int32_t>(lists[e].size());
    m_indptr[e + 1] = m_indptr[e] + counts[e];
  }
  int32_t r = 0;
  for (int e = 0; e < E; ++e) {
    for (int32_t s : lists[e]) {
      row_to_slot[r] = s;
      slot_to_row[s] = r;
      if (w_perm) w_perm[r] = w[s];
      if (x_perm)
        std::memcpy(x_perm + static_cast<size_t>(r) * H, x + static_cast<size_t>(s / k) * H,
                    sizeof(uint16_t) * H);
      ++r;
    }
  }
  return ORACLE_OK;
}

// ---------------------------------------------------------------------------
// Grouped SwiGLU expert MLP on expert-major rows, for a chosen set of rows.
// LightMoE README, "Grouped GEMM" (out[sum M_e, N] = a[rows_e] @ b[e].T with
// b: [num_experts, N, K]) and "MoE inference" (gate/up projection, gated
// activation, down projection, routing-weight application).  act / clamp
// choose the activation (act_forward); wgu is [E, 2I, H], or the up weight
// [E, I, H] for ReLU².  For row r of expert e (found from m_indptr):
//   g, u, hq as in gate_up_row;  o = down_row(hq)
//   h_out[i, n]  = bf16(hq[n])                           (optional)
//   gu_out[i, :] = [g | u] as float, 2I values (ReLU²: g, I values)  (optional)
//   y_out[i, c]  = bf16( w_perm[r] * o[c] )               (optional)
// The weight is applied to the down projection's float result before the
// single bf16 rounding of y.
int oracle_grouped_swiglu_rows(const uint16_t* x_perm, const int32_t* m_indptr, const uint16_t* wgu,
                               const uint16_t* wd, const float* w_perm, int R, int H, int I, int E,
                               const int32_t* rows, int nrows, uint16_t* h_out, float* gu_out,
                               uint16_t* y_out, int act, float clamp, int threads) {
  if (R < 0 || H < 1 || I < 1 || E < 1 || nrows < 0 || act < 0 || act > kActReLU2) return ORACLE_BAD_ARG;
  for (int i = 0; i < nrows; ++i) {
    if (rows[i] < 0 || rows[i] >= R || expert_of_row(m_indptr, E, rows[i]) < 0) return ORACLE_BAD_ARG;
  }
  parallel_for(nrows, threads, [&](int i) {
    int r = rows[i];
    int e = expert_of_row(m_indptr, E, r);
    std::vector<float> g(I), u(I), hq(I), o(H);
    const int nin = first_rows(act, I);
    const uint16_t* wgu_e = wgu + static_cast<size_t>(e) * nin * H;
    const uint16_t* wd_e = wd + static_cast<size_t>(e) * H * I;
    gate_up_row(x_perm + static_cast<size_t>(r) * H, wgu_e, H, I, g.data(), u.data(), hq.data(), act, clamp);
    if (h_out)
      for (int n = 0; n < I; ++n) h_out[static_cast<size_t>(i) * I + n] = float_to_bf16(hq[n]);
    if (gu_out)
      for (int n = 0; n < I; ++n) {
        gu_out[static_cast<size_t>(i) * nin + n] = g[n];
        if (gated(act)) gu_out[static_cast<size_t>(i) * nin + I + n] = u[n];
      }
    if (y_out) {
      down_row(hq.data(), wd_e, H, I, o.data());
      for (int c = 0; c < H; ++c)
        y_out[static_cast<size_t>(i) * H + c] = float_to_bf16(w_perm[r] * o[c]);
    }
  });
  return ORACLE_OK;
}

// ---------------------------------------------------------------------------
// Combine: routed rows back to token order.
// LigerCute README, "Forward pass" (final local combine); LightMoE README,
// "Highlights" (deterministic combine).
//   Y[t, c] = bf16( sum_{j=0..k-1} float(y_perm[slot_to_row[t*k+j], c]) )
// float sum, j ascending, for the listed tokens.
int oracle_combine(const uint16_t* y_perm, const int32_t* slot_to_row, int T, int H, int k,
                   const int32_t* toks, int ntok, uint16_t* y_out) {
  if (T < 0 || H < 1 || k < 1) return ORACLE_BAD_ARG;
  std::vector<float> acc(H);
  for (int i = 0; i < ntok; ++i) {
    int t = toks[i];
    if (t < 0 || t >= T) return ORACLE_BAD_ARG;
    std::fill(acc.begin(), acc.end(), 0.0f);
    for (int j = 0; j < k; ++j) {
      const uint16_t* row = y_perm + static_cast<size_t>(slot_to_row[static_cast<size_t>(t) * k + j]) * H;
      for (int c = 0; c < H; ++c) acc[c] += bf16_to_float(row[c]);
    }
    for (int c = 0; c < H; ++c) y_out[static_cast<size_t>(i) * H + c] = float_to_bf16(acc[c]);
  }
  return ORACLE_OK;
}

// ---------------------------------------------------------------------------
// Whole-layer forward, written per token (no dispatch):
//   for j = 0..k-1:  e = ids[t,j];  o = down_row(gate_up_row(x[t]))
//                    y_j[c] = bf16(w[t,j] * o[c])
//   Y[t, c] = bf16( sum_j float(y_j[c]) )        (j ascending)
// Same rounding points as dispatch -> grouped rows -> combine, so the two
// agree bit for bit (a test checks this).
int oracle_forward_tokens(const uint16_t* x, const uint16_t* wgu, const uint16_t* wd,
                          const int32_t* ids, const float* w, int T, int H, int I, int E, int k,
                          const int32_t* toks, int ntok, uint16_t* y_out, int act, float clamp, int threads) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || k < 1 || ntok < 0 || act < 0 || act > kActReLU2) return ORACLE_BAD_ARG;
  for (int i = 0; i < ntok; ++i) {
    if (toks[i] < 0 || toks[i] >= T) return ORACLE_BAD_ARG;
    for (int j = 0; j < k; ++j) {
      int e = ids[static_cast<size_t>(toks[i]) * k + j];
      if (e < 0 || e >= E) return ORACLE_BAD_ID;
    }
  }
  parallel_for(ntok, threads, [&](int i) {
    int t = toks[i];
    std::vector<float> g(I), u(I), hq(I), o(H), acc(H, 0.0f);
    for (int j = 0; j < k; ++j) {
      int e = ids[static_cast<size_t>(t) * k + j];
      float wj = w[static_cast<size_t>(t) * k + j];
      gate_up_row(x + static_cast<size_t>(t) * H, wgu + static_cast<size_t>(e) * first_rows(act, I) * H, H, I,
                  g.data(), u.data(), hq.data(), act, clamp);
      down_row(hq.data(), wd + static_cast<size_t>(e) * H * I, H, I, o.data());
      for (int c = 0; c < H; ++c) acc[c] += round_to_bf16(wj * o[c]);
    }
    for (int c = 0; c < H; ++c) y_out[static_cast<size_t>(i) * H + c] = float_to_bf16(acc[c]);
  });
  return ORACLE_OK;
}

// ---------------------------------------------------------------------------
// Backward, per token: input gradient and router-logit gradient.
// LigerCute README, "Backward pass" (expert-output gradients, recomputed
// activations, input gradient, routed dX reduced back to tokens); LightMoE
// README, "MoE training" (input-gradient and router-gradient kernels;
// differentiable_probs).  For token t, with loss L = <dY, Y>:
//   per j: (gamma_j, dg_j, du_j) = swiglu_row_backward(...)
//   dX[t, h] = bf16( sum_j sum_n ( dg_j[n]*Wgu[e_j, n, h] + du_j[n]*Wgu[e_j, I+n, h] ) )
//              (float; j ascending, then n ascending, gate term then up term;
//               ReLU²: the gate term alone, Wgu the up weight)
//   S = sum_i w_i * gamma_i                    (i ascending)
//   d_logits[t, ids_j] = w_j * (gamma_j - S);  every other entry is exactly 0
// gamma_j = dL/dw_j; the last line is the softmax Jacobian restricted to the
// selected k, so unselected logits get no gradient.
int oracle_backward_tokens(const uint16_t* x, const uint16_t* dy, const uint16_t* wgu, const uint16_t* wd,
                           const int32_t* ids, const float* w, int T, int H, int I, int E, int k,
                           const int32_t* toks, int ntok, uint16_t* dx_out, float* dlogits_out, int act,
                           float clamp, int threads) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || k < 1 || ntok < 0 || act < 0 || act > kActReLU2) return ORACLE_BAD_ARG;
  for (int i = 0; i < ntok; ++i) {
    if (toks[i] < 0 || toks[i] >= T) return ORACLE_BAD_ARG;
    for (int j = 0; j < k; ++j) {
      int e = ids[static_cast<size_t>(toks[i]) * k + j];
      if (e < 0 || e >= E) return ORACLE_BAD_ID;
    }
  }
  parallel_for(ntok, threads, [&](int i) {
    int t = toks[i];
    std::vector<float> g(I), u(I), hq(I), dHu(I), dg(I), du(I), acc(H, 0.0f), gam(k);
    for (int j = 0; j < k; ++j) {
      int e = ids[static_cast<size_t>(t) * k + j];
      float wj = w[static_cast<size_t>(t) * k + j];
      const uint16_t* wgu_e = wgu + static_cast<size_t>(e) * first_rows(act, I) * H;
      gate_up_row(x + static_cast<size_t>(t) * H, wgu_e, H, I, g.data(), u.data(), hq.data(), act, clamp);
      gam[j] = swiglu_row_backward(dy + static_cast<size_t>(t) * H, wd + static_cast<size_t>(e) * H * I, H, I,
                                   wj, g.data(), u.data(), hq.data(), dHu.data(), dg.data(), du.data(), act,
                                   clamp);
      for (int n = 0; n < I; ++n) {
        const uint16_t* wg = wgu_e + static_cast<size_t>(n) * H;
        const uint16_t* wu = gated(act) ? wgu_e + static_cast<size_t>(I + n) * H : nullptr;
        for (int h = 0; h < H; ++h) {
          acc[h] += dg[n] * bf16_to_float(wg[h]);
          if (wu) acc[h] += du[n] * bf16_to_float(wu[h]);
        }
      }
    }
    if (dx_out)
      for (int h = 0; h < H; ++h) dx_out[static_cast<size_t>(i) * H + h] = float_to_bf16(acc[h]);
    if (dlogits_out) {
      float S = 0.0f;
      for (int j = 0; j < k; ++j) S += w[static_cast<size_t>(t) * k + j] * gam[j];
      float* dl = dlogits_out + static_cast<size_t>(i) * E;
      for (int e = 0; e < E; ++e) dl[e] = 0.0f;
      for (int j = 0; j < k; ++j) {
        float wj = w[static_cast<size_t>(t) * k + j];
        dl[ids[static_cast<size_t>(t) * k + j]] = wj * (gam[j] - S);
      }
    }
  });
  return ORACLE_OK;
}

// ---------------------------------------------------------------------------
// Backward, per expert: weight gradients (overwritten, bf16).
// LigerCute README, "Backward pass" (expert-weight gradients accumulated
// across token batches); LightMoE README, "MoE training" (deterministic
// weight-gradient kernels).  For expert e, over its routed rows (t, j) with
// t ascending:
//   dW_gu[e, n, h]   = bf16( sum dg[n] * x[t, h] )        n < I
//   dW_gu[e, I+n, h] = bf16( sum du[n] * x[t, h] )          (gated activations only: ReLU²'s
//                                                          dW_up is [E, I, H])
//   dW_d[e, c, n]    = bf16( sum (w_j * dY[t, c]) * hq[n] )
// float sums in row order.  An expert with no rows gets exact zeros.
int oracle_backward_dw(const uint16_t* x, const uint16_t* dy, const uint16_t* wgu, const uint16_t* wd,
                       const int32_t* ids, const float* w, int T, int H, int I, int E, int k,
                       const int32_t* experts, int nexp, uint16_t* dwgu_out, uint16_t* dwd_out, int act,
                       float clamp, int threads) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || k < 1 || nexp < 0 || act < 0 || act > kActReLU2) return ORACLE_BAD_ARG;
  for (int i = 0; i < nexp; ++i)
    if (experts[i] < 0 || experts[i] >= E) return ORACLE_BAD_ARG;
  for (long long s = 0; s < static_cast<long long>(T) * k; ++s)
    if (ids[s] < 0 || ids[s] >= E) return ORACLE_BAD_ID;
  // Two passes with the same arithmetic as one loop per expert: (1) each routed row's dg, du
  // and hq (independent rows, so they run in parallel); (2) each block of output rows sums
  // its products over the expert's rows in row order.  Experts are taken in groups whose
  // per-row vectors fit a bounded buffer.
  const int nin = first_rows(act, I);
  const long long R = static_cast<long long>(T) * k;
  struct Row {
    int t;
    float wj;
  };
  std::vector<std::vector<Row>> rows_of(nexp);
  for (int i = 0; i < nexp; ++i)
    for (long long s = 0; s < R; ++s)  // t ascending, j ascending within t
      if (ids[s] == experts[i]) rows_of[i].push_back(Row{static_cast<int>(s / k), w[s]});
  const size_t cap_rows = std::max<size_t>(1, (size_t(256) << 20) / (3 * sizeof(float) * static_cast<size_t>(I)));
  constexpr int kBlk = 32;  // output rows per unit of the second pass
  for (int i0 = 0; i0 < nexp;) {
    int i1 = i0;
    std::vector<size_t> first{0};  // row offset of each expert of the group in the buffers
    while (i1 < nexp && (i1 == i0 || first.back() + rows_of[i1].size() <= cap_rows)) {
      first.push_back(first.back() + rows_of[i1].size());
      ++i1;
    }
    const size_t nrows = first.back();
    std::vector<int> owner(nrows);
    for (int i = i0; i < i1; ++i)
      for (size_t q = first[i - i0]; q < first[i - i0 + 1]; ++q) owner[q] = i;
    std::vector<float> dgv(nrows * I), duv(nrows * I), hqv(nrows * I);
    parallel_for(static_cast<int>(nrows), threads, [&](int q) {
      const int i = owner[q];
      const int e = experts[i];
      const Row& rw = rows_of[i][q - first[i - i0]];
      std::vector<float> g(I), u(I), dHu(I);
      gate_up_row(x + static_cast<size_t>(rw.t) * H, wgu + static_cast<size_t>(e) * nin * H, H, I, g.data(), u.data(),
                  hqv.data() + static_cast<size_t>(q) * I, act, clamp);
      swiglu_row_backward(dy + static_cast<size_t>(rw.t) * H, wd + static_cast<size_t>(e) * H * I, H, I, rw.wj,
                          g.data(), u.data(), hqv.data() + static_cast<size_t>(q) * I, dHu.data(),
                          dgv.data() + static_cast<size_t>(q) * I, duv.data() + static_cast<size_t>(q) * I, act, clamp);
    });
    // units: per expert of the group, I / kBlk blocks of gate(/up) rows n, then H / kBlk blocks of rows c
    const int ublk_gu = (I + kBlk - 1) / kBlk, ublk_d = (H + kBlk - 1) / kBlk;
    const int per_e = ublk_gu + ublk_d;
    parallel_for((i1 - i0) * per_e, threads, [&](int unit) {
      const int i = i0 + unit / per_e;
      const int b = unit % per_e;
      const std::vector<Row>& rws = rows_of[i];
      const size_t q0 = first[i - i0];
      if (b < ublk_gu) {
        const int n0 = b * kBlk, n1 = std::min(I, n0 + kBlk);
        std::vector<float> agu(static_cast<size_t>(n1 - n0) * H * 2, 0.0f);  // gate rows, then up rows
        for (size_t r = 0; r < rws.size(); ++r) {
          const float* dg = dgv.data() + (q0 + r) * I;
          const float* du = duv.data() + (q0 + r) * I;
          const uint16_t* xr = x + static_cast<size_t>(rws[r].t) * H;
          for (int n = n0; n < n1; ++n) {
            float* rg = agu.data() + static_cast<size_t>(n - n0) * H;
            float* ru = gated(act) ? agu.data() + static_cast<size_t>(n1 - n0 + n - n0) * H : nullptr;
            for (int h = 0; h < H; ++h) {
              float xv = bf16_to_float(xr[h]);
              rg[h] += dg[n] * xv;
              if (ru) ru[h] += du[n] * xv;
            }
          }
        }
        if (dwgu_out) {
          uint16_t* o = dwgu_out + static_cast<size_t>(i) * nin * H;
          for (int n = n0; n < n1; ++n) {
            for (int h = 0; h < H; ++h) {
              o[static_cast<size_t>(n) * H + h] = float_to_bf16(agu[static_cast<size_t>(n - n0) * H + h]);
              if (gated(act))
                o[static_cast<size_t>(I + n) * H + h] = float_to_bf16(agu[static_cast<size_t>(n1 - n0 + n - n0) * H + h]);
            }
          }
        }
      } else {
        const int c0 = (b - ublk_gu) * kBlk, c1 = std::min(H, c0 + kBlk);
        std::vector<float> ad(static_cast<size_t>(c1 - c0) * I, 0.0f);
        for (size_t r = 0; r < rws.size(); ++r) {
          const float wj = rws[r].wj;
          const float* hq = hqv.data() + (q0 + r) * I;
          const uint16_t* dyr = dy + static_cast<size_t>(rws[r].t) * H;
          for (int c = c0; c < c1; ++c) {
            float wdy = wj * bf16_to_float(dyr[c]);
            float* rd = ad.data() + static_cast<size_t>(c - c0) * I;
            for (int n = 0; n < I; ++n) rd[n] += wdy * hq[n];
          }
        }
        if (dwd_out) {
          uint16_t* o = dwd_out + static_cast<size_t>(i) * H * I + static_cast<size_t>(c0) * I;
          for (size_t q = 0; q < ad.size(); ++q) o[q] = float_to_bf16(ad[q]);
        }
      }
    });
    i0 = i1;
  }
  return ORACLE_OK;
}


// ---------------------------------------------------------------------------
// Router projection (the linear layer in front of route_topk; LightMoE README,
// "MoE training": routing policy belongs to the host framework, whose
// plainest router is one bias-optional linear layer).
//   logits[t, e] = ( sum_h x[t, h] * Wr[e, h] ) + bias[e]
// float, h ascending, the bias added once after the sum (bias may be NULL).
int oracle_router_logits(const uint16_t* x, const uint16_t* wr, const float* bias, int T, int H, int E,
                         float* logits, int threads) {
  if (T < 0 || H < 1 || E < 1) return ORACLE_BAD_ARG;
  parallel_for(T, threads, [&](int t) {
    const uint16_t* xr = x + static_cast<size_t>(t) * H;
    for (int e = 0; e < E; ++e) {
      const uint16_t* we = wr + static_cast<size_t>(e) * H;
      float acc = 0.0f;
      for (int h = 0; h < H; ++h) acc += bf16_to_float(xr[h]) * bf16_to_float(we[h]);
      logits[static_cast<size_t>(t) * E + e] = bias ? acc + bias[e] : acc;
    }
  });
  return ORACLE_OK;
}

// Backward of the router projection for an upstream gradient d_logits [T, E]
// (dense: every entry is used).  With L the layer loss:
//   dX[t, h]  = bf16( float(dx_in[t, h]) + sum_e d_logits[t, e] * Wr[e, h] )
//               (the router's input gradient added to the layer's dX, dx_in;
//                the sum over e ascending is formed first; dx_in may be NULL = 0)
//   dWr[e, h] = bf16( sum_t d_logits[t, e] * x[t, h] )      t ascending
//   dbias[e]  = sum_t d_logits[t, e]                          t ascending
// for the listed tokens (dx_out [ntok, H]) and experts (dwr_out [nexp, H],
// dbias_out [nexp]); any output may be NULL.
int oracle_router_backward(const float* dlogits, const uint16_t* x, const uint16_t* wr, const uint16_t* dx_in,
                           int T, int H, int E, const int32_t* toks, int ntok, uint16_t* dx_out,
                           const int32_t* experts, int nexp, uint16_t* dwr_out, float* dbias_out, int threads) {
  if (T < 0 || H < 1 || E < 1 || ntok < 0 || nexp < 0) return ORACLE_BAD_ARG;
  for (int i = 0; i < ntok; ++i)
    if (toks[i] < 0 || toks[i] >= T) return ORACLE_BAD_ARG;
  for (int i = 0; i < nexp; ++i)
    if (experts[i] < 0 || experts[i] >= E) return ORACLE_BAD_ARG;
  if (dx_out)
    parallel_for(ntok, threads, [&](int i) {
      const int t = toks[i];
      std::vector<float> acc(H, 0.0f);
      const float* dl = dlogits + static_cast<size_t>(t) * E;
      for (int e = 0; e < E; ++e) {
        const uint16_t* we = wr + static_cast<size_t>(e) * H;
        for (int h = 0; h < H; ++h) acc[h] += dl[e] * bf16_to_float(we[h]);
      }
      for (int h = 0; h < H; ++h) {
        const float base = dx_in ? bf16_to_float(dx_in[static_cast<size_t>(t) * H + h]) : 0.0f;
        dx_out[static_cast<size_t>(i) * H + h] = float_to_bf16(base + acc[h]);
      }
    });
  if (dwr_out || dbias_out)
    parallel_for(nexp, threads, [&](int i) {
      const int e = experts[i];
      std::vector<float> acc(H, 0.0f);
      float db = 0.0f;
      for (int t = 0; t < T; ++t) {
        const float d = dlogits[static_cast<size_t>(t) * E + e];
        const uint16_t* xr = x + static_cast<size_t>(t) * H;
        for (int h = 0; h < H; ++h) acc[h] += d * bf16_to_float(xr[h]);
        db += d;
      }
      if (dwr_out)
        for (int h = 0; h < H; ++h) dwr_out[static_cast<size_t>(i) * H + h] = float_to_bf16(acc[h]);
      if (dbias_out) dbias_out[i] = db;
    });
  return ORACLE_OK;
}

}  // extern "C"
