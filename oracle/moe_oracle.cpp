// CPU oracle for the MoE expert layer forward pass.
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU
// baseline may load this library.  It shares no code, header, table or helper with the
// CUDA library; it is a plain, slow, obviously correct restatement of what the layer
// computes, in fp64.
//
// What it follows (page titles of the source material):
//  * "Wide-EP ... (NVIDIA)" explainer, section "MoE basics": a router picks, for each
//    token, which experts it uses (DeepSeek-R1: 256 experts, 8 chosen); only the chosen
//    experts compute and their results are summed.
//  * "Efficient MoE training for biological foundation models" (NVIDIA BioNeMo blog
//    rewrite), section "GroupedLinear Optimizes Expert Computation": each expert keeps its
//    own matrices (GroupedLinear -> ScaledSwiGLU -> GroupedLinear); ScaledSwiGLU folds the
//    routing probabilities ("scales") into the SwiGLU activation.
//  * same page, section "MXFP8 Precision Reduces Memory Footprint": MXFP8 stores 8-bit
//    values with one scaling factor per block of 32 consecutive values.
//
// Readings where the pages are silent (each one is listed in the design notes):
//  * top-k order: key (-logit, id) ascending: highest logit first, equal logits go to the
//    lower expert id; +0.0 == -0.0; NaN logits are rejected (status -2).
//  * probabilities: softmax over the k selected logits, p_j = exp(l_j - l_1) / sum_i
//    exp(l_i - l_1), l_1 the largest selected logit.
//  * SwiGLU: h = p * silu(x W_gate) (.) (x W_up), silu(a) = a / (1 + exp(-a)); the
//    probability is applied to h, before the down projection.
//  * no token dropping; tokens with no local expert get a zero output row.
//  * y_t = sum over the token's local slots, in slot order, of h W_down.
//  * MXFP8 element = OCP FP8 E4M3 ("E4M3FN": bias 7, max normal 448, no infinities,
//    NaN = S.1111.111, subnormals kept), rounding to nearest even, saturating to +-448.
//    Scale = E8M0 power of two 2^X with X = floor(log2(amax)) - 8 clamped to [-127, 127];
//    an all-zero block gets code 127 (2^0).  Element = RNE(v / 2^X).
//  * MXFP8 blocks run along the contraction (K) dimension: x rows along d, W_gate/W_up
//    columns along d, W_down columns along f, h rows along f (after the probability).
//
// The backward (oracle_moe_backward) is pinned by central finite differences of the
// forward in fp64 (tests/test_backward_oracle.py).
//
// Parity pins: every function here is pinned by tests that do not call it back with
// its own formula (hand-worked example, numpy brute force with an independent top-k and
// an independent nearest-code quantiser, dense-MLP reductions, linearity and EP-slice
// additivity, exhaustive E4M3 decode against torch's float8_e4m3fn).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

enum DType { DT_F32 = 0, DT_BF16 = 1, DT_E4M3 = 2, DT_F64 = 3 };

inline double bf16_value(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

inline double load_value(const void* p, int dtype, int64_t i) {
  switch (dtype) {
    case DT_F32: return static_cast<double>(static_cast<const float*>(p)[i]);
    case DT_BF16: return bf16_value(static_cast<const uint16_t*>(p)[i]);
    case DT_F64: return static_cast<const double*>(p)[i];
    default: return NAN;
  }
}

// --- OCP FP8 E4M3 ("E4M3FN") -------------------------------------------------------
double e4m3_decode(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 0xF, m = c & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0) mag = std::ldexp(static_cast<double>(m), -9);           // m/8 * 2^-6
  else mag = std::ldexp(8.0 + m, e - 7 - 3);                           // (1+m/8) * 2^(e-7)
  return s ? -mag : mag;
}

// Round a non-negative real q (exactly representable) to the nearest integer, ties to even.
inline double rne(double q) {
  double fl = std::floor(q), fr = q - fl;
  if (fr > 0.5) return fl + 1.0;
  if (fr < 0.5) return fl;
  return (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

uint8_t e4m3_encode(double v) {
  if (std::isnan(v)) return 0x7F;
  const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  const double a = std::fabs(v);
  if (a >= 448.0) return sign | 0x7E;                         // saturate to max normal
  if (a < std::ldexp(1.0, -6)) {                              // subnormal grid, step 2^-9
    const int r = static_cast<int>(rne(std::ldexp(a, 9)));    // 0..8 (8 = min normal 0x08)
    return sign | static_cast<uint8_t>(r);
  }
  int ex;
  std::frexp(a, &ex);                                         // a = m * 2^ex, m in [0.5,1)
  int e = ex - 1;                                             // floor(log2 a), in [-6, 8]
  int r = static_cast<int>(rne(std::ldexp(a, 3 - e)));        // mantissa grid, in [8, 16]
  if (r == 16) { r = 8; e += 1; }
  return sign | static_cast<uint8_t>(((e + 7) << 3) | (r - 8));
}

// E8M0 shared exponent for one block: X = floor(log2(amax)) - 8 clamped to [-127,127];
// amax == 0 -> X = 0 (code 127).
int mx_block_exponent(double amax) {
  if (amax == 0.0) return 0;
  int ex;
  std::frexp(amax, &ex);
  int X = (ex - 1) - 8;
  return std::max(-127, std::min(127, X));
}

// Quantise 32 values v[i*stride] in place into codes/scale, return dequantised values.
void mx_quantize_block(const double* v, int64_t stride, uint8_t* codes, int64_t cstride,
                       uint8_t* scale, double* deq) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[i * stride]));
  const int X = mx_block_exponent(amax);
  *scale = static_cast<uint8_t>(X + 127);
  for (int i = 0; i < 32; ++i) {
    const uint8_t c = e4m3_encode(std::ldexp(v[i * stride], -X));
    if (codes) codes[i * cstride] = c;
    if (deq) deq[i * stride] = std::ldexp(e4m3_decode(c), X);
  }
}

inline double silu(double a) { return a / (1.0 + std::exp(-a)); }

// Top-k of one token.  Returns false on a NaN logit.
bool route_one(const float* lg, int E, int k, int32_t* ids, double* probs) {
  for (int e = 0; e < E; ++e)
    if (std::isnan(lg[e])) return false;
  std::vector<int32_t> idx(E);
  std::iota(idx.begin(), idx.end(), 0);
  std::partial_sort(idx.begin(), idx.begin() + k, idx.end(), [&](int32_t a, int32_t b) {
    const double la = lg[a], lb = lg[b];
    if (la != lb) return la > lb;   // -0.0 == +0.0 here
    return a < b;
  });
  const double l1 = lg[idx[0]];
  double s = 0.0;
  for (int j = 0; j < k; ++j) s += std::exp(static_cast<double>(lg[idx[j]]) - l1);
  for (int j = 0; j < k; ++j) {
    ids[j] = idx[j];
    probs[j] = std::exp(static_cast<double>(lg[idx[j]]) - l1) / s;
  }
  return true;
}

// One weight element of expert e, matrix [R, C] (user layout), dequantised if E4M3.
struct WeightView {
  const void* p;
  const uint8_t* scale;  // E4M3 only: [E_loc, R/32, C]
  int dtype;
  int64_t R, C;
  double at(int64_t e, int64_t r, int64_t c) const {
    const int64_t i = (e * R + r) * C + c;
    if (dtype == DT_E4M3) {
      const uint8_t s = scale[(e * (R / 32) + r / 32) * C + c];
      return std::ldexp(e4m3_decode(static_cast<const uint8_t*>(p)[i]), static_cast<int>(s) - 127);
    }
    return load_value(p, dtype, i);
  }
};

}  // namespace

extern "C" {

int oracle_version(void) { return 1; }

void oracle_e4m3_decode(const uint8_t* codes, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_decode(codes[i]);
}

void oracle_e4m3_encode(const double* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode(v[i]);
}

// MXFP8 quantisation of a tensor [n_outer, K, n_inner] in blocks of 32 along K.
// codes: same shape; scales: [n_outer, K/32, n_inner].  Returns -1 if K % 32 != 0.
int oracle_mx_quantize(const void* src, int src_dtype, int64_t n_outer, int64_t K, int64_t n_inner,
                       uint8_t* codes, uint8_t* scales, int nthreads) {
  if (K % 32 != 0) return -1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
  for (int64_t o = 0; o < n_outer; ++o) {
    std::vector<double> blk(32);
    for (int64_t kb = 0; kb < K / 32; ++kb)
      for (int64_t c = 0; c < n_inner; ++c) {
        const int64_t base = (o * K + kb * 32) * n_inner + c;
        for (int i = 0; i < 32; ++i) blk[i] = load_value(src, src_dtype, base + i * n_inner);
        mx_quantize_block(blk.data(), 1, codes + base, n_inner, scales + (o * (K / 32) + kb) * n_inner + c,
                          nullptr);
      }
  }
  return 0;
}

// Routing: ids [T,k] int32, probs [T,k] fp64.  Returns -2 on a NaN logit, -1 on bad args.
int oracle_route_topk(const float* logits, int64_t T, int E, int k, int32_t* ids, double* probs) {
  if (k < 1 || k > E) return -1;
  for (int64_t t = 0; t < T; ++t)
    if (!route_one(logits + t * E, E, k, ids + t * k, probs + t * k)) return -2;
  return 0;
}

// Permutation into expert-contiguous order (local experts [e0, e0+E_loc)).
// counts [E_loc], offsets [E_loc+1], row_src_token / row_slot [N], pair_to_row [T,k].
int oracle_permute(const int32_t* ids, int64_t T, int k, int e0, int E_loc, int32_t* counts,
                   int32_t* offsets, int32_t* row_src_token, int32_t* row_slot, int32_t* pair_to_row) {
  for (int e = 0; e < E_loc; ++e) counts[e] = 0;
  for (int64_t i = 0; i < T * k; ++i) {
    const int e = ids[i] - e0;
    if (e >= 0 && e < E_loc) counts[e] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E_loc; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int32_t> cursor(offsets, offsets + E_loc);
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      const int e = ids[t * k + j] - e0;
      if (e >= 0 && e < E_loc) {
        const int32_t row = cursor[e]++;
        row_src_token[row] = static_cast<int32_t>(t);
        row_slot[row] = j;
        pair_to_row[t * k + j] = row;
      } else {
        pair_to_row[t * k + j] = -1;
      }
    }
  return 0;
}

// Layer forward for a list of tokens, fp64.
//   x        [T, d]           x_dtype F32 or BF16
//   logits   [T, E]           fp32
//   W_gate/W_up [E_loc, d, f], W_down [E_loc, f, d]   w_dtype F32, BF16 or E4M3 (then the
//            *_scale arrays give E8M0 codes: [E_loc, d/32, f] and [E_loc, f/32, d])
//   mx_act   1: x rows and h rows are MXFP8-quantised (blocks of 32 along d and f)
//   tokens   [n_tokens] token indices; y [n_tokens, d] fp64 output.
int oracle_moe_forward(const void* x, int x_dtype, const float* logits, int64_t T, int d, int f, int E,
                       int k, int e0, int E_loc, int w_dtype, const void* W_gate, const void* W_up,
                       const void* W_down, const uint8_t* Wg_scale, const uint8_t* Wu_scale,
                       const uint8_t* Wd_scale, int mx_act, const int64_t* tokens, int64_t n_tokens,
                       double* y, int nthreads) {
  if (k < 1 || k > E || e0 < 0 || e0 + E_loc > E || d <= 0 || f <= 0) return -1;
  if ((mx_act || w_dtype == DT_E4M3) && (d % 32 != 0 || f % 32 != 0)) return -1;
  for (int64_t i = 0; i < n_tokens; ++i)
    if (tokens[i] < 0 || tokens[i] >= T) return -1;
  const WeightView Wg{W_gate, Wg_scale, w_dtype, d, f};
  const WeightView Wu{W_up, Wu_scale, w_dtype, d, f};
  const WeightView Wd{W_down, Wd_scale, w_dtype, f, d};
  int status = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t i = 0; i < n_tokens; ++i) {
    const int64_t t = tokens[i];
    std::vector<int32_t> ids(k);
    std::vector<double> probs(k), xt(d), g(f), u(f), h(f), o(d);
    double* yt = y + i * d;
    for (int m = 0; m < d; ++m) yt[m] = 0.0;
    if (!route_one(logits + t * E, E, k, ids.data(), probs.data())) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      status = -2;
      continue;
    }
    for (int c = 0; c < d; ++c) xt[c] = load_value(x, x_dtype, t * d + c);
    if (mx_act) {
      uint8_t s;
      for (int b = 0; b < d / 32; ++b) mx_quantize_block(&xt[b * 32], 1, nullptr, 1, &s, &xt[b * 32]);
    }
    for (int j = 0; j < k; ++j) {
      const int e = ids[j] - e0;
      if (e < 0 || e >= E_loc) continue;
      // gate and up projections: g = x W_gate, u = x W_up
      for (int n = 0; n < f; ++n) { g[n] = 0.0; u[n] = 0.0; }
      for (int c = 0; c < d; ++c) {
        const double xc = xt[c];
        for (int n = 0; n < f; ++n) {
          g[n] += xc * Wg.at(e, c, n);
          u[n] += xc * Wu.at(e, c, n);
        }
      }
      // scaled SwiGLU
      for (int n = 0; n < f; ++n) h[n] = probs[j] * silu(g[n]) * u[n];
      if (mx_act) {
        uint8_t s;
        for (int b = 0; b < f / 32; ++b) mx_quantize_block(&h[b * 32], 1, nullptr, 1, &s, &h[b * 32]);
      }
      // down projection, summed into y in slot order
      for (int m = 0; m < d; ++m) o[m] = 0.0;
      for (int n = 0; n < f; ++n) {
        const double hn = h[n];
        for (int m = 0; m < d; ++m) o[m] += hn * Wd.at(e, n, m);
      }
      for (int m = 0; m < d; ++m) yt[m] += o[m];
    }
  }
  return status;
}

// Down projection alone for given h rows (diagnostic for MXFP8: the oracle's GEMM2 applied
// to another producer's quantised h).  h_codes [n_rows, f] E4M3, h_scales [n_rows, f/32],
// row_expert [n_rows] local expert index; out [n_rows, d] fp64.
int oracle_down_proj_mx(const uint8_t* h_codes, const uint8_t* h_scales, const int32_t* row_expert,
                        int64_t n_rows, int d, int f, int E_loc, int w_dtype, const void* W_down,
                        const uint8_t* Wd_scale, double* out, int nthreads) {
  if (f % 32 != 0) return -1;
  const WeightView Wd{W_down, Wd_scale, w_dtype, f, d};
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t r = 0; r < n_rows; ++r) {
    double* o = out + r * d;
    for (int m = 0; m < d; ++m) o[m] = 0.0;
    const int e = row_expert[r];
    if (e < 0 || e >= E_loc) continue;
    for (int n = 0; n < f; ++n) {
      const double hn = std::ldexp(e4m3_decode(h_codes[r * f + n]),
                                   static_cast<int>(h_scales[r * (f / 32) + n / 32]) - 127);
      for (int m = 0; m < d; ++m) o[m] += hn * Wd.at(e, n, m);
    }
  }
  return 0;
}


// Layer backward (bf16/fp32/fp64 inputs, no MXFP8), fp64.  With L = sum_t dy_t . y_t, for
// each token t and local slot j (expert e, probability p_j, from route_one):
//   g = x W_gate_e, u = x W_up_e, s = sigmoid(g), a = g s (= silu(g)), h = p_j a u
//   dh = W_down_e dy_t                    (dh_n = sum_m W_down_e[n, m] dy_t[m])
//   dW_down_e[n, m] += h_n dy_t[m]
//   dp_j = sum_n dh_n a_n u_n
//   du = p_j dh a,  dg = p_j dh u s (1 + g (1 - s))      (d silu / dg = s (1 + g (1 - s)))
//   dx_t += W_gate_e dg + W_up_e du;  dW_gate_e[c, n] += x_c dg_n;  dW_up_e[c, n] += x_c du_n
// and for the token's k selected logits (softmax over them, dp = 0 for non-local slots):
//   dlogit_{id_j} = p_j (dp_j - sum_i p_i dp_i); the other E - k logits get 0.
//   tokens [n_tokens]: dx [n_tokens, d] and dlogits [n_tokens, E] are written for these.
//   experts [n_experts] (local indices): dWg, dWu [n_experts, d, f], dWd [n_experts, f, d]
//   summed over all T tokens.  Null outputs are skipped.
int oracle_moe_backward(const void* x, int x_dtype, const float* logits, int64_t T, int d, int f, int E, int k,
                        int e0, int E_loc, int w_dtype, const void* W_gate, const void* W_up, const void* W_down,
                        const void* dy, int dy_dtype, const int64_t* tokens, int64_t n_tokens, double* dx,
                        double* dlogits, const int32_t* experts, int n_experts, double* dWg, double* dWu,
                        double* dWd, int nthreads) {
  if (k < 1 || k > E || e0 < 0 || e0 + E_loc > E || d <= 0 || f <= 0 || w_dtype == DT_E4M3) return -1;
  for (int64_t i = 0; i < n_tokens; ++i)
    if (tokens[i] < 0 || tokens[i] >= T) return -1;
  for (int i = 0; i < n_experts; ++i)
    if (experts[i] < 0 || experts[i] >= E_loc) return -1;
  const WeightView Wg{W_gate, nullptr, w_dtype, d, f};
  const WeightView Wu{W_up, nullptr, w_dtype, d, f};
  const WeightView Wd{W_down, nullptr, w_dtype, f, d};
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
  int status = 0;
  // per-slot quantities of one (token, expert) pair
  auto pair_grads = [&](int64_t t, int e, double p, std::vector<double>& xt, std::vector<double>& dyt,
                        std::vector<double>& g, std::vector<double>& u, std::vector<double>& h,
                        std::vector<double>& dg, std::vector<double>& du) -> double {
    for (int c = 0; c < d; ++c) xt[c] = load_value(x, x_dtype, t * d + c);
    for (int m = 0; m < d; ++m) dyt[m] = load_value(dy, dy_dtype, t * d + m);
    for (int n = 0; n < f; ++n) { g[n] = 0.0; u[n] = 0.0; }
    for (int c = 0; c < d; ++c)
      for (int n = 0; n < f; ++n) {
        g[n] += xt[c] * Wg.at(e, c, n);
        u[n] += xt[c] * Wu.at(e, c, n);
      }
    double dp = 0.0;
    for (int n = 0; n < f; ++n) {
      const double sg = 1.0 / (1.0 + std::exp(-g[n]));
      const double a = g[n] * sg;
      h[n] = p * a * u[n];
      double dh = 0.0;
      for (int m = 0; m < d; ++m) dh += Wd.at(e, n, m) * dyt[m];
      dp += dh * a * u[n];
      du[n] = p * dh * a;
      dg[n] = p * dh * u[n] * sg * (1.0 + g[n] * (1.0 - sg));
    }
    return dp;
  };
  if (dx || dlogits) {
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < n_tokens; ++i) {
      const int64_t t = tokens[i];
      std::vector<int32_t> ids(k);
      std::vector<double> probs(k), dps(k, 0.0), xt(d), dyt(d), g(f), u(f), h(f), dg(f), du(f);
      if (!route_one(logits + t * E, E, k, ids.data(), probs.data())) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
        status = -2;
        continue;
      }
      if (dx)
        for (int c = 0; c < d; ++c) dx[i * d + c] = 0.0;
      for (int j = 0; j < k; ++j) {
        const int e = ids[j] - e0;
        if (e < 0 || e >= E_loc) continue;
        dps[j] = pair_grads(t, e, probs[j], xt, dyt, g, u, h, dg, du);
        if (dx)
          for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int n = 0; n < f; ++n) acc += Wg.at(e, c, n) * dg[n] + Wu.at(e, c, n) * du[n];
            dx[i * d + c] += acc;
          }
      }
      if (dlogits) {
        for (int q = 0; q < E; ++q) dlogits[i * E + q] = 0.0;
        double pdp = 0.0;
        for (int j = 0; j < k; ++j) pdp += probs[j] * dps[j];
        for (int j = 0; j < k; ++j) dlogits[i * E + ids[j]] = probs[j] * (dps[j] - pdp);
      }
    }
  }
  if (dWg || dWu || dWd) {
    // one expert per task; every token routed to it contributes
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int q = 0; q < n_experts; ++q) {
      const int e = experts[q];
      std::vector<int32_t> ids(k);
      std::vector<double> probs(k), xt(d), dyt(d), g(f), u(f), h(f), dg(f), du(f);
      double* gw = dWg ? dWg + static_cast<int64_t>(q) * d * f : nullptr;
      double* uw = dWu ? dWu + static_cast<int64_t>(q) * d * f : nullptr;
      double* dw = dWd ? dWd + static_cast<int64_t>(q) * f * d : nullptr;
      if (gw) std::fill(gw, gw + static_cast<int64_t>(d) * f, 0.0);
      if (uw) std::fill(uw, uw + static_cast<int64_t>(d) * f, 0.0);
      if (dw) std::fill(dw, dw + static_cast<int64_t>(f) * d, 0.0);
      for (int64_t t = 0; t < T; ++t) {
        if (!route_one(logits + t * E, E, k, ids.data(), probs.data())) continue;
        for (int j = 0; j < k; ++j) {
          if (ids[j] - e0 != e) continue;
          pair_grads(t, e, probs[j], xt, dyt, g, u, h, dg, du);
          for (int c = 0; c < d; ++c)
            for (int n = 0; n < f; ++n) {
              if (gw) gw[static_cast<int64_t>(c) * f + n] += xt[c] * dg[n];
              if (uw) uw[static_cast<int64_t>(c) * f + n] += xt[c] * du[n];
            }
          if (dw)
            for (int n = 0; n < f; ++n)
              for (int m = 0; m < d; ++m) dw[static_cast<int64_t>(n) * d + m] += h[n] * dyt[m];
        }
      }
    }
  }
  return status;
}

}  // extern "C"
