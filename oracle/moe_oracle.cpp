// Routed MoE FFN layer: the plain fp64 CPU oracle.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
// definition that the CUDA library is checked against.  Only the tests, the
// smoke check and the CPU-baseline leg of the benchmark may load it; the
// library never does, and this file shares no code, header, table or helper
// with the CUDA sources.
//
// What it computes (sources are the five web pages on the Strata engine; the
// model they describe has 48 layers, 512 experts per layer, 10 picked per
// token, plus a shared expert):
//   * router logits, one score per expert per token, and the choice of the top
//     K experts -- 'Strata はなぜ少ない VRAM でも速いのか' (modeldock.net),
//     section '問題：1,250 億パラメータと 12 GB' (512 experts per layer, the
//     router picks 10 per token);
//   * the shared expert, part of the weights every token uses -- same page and
//     section;
//   * the expert results summed before the next layer starts -- same page,
//     section '1 トークン、三者の分担';
//   * the pages give no formula, activation, normalisation or number format.
//     The readings taken here (softmax over all logits then renormalise the
//     kept K; SwiGLU experts; int4 symmetric group-32 weights with fp16
//     scales; RMSNorm before each layer of the stack) are the plain readings
//     listed in the design notes, each marked where it is used below.
//
// Everything is widened to double from the exact stored bytes (bf16 / fp32
// activations, fp32 router, packed int4 + fp16 scales or fp32 experts) and
// computed in double.  Library primitives used: std::exp, std::sqrt,
// std::stable_sort.
//
// Pins (tests/test_oracle_pins.py): brute-force full sort of all logits on
// tiny inputs including exact ties, closed-form two-expert weights, weights
// summing to one, the K = E case equal to the full softmax mixture computed
// by torch, the single-expert case equal to a dense SwiGLU FFN computed by
// torch, hand-packed int4 blocks (tests/golden), dispatch invariants and
// numpy's stable argsort, RMSNorm against its closed form.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

enum { ACT_F32 = 0, ACT_BF16 = 1 };
enum { W_F32 = 0, W_INT4_G32 = 1 };

// bf16 is the top half of an fp32 bit pattern.
double bf16_to_double(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
double f16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int ex = (h >> 10) & 0x1F;
  int fr = h & 0x3FF;
  double v;
  if (ex == 0) {
    v = std::ldexp(static_cast<double>(fr), -24);  // subnormal: fr * 2^-14 * 2^-10
  } else if (ex == 31) {
    v = fr ? NAN : INFINITY;
  } else {
    v = std::ldexp(1.0 + fr / 1024.0, ex - 15);
  }
  return sign ? -v : v;
}

double act_at(const void* x, int dtype, size_t i) {
  if (dtype == ACT_BF16) return bf16_to_double(static_cast<const uint16_t*>(x)[i]);
  return static_cast<double>(static_cast<const float*>(x)[i]);
}

// int4 plane: row-major, two values per byte, even column in the low nibble,
// two's complement in [-8, 7].
int int4_at(const uint8_t* row, int k) {
  int b = row[k >> 1];
  int n = (k & 1) ? (b >> 4) : (b & 0xF);
  return n >= 8 ? n - 16 : n;
}

// Row r of a weight matrix with `cols` columns, dequantised to double:
// value = q * scale, scale shared by each run of 32 consecutive columns.
void weight_row(int wfmt, const void* q, const void* s, int r, int cols, double* out) {
  if (wfmt == W_F32) {
    const float* w = static_cast<const float*>(q) + static_cast<size_t>(r) * cols;
    for (int k = 0; k < cols; ++k) out[k] = w[k];
    return;
  }
  const uint8_t* row = static_cast<const uint8_t*>(q) + static_cast<size_t>(r) * (cols / 2);
  const uint16_t* sc = static_cast<const uint16_t*>(s) + static_cast<size_t>(r) * (cols / 32);
  for (int g = 0; g < cols / 32; ++g) {
    const double scale = f16_to_double(sc[g]);  // one scale per run of 32 columns
    for (int k = 32 * g; k < 32 * g + 32; ++k) out[k] = int4_at(row, k) * scale;
  }
}

double silu(double z) { return z / (1.0 + std::exp(-z)); }

// One token through one SwiGLU expert: h = silu(W_gate x) * (W_up x), y = W_down h.
// Gate rows are rows 0..f-1 of the gate/up matrix, up rows are rows f..2f-1.
void expert_ffn(int d, int f, int wfmt, const void* gu, const void* gu_s, const void* dn, const void* dn_s,
                const double* x, double* y) {
  std::vector<double> row(std::max(d, f)), h(f);
  for (int i = 0; i < f; ++i) {
    weight_row(wfmt, gu, gu_s, i, d, row.data());
    double g = 0.0;
    for (int k = 0; k < d; ++k) g += row[k] * x[k];
    weight_row(wfmt, gu, gu_s, f + i, d, row.data());
    double u = 0.0;
    for (int k = 0; k < d; ++k) u += row[k] * x[k];
    h[i] = silu(g) * u;
  }
  for (int j = 0; j < d; ++j) {
    weight_row(wfmt, dn, dn_s, j, f, row.data());
    double acc = 0.0;
    for (int i = 0; i < f; ++i) acc += row[i] * h[i];
    y[j] = acc;
  }
}

// Router for one token: logits, softmax over all E, the K largest logits (ties
// to the lower expert index), weights renormalised over the kept K.
void route_token(int d, int E, int K, const double* x, const float* Wr, const float* bias, double* logits,
                 int32_t* idx, double* w, double* gap) {
  for (int e = 0; e < E; ++e) {
    double acc = 0.0;
    const float* wr = Wr + static_cast<size_t>(e) * d;
    for (int k = 0; k < d; ++k) acc += static_cast<double>(wr[k]) * x[k];
    if (bias) acc += bias[e];
    logits[e] = acc;
  }
  double mx = logits[0];
  for (int e = 1; e < E; ++e) mx = std::max(mx, logits[e]);
  std::vector<double> p(E);
  double z = 0.0;
  for (int e = 0; e < E; ++e) {
    p[e] = std::exp(logits[e] - mx);
    z += p[e];
  }
  for (int e = 0; e < E; ++e) p[e] /= z;

  std::vector<int> order(E);
  for (int e = 0; e < E; ++e) order[e] = e;
  // stable sort by logit, largest first: equal logits keep ascending index order
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return logits[a] > logits[b]; });
  double kept = 0.0;
  for (int k = 0; k < K; ++k) {
    idx[k] = order[k];
    kept += p[order[k]];
  }
  for (int k = 0; k < K; ++k) w[k] = p[idx[k]] / kept;
  if (gap) *gap = (K < E) ? logits[order[K - 1]] - logits[order[K]] : INFINITY;
}

// Weights for a given expert set (used when another valid choice at a near-tie is accepted).
void weights_for_set(int E, int K, const double* logits, const int32_t* idx, double* w) {
  double mx = logits[0];
  for (int e = 1; e < E; ++e) mx = std::max(mx, logits[e]);
  double z = 0.0;
  for (int e = 0; e < E; ++e) z += std::exp(logits[e] - mx);
  double kept = 0.0;
  for (int k = 0; k < K; ++k) kept += std::exp(logits[idx[k]] - mx) / z;
  for (int k = 0; k < K; ++k) w[k] = (std::exp(logits[idx[k]] - mx) / z) / kept;
}

}  // namespace

extern "C" {

int orc_version() { return 1; }

// Widen stored activations to double (exact).
int orc_widen(size_t n, const void* x, int x_dtype, double* out) {
  for (size_t i = 0; i < n; ++i) out[i] = act_at(x, x_dtype, i);
  return 0;
}

int orc_f16_to_double(size_t n, const uint16_t* h, double* out) {
  for (size_t i = 0; i < n; ++i) out[i] = f16_to_double(h[i]);
  return 0;
}

// Dequantise a whole [rows x cols] matrix (for pins).
int orc_dequant(int rows, int cols, int wfmt, const void* q, const void* s, double* out) {
  if (wfmt == W_INT4_G32 && (cols % 32) != 0) return 1;
  for (int r = 0; r < rows; ++r) weight_row(wfmt, q, s, r, cols, out + static_cast<size_t>(r) * cols);
  return 0;
}

// Router over T tokens.  logits [T*E] (may be null), idx [T*K], w [T*K], gap [T] (may be null).
int orc_route(int T, int d, int E, int K, const void* x, int x_dtype, const float* Wr, const float* bias,
              double* logits, int32_t* idx, double* w, double* gap, int nthreads) {
  if (K < 1 || K > E) return 1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int t = 0; t < T; ++t) {
    std::vector<double> xt(d), lg(E);
    for (int k = 0; k < d; ++k) xt[k] = act_at(x, x_dtype, static_cast<size_t>(t) * d + k);
    route_token(d, E, K, xt.data(), Wr, bias, lg.data(), idx + static_cast<size_t>(t) * K,
                w + static_cast<size_t>(t) * K, gap ? gap + t : nullptr);
    if (logits) std::copy(lg.begin(), lg.end(), logits + static_cast<size_t>(t) * E);
  }
  return 0;
}

// Weights of a given routing (idx [T*K]) from logits [T*E].
int orc_weights_for(int T, int E, int K, const double* logits, const int32_t* idx, double* w) {
  for (int t = 0; t < T; ++t)
    weights_for_set(E, K, logits + static_cast<size_t>(t) * E, idx + static_cast<size_t>(t) * K,
                    w + static_cast<size_t>(t) * K);
  return 0;
}

// Token -> expert dispatch: count per expert, exclusive prefix sum, and the
// assignments a = t*K + k stably sorted by expert, plus the ascending list of
// experts with at least one assignment.
int orc_dispatch(int T, int K, int E, const int32_t* idx, int32_t* counts, int32_t* offs, int32_t* perm,
                 int32_t* active, int32_t* n_active) {
  const int n = T * K;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int a = 0; a < n; ++a) {
    if (idx[a] < 0 || idx[a] >= E) return 1;
    counts[idx[a]]++;
  }
  offs[0] = 0;
  for (int e = 0; e < E; ++e) offs[e + 1] = offs[e] + counts[e];
  std::vector<int> order(n);
  for (int a = 0; a < n; ++a) order[a] = a;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return idx[a] < idx[b]; });
  for (int i = 0; i < n; ++i) perm[i] = order[i];
  int m = 0;
  for (int e = 0; e < E; ++e)
    if (counts[e] > 0) active[m++] = e;
  *n_active = m;
  return 0;
}

// One expert on one token (double in, double out).
int orc_expert(int d, int f, int wfmt, const void* gu, const void* gu_s, const void* dn, const void* dn_s,
               const double* x, double* y) {
  expert_ffn(d, f, wfmt, gu, gu_s, dn, dn_s, x, y);
  return 0;
}

// The layer: y_t = sum_k w_{t,k} * FFN_{idx_{t,k}}(x_t) + [shared] FFN_shared(x_t).
// Per-expert planes come as pointer tables of length E (entries of unused experts may be null).
// If idx_in is non-null that routing is used (weights recomputed for it); otherwise the oracle routes.
// idx_out / w_out (may be null) receive the routing used.  y [T*d] double.
int orc_layer(int T, int d, int f, int E, int K, int wfmt, int has_shared, const void* x, int x_dtype,
              const float* Wr, const float* bias, const void* const* gu, const void* const* gu_s,
              const void* const* dn, const void* const* dn_s, const void* sh_gu, const void* sh_gu_s,
              const void* sh_dn, const void* sh_dn_s, const int32_t* idx_in, int32_t* idx_out, double* w_out,
              double* y, int nthreads) {
  if (K < 1 || K > E) return 1;
  int bad = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
#endif
  for (int t = 0; t < T; ++t) {
    std::vector<double> xt(d), lg(E), w(K), o(d);
    std::vector<int32_t> id(K);
    for (int k = 0; k < d; ++k) xt[k] = act_at(x, x_dtype, static_cast<size_t>(t) * d + k);
    route_token(d, E, K, xt.data(), Wr, bias, lg.data(), id.data(), w.data(), nullptr);
    if (idx_in) {
      for (int k = 0; k < K; ++k) id[k] = idx_in[static_cast<size_t>(t) * K + k];
      weights_for_set(E, K, lg.data(), id.data(), w.data());
    }
    double* yt = y + static_cast<size_t>(t) * d;
    for (int j = 0; j < d; ++j) yt[j] = 0.0;
    for (int k = 0; k < K; ++k) {
      int e = id[k];
      if (e < 0 || e >= E || !gu[e] || !dn[e]) {
        bad++;
        continue;
      }
      expert_ffn(d, f, wfmt, gu[e], gu_s ? gu_s[e] : nullptr, dn[e], dn_s ? dn_s[e] : nullptr, xt.data(),
                 o.data());
      for (int j = 0; j < d; ++j) yt[j] += w[k] * o[j];
    }
    if (has_shared) {
      expert_ffn(d, f, wfmt, sh_gu, sh_gu_s, sh_dn, sh_dn_s, xt.data(), o.data());
      for (int j = 0; j < d; ++j) yt[j] += o[j];
    }
    if (idx_out)
      for (int k = 0; k < K; ++k) idx_out[static_cast<size_t>(t) * K + k] = id[k];
    if (w_out)
      for (int k = 0; k < K; ++k) w_out[static_cast<size_t>(t) * K + k] = w[k];
  }
  return bad ? 2 : 0;
}

// RMSNorm without a learned weight: x / sqrt(mean(x^2) + eps), per token.
int orc_rmsnorm(int T, int d, const void* x, int x_dtype, double eps, double* out) {
  for (int t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int k = 0; k < d; ++k) {
      double v = act_at(x, x_dtype, static_cast<size_t>(t) * d + k);
      ss += v * v;
    }
    double inv = 1.0 / std::sqrt(ss / d + eps);
    for (int k = 0; k < d; ++k)
      out[static_cast<size_t>(t) * d + k] = act_at(x, x_dtype, static_cast<size_t>(t) * d + k) * inv;
  }
  return 0;
}

}  // extern "C"
