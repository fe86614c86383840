// Plain, slow CPU oracle for the fused MoE router.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may load or call
// this file: only the tests, the package smoke check and the benchmark's
// CPU-baseline leg use it. It shares no code, header, table or constant with
// the CUDA library; both sides take their inputs from the seeded generators.
//
// Every step follows its definition literally, in FP64, with no blocking,
// fusion or reordering:
//   * gate projection  logits[m,e] = sum_h x[m,h] * W[e,h]  (sequential h loop)
//       qwisp issue #145, "Observation" (postNorm[H] -> gateLogits[E]);
//       dense_router_decode commit page, "DenseRouterDecodeKernel" (BF16 GEMM,
//       FP32 accumulator; here FP64 accumulation).
//   * NVFP4 weights    W[e,h] = e2m1(q[e,h]) * e4m3(s[e,h/16]) * g
//       dense_router_decode commit page, "NVFP4 blockscaled GEMM".
//   * scores           softmax over all E; or a = sqrt(softplus(l)) with the
//       stable softplus max(l,0) + log1p(exp(-|l|)) and key = a + bias
//       (commit page, "Numerically stable softplus"; the bias only selects,
//       the heap keeps "(score, index, unbiased act)"); or a = sigmoid(l) =
//       1 / (1 + exp(-l)) with key = a + bias in the same way (the same
//       biased-score contract with the sigmoid as the score). With a bias,
//       softmax follows that contract too: key = p + bias with p the full-E
//       softmax probability, weights the unbiased p renormalised (qwisp issue
//       #145, "Gates": the bias variant of the softmax route kernel).
//   * top-k            full stable sort of all E experts by (key desc, index
//       asc): equal keys keep the lower expert index first
//       (qwisp issue #145, "Bit-exactness": the tie-break order is part of
//       the contract).
//   * renormalise      w_j = s_j / sum_{i<k} s_i over the chosen k
//       (commit page, "top-k + renorm").
//   * gather + shared add (the table's consumer): FP32 fma accumulation of
//       the routed rows in slot order -> BF16 -> + shared BF16 -> BF16
//       (b70 lab note, "Exact arithmetic").
//   * route table      serial walk over (token, slot) in row-major order;
//       first sight of an expert appends it to the unique list
//       (b70 lab note, "Unique-route router screen": encounter-ordered
//       unique experts, per-expert token masks, slot-to-unique map, count).
//
// Readings where the pages are silent: without a bias the softmax selection
// key is the logit (softmax is strictly increasing, so the order is the same
// and FP64 probabilities cannot collapse two distinct logits into a false
// tie); with a bias it is the FP64 probability plus the bias; -0.0 and +0.0
// compare equal; if every chosen score is zero the weights are 1/k.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

constexpr int kF32 = 0, kBF16 = 1, kNVFP4 = 2;
constexpr int kSoftmax = 0, kSqrtSoftplus = 1, kSigmoid = 2;

double from_bf16(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// E2M1 magnitudes by code (sign bit 3): OCP microscaling FP4.
const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double e2m1(int code) {
  double v = kE2M1[code & 7];
  return (code & 8) ? -v : v;
}

// E4M3 (OCP FP8): sign, 4 exponent bits with bias 7, 3 mantissa bits,
// subnormals at exponent 0, a single NaN pattern S.1111.111, no infinity.
double e4m3(int code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return std::nan("");
  double v = (e == 0) ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

double sqrt_softplus(double z) {
  double sp = std::max(z, 0.0) + std::log1p(std::exp(-std::fabs(z)));
  return std::sqrt(sp);
}

double sigmoid(double z) { return 1.0 / (1.0 + std::exp(-z)); }

}  // namespace

extern "C" {

double orc_e2m1(int code) { return e2m1(code); }
double orc_e4m3(int code) { return e4m3(code); }
double orc_sqrt_softplus(double z) { return sqrt_softplus(z); }
double orc_sigmoid(double z) { return sigmoid(z); }

// Element h of row r of an [R, H] matrix of the given dtype, widened to FP64.
// NVFP4 rows: packed bytes [R, H/2], scales [R, H/16]; the global scale is
// applied by the caller.
static double elem(const void* p, int dtype, const uint8_t* scales, int H, int r, int h) {
  if (dtype == kF32) return static_cast<const float*>(p)[(size_t)r * H + h];
  if (dtype == kBF16) return from_bf16(static_cast<const uint16_t*>(p)[(size_t)r * H + h]);
  const uint8_t byte = static_cast<const uint8_t*>(p)[(size_t)r * (H / 2) + h / 2];
  const int code = (h % 2 == 0) ? (byte & 15) : (byte >> 4);
  return e2m1(code) * e4m3(scales[(size_t)r * (H / 16) + h / 16]);
}

// logits[m,e] in FP64. Returns 0, or -1 on a bad argument or a NaN scale.
int orc_logits(const void* x, int x_dtype, const void* W, int w_dtype,
               const uint8_t* w_scales, double g, int M, int H, int E, double* out) {
  if (x_dtype != kF32 && x_dtype != kBF16) return -1;
  if (w_dtype == kNVFP4) {
    if (H % 16 != 0 || !w_scales) return -1;
    for (size_t i = 0; i < (size_t)E * (H / 16); ++i)
      if (std::isnan(e4m3(w_scales[i]))) return -1;
  } else if (w_dtype != kF32 && w_dtype != kBF16) {
    return -1;
  }
  for (int m = 0; m < M; ++m) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h)
        acc += elem(x, x_dtype, nullptr, H, m, h) * elem(W, w_dtype, w_scales, H, e, h);
      out[(size_t)m * E + e] = (w_dtype == kNVFP4) ? g * acc : acc;
    }
  }
  return 0;
}

// The selection key and the weight score of every expert of one row of
// FP64 logits l[E] (b: that row's FP32 bias, or null).
//   softmax, no bias  score = exp(l - max) / sum_e exp(l_e - max), key = l
//   softmax, bias     score as above,                             key = score + b
//   sqrt-softplus     score = sqrt(max(l,0) + log1p(exp(-|l|))),   key = score + b
//   sigmoid           score = 1 / (1 + exp(-l)),                   key = score + b
static void row_keys(const double* l, const float* b, int E, int act, double* key,
                     double* score) {
  if (act == kSoftmax) {
    double mx = l[0];
    for (int e = 1; e < E; ++e) mx = std::max(mx, l[e]);
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += std::exp(l[e] - mx);
    for (int e = 0; e < E; ++e) {
      score[e] = std::exp(l[e] - mx) / z;
      key[e] = b ? score[e] + static_cast<double>(b[e]) : l[e];
    }
  } else {
    for (int e = 0; e < E; ++e) {
      score[e] = act == kSigmoid ? sigmoid(l[e]) : sqrt_softplus(l[e]);
      key[e] = score[e] + (b ? static_cast<double>(b[e]) : 0.0);
    }
  }
}

// Selection + renormalisation on FP64 logits [M, E].
//   bias: nullable FP32 [E], or per-row [M, E] when bias_per_row != 0 (used
//         by the adversarial tests).
//   out_idx [M,k], out_w [M,k]; out_keys (nullable) [M, kk] receives the
//   first kk = min(k+1, E) keys in sorted order (for the gap rule).
int orc_select(const double* logits, const float* bias, int bias_per_row, int M, int E,
               int k, int act, int32_t* out_idx, double* out_w, double* out_keys) {
  if (k < 1 || k > E || (act != kSoftmax && act != kSqrtSoftplus && act != kSigmoid)) return -1;
  const int kk = std::min(k + 1, E);
  std::vector<double> key(E), score(E);
  std::vector<int> order(E);
  for (int m = 0; m < M; ++m) {
    const double* l = logits + (size_t)m * E;
    const float* b = bias ? (bias_per_row ? bias + (size_t)m * E : bias) : nullptr;
    row_keys(l, b, E, act, key.data(), score.data());
    for (int e = 0; e < E; ++e) order[e] = e;
    std::stable_sort(order.begin(), order.end(),
                     [&](int a, int c) { return key[a] > key[c]; });
    double sum = 0.0;
    for (int j = 0; j < k; ++j) sum += score[order[j]];
    for (int j = 0; j < k; ++j) {
      out_idx[(size_t)m * k + j] = order[j];
      out_w[(size_t)m * k + j] = (sum > 0.0) ? score[order[j]] / sum : 1.0 / k;
    }
    if (out_keys)
      for (int j = 0; j < kk; ++j) out_keys[(size_t)m * kk + j] = key[order[j]];
  }
  return 0;
}

// Every expert's key and score ([M, E] each), as orc_select ranks and
// weights them; used to judge rows whose order is decided within rounding.
int orc_keys(const double* logits, const float* bias, int bias_per_row, int M, int E, int act,
             double* out_key, double* out_score) {
  if (E < 1 || (act != kSoftmax && act != kSqrtSoftplus && act != kSigmoid)) return -1;
  for (int m = 0; m < M; ++m) {
    const float* b = bias ? (bias_per_row ? bias + (size_t)m * E : bias) : nullptr;
    row_keys(logits + (size_t)m * E, b, E, act, out_key + (size_t)m * E,
             out_score + (size_t)m * E);
  }
  return 0;
}

// Diagnostic for the softmax key reading: the same selection, but sorted by
// the FP64 probability instead of the logit.
int orc_select_by_prob(const double* logits, int M, int E, int k, int32_t* out_idx) {
  if (k < 1 || k > E) return -1;
  std::vector<double> p(E);
  std::vector<int> order(E);
  for (int m = 0; m < M; ++m) {
    const double* l = logits + (size_t)m * E;
    double mx = l[0];
    for (int e = 1; e < E; ++e) mx = std::max(mx, l[e]);
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += std::exp(l[e] - mx);
    for (int e = 0; e < E; ++e) p[e] = std::exp(l[e] - mx) / z;
    for (int e = 0; e < E; ++e) order[e] = e;
    std::stable_sort(order.begin(), order.end(), [&](int a, int c) { return p[a] > p[c]; });
    for (int j = 0; j < k; ++j) out_idx[(size_t)m * k + j] = order[j];
  }
  return 0;
}

// Serial unique-route table for groups of T tokens with k slots each.
//   idx    [G, T, k]
//   unique [G, T*k]  encounter-ordered unique experts, -1 past the count
//   mask   [G, T*k]  bit t set when token t routes to unique[u]; 0 past count
//   map    [G, T, k] position u of each (token, slot) in unique
//   count  [G]
int orc_route_table(const int32_t* idx, int G, int T, int k, int32_t* unique,
                    uint8_t* mask, uint8_t* map, int32_t* count) {
  if (T < 1 || T > 8 || k < 1) return -1;
  const int n = T * k;
  for (int g = 0; g < G; ++g) {
    std::vector<int32_t> uq;
    std::vector<uint8_t> mk;
    for (int t = 0; t < T; ++t) {
      for (int s = 0; s < k; ++s) {
        const size_t pos = ((size_t)g * T + t) * k + s;
        const int32_t v = idx[pos];
        size_t u = 0;
        while (u < uq.size() && uq[u] != v) ++u;
        if (u == uq.size()) {
          uq.push_back(v);
          mk.push_back(0);
        }
        mk[u] = static_cast<uint8_t>(mk[u] | (1u << t));
        map[pos] = static_cast<uint8_t>(u);
      }
    }
    count[g] = static_cast<int32_t>(uq.size());
    for (int u = 0; u < n; ++u) {
      unique[(size_t)g * n + u] = u < (int)uq.size() ? uq[u] : -1;
      mask[(size_t)g * n + u] = u < (int)uq.size() ? mk[u] : 0;
    }
  }
  return 0;
}


// Consumer side of the unique-route table (b70 lab note, "MTP1 M=2
// gather/shared-add gate", "Exact arithmetic": FP32 routed accumulation ->
// BF16 -> add shared BF16 -> BF16; "Real route-direct result": one expert
// output row per unique (token, expert) route, reused by duplicate slots).
//   y      BF16 [G, T*k, T, D]  row (u, t): unique expert u's output for token t
//   map    [G, T, k]            unique position of slot s of token t (route_table)
//   w      FP32 [G, T, k]       the router's weights
//   shared BF16 [G, T, D]       the shared expert's output
//   out    BF16 [G, T, D]
// For each (g, t, d): acc = 0; for s = 0..k-1 in slot order,
// acc = fma(w[t][s], y[map[t][s]][t][d], acc) in FP32 (one rounding each);
// then out = bf16(float(bf16(acc)) + float(shared)), the add in FP32 and
// both conversions round-to-nearest-even.
static uint16_t to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);  // quiet NaN
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static float bf16_value(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

int orc_gather_add(const uint16_t* y, const uint8_t* map, const float* w, const uint16_t* shared,
                   int G, int T, int k, int D, uint16_t* out) {
  if (G < 0 || T < 1 || T > 8 || k < 1 || D < 1) return -1;
  const int n = T * k;
  for (int g = 0; g < G; ++g) {
    for (int t = 0; t < T; ++t) {
      const uint8_t* mp = map + ((size_t)g * T + t) * k;
      const float* wt = w + ((size_t)g * T + t) * k;
      for (int s = 0; s < k; ++s)
        if (mp[s] >= n) return -1;
      for (int d = 0; d < D; ++d) {
        float acc = 0.0f;
        for (int s = 0; s < k; ++s) {
          const size_t row = ((size_t)g * n + mp[s]) * T + t;
          acc = std::fmaf(wt[s], bf16_value(y[row * D + d]), acc);
        }
        const float sum = bf16_value(to_bf16(acc)) + bf16_value(shared[((size_t)g * T + t) * D + d]);
        out[((size_t)g * T + t) * D + d] = to_bf16(sum);
      }
    }
  }
  return 0;
}

}  // extern "C"
