// Oracle of the quantized MoE expert layer -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, CPU reference of what the layer computes, used by the test
// suite, the smoke check and the benchmark's CPU-baseline leg to judge the
// CUDA path.  The product never links, loads or calls it; it shares no code,
// header, table or helper with the CUDA library.  Accumulation is in fp64;
// quantisation decisions are taken in fp32 (the precision the pages leave
// to the implementation), element by element, in the order the definitions
// state, with no blocking or reordering.
//
// What it follows:
//   * Weight formats: "fp6 uses six-bit e2m3 values with a power-of-two scale
//     per 128 weights; nvfp4 uses four-bit values with a scale per 16"
//     (knivesysl README, "formats"); the e4m3 block scale with an fp32 tensor
//     scale is the two-level NVFP4 recipe; the element encodings are the OCP
//     Microscaling (MX) v1.0 e2m1 / e2m3 / e4m3 / e8m0 formats.
//   * Byte-exact quantisers need correctly rounded IEEE division (Strata on an
//     Intel Arc, "The engine itself on Intel: the SYCL port", build step 4):
//     every division below is one IEEE fp32 division, round to nearest even.
//   * Router top-k and the always-on shared expert are the "router_top10" and
//     "shared_expert" kernels of that same section's parity table; "each token
//     brings its own 8 experts" (nextsycl README, "Lessons learned").
//   * The expert is a SwiGLU FFN: y = W_down (silu(W_gate x) * (W_up x)).
//
// Readings where the pages are silent (R1, R2, ...; the same labels name them in
// the design notes):
//   R1 NVFP4 tensor scale ts = amax(W) / (6 * 448), one per (expert, matrix);
//      block scale s_b = e4m3_rne((amax_b / 6) / ts); q = e2m1_rne(w / (s_b*ts)).
//   R2 blocks run along K (the reduction dimension), contiguous.
//   R3 rounding to a code grid is round-to-nearest, ties to the even code,
//      saturating at the largest finite magnitude; zero is always +0.
//   R4 an all-zero NVFP4 block (or s_b = 0) gets code 0; an all-zero FP6 block
//      gets exponent 0 (byte 127) and code 0.
//   R5 FP6 block exponent E_b = the smallest integer with amax_b <= 7.5 * 2^E_b.
//   R6 dequantised weight = (value(code) * value(block scale)) * ts, in fp32.
//   R7 router logit = fp32(sum_h x_h * Wr_eh in fp64) + bias_e (fp32 add).
//   R8 softmax over all E logits, top-k by probability (ties -> lower expert
//      index), renormalised over the k selected (fp64, rounded to fp32).
//   R9 dispatch order: expert-major, then token, then rank j (stable).
//   R10 shared expert: always on, weight 1, same format and I as the routed.
//   R11 output = fp32(sum_j g_j * y_j + y_shared), summed in fp64.
//   R19 optional sigmoid router: s_e = sigmoid(x . Wr_e), top-k by s_e + b_e (the
//      bias selects only), gates s_j / sum of the picked s.
//   R20 W4A4 (optional, act_fp4): the activations of each product are quantised
//      to NVFP4 too, per row with the weight recipe (R1, R3, R4, R6): x of a
//      token before gate/up, and a = silu(g) * u, rounded to fp32, per
//      (token, expert) row before down; the products then take the dequantised
//      values.
//   R17 MXFP4 (OCP MX v1.0 FP4): blocks of 32 along K share an e8m0 scale
//      X = 2^(floor(log2 amax_b) - 2) (2 = the largest e2m1 exponent), clamped
//      to [2^-127, 2^127]; q = e2m1_rne(w / X), saturating at 6; an all-zero
//      block gets X = 2^0 (byte 127) and code 0; value = value(q) * X.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------- code values
// OCP MX element encodings, written from their definition:
//   value = (-1)^s * 2^(e - bias) * (1 + m / 2^M)   for e > 0
//   value = (-1)^s * 2^(1 - bias) * (m / 2^M)       for e = 0 (subnormal)

double e2m1_value(int code) {  // s | e1 e0 | m0, bias 1
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? std::ldexp(m / 2.0, 0) : std::ldexp(1.0 + m / 2.0, e - 1);
  return s ? -mag : mag;
}

double e2m3_value(int code) {  // s | e1 e0 | m2 m1 m0, bias 1
  int s = (code >> 5) & 1, e = (code >> 3) & 3, m = code & 7;
  double mag = (e == 0) ? std::ldexp(m / 8.0, 0) : std::ldexp(1.0 + m / 8.0, e - 1);
  return s ? -mag : mag;
}

double e4m3_value(int code) {  // s | e3..e0 | m2 m1 m0, bias 7; S.1111.111 is NaN, no infinities
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return std::nan("");
  double mag = (e == 0) ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

double ue8m0_value(int b) {  // unsigned exponent, bias 127; 0xFF is NaN
  if (b == 255) return std::nan("");
  return std::ldexp(1.0, b - 127);
}

// Nearest of the non-negative codes 0..n-1 of a monotone grid (mag(c)),
// ties to the even code; values past the largest magnitude saturate to it.
template <class F>
int nearest_code(double v, int n, F mag) {
  int best = 0;
  double bd = std::fabs(v - mag(0));
  for (int c = 1; c < n; ++c) {
    double d = std::fabs(v - mag(c));
    if (d < bd || (d == bd && (c % 2 == 0))) {
      best = c;
      bd = d;
    }
  }
  return best;
}

int e2m1_rne(float v) {  // signed; returns the 4-bit code (never -0)
  int c = nearest_code(std::fabs((double)v), 8, [](int k) { return e2m1_value(k); });
  return (v < 0 && c != 0) ? (c | 8) : c;
}

int e2m3_rne(float v) {  // signed; returns the 6-bit code (never -0)
  int c = nearest_code(std::fabs((double)v), 32, [](int k) { return e2m3_value(k); });
  return (v < 0 && c != 0) ? (c | 32) : c;
}

int e4m3_rne(float v) {  // v >= 0; codes 0..0x7E (0x7F is NaN)
  return nearest_code((double)v, 127, [](int k) { return e4m3_value(k); });
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------- exported code tables
double orc_e2m1_value(int code) { return e2m1_value(code & 15); }
double orc_e2m3_value(int code) { return e2m3_value(code & 63); }
double orc_e4m3_value(int code) { return e4m3_value(code & 255); }
double orc_ue8m0_value(int b) { return ue8m0_value(b & 255); }
int orc_e2m1_rne(float v) { return e2m1_rne(v); }
int orc_e2m3_rne(float v) { return e2m3_rne(v); }
int orc_e4m3_rne(float v) { return e4m3_rne(v); }

// ---------------------------------------------------------------- quantisers
// NVFP4, readings R1-R4.  W [rows x K] fp32 row-major, K % 16 == 0.
// codes [rows x K/2]: two e2m1 codes per byte, the even column in the low nibble.
// scales [rows x K/16]: e4m3 bytes.  *tscale: the fp32 tensor scale.
int orc_quantize_nvfp4(const float* W, int rows, int K, uint8_t* codes, uint8_t* scales,
                       float* tscale) {
  if (rows <= 0 || K <= 0 || K % 16 != 0) return -1;
  float A = 0.0f;
  for (long i = 0; i < (long)rows * K; ++i) A = std::max(A, std::fabs(W[i]));
  const float ts = (A > 0.0f) ? A / 2688.0f : 0.0f;  // 2688 = 6 * 448
  *tscale = ts;
  for (int r = 0; r < rows; ++r) {
    for (int b = 0; b < K / 16; ++b) {
      const float* w = W + (long)r * K + b * 16;
      float amax = 0.0f;
      for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(w[i]));
      int s = 0;
      if (ts > 0.0f) {
        float sv = (amax / 6.0f) / ts;
        s = e4m3_rne(sv);
      }
      scales[(long)r * (K / 16) + b] = (uint8_t)s;
      const float sval = (float)e4m3_value(s);
      for (int i = 0; i < 16; ++i) {
        int q = 0;
        if (s != 0) {
          float denom = sval * ts;
          q = e2m1_rne(w[i] / denom);
        }
        long col = (long)b * 16 + i;
        uint8_t& byte = codes[(long)r * (K / 2) + col / 2];
        if (col % 2 == 0)
          byte = (uint8_t)q;
        else
          byte = (uint8_t)(byte | (q << 4));
      }
    }
  }
  return 0;
}

// FP6 e2m3 with a power-of-two block scale, readings R2-R5.  K % 128 == 0.
// codes [rows x K]: one 6-bit code per byte.  exps [rows x K/128]: ue8m0 bytes.
int orc_quantize_fp6(const float* W, int rows, int K, uint8_t* codes, uint8_t* exps) {
  if (rows <= 0 || K <= 0 || K % 128 != 0) return -1;
  for (int r = 0; r < rows; ++r) {
    for (int b = 0; b < K / 128; ++b) {
      const float* w = W + (long)r * K + b * 128;
      float amax = 0.0f;
      for (int i = 0; i < 128; ++i) amax = std::max(amax, std::fabs(w[i]));
      int E = 0;
      if (amax > 0.0f) {
        E = -127;
        while (std::ldexp(7.5, E) < (double)amax) ++E;  // smallest E with amax <= 7.5 * 2^E
        if (E > 127) return -2;
      }
      exps[(long)r * (K / 128) + b] = (uint8_t)(E + 127);
      for (int i = 0; i < 128; ++i) {
        // w / 2^E is exact; the grid decision is taken on that exact value
        double v = (amax > 0.0f) ? std::ldexp((double)w[i], -E) : 0.0;
        codes[(long)r * K + b * 128 + i] = (uint8_t)e2m3_rne((float)v);
      }
    }
  }
  return 0;
}

// MXFP4, reading R17.  K % 32 == 0.  codes [rows x K/2] as for NVFP4;
// exps [rows x K/32]: ue8m0 bytes.
int orc_quantize_mxfp4(const float* W, int rows, int K, uint8_t* codes, uint8_t* exps) {
  if (rows <= 0 || K <= 0 || K % 32 != 0) return -1;
  for (int r = 0; r < rows; ++r) {
    for (int b = 0; b < K / 32; ++b) {
      const float* w = W + (long)r * K + b * 32;
      float amax = 0.0f;
      for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(w[i]));
      int E = 0;
      if (amax > 0.0f) {
        int e2;
        std::frexp((double)amax, &e2);  // amax = f * 2^e2, f in [0.5, 1): floor(log2 amax) = e2 - 1
        E = std::min(127, std::max(-127, e2 - 1 - 2));
      }
      exps[(long)r * (K / 32) + b] = (uint8_t)(E + 127);
      for (int i = 0; i < 32; ++i) {
        // w / 2^E is exact; the grid decision is taken on that exact value
        const double v = (amax > 0.0f) ? std::ldexp((double)w[i], -E) : 0.0;
        const int q = e2m1_rne((float)v);
        const long col = (long)b * 32 + i;
        uint8_t& byte = codes[(long)r * (K / 2) + col / 2];
        if (col % 2 == 0)
          byte = (uint8_t)q;
        else
          byte = (uint8_t)(byte | (q << 4));
      }
    }
  }
  return 0;
}

// ---------------------------------------------------------------- dequantisers (R6)
int orc_dequant_nvfp4(const uint8_t* codes, const uint8_t* scales, float tscale, int rows, int K,
                      float* out) {
  if (K % 16 != 0) return -1;
  for (int r = 0; r < rows; ++r)
    for (int c = 0; c < K; ++c) {
      uint8_t byte = codes[(long)r * (K / 2) + c / 2];
      int q = (c % 2 == 0) ? (byte & 15) : (byte >> 4);
      float cs = (float)(e2m1_value(q) * e4m3_value(scales[(long)r * (K / 16) + c / 16]));
      out[(long)r * K + c] = cs * tscale;
    }
  return 0;
}

int orc_dequant_mxfp4(const uint8_t* codes, const uint8_t* exps, int rows, int K, float* out) {
  if (K % 32 != 0) return -1;
  for (int r = 0; r < rows; ++r)
    for (int c = 0; c < K; ++c) {
      uint8_t byte = codes[(long)r * (K / 2) + c / 2];
      int q = (c % 2 == 0) ? (byte & 15) : (byte >> 4);
      double v = e2m1_value(q) * ue8m0_value(exps[(long)r * (K / 32) + c / 32]);
      out[(long)r * K + c] = (float)v;
    }
  return 0;
}

int orc_dequant_fp6(const uint8_t* codes, const uint8_t* exps, int rows, int K, float* out) {
  if (K % 128 != 0) return -1;
  for (int r = 0; r < rows; ++r)
    for (int c = 0; c < K; ++c) {
      double v = e2m3_value(codes[(long)r * K + c] & 63) *
                 ue8m0_value(exps[(long)r * (K / 128) + c / 128]);
      out[(long)r * K + c] = (float)v;
    }
  return 0;
}

// ---------------------------------------------------------------- the layer
// Canonical weights of every expert matrix, indexed [expert * 3 + matrix],
// expert == E for the shared expert, matrix 0 gate [I x H], 1 up [I x H],
// 2 down [H x I].  Pointers of experts a call does not touch may be null.
struct orc_layer {
  int format;  // 1 NVFP4, 2 FP6 e2m3, 3 MXFP4
  int H, I, E, k, shared;
  const uint8_t* const* codes;
  const uint8_t* const* scales;  // e4m3 block scales (NVFP4) or ue8m0 exponents (FP6, MXFP4)
  const float* tscales;          // NVFP4 tensor scales [(E + shared) * 3]; unused otherwise
  const uint16_t* router;        // bf16 bits [E x H]
  const float* bias;             // fp32 [E] or null
  int act_fp4;                   // 1: W4A4, activations quantised to NVFP4 per row (R20)
};

}  // extern "C"

namespace {

double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// One dequantised row of an expert matrix (R6).
void dequant_row(const orc_layer& L, int expert, int matrix, int row, int K, float* out) {
  const int m = expert * 3 + matrix;
  if (L.format == 1) {
    const uint8_t* c = L.codes[m] + (long)row * (K / 2);
    const uint8_t* s = L.scales[m] + (long)row * (K / 16);
    orc_dequant_nvfp4(c, s, L.tscales[m], 1, K, out);
  } else if (L.format == 3) {
    const uint8_t* c = L.codes[m] + (long)row * (K / 2);
    const uint8_t* s = L.scales[m] + (long)row * (K / 32);
    orc_dequant_mxfp4(c, s, 1, K, out);
  } else {
    const uint8_t* c = L.codes[m] + (long)row * K;
    const uint8_t* s = L.scales[m] + (long)row * (K / 128);
    orc_dequant_fp6(c, s, 1, K, out);
  }
}

// R20: one activation row (fp32 values) through the NVFP4 recipe and back.
void act_fp4_row(std::vector<double>& v) {
  const int K = (int)v.size();
  std::vector<float> f((size_t)K), back((size_t)K);
  std::vector<uint8_t> codes((size_t)K / 2), scales((size_t)K / 16);
  for (int i = 0; i < K; ++i) f[i] = (float)v[i];
  float ts = 0.f;
  orc_quantize_nvfp4(f.data(), 1, K, codes.data(), scales.data(), &ts);
  orc_dequant_nvfp4(codes.data(), scales.data(), ts, 1, K, back.data());
  for (int i = 0; i < K; ++i) v[i] = (double)back[i];
}

// y[h] = sum_i Wd'[h,i] * a_i with a_i = silu(g_i) * u_i, g = Wg' x, u = Wu' x (fp64).
void expert_ffn(const orc_layer& L, int expert, const double* x_in, double* y) {
  const int H = L.H, I = L.I;
  std::vector<float> row((size_t)std::max(H, I));
  std::vector<double> a((size_t)I), xq(x_in, x_in + H);
  if (L.act_fp4) act_fp4_row(xq);
  const double* x = xq.data();
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    dequant_row(L, expert, 0, i, H, row.data());
    for (int h = 0; h < H; ++h) g += (double)row[h] * x[h];
    dequant_row(L, expert, 1, i, H, row.data());
    for (int h = 0; h < H; ++h) u += (double)row[h] * x[h];
    double silu = g / (1.0 + std::exp(-g));
    a[i] = silu * u;
  }
  if (L.act_fp4) act_fp4_row(a);
  for (int h = 0; h < H; ++h) {
    dequant_row(L, expert, 2, h, I, row.data());
    double acc = 0.0;
    for (int i = 0; i < I; ++i) acc += (double)row[i] * a[i];
    y[h] = acc;
  }
}

template <class F>
void parallel_for(int n, int threads, F f) {
  if (threads <= 1 || n <= 1) {
    for (int i = 0; i < n; ++i) f(i);
    return;
  }
  std::vector<std::thread> pool;
  for (int t = 0; t < threads; ++t)
    pool.emplace_back([&, t] {
      for (int i = t; i < n; i += threads) f(i);
    });
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// R7: logits [T x E] fp32.
int orc_router_logits(const orc_layer* L, const uint16_t* x, int T, float* logits) {
  const int H = L->H, E = L->E;
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h)
        acc += bf16_value(x[(long)t * H + h]) * bf16_value(L->router[(long)e * H + h]);
      float l = (float)acc;
      if (L->bias) l = l + L->bias[e];
      logits[(long)t * E + e] = l;
    }
  return 0;
}

// R8: softmax over all E, top-k by probability, renormalised over the k.
int orc_topk_gates(const float* logits, int T, int E, int k, int32_t* idx, float* gates) {
  if (k < 1 || k > E) return -1;
  std::vector<double> p((size_t)E);
  std::vector<int> order((size_t)E);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (long)t * E;
    double mx = l[0];
    for (int e = 1; e < E; ++e) mx = std::max(mx, (double)l[e]);
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += std::exp((double)l[e] - mx);
    for (int e = 0; e < E; ++e) p[e] = std::exp((double)l[e] - mx) / z;
    for (int e = 0; e < E; ++e) order[e] = e;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return p[a] > p[b]; });
    double s = 0.0;
    for (int j = 0; j < k; ++j) s += p[order[j]];
    for (int j = 0; j < k; ++j) {
      idx[(long)t * k + j] = order[j];
      gates[(long)t * k + j] = (float)(p[order[j]] / s);
    }
  }
  return 0;
}

// R19: the sigmoid router with a selection bias.  logits are x . Wr_e without
// the bias; s_e = 1 / (1 + exp(-l_e)); the k experts with the largest
// s_e + b_e (ties -> lower index) are picked, the bias deciding the
// selection only; g_j = s_j / (sum of the picked s), in fp64, rounded to fp32.
int orc_topk_gates_sigmoid(const float* logits, const float* bias, int T, int E, int k,
                           int32_t* idx, float* gates) {
  if (k < 1 || k > E) return -1;
  std::vector<double> s((size_t)E), key((size_t)E);
  std::vector<int> order((size_t)E);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (long)t * E;
    for (int e = 0; e < E; ++e) {
      s[e] = 1.0 / (1.0 + std::exp(-(double)l[e]));
      key[e] = s[e] + (bias ? (double)bias[e] : 0.0);
      order[e] = e;
    }
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return key[a] > key[b]; });
    double z = 0.0;
    for (int j = 0; j < k; ++j) z += s[order[j]];
    for (int j = 0; j < k; ++j) {
      idx[(long)t * k + j] = order[j];
      gates[(long)t * k + j] = (float)(s[order[j]] / z);
    }
  }
  return 0;
}

// R9: counts [E], offsets [E + 1] (exclusive scan), perm [T*k]: slot ids
// s = t*k + j listed expert-major, then by slot id.
int orc_dispatch(const int32_t* idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
                 int32_t* perm) {
  const long S = (long)T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long s = 0; s < S; ++s) {
    if (idx[s] < 0 || idx[s] >= E) return -1;
    counts[idx[s]]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  long n = 0;
  for (int e = 0; e < E; ++e)
    for (long s = 0; s < S; ++s)
      if (idx[s] == e) perm[n++] = (int32_t)s;
  return 0;
}

// R10/R11 with the routing given: out [T x H] fp32 = sum_j gates[t,j] * y_{idx[t,j]}(x_t)
// (+ the shared expert's y when the layer has one).
int orc_combine(const orc_layer* L, const uint16_t* x, int T, const int32_t* idx,
                const float* gates, float* out, int threads) {
  const int H = L->H, k = L->k;
  parallel_for(T, threads, [&](int t) {
    std::vector<double> xt((size_t)H), y((size_t)H), acc((size_t)H, 0.0);
    for (int h = 0; h < H; ++h) xt[h] = bf16_value(x[(long)t * H + h]);
    for (int j = 0; j < k; ++j) {
      expert_ffn(*L, idx[(long)t * k + j], xt.data(), y.data());
      double g = gates[(long)t * k + j];
      for (int h = 0; h < H; ++h) acc[h] += g * y[h];
    }
    if (L->shared) {
      expert_ffn(*L, L->E, xt.data(), y.data());
      for (int h = 0; h < H; ++h) acc[h] += y[h];
    }
    for (int h = 0; h < H; ++h) out[(long)t * H + h] = (float)acc[h];
  });
  return 0;
}

// The whole layer: router logits, softmax / top-k / renormalise, experts, combine.
int orc_moe_forward(const orc_layer* L, const uint16_t* x, int T, float* logits, int32_t* idx,
                    float* gates, float* out, int threads) {
  int rc = orc_router_logits(L, x, T, logits);
  if (rc) return rc;
  rc = orc_topk_gates(logits, T, L->E, L->k, idx, gates);
  if (rc) return rc;
  return orc_combine(L, x, T, idx, gates, out, threads);
}

// One expert's SwiGLU FFN for T tokens: y [T x H] (fp64 accumulate, fp32 out).
int orc_expert_ffn(const orc_layer* L, int expert, const uint16_t* x, int T, float* y) {
  std::vector<double> xt((size_t)L->H), yt((size_t)L->H);
  for (int t = 0; t < T; ++t) {
    for (int h = 0; h < L->H; ++h) xt[h] = bf16_value(x[(long)t * L->H + h]);
    expert_ffn(*L, expert, xt.data(), yt.data());
    for (int h = 0; h < L->H; ++h) y[(long)t * L->H + h] = (float)yt[h];
  }
  return 0;
}

}  // extern "C"
