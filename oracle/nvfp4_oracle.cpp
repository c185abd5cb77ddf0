// NVFP4 rollout-linear oracle: TEST INFRASTRUCTURE, not part of the product.
//
// Only the tests, the smoke check and the benchmark's CPU-baseline leg load this
// library. It is a plain, slow, single-threaded CPU restatement of what the
// GPU path computes, written from the definitions, and shares no code, header,
// table or constant with the CUDA sources.
//
// Sources of each definition:
//  * NVFP4 format: 4-bit E2M1 values on the grid {0, .5, 1, 1.5, 2, 3, 4, 6} that
//    share a per-block scale (QeRL explainer, section "NVFP4量子化とLoRA"; TRACE
//    summary, section "仕組みの工学的な理解": a few values share one scale, each
//    value is 4 bits). The block is 16 elements, the block scale is an E4M3 byte
//    equal to RNE(block_amax / 6 / g), and g = tensor_amax / (6 * 448) is an fp32
//    per-tensor scale (the benchmark spec of the recipe).
//  * Rounding direction as a per-value choice between the two neighbouring grid
//    points (TRACE summary, same section; "rollout-guided QAT" and the cache of
//    mantissa information, section "TRACE の中心的なアイデア").
//  * AQN: RMSNorm whose weight is w + z, z a Gaussian per-channel noise vector
//    (QeRL explainer, section "ゼロオーバーヘッド：レイヤー正規化への統合"), with
//    an exponential noise schedule (section "AQNの仕組み").
//  * LoRA linear: Y = x deq(W)^T + s (x A^T) B^T (QeRL explainer, section
//    "NVFP4量子化とLoRA": frozen quantized base plus low-rank trainable factors).
//  * FP4 KV cache (TRACE summary, section "実験結果と性能": rollouts with FP4 weights,
//    activations and KV cache): every cached key/value row of a head is NVFP4-encoded
//    like any tensor (16-element blocks along the head dimension, E4M3 block scales)
//    with a per-tensor g given by the caller, and decode attention reads the dequantized
//    rows: out = softmax(scale q K^T) V over the sequence's cached tokens, query head h
//    reading KV head h / (Hq / Hkv) (grouped-query attention).
//  * AIS mixing coefficient (AIS summary, section 2.1 "混合係数": alpha_ess from the
//    coefficient of variation of the truncated weights, alpha_mis from the mean
//    absolute log-prob mismatch and a saturation threshold delta, alpha_var from a
//    variance amplification ratio and a tolerance gamma, alpha = clip(alpha_ess -
//    beta alpha_var, 0, 1) alpha_mis; section 2.2: the rectified weight
//    w~ = 1 + alpha (min(rho, C) - 1)).
//
// Readings taken where the definition leaves a step open:
//  * Both roundings (the E4M3 block scale and the E2M1 element code) apply to the
//    exact real quotient: the scale byte is the E4M3 value nearest to
//    bamax / (6 g), the code is the grid point nearest to x / (dec(s) g), ties to
//    the even encoding, both saturating at the largest finite value.
//    Each decision is taken by comparing the input against an exact midpoint
//    times the exact divisor, all in double, where every such product is exact
//    (at most 31 significant bits).
//  * g is the fp32 quotient amax / 2688 rounded to nearest (one IEEE division).
//  * Signs are kept, also on zero codes (-0.1 in a block of large values -> 0x8).
//  * A block whose scale byte is 0 (and every block when g == 0) gets codes
//    sign|0.
//  * Guided rounding: with a = |x| / (dec(s) g): a >= 6 gives 6; an exact grid
//    point is kept; otherwise mask bit 1 takes the larger-magnitude neighbour and
//    bit 0 the smaller one. The scale byte is the plain one.
//  * Recording (the rollout side of TRACE, section "仕組みの工学的な理解": the
//    rollout engine quantizes and keeps a record of the result, which the training
//    side later consults to take the same rounding decisions): the record bit of an
//    element is 1 when the plain code's magnitude exceeds |x| / S (the value was
//    rounded up in magnitude) and 0 otherwise (rounded down, on the grid, saturated,
//    or a zero scale). Guided rounding with that mask gives the plain codes back.
//  * AIS readings: one importance ratio per token, rho = exp(logp_train - logp_rollout)
//    (training over rollout probability of the sampled token); w = min(rho, C); the
//    CV, means and standard deviations are over the batch's N tokens with weight 1/N
//    (population statistics); the variance amplification Delta sigma is the relative
//    growth of the advantages' spread under the weights, std(w * A) / std(A) - 1 with A
//    the per-token advantage (0 when the weights are all 1, so that a batch without
//    mismatch is not penalised), and 0 when std(A) = 0.
//  * Replay from the cache (section "TRACE の中心的なアイデア": the scale information
//    is kept with the rounding bits): codes are the guided codes against the recorded
//    scale byte and g, with no amax and no scale search. A recorded byte above 0x7E
//    (the quantizer never writes one) is read as 0x7E; g <= 0 or NaN gives sign|0.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

const double kGrid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double e2m1_value(int code) {
  const double m = kGrid[code & 7];
  return (code & 8) ? -m : m;
}

// OCP FP8 E4M3 ("E4M3FN"): sign, 4 exponent bits (bias 7), 3 mantissa bits,
// subnormals m/8 * 2^-6, no infinities, S.1111.111 is NaN.
double e4m3_value(int byte) {
  const int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
  if (e == 15 && m == 7) return NAN;
  const double v = (e == 0) ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

// Non-negative E4M3 byte nearest to num / den (num >= 0, den > 0), ties to the
// even byte, saturating to 0x7E (448). Walks the 127 finite values upward.
int e4m3_encode_ratio(double num, double den) {
  if (num >= 448.0 * den) return 0x7E;
  for (int b = 0; b < 0x7E; ++b) {
    const double mid = 0.5 * (e4m3_value(b) + e4m3_value(b + 1));
    const double t = mid * den;
    if (num < t) return b;
    if (num == t) return (b & 1) ? b + 1 : b;
  }
  return 0x7E;
}

// E2M1 code of x for the real scale S = dec(s) * g: sign bit, then the grid
// index nearest to |x| / S, ties to the even index, saturating at 7.
int e2m1_encode(double x, double S) {
  const int sign = std::signbit(x) ? 8 : 0;
  if (S == 0.0) return sign;
  const double a = std::fabs(x);
  for (int k = 0; k < 7; ++k) {
    const double t = 0.5 * (kGrid[k] + kGrid[k + 1]) * S;
    if (a < t) return sign | k;
    if (a == t) return sign | ((k & 1) ? k + 1 : k);
  }
  return sign | 7;
}

// Guided E2M1 code: `up` selects the larger-magnitude neighbour of |x| / S.
int e2m1_encode_guided(double x, double S, int up) {
  const int sign = std::signbit(x) ? 8 : 0;
  if (S == 0.0) return sign;
  const double a = std::fabs(x);
  if (a >= 6.0 * S) return sign | 7;
  int k = 0;
  while (k < 7 && kGrid[k + 1] * S <= a) ++k;
  if (a == kGrid[k] * S) return sign | k;
  return sign | (up ? k + 1 : k);
}

// Record bit of x under the real scale S: 1 when the plain code rounds |x| / S up
// in magnitude.
int e2m1_round_up(double x, double S) {
  if (S == 0.0) return 0;
  const int c = e2m1_encode(x, S);
  return kGrid[c & 7] * S > std::fabs(x) ? 1 : 0;
}

double load_elem(const void* x, int dtype, int64_t i) {
  if (dtype == 0) {  // bf16 bit pattern
    const uint32_t u = static_cast<uint32_t>(static_cast<const uint16_t*>(x)[i]) << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
  }
  return static_cast<const float*>(x)[i];
}

double bf16_value(uint16_t b) {
  const uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

void quantize_rows(const void* x, int dtype, int64_t cols, int64_t row0, int64_t row1, float g,
                   const uint32_t* mask, uint8_t* codes, uint8_t* scales, uint32_t* record = nullptr) {
  const int64_t nblk = cols / 16;
  for (int64_t r = row0; r < row1; ++r) {
    for (int64_t b = 0; b < nblk; ++b) {
      const int64_t base = r * cols + b * 16;
      double bamax = 0.0;
      for (int i = 0; i < 16; ++i) bamax = std::fmax(bamax, std::fabs(load_elem(x, dtype, base + i)));
      const int s = (g == 0.0f) ? 0 : e4m3_encode_ratio(bamax, 6.0 * static_cast<double>(g));
      scales[r * nblk + b] = static_cast<uint8_t>(s);
      const double S = e4m3_value(s) * static_cast<double>(g);
      for (int i = 0; i < 16; ++i) {
        const int64_t idx = base + i;
        const double v = load_elem(x, dtype, idx);
        int c;
        if (mask) {
          const int up = (mask[idx / 32] >> (idx % 32)) & 1;
          c = e2m1_encode_guided(v, S, up);
        } else {
          c = e2m1_encode(v, S);
        }
        if (record) {
          const uint32_t bit = static_cast<uint32_t>(e2m1_round_up(v, S)) << (idx % 32);
          record[idx / 32] = (record[idx / 32] & ~(1u << (idx % 32))) | bit;
        }
        uint8_t& byte = codes[idx / 2];
        if ((idx & 1) == 0) byte = static_cast<uint8_t>((byte & 0xF0) | c);
        else byte = static_cast<uint8_t>((byte & 0x0F) | (c << 4));
      }
    }
  }
}

}  // namespace

extern "C" {

double oracle_e2m1_value(int code) { return e2m1_value(code); }
double oracle_e4m3_value(int byte) { return e4m3_value(byte); }
int oracle_e4m3_encode_ratio(double num, double den) { return e4m3_encode_ratio(num, den); }
int oracle_e2m1_encode(double x, double S) { return e2m1_encode(x, S); }
int oracle_e2m1_encode_guided(double x, double S, int up) { return e2m1_encode_guided(x, S, up); }

// max |x_i| over [i0, i1); dtype 0 = bf16 bits, 1 = fp32.
float oracle_amax(const void* x, int dtype, int64_t i0, int64_t i1) {
  double m = 0.0;
  for (int64_t i = i0; i < i1; ++i) m = std::fmax(m, std::fabs(load_elem(x, dtype, i)));
  return static_cast<float>(m);
}

// g = amax / (6 * 448), one fp32 division rounded to nearest.
float oracle_global_scale(float amax) { return amax / 2688.0f; }

// Rows [row0, row1) of the NVFP4 encoding of x (rows x cols, cols % 16 == 0)
// with per-tensor scale g. codes: rows x cols/2 bytes, element 2j in the low
// nibble of byte j; scales: rows x cols/16 E4M3 bytes.
void oracle_quantize_rows(const void* x, int dtype, int64_t cols, int64_t row0, int64_t row1, float g,
                          uint8_t* codes, uint8_t* scales) {
  quantize_rows(x, dtype, cols, row0, row1, g, nullptr, codes, scales);
}

// Same with the rounding direction of every non-grid element taken from
// mask bit (i % 32) of word i / 32, i the flat row-major element index.
void oracle_quantize_guided_rows(const void* x, int dtype, int64_t cols, int64_t row0, int64_t row1,
                                 float g, const uint32_t* mask, uint8_t* codes, uint8_t* scales) {
  quantize_rows(x, dtype, cols, row0, row1, g, mask, codes, scales);
}

// Plain encoding of rows [row0, row1) as oracle_quantize_rows, and the record bit of every
// element written to bit (i % 32) of record[i / 32], i the flat row-major index.
void oracle_quantize_record_rows(const void* x, int dtype, int64_t cols, int64_t row0, int64_t row1, float g,
                                 uint8_t* codes, uint8_t* scales, uint32_t* record) {
  quantize_rows(x, dtype, cols, row0, row1, g, nullptr, codes, scales, record);
}

int oracle_e2m1_round_up(double x, double S) { return e2m1_round_up(x, S); }

// Codes of rows [row0, row1) from a cache: scale byte scales[r * cols/16 + b] and g as
// recorded, rounding direction from the mask (same layout as the guided encoding).
void oracle_quantize_cached_rows(const void* x, int dtype, int64_t cols, int64_t row0, int64_t row1, float g,
                                 const uint8_t* scales, const uint32_t* mask, uint8_t* codes) {
  const int64_t nblk = cols / 16;
  for (int64_t r = row0; r < row1; ++r)
    for (int64_t b = 0; b < nblk; ++b) {
      const int s = scales[r * nblk + b] > 0x7E ? 0x7E : scales[r * nblk + b];
      const double S = (g > 0.0f) ? e4m3_value(s) * static_cast<double>(g) : 0.0;
      for (int i = 0; i < 16; ++i) {
        const int64_t idx = r * cols + b * 16 + i;
        const int up = (mask[idx / 32] >> (idx % 32)) & 1;
        const int c = e2m1_encode_guided(load_elem(x, dtype, idx), S, up);
        uint8_t& byte = codes[idx / 2];
        if ((idx & 1) == 0) byte = static_cast<uint8_t>((byte & 0xF0) | c);
        else byte = static_cast<uint8_t>((byte & 0x0F) | (c << 4));
      }
    }
}

// deq(code, s, g) = e2m1(code) * e4m3(s) * g, exact in double; rows [row0, row1).
void oracle_dequantize_rows(const uint8_t* codes, const uint8_t* scales, float g, int64_t cols,
                            int64_t row0, int64_t row1, double* out) {
  const int64_t nblk = cols / 16;
  for (int64_t r = row0; r < row1; ++r)
    for (int64_t k = 0; k < cols; ++k) {
      const int64_t idx = r * cols + k;
      const int c = (codes[idx / 2] >> ((idx & 1) * 4)) & 15;
      out[idx] = e2m1_value(c) * e4m3_value(scales[r * nblk + k / 16]) * static_cast<double>(g);
    }
}

// Decode attention over an NVFP4 KV cache, in fp64. q: [B][Hq][D] bf16 bits; caches: codes
// [B][Lmax][Hkv][D/2], scales [B][Lmax][Hkv][D/16] for K and V, with per-tensor scales gk, gv;
// lens[b] tokens of sequence b are attended (0 < lens[b] <= Lmax); out: [B][Hq][D] doubles.
void oracle_attention_decode(const uint16_t* q, const uint8_t* kc, const uint8_t* ks, float gk, const uint8_t* vc,
                             const uint8_t* vs, float gv, const int32_t* lens, int64_t B, int64_t Hq, int64_t Hkv,
                             int64_t D, int64_t Lmax, double scale, double* out) {
  const int64_t group = Hq / Hkv;
  const auto deq = [&](const uint8_t* codes, const uint8_t* scales, float g, int64_t row, int64_t d) {
    const int c = (codes[row * (D / 2) + d / 2] >> ((d & 1) * 4)) & 15;
    return e2m1_value(c) * e4m3_value(scales[row * (D / 16) + d / 16]) * static_cast<double>(g);
  };
  for (int64_t b = 0; b < B; ++b)
    for (int64_t h = 0; h < Hq; ++h) {
      const int64_t kvh = h / group, L = lens[b];
      std::vector<double> sc(L);
      double mx = -INFINITY;
      for (int64_t t = 0; t < L; ++t) {
        const int64_t row = (b * Lmax + t) * Hkv + kvh;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d) dot += bf16_value(q[(b * Hq + h) * D + d]) * deq(kc, ks, gk, row, d);
        sc[t] = scale * dot;
        mx = std::fmax(mx, sc[t]);
      }
      double den = 0.0;
      for (int64_t t = 0; t < L; ++t) {
        sc[t] = std::exp(sc[t] - mx);
        den += sc[t];
      }
      for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t t = 0; t < L; ++t) acc += sc[t] * deq(vc, vs, gv, (b * Lmax + t) * Hkv + kvh, d);
        out[(b * Hq + h) * D + d] = acc / den;
      }
    }
}

// AIS over a batch of n tokens. stats (8 doubles): alpha, alpha_ess, alpha_mis, alpha_var,
// the mean |logp_train - logp_rollout|, CV^2 of the truncated weights, Delta sigma, and mean(w). w_out (n doubles, may be null): the rectified weights.
void oracle_ais(int64_t n, const float* logp_rollout, const float* logp_train, const float* adv, double C,
                double delta, double gamma, double beta, double* stats, double* w_out) {
  if (n <= 0) return;
  std::vector<double> w(n);
  double sum_d = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    const double d = static_cast<double>(logp_train[i]) - static_cast<double>(logp_rollout[i]);
    sum_d += std::fabs(d);
    w[i] = std::fmin(std::exp(d), C);
  }
  const double N = static_cast<double>(n);
  double mw = 0.0, ma = 0.0, mwa = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    mw += w[i];
    ma += adv[i];
    mwa += w[i] * adv[i];
  }
  mw /= N;
  ma /= N;
  mwa /= N;
  double vw = 0.0, va = 0.0, vwa = 0.0;  // two-pass population variances
  for (int64_t i = 0; i < n; ++i) {
    vw += (w[i] - mw) * (w[i] - mw);
    va += (adv[i] - ma) * (adv[i] - ma);
    vwa += (w[i] * adv[i] - mwa) * (w[i] * adv[i] - mwa);
  }
  vw /= N;
  va /= N;
  vwa /= N;
  const double cv2 = vw / (mw * mw);
  const double a_ess = 1.0 / std::sqrt(1.0 + cv2);
  const double dbar = sum_d / N;
  const double a_mis = std::fmin(1.0, dbar / delta);
  const double amp = va > 0.0 ? std::sqrt(vwa) / std::sqrt(va) - 1.0 : 0.0;
  const double a_var = std::fmax(0.0, (amp - gamma) / gamma);
  const double alpha = std::fmin(1.0, std::fmax(0.0, a_ess - beta * a_var)) * a_mis;
  stats[0] = alpha;
  stats[1] = a_ess;
  stats[2] = a_mis;
  stats[3] = a_var;
  stats[4] = dbar;
  stats[5] = cv2;
  stats[6] = amp;
  stats[7] = mw;
  if (w_out)
    for (int64_t i = 0; i < n; ++i) w_out[i] = 1.0 + alpha * (w[i] - 1.0);
}

// AQN noise schedule: sigma_k = sigma0 * (sigmaK / sigma0)^(k / K).
double oracle_aqn_sigma(double sigma0, double sigmaK, int64_t k, int64_t K) {
  return sigma0 * std::pow(sigmaK / sigma0, static_cast<double>(k) / static_cast<double>(K));
}

// Rows [row0, row1) of y = (w + sigma * eps) * x / sqrt(mean_j x_j^2 + delta), in double.
// x: M x H bf16 bits; w, eps: H fp32 (eps may be null: no noise).
void oracle_rmsnorm_aqn_rows(const uint16_t* x, int64_t H, int64_t row0, int64_t row1, const float* w,
                             const float* eps, float sigma, float delta, double* y) {
  for (int64_t m = row0; m < row1; ++m) {
    double ss = 0.0;
    for (int64_t j = 0; j < H; ++j) {
      const double v = bf16_value(x[m * H + j]);
      ss += v * v;
    }
    const double inv = 1.0 / std::sqrt(ss / static_cast<double>(H) + static_cast<double>(delta));
    for (int64_t j = 0; j < H; ++j) {
      const double z = eps ? static_cast<double>(sigma) * static_cast<double>(eps[j]) : 0.0;
      y[m * H + j] = (static_cast<double>(w[j]) + z) * bf16_value(x[m * H + j]) * inv;
    }
  }
}

// LoRA down-projection U = xl A^T: xl nrows x K (double), A r x K bf16 bits, U nrows x r.
void oracle_lora_down(const double* xl, int64_t nrows, int64_t K, const uint16_t* A, int32_t r, double* U) {
  for (int64_t m = 0; m < nrows; ++m)
    for (int32_t j = 0; j < r; ++j) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += xl[m * K + k] * bf16_value(A[j * K + k]);
      U[m * r + j] = acc;
    }
}

// Columns [n0, n1) of Y = xq deq(W)^T + s U B^T, Y nrows x N (double).
// xq: nrows x K (double) operand of the base GEMM; W: N x K NVFP4 (codes, scales, g);
// U: nrows x r from oracle_lora_down (ignored when r == 0); B: N x r bf16 bits.
void oracle_linear_cols(const double* xq, int64_t nrows, int64_t K, const uint8_t* codes,
                        const uint8_t* scales, float g, int64_t N, int64_t n0, int64_t n1,
                        const double* U, const uint16_t* B, int32_t r, double s, double* Y) {
  std::vector<double> wrow(static_cast<size_t>(K));
  for (int64_t n = n0; n < n1; ++n) {
    for (int64_t k = 0; k < K; ++k) {
      const int64_t idx = n * K + k;
      const int c = (codes[idx / 2] >> ((idx & 1) * 4)) & 15;
      wrow[k] = e2m1_value(c) * e4m3_value(scales[n * (K / 16) + k / 16]) * static_cast<double>(g);
    }
    for (int64_t m = 0; m < nrows; ++m) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += xq[m * K + k] * wrow[k];
      double lora = 0.0;
      for (int32_t j = 0; j < r; ++j) lora += U[m * r + j] * bf16_value(B[n * r + j]);
      Y[m * N + n] = acc + s * lora;
    }
  }
}

}  // extern "C"
