// fp8rl CPU oracle -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, deliberately unoptimised restatement of what the FP8 rollout
// hot path computes, used to check the CUDA library.  Only the test suite, the
// smoke check and the benchmark's CPU-baseline leg may load it; the product
// path never does.  It shares no source, header, table or constant with the
// CUDA library under fp8_precision_rollout_gb300/csrc.
//
// Sources (web pages on "FP8-RL: A Practical and Stable Low-Precision Stack
// for LLM Reinforcement Learning", arXiv 2601.18150):
//   [S341]  long-form summary, section 3.4.1 "Blockwise FP8 Quantization for
//           Linear Layers" (E4M3 format facts; the equation W_hat = round(W/scale);
//           128x128 weight blocks, 1x128 activation tiles)
//   [S342]  same page, section 3.4.2 "Dynamic Weight Synchronization Pipeline",
//           Phase 2 step 2 (scale from block max-abs, divide, round to E4M3) and
//           Phase 3 (FP8 x FP8 matmul, FP32 accumulation, BF16 output)
//   [S343]  same page, section 3.4.3 (importance weight w = pi_theta / pi_fp8,
//           truncated IS with C = 2)
//   [S344]  same page, section 3.4.4 "KV-Cache Quantization" (per-layer or
//           per-head K/V scales computed from observed K/V)
//   [OCP]   E4M3 encoding of Micikevicius et al. "FP8 Formats for Deep
//           Learning" (cited by the summary, section 2): bias 7, no infinities,
//           S.1111.111 is NaN, largest finite magnitude 448.
//
// Readings taken where the pages are silent:
//   * scale s = fl32(amax / 448) in IEEE binary32 division;
//   * quantised code = E4M3_RNE_satfinite(fl32(x / s)): two roundings, first
//     the binary32 quotient, then round-to-nearest-even into E4M3 with
//     saturation to +-448; the sign of zero is kept;
//   * an all-zero block has s = 0 and codes +-0 (0x00 / 0x80);
//   * KV scale per (tensor, head) = fl32(amax / 448) over all tokens and dims.
//
// Build: g++ -O2 -ffp-contract=off -shared -fPIC -pthread (see oracle/build.py).
// No fast-math and no FMA contraction: every float/double operation below is
// one IEEE operation, rounded to nearest-even.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------- helpers --

// Run f(lo, hi) over [0, n) split into contiguous chunks on `threads` threads.
template <class F>
void parallel_for(int64_t n, int threads, F f) {
  if (threads <= 1 || n < 2) {
    f((int64_t)0, n);
    return;
  }
  int64_t t = std::min<int64_t>(threads, n);
  std::vector<std::thread> pool;
  int64_t chunk = (n + t - 1) / t;
  for (int64_t i = 0; i < t; ++i) {
    int64_t lo = i * chunk, hi = std::min(n, lo + chunk);
    if (lo >= hi) break;
    pool.emplace_back([=] { f(lo, hi); });
  }
  for (auto& th : pool) th.join();
}

// BF16 is the upper half of a binary32: widening is exact.
float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// ------------------------------------------------------------ E4M3 codec --

// [OCP] value of an E4M3 code: sign bit, 4-bit exponent field e (bias 7),
// 3-bit mantissa field m.  e == 0 is subnormal: m * 2^-9.  e == 15, m == 7 is
// NaN (the format has no infinities).  Otherwise (1 + m/8) * 2^(e-7).
double e4m3_decode(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  if (e == 0xF && m == 0x7) return std::nan("");
  double mag = (e == 0) ? std::ldexp((double)m, -9)
                        : std::ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -mag : mag;
}

// [OCP] + [S341] "round to the nearest representable FP8 value": exact
// round-to-nearest-even of the real value |x| onto the E4M3 grid, saturating
// at 448 (so +-inf and anything that would round past 448 give +-448), sign
// kept (including the sign of zero), NaN -> 0x7F.
uint8_t e4m3_encode(float x) {
  if (std::isnan(x)) return 0x7F;
  uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  double a = std::fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;
  int code;
  if (a < std::ldexp(1.0, -6)) {
    // below the smallest normal 2^-6 the grid spacing is 2^-9; code = count
    // of quanta (8 quanta is exactly the smallest normal, code 0x08).
    double quanta = std::nearbyint(a * 512.0);  // exact scaling, then RNE
    code = (int)quanta;
  } else {
    int ex;
    std::frexp(a, &ex);        // a = f * 2^ex, f in [0.5, 1)
    int E = ex - 1;            // a in [2^E, 2^(E+1)), E in [-6, 8]
    // eighths of 2^E: in [8, 16]; 16 carries into the next binade, which the
    // code arithmetic below absorbs (mantissa 0 of exponent E+1).
    double eighths = std::nearbyint(std::ldexp(a, 3 - E));
    code = (E + 7) * 8 + (int)eighths - 8;
  }
  if (code > 0x7E) code = 0x7E;  // unreachable for a < 448; kept as a guard
  return (uint8_t)(sign | code);
}

// [S341]/[S342]: divide by the block scale in binary32, then round to E4M3.
// An all-zero block (s == 0) keeps its signed zeros.
uint8_t quantize_one(float x, float s) {
  float q = (s == 0.0f) ? x : x / s;
  return e4m3_encode(q);
}

// [S341]: the scale maps the block's largest magnitude onto 448.
float scale_from_amax(float amax) { return amax / 448.0f; }

}  // namespace


// ------------------------------------------------------- MoE glue (SiLU) --

// The MoE glue between the expert GEMMs (summary page, section 3.4.1 names
// the expert layers fc1/fc2 among the quantized linears; the pages fix no
// activation arithmetic).  Reading: the gated activation of the Qwen3 family,
//   y = BF16_RNE( silu(g) * u ),   silu(g) = g / (1 + e^-g),
// the real-number product rounded ONCE to the nearest BF16 value (ties to
// even, overflow to +-inf, underflow to a subnormal or a signed zero).  For
// finite non-zero g, silu(g) is transcendental (Lindemann), so the product is
// never exactly a rounding midpoint.  Special values follow the IEEE
// evaluation of g * sigma(g) * u: a NaN input gives NaN; silu(+inf) = +inf;
// silu(-inf) = -inf * 0 = NaN; silu(+-0) = +-0; then +-0 * inf = NaN, a
// non-zero finite silu times +-inf is +-inf, and times +-0 is a signed zero.
//
// Here the product is formed in float64 (relative error below 2^-50) and
// rounded to BF16 exactly from that value.  Inputs whose float64 value lies
// within 2^-40 (relative) of a BF16 rounding midpoint are reported to the
// caller, which decides them in 80-digit decimal arithmetic.

const uint16_t kBf16QuietNaN = 0x7FC0;

// Nearest BF16 (bit pattern) to the finite float64 x, ties to even; sets
// *hard when x is within 2^-40 (relative) of a rounding midpoint.  A value
// exactly on a midpoint with tie_dir != 0 stands for a true value just beside
// it: tie_dir > 0 rounds to the larger magnitude, tie_dir < 0 to the smaller.
uint16_t bf16_nearest(double x, int tie_dir, bool* hard) {
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0x0000;
  const double a = std::fabs(x);
  if (a == 0.0) return sign;
  if (a >= std::ldexp(1.0, 128)) return sign | 0x7F80;
  int ex;
  std::frexp(a, &ex);
  const int e = ex - 1;                        // a in [2^e, 2^(e+1))
  const int qe = (e < -126 ? -126 : e) - 7;    // spacing of BF16 values around a
  const double t = std::ldexp(a, -qe);         // exact: a in units of the spacing
  double n = std::floor(t);
  const double frac = t - n;                   // exact
  if (frac == 0.5 && tie_dir != 0) {
    if (tie_dir > 0) n += 1.0;
  } else {
    if (std::fabs(frac - 0.5) <= std::ldexp(t, -40)) *hard = true;
    if (frac > 0.5 || (frac == 0.5 && std::fmod(n, 2.0) != 0.0)) n += 1.0;
  }
  const double v = std::ldexp(n, qe);          // a BF16 value (or 2^128)
  if (v >= std::ldexp(1.0, 128)) return sign | 0x7F80;
  const float f = (float)v;                    // exact
  uint32_t b;
  std::memcpy(&b, &f, 4);
  return (uint16_t)(sign | (b >> 16));
}

// y = BF16_RNE(silu(g) * u) for BF16 inputs (bit patterns).
//
// Two families of products sit exactly on a BF16 midpoint in float64 while
// the true product does not, and their direction is known:
//   * g > 0 with e^-g below half a float64 ulp of 1: float64 gives silu = g,
//     while silu(g) = g - g e^-g / (1 + e^-g) is strictly smaller, so the
//     true |x| lies just below |g u|;
//   * |g| so small that e^-g rounds to 1: float64 gives silu = g / 2, while
//     silu(g) = g/2 + g^2/4 - ... lies strictly above g/2, so the true x lies
//     just beside (g/2) u, on the larger-magnitude side when g > 0 and the
//     smaller when g < 0.
// Any other product closer than 2^-40 to a midpoint is flagged.
uint16_t silu_mul_bf16_one(uint16_t gb, uint16_t ub, bool* hard) {
  const double g = bf16_to_float(gb), u = bf16_to_float(ub);
  if (std::isnan(g) || std::isnan(u)) return kBf16QuietNaN;
  const uint16_t sx = (std::signbit(g) != std::signbit(u)) ? 0x8000 : 0x0000;
  if (std::isinf(g)) {
    if (g < 0 || u == 0.0) return kBf16QuietNaN;
    return (uint16_t)(sx | 0x7F80);
  }
  if (g == 0.0) return std::isinf(u) ? kBf16QuietNaN : sx;
  // g finite and non-zero: silu(g) is non-zero with the sign of g
  if (std::isinf(u)) return (uint16_t)(sx | 0x7F80);
  if (u == 0.0) return sx;
  double s;
  int tie_dir = 0;
  if (g > 0) {
    const double e = std::exp(-g);
    s = g / (1.0 + e);
    if (1.0 + e == 1.0) tie_dir = -1;          // float64 silu = g; true silu < g
    else if (e == 1.0) tie_dir = +1;           // float64 silu = g/2; true silu > g/2
  } else {
    const double e = std::exp(g);              // 0 below about -745: |y| rounds to 0 there
    s = g * e / (1.0 + e);
    if (e == 1.0) tie_dir = -1;                // float64 silu = g/2; true |silu| < |g|/2
  }
  const double x = s * u;
  if (x == 0.0) return sx;                     // |x| < 2^-900: far below the smallest BF16
  return bf16_nearest(x, tie_dir, hard);
}

// binary32 -> BF16, round to nearest even (NaN stays a quiet NaN).
uint16_t float_to_bf16(float f) {
  uint32_t b;
  std::memcpy(&b, &f, 4);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((b >> 16) | 0x0040u);
  b += 0x7FFFu + ((b >> 16) & 1u);
  return (uint16_t)(b >> 16);
}

// Collects the indices of flagged inputs from a parallel loop.
struct HardList {
  std::vector<std::vector<int64_t>> per_thread;
  explicit HardList(int threads) : per_thread((size_t)std::max(threads, 1)) {}
  int64_t emit(int64_t* out, int64_t max_out) const {
    int64_t cnt = 0;
    for (auto& v : per_thread)
      for (int64_t i : v) {
        if (cnt < max_out) out[cnt] = i;
        ++cnt;
      }
    return cnt;
  }
};

extern "C" {

// ------------------------------------------------------------- the codec --

double orc_e4m3_decode(uint8_t code) { return e4m3_decode(code); }
uint8_t orc_e4m3_encode(float x) { return e4m3_encode(x); }

void orc_e4m3_encode_array(const float* x, uint8_t* out, int64_t n, int threads) {
  parallel_for(n, threads, [&](int64_t lo, int64_t hi) {
    for (int64_t i = lo; i < hi; ++i) out[i] = e4m3_encode(x[i]);
  });
}

void orc_e4m3_decode_array(const uint8_t* c, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_decode(c[i]);
}

// Element map of every quantizer: code of x under scale s.
void orc_quantize_values(const float* x, const float* s, uint8_t* out, int64_t n,
                         int threads) {
  parallel_for(n, threads, [&](int64_t lo, int64_t hi) {
    for (int64_t i = lo; i < hi; ++i) out[i] = quantize_one(x[i], s[i]);
  });
}

// ----------------------------------------------- 128x128 weight blocks ----
// [S341] eq. W_hat_ij = round(W_ij / scale_ij), W in R^{n x k} (BF16),
// scale_ij from the max-abs of the 128x128 block holding (i, j); [S342] Phase 2
// step 2.  Layout: w[i*ldw + j] BF16 bits, q[i*ldq + j] codes, scales
// [ceil(n/128), ceil(k/128)] row-major.  Partial edge blocks take the max over
// their valid elements only.
void orc_quantize_weights_blockwise(const uint16_t* w, int64_t n, int64_t k,
                                    int64_t ldw, uint8_t* q, int64_t ldq,
                                    float* scales, int threads) {
  int64_t nb = (n + 127) / 128, kb = (k + 127) / 128;
  parallel_for(nb * kb, threads, [&](int64_t lo, int64_t hi) {
    for (int64_t b = lo; b < hi; ++b) {
      int64_t bi = b / kb, bj = b % kb;
      int64_t i0 = bi * 128, i1 = std::min(n, i0 + 128);
      int64_t j0 = bj * 128, j1 = std::min(k, j0 + 128);
      float amax = 0.0f;
      for (int64_t i = i0; i < i1; ++i)
        for (int64_t j = j0; j < j1; ++j)
          amax = std::max(amax, std::fabs(bf16_to_float(w[i * ldw + j])));
      float s = scale_from_amax(amax);
      scales[bi * kb + bj] = s;
      for (int64_t i = i0; i < i1; ++i)
        for (int64_t j = j0; j < j1; ++j)
          q[i * ldq + j] = quantize_one(bf16_to_float(w[i * ldw + j]), s);
    }
  });
}

// ------------------------------------------------ 1x128 activation groups --
// [S341] (1x128 activation tiles, after DeepSeek-V3) and the dynamic
// activation quantization of [S342] Phase 3: per token, per 128-wide group of
// the hidden dimension, the same scale and rounding rule as the weights.
// Layout: a[r*lda + c] BF16, q[r*k + c] codes (dense), scales stored
// group-major: scales[g*m + r] for g in [0, ceil(k/128)).
void orc_quantize_act_groupwise(const uint16_t* a, int64_t m, int64_t k,
                                int64_t lda, uint8_t* q, float* scales,
                                int threads) {
  int64_t g_count = (k + 127) / 128;
  parallel_for(m, threads, [&](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) {
      for (int64_t g = 0; g < g_count; ++g) {
        int64_t c0 = g * 128, c1 = std::min(k, c0 + 128);
        float amax = 0.0f;
        for (int64_t c = c0; c < c1; ++c)
          amax = std::max(amax, std::fabs(bf16_to_float(a[r * lda + c])));
        float s = scale_from_amax(amax);
        scales[g * m + r] = s;
        for (int64_t c = c0; c < c1; ++c)
          q[r * k + c] = quantize_one(bf16_to_float(a[r * lda + c]), s);
      }
    }
  });
}

// ---------------------------------------------------------- FP8 KV cache --
// [S344]: K and V are stored as E4M3 with per-head scales computed from the
// K/V values observed in the calibration forward.  x is [rows, heads, hd]
// BF16 (rows = sequences x tokens).  Calibration: amax over rows and hd for
// each head, s[h] = fl32(amax/448).  Quantization: code = E4M3(fl32(x/s[h])).
void orc_kv_calibrate(const uint16_t* x, int64_t rows, int heads, int hd,
                      float* scales, int threads) {
  std::vector<float> part((size_t)std::max(threads, 1) * heads, 0.0f);
  int64_t nthreads = std::max(threads, 1);
  int64_t chunk = (rows + nthreads - 1) / nthreads;
  parallel_for(nthreads, threads, [&](int64_t tlo, int64_t thi) {
    for (int64_t t = tlo; t < thi; ++t) {
      int64_t r0 = t * chunk, r1 = std::min(rows, r0 + chunk);
      for (int64_t r = r0; r < r1; ++r)
        for (int h = 0; h < heads; ++h)
          for (int d = 0; d < hd; ++d) {
            float v = std::fabs(bf16_to_float(x[(r * heads + h) * hd + d]));
            part[t * heads + h] = std::max(part[t * heads + h], v);
          }
    }
  });
  for (int h = 0; h < heads; ++h) {
    float amax = 0.0f;
    for (int64_t t = 0; t < nthreads; ++t) amax = std::max(amax, part[t * heads + h]);
    scales[h] = scale_from_amax(amax);
  }
}

void orc_kv_quantize(const uint16_t* x, int64_t rows, int heads, int hd,
                     const float* scales, uint8_t* q, int threads) {
  parallel_for(rows, threads, [&](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r)
      for (int h = 0; h < heads; ++h)
        for (int d = 0; d < hd; ++d) {
          int64_t i = (r * heads + h) * hd + d;
          q[i] = quantize_one(bf16_to_float(x[i]), scales[h]);
        }
  });
}

// ------------------------------------------------ blockwise W8A8 GEMM -----
// [S342] Phase 3 / [S341]: Y = A W^T from FP8 codes, each operand dequantized
// by its own scale set, accumulated without loss, BF16 rounding left to the
// caller.  Here in float64:
//   Y[m,n] = sum_k (dec(qa[m,k]) * sa[k/128, m]) * (dec(qw[n,k]) * sw[n/128, k/128])
// Each dequantized operand is exact in float64 (a 4-bit significand times a
// binary32 scale); the only rounding is the float64 running sum over k.
// Also returns B[m,n] = sum_k |A_deq[m,k]| * |W_deq[n,k]| for the error bound.
// rows/cols select which outputs to compute (sampled checks of big launches).
// qa [M, K] codes, sa [K/128, M], qw [N, K], sw [ceil(N/128), K/128].
void orc_gemm_w8a8_sampled(const uint8_t* qa, const float* sa, const uint8_t* qw,
                           const float* sw, int64_t M, int64_t N, int64_t K,
                           const int64_t* rows, int64_t nr, const int64_t* cols,
                           int64_t nc, double* y, double* absprod, int threads) {
  int64_t kb_count = K / 128;
  parallel_for(nr, threads, [&](int64_t lo, int64_t hi) {
    std::vector<double> arow((size_t)K);
    for (int64_t ri = lo; ri < hi; ++ri) {
      int64_t m = rows[ri];
      for (int64_t kk = 0; kk < K; ++kk)
        arow[kk] = e4m3_decode(qa[m * K + kk]) * (double)sa[(kk / 128) * M + m];
      for (int64_t ci = 0; ci < nc; ++ci) {
        int64_t n = cols[ci];
        double acc = 0.0, acc_abs = 0.0;
        for (int64_t kk = 0; kk < K; ++kk) {
          double wv = e4m3_decode(qw[n * K + kk]) *
                      (double)sw[(n / 128) * kb_count + kk / 128];
          acc += arow[kk] * wv;
          acc_abs += std::fabs(arow[kk]) * std::fabs(wv);
        }
        y[ri * nc + ci] = acc;
        absprod[ri * nc + ci] = acc_abs;
      }
    }
  });
}

// Grouped (MoE expert) variant: rows [offsets[e], offsets[e+1]) of A are the
// tokens routed to expert e and multiply expert e's weights qw[e] ([N, K]) with
// scales sw[e] ([N/128, K/128]).  A row outside every segment has no output.
// rows are global row indices into A.
void orc_grouped_gemm_w8a8_sampled(const uint8_t* qa, const float* sa,
                                   const uint8_t* qw, const float* sw,
                                   const int32_t* offsets, int32_t E,
                                   int64_t M, int64_t N, int64_t K,
                                   const int64_t* rows, int64_t nr,
                                   const int64_t* cols, int64_t nc, double* y,
                                   double* absprod, int threads) {
  int64_t kb_count = K / 128, nb_count = (N + 127) / 128;
  parallel_for(nr, threads, [&](int64_t lo, int64_t hi) {
    std::vector<double> arow((size_t)K);
    for (int64_t ri = lo; ri < hi; ++ri) {
      int64_t m = rows[ri];
      int32_t e = -1;
      for (int32_t j = 0; j < E; ++j)
        if (m >= offsets[j] && m < offsets[j + 1]) { e = j; break; }
      if (e < 0) {
        for (int64_t ci = 0; ci < nc; ++ci) {
          y[ri * nc + ci] = std::nan("");
          absprod[ri * nc + ci] = std::nan("");
        }
        continue;
      }
      const uint8_t* qwe = qw + (int64_t)e * N * K;
      const float* swe = sw + (int64_t)e * nb_count * kb_count;
      for (int64_t kk = 0; kk < K; ++kk)
        arow[kk] = e4m3_decode(qa[m * K + kk]) * (double)sa[(kk / 128) * M + m];
      for (int64_t ci = 0; ci < nc; ++ci) {
        int64_t n = cols[ci];
        double acc = 0.0, acc_abs = 0.0;
        for (int64_t kk = 0; kk < K; ++kk) {
          double wv = e4m3_decode(qwe[n * K + kk]) *
                      (double)swe[(n / 128) * kb_count + kk / 128];
          acc += arow[kk] * wv;
          acc_abs += std::fabs(arow[kk]) * std::fabs(wv);
        }
        y[ri * nc + ci] = acc;
        absprod[ri * nc + ci] = acc_abs;
      }
    }
  });
}

// --------------------------------------------- truncated IS weights (TIS) --
// [S343]: w = pi_theta(a|s) / pi_fp8(a|s) = exp(logp_train - logp_rollout)
// per token.  Reading: the difference is one binary32 subtraction and the
// weight is the correctly rounded binary32 value of e^delta (the one result
// two independent implementations can agree on bit for bit).  This routine
// returns that rounded exponential; clipping to C and the mask are applied by
// the Python side of the oracle.
//
// e^delta is formed in float64 by the C library and rounded once to binary32.
// The C library's exp is accurate to well under 2^-50 relative, so the
// binary32 rounding can only be wrong when the float64 value lies within that
// distance of a binary32 rounding boundary (a midpoint between neighbouring
// floats).  Such inputs are listed in `hard` (indices) with the two candidate
// floats, and are decided exactly by the caller with a 60-digit decimal exp.
// Returns the number of hard cases written (at most max_hard).
int64_t orc_tis_exp(const float* lt, const float* lr, int64_t n, float* e32,
                    int64_t* hard, int64_t max_hard, int threads) {
  const double rel = std::ldexp(1.0, -40);
  std::vector<std::vector<int64_t>> found((size_t)std::max(threads, 1));
  int64_t nthreads = std::max(threads, 1);
  int64_t chunk = (n + nthreads - 1) / nthreads;
  parallel_for(nthreads, threads, [&](int64_t tlo, int64_t thi) {
    for (int64_t t = tlo; t < thi; ++t) {
      int64_t i0 = t * chunk, i1 = std::min(n, i0 + chunk);
      for (int64_t i = i0; i < i1; ++i) {
        float delta = lt[i] - lr[i];
        double e = std::exp((double)delta);
        float f = (float)e;
        e32[i] = f;
        if (!std::isfinite(e) || e == 0.0 || (double)f == e) continue;
        // the rounding boundary on e's side of f
        float g = std::nextafter(f, (e > (double)f) ? INFINITY : -INFINITY);
        double mid;
        if (std::isinf(f) || std::isinf(g))   // boundary between FLT_MAX and overflow
          mid = std::ldexp(2.0 - std::ldexp(1.0, -24), 127);
        else
          mid = ((double)f + (double)g) * 0.5;  // exact in float64
        if (std::fabs(e - mid) <= rel * std::fabs(e)) found[t].push_back(i);
      }
    }
  });
  int64_t cnt = 0;
  for (auto& v : found)
    for (int64_t i : v) {
      if (cnt < max_hard) hard[cnt] = i;
      ++cnt;
    }
  return cnt;
}

void orc_float_to_bf16(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = float_to_bf16(x[i]);
}

// y[i] = BF16_RNE(silu(g[i]) * u[i]) over n pairs of BF16 bit patterns.
// Indices whose rounding the float64 value cannot decide go to `hard`;
// returns how many there are (all are counted, at most max_hard written).
int64_t orc_silu_mul_pairs(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* y,
                           int64_t* hard, int64_t max_hard, int threads) {
  HardList found(threads);
  const int64_t nthreads = std::max(threads, 1);
  const int64_t chunk = (n + nthreads - 1) / nthreads;
  parallel_for(nthreads, threads, [&](int64_t tlo, int64_t thi) {
    for (int64_t t = tlo; t < thi; ++t) {
      const int64_t i0 = t * chunk, i1 = std::min(n, i0 + chunk);
      for (int64_t i = i0; i < i1; ++i) {
        bool h = false;
        y[i] = silu_mul_bf16_one(g[i], u[i], &h);
        if (h) found.per_thread[t].push_back(i);
      }
    }
  });
  return found.emit(hard, max_hard);
}

// Gated activation of one MoE expert layer: h is BF16 [m, 2*inter] (row
// stride ldh) holding gate (columns [0, inter)) then up ([inter, 2*inter));
// y = BF16_RNE(silu(gate) * up), BF16 [m, inter] dense.  Flagged elements
// (flat index r * inter + c) go to `hard` as in orc_silu_mul_pairs.
int64_t orc_silu_mul_bf16(const uint16_t* h, int64_t m, int64_t inter, int64_t ldh, uint16_t* y,
                          int64_t* hard, int64_t max_hard, int threads) {
  HardList found(threads);
  const int64_t nthreads = std::max(threads, 1);
  const int64_t chunk = (m + nthreads - 1) / nthreads;
  parallel_for(nthreads, threads, [&](int64_t tlo, int64_t thi) {
    for (int64_t t = tlo; t < thi; ++t) {
      const int64_t r0 = t * chunk, r1 = std::min(m, r0 + chunk);
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = 0; c < inter; ++c) {
          bool hd = false;
          y[r * inter + c] = silu_mul_bf16_one(h[r * ldh + c], h[r * ldh + inter + c], &hd);
          if (hd) found.per_thread[t].push_back(r * inter + c);
        }
    }
  });
  return found.emit(hard, max_hard);
}

}  // extern "C"
