// fp_exact.cuh -- exactly rounded binary32 building blocks of the hot path.
//
// Everything here is written against IEEE-754 round-to-nearest-even and uses
// explicitly rounded operations (never contracted into FMAs by the compiler),
// so that each function returns the same bits on the device and in a host
// build compiled with -ffp-contract=off.
//
//  * quotient by a block scale, fl32(x / s), at the cost of one multiply and
//    two FMAs: the correction step of P. Markstein ("Computation of elementary
//    functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
//    1990; also "IA-64 and Elementary Functions", 2000).  With y = RN(1/s) and
//    q0 = RN(x*y) within one ulp of x/s, r = x - q0*s is exact and
//    RN(q0 + r*y) = RN(x/s), provided no intermediate underflows or
//    overflows.  The fast form is used for scales in [2^-60, 2^126]: there,
//    any |x| small enough for r to underflow (|x| < 2^-71) has |x/s| < 2^-11,
//    whose E4M3 code is +-0 whatever the last bits of the quotient, so every
//    code equals that of the IEEE quotient.  Other scales (tiny, huge,
//    negative, non-finite) take IEEE division.
//  * e^d correctly rounded to binary32 (the TIS weight): a float-float
//    evaluation after Tang's table-driven method (P.T.P. Tang, "Table-driven
//    implementation of the exponential function in IEEE floating-point
//    arithmetic", ACM TOMS 15(2), 1989) with 32 table entries and a degree-6
//    Taylor polynomial, accurate to ~2^-44 relative; inputs whose result lies
//    within 2^-40 of a binary32 rounding boundary, or outside |d| <= 87, are
//    recomputed more accurately (~2^-64 relative): reduction by ln2/32 in
//    double-double, e^r - 1 - r by a degree-7 polynomial in double, and a
//    double-double table of 2^(j/32).  Over all binary32 d no value e^d lies
//    closer than 2^-52.6 (relative) to a rounding boundary -- found by
//    enumerating every input within 2^-40 of one with a 60-digit decimal
//    exponential -- so that accuracy decides every rounding correctly.
#pragma once

#include <stdint.h>
#include <math.h>

#if defined(__CUDACC__)
#define FP8RL_HD __host__ __device__ __forceinline__
#define FP8RL_HD_OUTLINE static __host__ __device__ __noinline__
#else
#define FP8RL_HD inline
#define FP8RL_HD_OUTLINE inline
#endif

namespace fp8rl {
namespace fx {

// ---- explicitly rounded primitives (device intrinsics; host IEEE ops) ------
#if defined(__CUDA_ARCH__)
FP8RL_HD float fadd(float a, float b) { return __fadd_rn(a, b); }
FP8RL_HD float fsub(float a, float b) { return __fsub_rn(a, b); }
FP8RL_HD float fmul(float a, float b) { return __fmul_rn(a, b); }
FP8RL_HD float ffma(float a, float b, float c) { return __fmaf_rn(a, b, c); }
FP8RL_HD float fdiv(float a, float b) { return __fdiv_rn(a, b); }
FP8RL_HD float frcp(float a) { return __frcp_rn(a); }
FP8RL_HD double dadd(double a, double b) { return __dadd_rn(a, b); }
FP8RL_HD double dsub(double a, double b) { return __dsub_rn(a, b); }
FP8RL_HD double dmul(double a, double b) { return __dmul_rn(a, b); }
FP8RL_HD double dfma(double a, double b, double c) { return __fma_rn(a, b, c); }
FP8RL_HD double ddiv(double a, double b) { return __ddiv_rn(a, b); }
FP8RL_HD float d2f(double a) { return __double2float_rn(a); }
FP8RL_HD uint32_t f2u(float f) { return __float_as_uint(f); }
FP8RL_HD float u2f(uint32_t u) { return __uint_as_float(u); }
#else
FP8RL_HD float fadd(float a, float b) { return a + b; }
FP8RL_HD float fsub(float a, float b) { return a - b; }
FP8RL_HD float fmul(float a, float b) { return a * b; }
FP8RL_HD float ffma(float a, float b, float c) { return fmaf(a, b, c); }
FP8RL_HD float fdiv(float a, float b) { return a / b; }
FP8RL_HD float frcp(float a) { return 1.0f / a; }
FP8RL_HD double dadd(double a, double b) { return a + b; }
FP8RL_HD double dsub(double a, double b) { return a - b; }
FP8RL_HD double dmul(double a, double b) { return a * b; }
FP8RL_HD double dfma(double a, double b, double c) { return fma(a, b, c); }
FP8RL_HD double ddiv(double a, double b) { return a / b; }
FP8RL_HD float d2f(double a) { return (float)a; }
FP8RL_HD uint32_t f2u(float f) { union { float f; uint32_t u; } v; v.f = f; return v.u; }
FP8RL_HD float u2f(uint32_t u) { union { float f; uint32_t u; } v; v.u = u; return v.f; }
#endif

// ---------------------------------------------------- quotient by a scale --

// Per-scale set-up for the element map x -> fl32(x / s).
struct ScaleDiv {
  float s;
  float y;     // RN(1/s) when mode == 1
  int mode;    // 0: s == 0 (the value passes through); 1: Markstein; 2: IEEE divide
};

FP8RL_HD ScaleDiv make_scale_div(float s) {
  ScaleDiv d;
  d.s = s;
  d.y = 0.0f;
  if (s == 0.0f) {
    d.mode = 0;
  } else if (s >= 0x1p-60f && s <= 0x1p126f) {    // see the range note above
    d.mode = 1;
    d.y = frcp(s);
  } else {
    d.mode = 2;
  }
  return d;
}

// fl32(x / s) when mode == 1, |x / s| < 2^127 and |x| >= 2^-71; for smaller
// |x| the result is within a few ulps of a quotient below 2^-11 (guarded
// variant below for arbitrary caller scales).  The residual is formed as
// q0*s - x and applied with -y: the same value as Markstein's
// q0 + (x - q0*s)*y for every non-zero x, and for x = -0 it yields -0 (the
// form with x - q0*s would return +0), so the sign of zero needs no fix-up.
FP8RL_HD float markstein_quotient(float x, float s, float y) {
  const float q0 = fmul(x, y);
  const float rp = ffma(q0, s, -x);
  return ffma(rp, -y, q0);
}

// The element map's binary32 quotient under a prepared scale.  kGuard adds
// the overflow guard needed when s is a caller-provided number rather than
// amax/448 (then |x/s| may exceed 448 by any amount; every |q| >= 1024
// saturates to 448 in E4M3 regardless of its exact value).
template <bool kGuard>
FP8RL_HD float scaled_quotient(float x, const ScaleDiv& d) {
  if (d.mode == 1) {
    float q = markstein_quotient(x, d.s, d.y);
    if (kGuard) {
      float q0 = fmul(x, d.y);
      if (!(fabsf(q0) < 1024.0f)) q = q0;
    }
    return q;
  }
  if (d.mode == 0) return x;
  return fdiv(x, d.s);
}

// ---------------------------------------------- correctly rounded e^d ------

// Tables of the exponential, built on the host by make_exp_tables():
// 2^(j/32), j = 0..31, as float-float pairs (fast path) and as double-double
// pairs (accurate path).
struct Exp2Table {
  float hi[32];
  float lo[32];
  double dhi[32];
  double dlo[32];
};

FP8RL_HD void two_sum(float a, float b, float& s, float& e) {
  s = fadd(a, b);
  float bb = fsub(s, a);
  e = fadd(fsub(a, fsub(s, bb)), fsub(b, bb));
}
FP8RL_HD void fast_two_sum(float a, float b, float& s, float& e) {  // needs |a| >= |b| or a == 0
  s = fadd(a, b);
  e = fsub(b, fsub(s, a));
}
FP8RL_HD void two_prod(float a, float b, float& p, float& e) {
  p = fmul(a, b);
  e = ffma(a, b, -p);
}

// Fast path, in parts so that a caller can fetch the table entry its own way
// (the CUDA kernel takes it from lane registers with a warp shuffle):
// exp_fast_k() gives the reduction multiple kf of d, exp_fast_index_k() the
// table index j (any d, also out of range), and exp_rn32_fast_with_k()
// finishes with th + tl = 2^(j/32).  It returns false when the input must
// take exp_rn32_slow (|d| > 87, NaN, or a result too close to a rounding
// boundary to decide here).
// ln2/32 is split in three: L1 has 12 significant bits so that k*L1 is exact
// for |k| < 2^12; L2 and L3 carry the next 48 bits.
constexpr float kExpInvL = 0x1.715476p+5f;      // ~32/ln2; only sets the reduction range
constexpr float kExpL1 = 0x1.62ep-6f;
constexpr float kExpL2 = 0x1.0bfbe8p-20f;
constexpr float kExpL3 = 0x1.cf79acp-45f;

// kf = rint(d * 32/ln2), the reduction multiple of ln2/32 (finite or not).
FP8RL_HD float exp_fast_k(float d) { return rintf(fmul(d, kExpInvL)); }

FP8RL_HD int exp_fast_index_k(float kf) {
  return fabsf(kf) < 65536.0f ? (((int)kf) & 31) : 0;   // out-of-range d: any valid index
}

// e^d rounded to binary32, or false (see above); kf = exp_fast_k(d).
FP8RL_HD bool exp_rn32_fast_with_k(float d, float kf, float th, float tl, float* out) {
  if (!(fabsf(d) <= 87.0f)) return false;
  int k = (int)kf;
  // r = d - k*ln2/32 as r_hi + r_lo, |r| <= ~ln2/64
  float a = ffma(-kf, kExpL1, d);                    // exact
  float p_hi, p_lo;
  two_prod(kf, kExpL2, p_hi, p_lo);
  float r_hi, e1;
  two_sum(a, -p_hi, r_hi, e1);
  float r_lo = fsub(fsub(e1, p_lo), fmul(kf, kExpL3));
  fast_two_sum(r_hi, r_lo, r_hi, r_lo);
  // e^r - 1 = r + r^2/2 + r^3/6 + r^4/24 + r^5/120 + r^6/720 (+ < 2^-55)
  float sq_hi, sq_lo;
  two_prod(r_hi, r_hi, sq_hi, sq_lo);
  float half = fmul(0.5f, sq_hi);                // exact
  float half_lo = fadd(ffma(r_hi, r_lo, fmul(0.5f, sq_lo)), fmul(half, r_lo));
  float t = ffma(r_hi, 1.0f / 720.0f, 1.0f / 120.0f);
  t = ffma(r_hi, t, 1.0f / 24.0f);
  t = ffma(r_hi, t, 1.0f / 6.0f);
  float tail = fmul(fmul(sq_hi, r_hi), t);
  float s1, e2;
  fast_two_sum(r_hi, half, s1, e2);
  float p_lo2 = fadd(fadd(fadd(e2, r_lo), half_lo), tail);
  // 2^(j/32) * (1 + P), k = 32 m + j
  const int j = k & 31;
  const int m = (k - j) / 32;
  float m_hi, m_lo;
  two_prod(th, s1, m_hi, m_lo);
  float rest = fadd(fadd(fadd(m_lo, fmul(th, p_lo2)), tl), fmul(tl, fadd(s1, p_lo2)));
  float y1, e3;
  fast_two_sum(th, m_hi, y1, e3);
  float yl0 = fadd(e3, rest);
  float yh, yl;
  fast_two_sum(y1, yl0, yh, yl);
  // distance to the rounding boundary on yl's side of yh (yh > 0)
  uint32_t b = f2u(yh);
  float nb = u2f(yl >= 0.0f ? b + 1u : b - 1u);
  float half_ulp = fmul(fsub(nb, yh), 0.5f);
  float dist = fsub(fabsf(half_ulp), fabsf(yl));
  if (dist <= fmul(yh, 0x1p-40f)) return false;
  *out = fmul(yh, u2f((uint32_t)(m + 127) << 23));   // exact: the result is normal
  return true;
}

// double-double helpers for the slow path
struct dd { double hi, lo; };
FP8RL_HD dd dd_fast(double a, double b) {
  double s = dadd(a, b);
  return dd{s, dsub(b, dsub(s, a))};
}
FP8RL_HD dd dd_two_sum(double a, double b) {
  double s = dadd(a, b);
  double bb = dsub(s, a);
  return dd{s, dadd(dsub(a, dsub(s, bb)), dsub(b, bb))};
}
FP8RL_HD dd dd_mul(dd a, dd b) {
  double p = dmul(a.hi, b.hi);
  double e = dfma(a.hi, b.hi, -p);
  e = dadd(e, dadd(dmul(a.hi, b.lo), dmul(a.lo, b.hi)));
  return dd_fast(p, e);
}
FP8RL_HD dd dd_add_one(dd a) {
  dd s = dd_two_sum(1.0, a.hi);
  return dd_fast(s.hi, dadd(s.lo, a.lo));
}

// Correct binary32 rounding of the double-double value H + L.
FP8RL_HD float dd_round_to_float(double H, double L) {
  float f = d2f(H);
  double fd = (double)f;
  if (fd == H) return f;
  float g = nextafterf(f, H > fd ? INFINITY : -INFINITY);
  double mid;
  if (isinf(f) || isinf(g))
    mid = copysign(0x1p128 - 0x1p103, H);          // FLT_MAX / overflow boundary
  else
    mid = dmul(dadd(fd, (double)g), 0.5);          // exact
  if (H == mid && L != 0.0) return ((L > 0.0) == (g > f)) ? g : f;
  return f;
}

// Accurate path: any binary32 d.  Kept out of line: it runs for a few lanes
// in ten thousand, and inlining it at every call site would bloat the fast
// path.
FP8RL_HD_OUTLINE float exp_rn32_slow(float d, const Exp2Table& T) {
  if (d != d) return d;
  if (d > 89.0f) return INFINITY;      // e^89 > 2^128: rounds to +inf
  if (d < -104.0f) return 0.0f;        // e^-104 < 2^-150: rounds to +0
  // ln2/32 as a double-double (ln 2 = 0x1.62e42fefa39ef35793c7673007e6p-1)
  const double kCHi = 0x1.62e42fefa39efp-6;
  const double kCLo = 0x1.abc9e3b39803fp-61;
  const double x = (double)d;
  const double kf = rint(dmul(x, 0x1.71547652b82fep+5));   // ~32/ln2; |k| <= 4800
  const int k = (int)kf;
  const int j = k & 31;
  const int m = (k - j) / 32;
  // r = x - k ln2/32 as rh + rl, |r| <= ~0.0109
  const double p1 = dmul(kf, kCHi);
  const double p1e = dfma(kf, kCHi, -p1);
  dd r = dd_two_sum(x, -p1);
  r = dd_fast(r.hi, dsub(dsub(r.lo, p1e), dmul(kf, kCLo)));
  // q = e^rh - 1 - rh (degree 7, truncation < 2^-67), in double
  const double rh = r.hi;
  double q = dfma(rh, 1.0 / 5040.0, 1.0 / 720.0);
  q = dfma(rh, q, 1.0 / 120.0);
  q = dfma(rh, q, 1.0 / 24.0);
  q = dfma(rh, q, 1.0 / 6.0);
  q = dfma(rh, q, 0.5);
  q = dmul(dmul(rh, rh), q);
  // e^r = 1 + rh + (rl + q + rh*rl) as a double-double
  dd e = dd_two_sum(1.0, rh);
  e = dd_fast(e.hi, dadd(e.lo, dadd(r.lo, dfma(rh, r.lo, q))));
  const dd v = dd_mul(e, dd{T.dhi[j], T.dlo[j]});
  return dd_round_to_float(ldexp(v.hi, m), ldexp(v.lo, m));
}

// Host-side construction of the tables.  2^(j/32) = e^(j ln2/32) is formed
// in double-double by a Taylor series of e^(x/256) followed by eight
// squarings (~2^-95); the float-float pairs keep its leading 48 bits.
inline dd dd_exp_host(dd x) {
  dd inv[16];
  for (int i = 1; i < 16; ++i) {
    inv[i].hi = 1.0 / i;
    inv[i].lo = fma(-inv[i].hi, (double)i, 1.0) / i;   // exact residual
  }
  const dd r{x.hi * 0x1p-8, x.lo * 0x1p-8};
  dd p{1.0, 0.0};
  for (int i = 15; i >= 1; --i) p = dd_add_one(dd_mul(dd_mul(p, r), inv[i]));
  for (int i = 0; i < 8; ++i) p = dd_mul(p, p);
  return p;
}

inline Exp2Table make_exp_tables() {
  Exp2Table T;
  const double kCHi = 0x1.62e42fefa39efp-6, kCLo = 0x1.abc9e3b39803fp-61;  // ln2/32
  for (int j = 0; j < 32; ++j) {
    const double ph = j * kCHi;
    const double pe = fma((double)j, kCHi, -ph);
    const dd x = dd_fast(ph, pe + j * kCLo);
    const dd v = dd_exp_host(x);
    T.dhi[j] = v.hi;
    T.dlo[j] = v.lo;
    T.hi[j] = (float)v.hi;
    T.lo[j] = (float)((v.hi - (double)T.hi[j]) + v.lo);
  }
  return T;
}

}  // namespace fx
}  // namespace fp8rl
