// quant.cu -- the per-token quantizers of the FP8 rollout hot path.
//
//   * per-token 1x128-group activation quantization (FP8-RL summary, sections
//     3.4.1/3.4.2 Phase 3, dynamic quantization), plain and gathering the
//     routed rows of an MoE layer,
//   * the MoE glue y = BF16_RNE(SiLU(gate) * up), alone or with the 1x128
//     quantization of y, between the expert GEMMs,
//   * FP8 E4M3 KV-cache quantization with per-head scales, given or
//     calibrated from the tensor (section 3.4.4).
//
// All apply the element map of quant_common.cuh: scale = fl32(amax/448),
// code = E4M3_RNE_satfinite(fl32(x/scale)), with the exact Markstein quotient
// of fp_exact.cuh.  Every kernel reads its input once with 16-byte
// non-allocating loads and writes packed 8-byte code vectors; amax is a
// bf16x2 max over |x| bit patterns, then warp shuffles.  (The 128x128 weight
// re-quantization is in wquant.cu.)
#include <algorithm>
#include <cstring>
#include <mutex>

#include "quant_common.cuh"

namespace fp8rl {
namespace {

// Programmatic dependent launch: lets the next kernel in the stream, if it was
// launched with programmatic serialization allowed (the GEMMs are), start its
// launch and prologue now.  It still waits (griddepcontrol.wait) for this
// grid to complete before it reads memory, so this changes timing only.
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------ 1x128 activation groups --

// Groups are numbered row-major over the whole matrix, f = r * kb + g (kb =
// ceil(k/128) groups per row), and a warp task is 8 consecutive groups -- so
// tasks may span rows and every lane has work even when kb is not a multiple
// of 8.  4 lanes per group, each lane 4 x 16-byte chunks (chunk slot + 4i of
// its group).  Scales go to the group-major array scales[g * m + r].
// kGather: output row r is source row rows[r] of a (m_src rows); an index out
// of range leaves the row zero and sets kStatusBadIndex.
template <bool kGather>
__global__ void __launch_bounds__(256) aquant_kernel(const uint16_t* __restrict__ a, int64_t m,
                                                     int64_t k, int64_t lda,
                                                     uint8_t* __restrict__ q,
                                                     float* __restrict__ scales,
                                                     int64_t n_tasks, int kb,
                                                     const int32_t* __restrict__ rows,
                                                     int64_t m_src, uint32_t* status) {
  allow_dependent_launch();   // the GEMM that reads these codes may launch now
  const int lane = threadIdx.x & 31;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int slot = lane & 3;
  const int64_t groups = m * kb;
  for (int64_t task = gw; task < n_tasks; task += nw) {
    const int64_t f = task * 8 + (lane >> 2);
    const bool valid = f < groups;
    const int64_t r = valid ? f / kb : 0;
    const int g = (int)(f - r * kb);
    const int64_t gcol = (int64_t)g * 128;
    int64_t src = r;
    bool load = valid;
    if (kGather && valid) {
      src = __ldg(rows + r);
      if (src < 0 || src >= m_src) {
        load = false;
        if (slot == 0 && g == 0) atomicOr(status, kStatusBadIndex);
      }
    }
    const uint16_t* arow = a + (load ? src : 0) * lda;
    uint4 v[4];
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t col = gcol + (slot + 4 * i) * 8;
      v[i] = (load && col < k) ? ld_stream(arow + col) : make_uint4(0, 0, 0, 0);
      m2 = absmax8(m2, v[i]);
    }
    const float amax = warp_max(bf16x2_maxf(m2), 4);
    const float s = fx::fdiv(amax, 448.0f);
    if (slot == 0 && valid) scales[(int64_t)g * m + r] = s;
    const ScaleDiv sd = make_scale_div(s);
    uint8_t* qrow = q + r * k;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t col = gcol + (slot + 4 * i) * 8;
      if (valid && col < k) *reinterpret_cast<uint2*>(qrow + col) = quant8_any<false>(v[i], sd);
    }
  }
}

// ------------------------------------------------------------- MoE glue --
//
// y = BF16_RNE(silu(g) * u), silu(g) = g / (1 + e^-g): the real product rounded
// once to the nearest BF16 (declared in fp8rl.h).  silu depends on the BF16
// gate alone, so each device holds it for all 65536 gate patterns as an
// unevaluated float-float pair hi + lo (relative error near 2^-48), formed in
// double precision once, when the library first meets the device.  The
// product hi*u + lo*u carries an exact FMA error term, and the BF16 rounding
// of that float-float value is decided from the binary32 product's bits, so
// y is the correctly rounded product unless it lies within about 2^-46 of a
// rounding midpoint (none does: the GPU tests compare every gate with every
// up mantissa and exponent against the oracle).
//
// Entries by the gate's exponent field eg and sign ("scale" K: the pair
// holds silu(g) * 2^K):
//   |g| < 2^-60 (eg < 67):   K = 100;
//   -128 < g <= -64:          K = 140;   -256 < g <= -128: K = 240;
//   g <= -256:                hi = 0 (|y| is below half the smallest BF16
//                             for every finite u);
//   otherwise:                K = 0 ("natural" entries);
//   +-0, +-inf, NaN:          unused (special values).
// Where the remainder silu*2^K - hi underflows binary32, lo is the smallest
// subnormal with the remainder's sign: products g*u or (g/2)*u that are
// exactly BF16 midpoints round in that direction.
// g_silu_pair holds (hi, lo) of every entry; g_silu_hi holds hi for the
// natural entries and 0 for all others, so the fast path reads 4 bytes and a
// zero product sends everything else to the general path.
__device__ float2 g_silu_pair[65536];
__device__ float g_silu_hi[65536];

__device__ __forceinline__ int silu_scale(uint32_t gb) {
  const uint32_t eg = (gb >> 7) & 0xFFu;
  if (eg < 67u) return 100;
  if ((gb & 0x8000u) && eg == 133u) return 140;
  if ((gb & 0x8000u) && eg >= 134u) return 240;
  return 0;
}

__global__ void silu_table_kernel() {
  const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 65536u) return;
  const float gf = __uint_as_float(i << 16);
  const uint32_t eg = (i >> 7) & 0xFFu;
  float hi = 0.0f, lo = 0.0f;
  if (eg != 0xFFu && gf != 0.0f && !((i & 0x8000u) && eg >= 135u)) {
    const double g = (double)gf;
    const double sc = ldexp(1.0, silu_scale(i));
    double a, b;          // silu(g) * 2^K = a + b, |b| far below |a|
    float sticky;         // sign of the remainder if it underflows
    if (eg < 115u) {      // |g| < 2^-12: g/2 + g^2/4 - g^4/96 (next term below 2^-70 relative)
      const double g2 = fx::dmul(g, g);
      a = fx::dmul(fx::dmul(g, 0.5), sc);
      b = fx::dmul(fx::dsub(fx::dmul(g2, 0.25), fx::ddiv(fx::dmul(g2, g2), 96.0)), sc);
      sticky = 0x1p-149f;             // silu(g) - g/2 > 0
    } else if (!(i & 0x8000u)) {      // g >= 2^-12: silu = g - c, c = g e^-g / (1 + e^-g)
      const double e = exp(-g);
      a = g;
      b = -fx::ddiv(fx::dmul(g, e), fx::dadd(1.0, e));
      sticky = -0x1p-149f;            // silu(g) < g
    } else {                          // g <= -2^-12: g e^g / (1 + e^g)
      const double e = exp(g);
      a = fx::dmul(fx::ddiv(fx::dmul(g, e), fx::dadd(1.0, e)), sc);
      b = 0.0;
      sticky = 0.0f;
    }
    hi = fx::d2f(fx::dadd(a, b));
    lo = fx::d2f(fx::dadd(fx::dsub(a, (double)hi), b));
    if (lo == 0.0f) lo = sticky;
  }
  g_silu_pair[i] = make_float2(hi, lo);
  g_silu_hi[i] = silu_scale(i) == 0 ? hi : 0.0f;
}

// The general path: special values, the scaled entries and products below
// 2^-100.  Works on magnitudes: |x| = (P + T) 2^(eh + eu - K) with P the
// binary32 product of the two significands in [1, 4) and T its exact error
// plus the table's lo term; rounds to the BF16 spacing at |x| (subnormal
// spacing 2^-133 below 2^-126).
__device__ __noinline__ uint32_t silu_mul_bf16_general(uint32_t gb, uint32_t ub) {
  const float2 t = g_silu_pair[gb];
  const float hs = t.x, ls = t.y;
  const uint32_t sx = (gb ^ ub) & 0x8000u;
  const uint32_t ag = gb & 0x7FFFu, au = ub & 0x7FFFu;
  if (ag > 0x7F80u || au > 0x7F80u) return 0x7FC0u;          // a NaN input
  if (ag == 0x7F80u) {                                        // g = +-inf
    if ((gb & 0x8000u) || au == 0u) return 0x7FC0u;           // silu(-inf) = -inf * 0; inf * 0
    return (ub & 0x8000u) | 0x7F80u;
  }
  if (ag == 0u) return au == 0x7F80u ? 0x7FC0u : sx;          // silu(+-0) = +-0
  if (au == 0x7F80u) return sx | 0x7F80u;                     // non-zero silu times +-inf
  if (au == 0u || hs == 0.0f) return sx;                      // a signed zero
  const int K = silu_scale(gb);
  const uint32_t hb = __float_as_uint(hs);                    // a normal number
  const int eh = (int)((hb >> 23) & 0xFFu) - 127;             // in [-121, 54] here
  const float mh = __uint_as_float((hb & 0x007FFFFFu) | 0x3F800000u);
  float ln = fx::fmul(fabsf(ls), __uint_as_float((uint32_t)(127 - eh) << 23));
  if ((__float_as_uint(ls) ^ hb) & 0x80000000u) ln = -ln;     // > 0 increases |x|
  uint32_t ubits = au << 16;
  int eu = -127;
  if ((au >> 7) == 0u) {                                      // subnormal u: scale by 2^64 (exact)
    ubits = __float_as_uint(fx::fmul(__uint_as_float(ubits), 0x1p64f));
    eu -= 64;
  }
  eu += (int)((ubits >> 23) & 0xFFu);
  const float mu = __uint_as_float((ubits & 0x007FFFFFu) | 0x3F800000u);
  const float P = fx::fmul(mh, mu);
  const float E1 = fx::ffma(mh, mu, -P);                     // exact error of P
  const float T = E1 == 0.0f ? fx::fmul(ln, mu) : fx::ffma(ln, mu, E1);   // keeps ln's sign
  const int ep = P >= 2.0f ? 1 : 0;
  const int E = ep + eh + eu - K;                             // |x| in [2^E, 2^(E+1)) before rounding
  if (E > 127) return sx | 0x7F80u;
  int qe = ep - 7;                                            // BF16 spacing in P's units
  if (E < -126) qe = min(qe - 126 - E, ep + 2);               // subnormal spacing (or all to zero)
  const float Q = __uint_as_float((uint32_t)(127 + qe) << 23);
  const float nq = truncf(fx::fmul(P, __uint_as_float((uint32_t)(127 - qe) << 23)));
  const float f = fx::fsub(P, fx::fmul(nq, Q));               // exact
  const float d = fx::fadd(fx::fsub(f, fx::fmul(0.5f, Q)), T);
  const bool up = d != 0.0f ? d > 0.0f : !(__float_as_uint(T) >> 31);
  const uint32_t n = (uint32_t)nq + (up ? 1u : 0u);
  uint32_t bits = E >= -126 ? ((uint32_t)(E + 127) << 7) + n - 128u : n;
  if (bits > 0x7F80u) bits = 0x7F80u;
  return sx | bits;
}

// y = BF16_RNE(silu(g) * u) for BF16 bit patterns gb, ub (low 16 bits), with
// hi = g_silu_hi[gb] already loaded.  Fast path: a natural entry with
// |hi * u| >= 2^-100 (then hi*u - p is exact).
__device__ __forceinline__ uint32_t silu_mul_bf16_hi(uint32_t gb, uint32_t ub, float hi) {
  const float u = __uint_as_float(ub << 16);
  const float p = fx::fmul(hi, u);
  if (fabsf(p) >= 0x1p-100f) {
    const uint32_t b = __float_as_uint(p);
    if ((b & 0xFFFFu) - 0x7FFCu <= 8u) {
      // within 4 binary32 ulps of a BF16 midpoint m: the sign of
      // (p - m) + (hi*u - p) + lo*u decides.  An exact product leaves a zero
      // error term; then lo*u alone keeps its sign even when it underflows.
      const float lo = __ldg(&g_silu_pair[gb].y);
      const float e = fx::ffma(hi, u, -p);
      const float c = e == 0.0f ? fx::fmul(lo, u) : fx::ffma(lo, u, e);
      const float m = __uint_as_float((b & 0xFFFF0000u) | 0x8000u);
      const float d = fx::fadd(fx::fsub(p, m), c);
      const uint32_t ds = __float_as_uint(d != 0.0f ? d : c);
      return (b >> 16) + (((ds ^ b) >> 31) ? 0u : 1u);
    }
    return (b + 0x7FFFu + ((b >> 16) & 1u)) >> 16;            // p decides alone
  }
  return silu_mul_bf16_general(gb, ub);
}

// 8 outputs from a 16-byte vector of gates and one of ups.  The 8 table
// lookups are issued before any of them is used (their latency, not the
// arithmetic, sets the kernels' pace).
__device__ __forceinline__ uint4 silu_mul8(const uint4& gv, const uint4& uv) {
  const uint32_t g[4] = {gv.x, gv.y, gv.z, gv.w};
  const uint32_t u[4] = {uv.x, uv.y, uv.z, uv.w};
  float hi[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    hi[2 * j] = __ldg(&g_silu_hi[g[j] & 0xFFFFu]);
    hi[2 * j + 1] = __ldg(&g_silu_hi[g[j] >> 16]);
  }
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    o[j] = silu_mul_bf16_hi(g[j] & 0xFFFFu, u[j] & 0xFFFFu, hi[2 * j]) |
           (silu_mul_bf16_hi(g[j] >> 16, u[j] >> 16, hi[2 * j + 1]) << 16);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// y[r, c] = BF16_RNE(silu(h[r, c]) * h[r, inter + c]); 8 outputs per thread
// and step (16-byte loads and stores), grid-stride over the row vectors.
__global__ void __launch_bounds__(256) silu_mul_kernel(const uint16_t* __restrict__ h, int64_t inter,
                                                       int64_t ldh, uint16_t* __restrict__ y,
                                                       int64_t ldy, int64_t n_vec) {
  const int64_t vpr = inter / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n_vec; v += stride) {
    const int64_t r = v / vpr, c = (v - r * vpr) * 8;
    const uint4 gv = ld_stream(h + r * ldh + c);
    const uint4 uv = ld_stream(h + r * ldh + inter + c);
    *reinterpret_cast<uint4*>(y + r * ldy + c) = silu_mul8(gv, uv);
  }
}

// Gated activation + 1x128 quantization: the task layout of aquant_kernel
// over the [m, inter] output; each lane forms its 4 x 8 outputs from the
// gate and up halves of its row, then quantizes them like aquant_kernel.
__global__ void __launch_bounds__(256, 3) silu_quant_kernel(const uint16_t* __restrict__ h, int64_t m,
                                                         int64_t inter, int64_t ldh,
                                                         uint8_t* __restrict__ q,
                                                         float* __restrict__ scales,
                                                         int64_t n_tasks, int kb) {
  allow_dependent_launch();   // the grouped GEMM that reads these codes may launch now
  const int lane = threadIdx.x & 31;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int slot = lane & 3;
  const int64_t groups = m * kb;
  for (int64_t task = gw; task < n_tasks; task += nw) {
    const int64_t f = task * 8 + (lane >> 2);
    const bool valid = f < groups;
    const int64_t r = valid ? f / kb : 0;
    const int g = (int)(f - r * kb);
    const int64_t gcol = (int64_t)g * 128;
    const uint16_t* hrow = h + r * ldh;
    uint4 gv[4], uv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t col = gcol + (slot + 4 * i) * 8;
      if (valid && col < inter) {
        gv[i] = ld_stream(hrow + col);
        uv[i] = ld_stream(hrow + inter + col);
      }
    }
    uint4 v[4];
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t col = gcol + (slot + 4 * i) * 8;
      v[i] = (valid && col < inter) ? silu_mul8(gv[i], uv[i]) : make_uint4(0, 0, 0, 0);
      m2 = absmax8(m2, v[i]);
    }
    const float amax = warp_max(bf16x2_maxf(m2), 4);
    const float s = fx::fdiv(amax, 448.0f);
    if (slot == 0 && valid) scales[(int64_t)g * m + r] = s;
    const ScaleDiv sd = make_scale_div(s);
    uint8_t* qrow = q + r * inter;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t col = gcol + (slot + 4 * i) * 8;
      if (valid && col < inter) *reinterpret_cast<uint2*>(qrow + col) = quant8_any<false>(v[i], sd);
    }
  }
}

// ----------------------------------------------------------- KV cache -----

// Thread t of a 256-thread CTA owns 16-byte vector slot t % vpr of a row
// (vpr = heads*head_dim/8 vectors per row), so its head is fixed; the CTA
// walks rows 256/vpr at a time with a grid stride.
struct KVMap {
  int vpr, rpp, hd;
  __device__ __forceinline__ bool active(int t) const { return t / vpr < rpp; }
};

__global__ void __launch_bounds__(256) kv_amax_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                      KVMap mp, uint32_t* __restrict__ amax_out,
                                                      int heads) {
  __shared__ uint32_t sm[256];
  const int t = threadIdx.x;
  sm[t] = 0;
  __syncthreads();
  if (mp.active(t)) {
    const int v = t % mp.vpr, rsub = t / mp.vpr;
    const int64_t row_elems = (int64_t)mp.vpr * 8;
    const int64_t stride = (int64_t)gridDim.x * mp.rpp;
    uint32_t m2 = 0;
    int64_t r = (int64_t)blockIdx.x * mp.rpp + rsub;
    for (; r + 3 * stride < rows; r += 4 * stride) {
      uint4 a0 = ld_stream(x + r * row_elems + v * 8);
      uint4 a1 = ld_stream(x + (r + stride) * row_elems + v * 8);
      uint4 a2 = ld_stream(x + (r + 2 * stride) * row_elems + v * 8);
      uint4 a3 = ld_stream(x + (r + 3 * stride) * row_elems + v * 8);
      m2 = absmax8(absmax8(absmax8(absmax8(m2, a0), a1), a2), a3);
    }
    for (; r < rows; r += stride) m2 = absmax8(m2, ld_stream(x + r * row_elems + v * 8));
    const float am = bf16x2_maxf(m2);
    atomicMax(&sm[(v * 8) / mp.hd], __float_as_uint(am));   // non-negative: int order = float order
  }
  __syncthreads();
  if (t < heads && sm[t] != 0) atomicMax(&amax_out[t], sm[t]);
}

template <bool kCalibrated>
__global__ void __launch_bounds__(256) kv_quant_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                       KVMap mp, const float* __restrict__ scales_in,
                                                       const uint32_t* __restrict__ amax_ws,
                                                       float* __restrict__ scales_out,
                                                       uint8_t* __restrict__ q, int heads) {
  const int t = threadIdx.x;
  if (kCalibrated && blockIdx.x == 0 && t < heads)
    scales_out[t] = fx::fdiv(__uint_as_float(amax_ws[t]), 448.0f);
  if (!mp.active(t)) return;
  const int v = t % mp.vpr, rsub = t / mp.vpr;
  const int h = (v * 8) / mp.hd;
  const float s = kCalibrated ? fx::fdiv(__uint_as_float(amax_ws[h]), 448.0f) : scales_in[h];
  const ScaleDiv sd = make_scale_div(s);
  const int64_t row_elems = (int64_t)mp.vpr * 8;
  const int64_t stride = (int64_t)gridDim.x * mp.rpp;
  int64_t r = (int64_t)blockIdx.x * mp.rpp + rsub;
  for (; r + 3 * stride < rows; r += 4 * stride) {
    uint4 a0 = ld_stream(x + r * row_elems + v * 8);
    uint4 a1 = ld_stream(x + (r + stride) * row_elems + v * 8);
    uint4 a2 = ld_stream(x + (r + 2 * stride) * row_elems + v * 8);
    uint4 a3 = ld_stream(x + (r + 3 * stride) * row_elems + v * 8);
    *reinterpret_cast<uint2*>(q + r * row_elems + v * 8) = quant8_any<!kCalibrated>(a0, sd);
    *reinterpret_cast<uint2*>(q + (r + stride) * row_elems + v * 8) = quant8_any<!kCalibrated>(a1, sd);
    *reinterpret_cast<uint2*>(q + (r + 2 * stride) * row_elems + v * 8) = quant8_any<!kCalibrated>(a2, sd);
    *reinterpret_cast<uint2*>(q + (r + 3 * stride) * row_elems + v * 8) = quant8_any<!kCalibrated>(a3, sd);
  }
  for (; r < rows; r += stride)
    *reinterpret_cast<uint2*>(q + r * row_elems + v * 8) =
        quant8_any<!kCalibrated>(ld_stream(x + r * row_elems + v * 8), sd);
}

int grid_for(int64_t work_ctas, const DeviceState* ds, int per_sm) {
  int64_t cap = (int64_t)ds->sm_count * per_sm;
  return (int)std::max<int64_t>(1, std::min<int64_t>(work_ctas, cap));
}

}  // namespace
}  // namespace fp8rl

using namespace fp8rl;

extern "C" fp8rl_status fp8rl_quantize_act_groupwise(const void* a, int64_t m, int64_t k,
                                                     int64_t lda, uint8_t* q, float* scales,
                                                     cudaStream_t stream) {
  if (!a || !q || !scales) return fail(FP8RL_ERR_INVALID_ARG, "null pointer");
  if (m < 1 || k < 1 || lda < k)
    return fail(FP8RL_ERR_INVALID_ARG, "need m, k >= 1 and lda >= k (m=%lld k=%lld lda=%lld)",
                (long long)m, (long long)k, (long long)lda);
  if (k % 8 || lda % 8) return fail(FP8RL_ERR_ALIGNMENT, "k and lda must be multiples of 8");
  if (!aligned(a, 16) || !aligned(q, 8) || !aligned(scales, 4))
    return fail(FP8RL_ERR_ALIGNMENT, "a must be 16-byte and q 8-byte aligned");
  DeviceState* ds = nullptr;
  fp8rl_status st = device_state(&ds);
  if (st != FP8RL_OK) return st;
  const int kb = (int)((k + 127) / 128);
  const int64_t tasks = (m * kb + 7) / 8;
  const int64_t ctas = (tasks + 7) / 8;
  static const int per_sm = resident_ctas_per_sm(aquant_kernel<false>, 256);
  aquant_kernel<false><<<grid_for(ctas, ds, per_sm), 256, 0, stream>>>(
      reinterpret_cast<const uint16_t*>(a), m, k, lda, q, scales, tasks, kb, nullptr, m, ds->status);
  st = cuda_check(cudaGetLastError(), "aquant_kernel launch");
  return st == FP8RL_OK ? ok() : st;
}

extern "C" fp8rl_status fp8rl_quantize_act_gather(const void* a, int64_t m_src, int64_t k,
                                                  int64_t lda, const int32_t* rows, int64_t m,
                                                  uint8_t* q, float* scales, cudaStream_t stream) {
  if (m < 0 || m_src < 0 || k < 1 || lda < k)
    return fail(FP8RL_ERR_INVALID_ARG, "need m, m_src >= 0, k >= 1 and lda >= k");
  if (m == 0) return ok();
  if (!a || !rows || !q || !scales) return fail(FP8RL_ERR_INVALID_ARG, "null pointer");
  if (k % 8 || lda % 8) return fail(FP8RL_ERR_ALIGNMENT, "k and lda must be multiples of 8");
  if (!aligned(a, 16) || !aligned(q, 8) || !aligned(scales, 4) || !aligned(rows, 4))
    return fail(FP8RL_ERR_ALIGNMENT, "a must be 16-byte, q 8-byte and rows 4-byte aligned");
  DeviceState* ds = nullptr;
  fp8rl_status st = device_state(&ds);
  if (st != FP8RL_OK) return st;
  const int kb = (int)((k + 127) / 128);
  const int64_t tasks = (m * kb + 7) / 8;
  const int64_t ctas = (tasks + 7) / 8;
  static const int per_sm = resident_ctas_per_sm(aquant_kernel<true>, 256);
  aquant_kernel<true><<<grid_for(ctas, ds, per_sm), 256, 0, stream>>>(
      reinterpret_cast<const uint16_t*>(a), m, k, lda, q, scales, tasks, kb, rows, m_src,
      ds->status);
  st = cuda_check(cudaGetLastError(), "aquant_kernel (gather) launch");
  return st == FP8RL_OK ? ok() : st;
}

namespace fp8rl {
fp8rl_status init_glue_tables() {
  silu_table_kernel<<<65536 / 256, 256>>>();
  fp8rl_status st = cuda_check(cudaGetLastError(), "silu_table_kernel launch");
  if (st != FP8RL_OK) return st;
  return cuda_check(cudaDeviceSynchronize(), "building the SiLU table");
}
}  // namespace fp8rl

extern "C" fp8rl_status fp8rl_silu_mul_quantize(const void* h, int64_t m, int64_t inter,
                                                int64_t ldh, uint8_t* q, float* scales,
                                                cudaStream_t stream) {
  if (m < 0 || inter < 1 || ldh < 2 * inter)
    return fail(FP8RL_ERR_INVALID_ARG, "need m >= 0, inter >= 1 and ldh >= 2 * inter");
  if (m == 0) return ok();
  if (!h || !q || !scales) return fail(FP8RL_ERR_INVALID_ARG, "null pointer");
  if (inter % 8 || ldh % 8) return fail(FP8RL_ERR_ALIGNMENT, "inter and ldh must be multiples of 8");
  if (!aligned(h, 16) || !aligned(q, 8) || !aligned(scales, 4))
    return fail(FP8RL_ERR_ALIGNMENT, "h must be 16-byte and q 8-byte aligned");
  DeviceState* ds = nullptr;
  fp8rl_status st = device_state(&ds);
  if (st != FP8RL_OK) return st;
  const int kb = (int)((inter + 127) / 128);
  const int64_t tasks = (m * kb + 7) / 8;
  const int64_t ctas = (tasks + 7) / 8;
  static const int per_sm = resident_ctas_per_sm(silu_quant_kernel, 256);
  silu_quant_kernel<<<grid_for(ctas, ds, per_sm), 256, 0, stream>>>(
      reinterpret_cast<const uint16_t*>(h), m, inter, ldh, q, scales, tasks, kb);
  st = cuda_check(cudaGetLastError(), "silu_quant_kernel launch");
  return st == FP8RL_OK ? ok() : st;
}

extern "C" fp8rl_status fp8rl_silu_mul_bf16(const void* h, int64_t m, int64_t inter, int64_t ldh,
                                            void* y, int64_t ldy, cudaStream_t stream) {
  if (m < 0 || inter < 1 || ldh < 2 * inter || ldy < inter)
    return fail(FP8RL_ERR_INVALID_ARG, "need m >= 0, inter >= 1, ldh >= 2 * inter, ldy >= inter");
  if (m == 0) return ok();
  if (!h || !y) return fail(FP8RL_ERR_INVALID_ARG, "null pointer");
  if (inter % 8 || ldh % 8 || ldy % 8)
    return fail(FP8RL_ERR_ALIGNMENT, "inter, ldh and ldy must be multiples of 8");
  if (!aligned(h, 16) || !aligned(y, 16))
    return fail(FP8RL_ERR_ALIGNMENT, "h and y must be 16-byte aligned");
  DeviceState* ds = nullptr;
  fp8rl_status st = device_state(&ds);
  if (st != FP8RL_OK) return st;
  const int64_t n_vec = m * (inter / 8);
  static const int per_sm = resident_ctas_per_sm(silu_mul_kernel, 256);
  silu_mul_kernel<<<grid_for((n_vec + 255) / 256, ds, per_sm), 256, 0, stream>>>(
      reinterpret_cast<const uint16_t*>(h), inter, ldh, reinterpret_cast<uint16_t*>(y), ldy, n_vec);
  st = cuda_check(cudaGetLastError(), "silu_mul_kernel launch");
  return st == FP8RL_OK ? ok() : st;
}

extern "C" fp8rl_status fp8rl_quantize_kv_fp8(const void* x, int64_t rows, int32_t heads,
                                              int32_t head_dim, int32_t mode, float* scales,
                                              uint8_t* q, cudaStream_t stream) {
  if (!x || !scales || !q) return fail(FP8RL_ERR_INVALID_ARG, "null pointer");
  if (rows < 0 || heads < 1 || head_dim < 1)
    return fail(FP8RL_ERR_INVALID_ARG, "need rows >= 0, heads >= 1, head_dim >= 1");
  if (mode != FP8RL_KV_GIVEN && mode != FP8RL_KV_CALIBRATE)
    return fail(FP8RL_ERR_INVALID_ARG, "mode must be FP8RL_KV_GIVEN or FP8RL_KV_CALIBRATE");
  if (head_dim % 8) return fail(FP8RL_ERR_ALIGNMENT, "head_dim must be a multiple of 8");
  if ((int64_t)heads * head_dim > 2048 || heads > 256)
    return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "need heads*head_dim <= 2048 and heads <= 256");
  if (!aligned(x, 16) || !aligned(q, 8) || !aligned(scales, 4))
    return fail(FP8RL_ERR_ALIGNMENT, "x must be 16-byte and q 8-byte aligned");
  DeviceState* ds = nullptr;
  fp8rl_status st = device_state(&ds);
  if (st != FP8RL_OK) return st;
  KVMap mp;
  mp.vpr = heads * head_dim / 8;
  mp.rpp = 256 / mp.vpr;
  mp.hd = head_dim;
  const int64_t ctas = rows > 0 ? (rows + mp.rpp - 1) / mp.rpp : 1;
  const int grid = grid_for(ctas, ds, 8);
  const uint16_t* xb = reinterpret_cast<const uint16_t*>(x);
  if (mode == FP8RL_KV_CALIBRATE) {
    st = cuda_check(cudaMemsetAsync(ds->kv_amax, 0, sizeof(uint32_t) * heads, stream),
                    "clearing calibration slots");
    if (st != FP8RL_OK) return st;
    kv_amax_kernel<<<grid, 256, 0, stream>>>(xb, rows, mp, ds->kv_amax, heads);
    st = cuda_check(cudaGetLastError(), "kv_amax_kernel launch");
    if (st != FP8RL_OK) return st;
    kv_quant_kernel<true><<<grid, 256, 0, stream>>>(xb, rows, mp, nullptr, ds->kv_amax, scales,
                                                    q, heads);
  } else {
    kv_quant_kernel<false><<<grid, 256, 0, stream>>>(xb, rows, mp, scales, nullptr, nullptr, q,
                                                     heads);
  }
  st = cuda_check(cudaGetLastError(), "kv_quant_kernel launch");
  return st == FP8RL_OK ? ok() : st;
}

// ------------------------------------------ allocation-free KV calibration --
//
// Same computation as fp8rl_quantize_kv_fp8(..., FP8RL_KV_CALIBRATE, ...), for
// callers that cannot have the library allocate device memory: the per-head
// max slots live in the file-scope array below instead of the library
// workspace.  Nothing here calls cudaMalloc, cudaFree or any other allocating
// routine.  The array persists in every device that loads the library until
// the process exits, is shared by every call of this entry point on that
// device, and is cleared on the stream at the start of each call.

constexpr int kNoAllocMaxHeads = 256;                 // 1 KB of device memory
static __device__ __align__(256) uint32_t g_kv_amax_noalloc[kNoAllocMaxHeads];

namespace {
struct NoAllocDevice {
  uint32_t* amax = nullptr;   // device address of g_kv_amax_noalloc
  int sm_count = 0;
};
std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc[64];
}  // namespace

extern "C" fp8rl_status fp8rl_quantize_kv_fp8_calibrate_noalloc(const void* x, int64_t rows,
                                                               int32_t heads, int32_t head_dim,
                                                               float* scales, uint8_t* q,
                                                               cudaStream_t stream) {
  if (!x || !scales || !q) return fail(FP8RL_ERR_INVALID_ARG, "null pointer");
  if (rows < 0 || heads < 1 || head_dim < 1)
    return fail(FP8RL_ERR_INVALID_ARG, "need rows >= 0, heads >= 1, head_dim >= 1");
  if (heads > kNoAllocMaxHeads)
    return fail(FP8RL_ERR_UNSUPPORTED_SHAPE,
                "the allocation-free variant supports at most %d heads (got %d): its scratch is a "
                "fixed %d-entry device array",
                kNoAllocMaxHeads, heads, kNoAllocMaxHeads);
  if (head_dim % 8) return fail(FP8RL_ERR_ALIGNMENT, "head_dim must be a multiple of 8");
  if ((int64_t)heads * head_dim > 2048)
    return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "need heads*head_dim <= 2048");
  if (!aligned(x, 16) || !aligned(q, 8) || !aligned(scales, 4))
    return fail(FP8RL_ERR_ALIGNMENT, "x must be 16-byte and q 8-byte aligned");
  int dev = -1;
  fp8rl_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != FP8RL_OK) return st;
  if (dev < 0 || dev >= 64) return fail(FP8RL_ERR_UNSUPPORTED_DEVICE, "device %d", dev);
  NoAllocDevice nd;
  {
    // First call on this device (with it current): resolve the array's device
    // address and the SM count.  Later calls reuse them.
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocDevice& slot = g_noalloc[dev];
    if (!slot.amax) {
      int major = 0, minor = 0, sms = 0;
      st = cuda_check(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev),
                      "cudaDeviceGetAttribute");
      if (st == FP8RL_OK)
        st = cuda_check(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev),
                        "cudaDeviceGetAttribute");
      if (st == FP8RL_OK)
        st = cuda_check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
                        "cudaDeviceGetAttribute");
      if (st != FP8RL_OK) return st;
      if (!(major == 10 && minor == 3))
        return fail(FP8RL_ERR_UNSUPPORTED_DEVICE,
                    "fp8rl is built for sm_103a (GB300); device %d is sm_%d%d", dev, major, minor);
      void* ptr = nullptr;
      st = cuda_check(cudaGetSymbolAddress(&ptr, g_kv_amax_noalloc),
                      "cudaGetSymbolAddress(g_kv_amax_noalloc)");
      if (st != FP8RL_OK) return st;
      slot.amax = static_cast<uint32_t*>(ptr);
      slot.sm_count = sms;
    }
    nd = slot;
  }
  KVMap mp;
  mp.vpr = heads * head_dim / 8;
  mp.rpp = 256 / mp.vpr;
  mp.hd = head_dim;
  const int64_t ctas = rows > 0 ? (rows + mp.rpp - 1) / mp.rpp : 1;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ctas, (int64_t)nd.sm_count * 8));
  const uint16_t* xb = reinterpret_cast<const uint16_t*>(x);
  // the slots keep the previous call's maxima: clear the ones this call uses
  st = cuda_check(cudaMemsetAsync(nd.amax, 0, sizeof(uint32_t) * heads, stream),
                  "clearing the allocation-free calibration slots");
  if (st != FP8RL_OK) return st;
  kv_amax_kernel<<<grid, 256, 0, stream>>>(xb, rows, mp, nd.amax, heads);
  st = cuda_check(cudaGetLastError(), "kv_amax_kernel launch");
  if (st != FP8RL_OK) return st;
  kv_quant_kernel<true><<<grid, 256, 0, stream>>>(xb, rows, mp, nullptr, nd.amax, scales, q, heads);
  st = cuda_check(cudaGetLastError(), "kv_quant_kernel launch");
  return st == FP8RL_OK ? ok() : st;
}
