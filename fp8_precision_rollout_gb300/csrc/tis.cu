// tis.cu -- token-level truncated importance-sampling weights.
//
// FP8-RL summary, section 3.4.3: the weight of a token is the ratio of the
// training policy's probability to the FP8 rollout policy's,
// w = exp(logp_train - logp_rollout), truncated at C (= 2 in all of the pages'
// experiments; the same section also states the two-sided range [1/C, C]).
// Here d = fl32(logp_train - logp_rollout), e = RN32(e^d) exactly (see
// fp_exact.cuh), w = min(e, c_hi), then max(w, c_lo) when c_lo > 0, NaN kept,
// and w = 0 for masked-out tokens.  Elementwise: 16-byte loads, 8 to 16 tokens
// per thread per round with all loads issued first, sized so that one resident
// wave covers the input (grid-stride beyond that); each lane holds
// one entry of the 2^(j/32) table in registers and lanes fetch theirs with a
// warp shuffle.
#include <algorithm>
#include <cmath>

#include "fp_exact.cuh"
#include "internal.h"

namespace fp8rl {
namespace {

// One token.  th_lane / tl_lane hold 2^(lane/32) (float-float) in this lane;
// every lane of the warp calls this together (the table lookup is a warp
// shuffle), before any per-lane branch.
// e = RN32(e^d).  Every lane of the warp calls this together (warp shuffles).
__device__ __forceinline__ float tis_e(float d, float th_lane, float tl_lane, const fx::Exp2Table& T) {
  const float kf = fx::exp_fast_k(d);
  const int j = fx::exp_fast_index_k(kf);
  const float th = __shfl_sync(0xFFFFFFFFu, th_lane, j);
  const float tl = __shfl_sync(0xFFFFFFFFu, tl_lane, j);
  float e;
  if (!fx::exp_rn32_fast_with_k(d, kf, th, tl, &e)) e = fx::exp_rn32_slow(d, T);
  return e;
}

__device__ __forceinline__ float tis_one(float lt, float lr, float c_hi, float c_lo, float th_lane,
                                         float tl_lane, const fx::Exp2Table& T) {
  const float e = tis_e(fx::fsub(lt, lr), th_lane, tl_lane, T);
  float w = (e > c_hi) ? c_hi : e;
  if (c_lo > 0.0f && e < c_lo) w = c_lo;
  return w;
}

__device__ __forceinline__ float4 tis_four(float4 a, float4 b, float c_hi, float c_lo,
                                           float th_lane, float tl_lane, const fx::Exp2Table& T) {
  float4 r;
  r.x = tis_one(a.x, b.x, c_hi, c_lo, th_lane, tl_lane, T);
  r.y = tis_one(a.y, b.y, c_hi, c_lo, th_lane, tl_lane, T);
  r.z = tis_one(a.z, b.z, c_hi, c_lo, th_lane, tl_lane, T);
  r.w = tis_one(a.w, b.w, c_hi, c_lo, th_lane, tl_lane, T);
  return r;
}

__device__ __forceinline__ void tis_store4(float4 r, int64_t i, const uint8_t* __restrict__ mask,
                                           float* __restrict__ w) {
  if (mask) {
    const uint32_t mk = __ldg(reinterpret_cast<const unsigned int*>(mask) + i);
    if (!(mk & 0xFFu)) r.x = 0.0f;
    if (!(mk & 0xFF00u)) r.y = 0.0f;
    if (!(mk & 0xFF0000u)) r.z = 0.0f;
    if (!(mk & 0xFF000000u)) r.w = 0.0f;
  }
  reinterpret_cast<float4*>(w)[i] = r;
}

// A warp task is 32*V consecutive 4-token vectors: lane l takes vectors
// l + 32u (u < V), all loaded before any is computed.  The host picks the
// smallest V in [2, 4] for which one resident wave of warps covers the whole
// input, so no token waits for a second round of load latency.  Warp-uniform
// trip count so every lane reaches the shuffles.
template <int V>
__global__ void __launch_bounds__(256) tis_kernel(const float* __restrict__ lt,
                                                  const float* __restrict__ lr,
                                                  const uint8_t* __restrict__ mask, int64_t n,
                                                  float c_hi, float c_lo, float* __restrict__ w,
                                                  const __grid_constant__ fx::Exp2Table T) {
  const int lane = threadIdx.x & 31;
  const float th_lane = T.hi[lane];
  const float tl_lane = T.lo[lane];
  const int64_t n4 = n >> 2;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const float4* lt4 = reinterpret_cast<const float4*>(lt);
  const float4* lr4 = reinterpret_cast<const float4*>(lr);
  for (int64_t v0 = gw * (32 * V); v0 < n4; v0 += nwarps * (32 * V)) {
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 a[V], b[V];
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const int64_t i = v0 + lane + 32 * u;
      a[u] = i < n4 ? __ldg(lt4 + i) : z;
      b[u] = i < n4 ? __ldg(lr4 + i) : z;
    }
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const int64_t i = v0 + lane + 32 * u;
      const float4 r = tis_four(a[u], b[u], c_hi, c_lo, th_lane, tl_lane, T);
      if (i < n4) tis_store4(r, i, mask, w);
    }
  }
  // ragged tail (n % 4 tokens): the first warp of block 0
  const int64_t tail = n - (n4 << 2);
  if (blockIdx.x == 0 && threadIdx.x < 32) {
    const int64_t j = (n4 << 2) + lane;
    const bool in = lane < tail;
    float r = tis_one(in ? lt[j] : 0.f, in ? lr[j] : 0.f, c_hi, c_lo, th_lane, tl_lane, T);
    if (in) {
      if (mask && !mask[j]) r = 0.0f;
      w[j] = r;
    }
  }
}

// ------------------------------------------ weights + mismatch statistics --

// Float-float running sum (hi + lo), exact up to ~2^-44 relative: FP64 is
// slow on this part, so FP32 two-sums carry the extra precision.
struct FF {
  float hi = 0.f, lo = 0.f;
  // Once hi is +-inf or NaN it alone carries the IEEE sum (lo would be NaN).
  __device__ __forceinline__ void add(float x) {
    float s, e;
    fx::two_sum(hi, x, s, e);
    hi = s;
    lo = fabsf(s) <= 3.402823466e38f ? fx::fadd(lo, e) : 0.f;
  }
  __device__ __forceinline__ void add(FF o) {
    add(o.hi);
    lo = fabsf(hi) <= 3.402823466e38f ? fx::fadd(lo, o.lo) : 0.f;
  }
  __device__ __forceinline__ double value() const { return (double)hi + (double)lo; }
};

// Running statistics of one thread: FP32 partial sums over at most 8 tokens
// (two 4-token vectors), then folded into float-float sums.
struct IsAcc {
  float k1 = 0.f, k3 = 0.f, r = 0.f, l = 0.f;
  FF K1, K3, R, L;
  int nv = 0, nc = 0;
  __device__ __forceinline__ void fold() {
    K1.add(k1);
    K3.add(k3);
    R.add(r);
    L.add(l);
    k1 = k3 = r = l = 0.f;
  }
};

__device__ __forceinline__ FF warp_sum(FF v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    FF w;
    w.hi = __shfl_xor_sync(0xFFFFFFFFu, v.hi, o);
    w.lo = __shfl_xor_sync(0xFFFFFFFFu, v.lo, o);
    v.add(w);
  }
  return v;
}

// One token: weight by mode (0 = truncate, 1 = mask), statistics if valid;
// `loss` is the token's loss (0 when the call has none), weighted by w.
template <int kMode>
__device__ __forceinline__ float is_one(float lt, float lr, float loss, bool valid, float c_hi,
                                        float c_lo, float th_lane, float tl_lane,
                                        const fx::Exp2Table& T, IsAcc& acc) {
  const float d = fx::fsub(lt, lr);
  const float e = tis_e(d, th_lane, tl_lane, T);
  float w;
  bool changed;
  if (kMode == 0) {
    w = (e > c_hi) ? c_hi : e;
    changed = e > c_hi;
    if (c_lo > 0.0f && e < c_lo) {
      w = c_lo;
      changed = true;
    }
  } else {
    const bool keep = (e >= c_lo) && (e <= c_hi);
    w = keep ? e : 0.0f;
    changed = !keep;
  }
  if (!valid) return 0.0f;
  acc.k1 = fx::fadd(acc.k1, fx::fsub(lr, lt));
  acc.k3 = fx::fadd(acc.k3, fx::fsub(fx::fsub(e, 1.0f), d));
  acc.r = fx::fadd(acc.r, e);
  acc.l = fx::fadd(acc.l, fx::fmul(w, loss));
  acc.nv += 1;
  acc.nc += changed ? 1 : 0;
  return w;
}

template <int kMode>
__device__ __forceinline__ float4 is_four(float4 a, float4 b, float4 ls, uint32_t valid4, float c_hi,
                                          float c_lo, float th_lane, float tl_lane,
                                          const fx::Exp2Table& T, IsAcc& acc) {
  float4 r;
  r.x = is_one<kMode>(a.x, b.x, ls.x, valid4 & 1u, c_hi, c_lo, th_lane, tl_lane, T, acc);
  r.y = is_one<kMode>(a.y, b.y, ls.y, valid4 & 2u, c_hi, c_lo, th_lane, tl_lane, T, acc);
  r.z = is_one<kMode>(a.z, b.z, ls.z, valid4 & 4u, c_hi, c_lo, th_lane, tl_lane, T, acc);
  r.w = is_one<kMode>(a.w, b.w, ls.w, valid4 & 8u, c_hi, c_lo, th_lane, tl_lane, T, acc);
  return r;
}

// Valid-token bits of 4-token vector i (bit t: token 4i + t).
__device__ __forceinline__ uint32_t valid_bits(const uint8_t* __restrict__ mask, int64_t i, bool in) {
  if (!in) return 0u;
  if (!mask) return 0xFu;
  const uint32_t mk = __ldg(reinterpret_cast<const unsigned int*>(mask) + i);
  return ((mk & 0xFFu) ? 1u : 0u) | ((mk & 0xFF00u) ? 2u : 0u) | ((mk & 0xFF0000u) ? 4u : 0u) |
         ((mk & 0xFF000000u) ? 8u : 0u);
}

// Same traversal as tis_kernel; the statistics are reduced per CTA and added
// to stats[nstats] (cleared beforehand) with one FP64 atomic each; nstats = 6
// adds the loss-weighted sum (loss non-null), 5 otherwise.
template <int kMode, bool kW, int V>
__global__ void __launch_bounds__(256) is_stats_kernel(const float* __restrict__ lt,
                                                       const float* __restrict__ lr,
                                                       const uint8_t* __restrict__ mask,
                                                       const float* __restrict__ loss, int64_t n,
                                                       float c_hi, float c_lo, float* __restrict__ w,
                                                       double* __restrict__ stats, int nstats,
                                                       const __grid_constant__ fx::Exp2Table T) {
  __shared__ double red[8][6];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float th_lane = T.hi[lane];
  const float tl_lane = T.lo[lane];
  const int64_t n4 = n >> 2;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const float4* lt4 = reinterpret_cast<const float4*>(lt);
  const float4* lr4 = reinterpret_cast<const float4*>(lr);
  const float4* ls4 = reinterpret_cast<const float4*>(loss);
  IsAcc acc;
  for (int64_t v0 = gw * (32 * V); v0 < n4; v0 += nwarps * (32 * V)) {
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 a[V], b[V], l4[V];
    uint32_t mb[V];
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const int64_t i = v0 + lane + 32 * u;
      a[u] = i < n4 ? __ldg(lt4 + i) : z;
      b[u] = i < n4 ? __ldg(lr4 + i) : z;
      l4[u] = (loss && i < n4) ? __ldg(ls4 + i) : z;
      mb[u] = valid_bits(mask, i, i < n4);
    }
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const int64_t i = v0 + lane + 32 * u;
      const float4 r = is_four<kMode>(a[u], b[u], l4[u], mb[u], c_hi, c_lo, th_lane, tl_lane, T, acc);
      if (kW && i < n4) reinterpret_cast<float4*>(w)[i] = r;
      if ((u & 1) || u == V - 1) acc.fold();   // FP32 partials over at most 8 tokens
    }
  }
  // ragged tail (n % 4 tokens): the first warp of block 0
  const int64_t tail = n - (n4 << 2);
  if (blockIdx.x == 0 && warp == 0 && tail > 0) {
    const int64_t j = (n4 << 2) + lane;
    const bool in = lane < tail;
    const bool valid = in && (!mask || mask[j]);
    const float r = is_one<kMode>(in ? lt[j] : 0.f, in ? lr[j] : 0.f, (loss && in) ? loss[j] : 0.f,
                                  valid, c_hi, c_lo, th_lane, tl_lane, T, acc);
    acc.fold();
    if (kW && in) w[j] = r;
  }
  int nv = acc.nv, nc = acc.nc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    nv += __shfl_xor_sync(0xFFFFFFFFu, nv, o);
    nc += __shfl_xor_sync(0xFFFFFFFFu, nc, o);
  }
  const FF k1 = warp_sum(acc.K1), k3 = warp_sum(acc.K3), rr = warp_sum(acc.R);
  const FF ll = warp_sum(acc.L);
  if (lane == 0) {
    red[warp][0] = (double)nv;
    red[warp][1] = k1.value();
    red[warp][2] = k3.value();
    red[warp][3] = rr.value();
    red[warp][4] = (double)nc;
    red[warp][5] = ll.value();
  }
  __syncthreads();
  if ((int)threadIdx.x < nstats) {
    double t = 0.0;
    for (int k = 0; k < (int)(blockDim.x >> 5); ++k) t += red[k][threadIdx.x];
    atomicAdd(stats + threadIdx.x, t);
  }
}

// Vectors per lane V in [2, 4] and grid: the smallest V for which one
// resident wave of warps (per_sm[V - 2] CTAs of 8 warps per SM) takes every
// 4-token vector in a single task.  Inputs too large for that run V = 2 in a
// grid-stride loop (the fewest registers, the most resident warps).
struct WaveFit {
  int v;
  int64_t ctas;
};
WaveFit fit_wave(int64_t n, int sms, const int per_sm[3]) {
  const int64_t n4 = std::max<int64_t>(n >> 2, 1);
  for (int v = 2; v <= 4; ++v) {
    const int64_t tasks = (n4 + 32 * v - 1) / (32 * v);
    const int64_t ctas = (tasks + 7) / 8;
    const int64_t cap = (int64_t)sms * std::max(per_sm[v - 2], 1);
    if (ctas <= cap) return {v, ctas};
  }
  return {2, (int64_t)sms * std::max(per_sm[0], 1)};
}

template <int kMode, bool kW>
void launch_is_stats_v(int sms, cudaStream_t stream, const float* lt, const float* lr,
                       const uint8_t* mask, const float* loss, int64_t n, float c_hi, float c_lo,
                       float* w, double* stats, int nstats, const fx::Exp2Table& T) {
  static const int per_sm[3] = {resident_ctas_per_sm(is_stats_kernel<kMode, kW, 2>, 256),
                                resident_ctas_per_sm(is_stats_kernel<kMode, kW, 3>, 256),
                                resident_ctas_per_sm(is_stats_kernel<kMode, kW, 4>, 256)};
  const WaveFit f = fit_wave(n, sms, per_sm);
  const int v = f.v;
  const unsigned grid = (unsigned)f.ctas;
  if (v == 2)
    is_stats_kernel<kMode, kW, 2><<<grid, 256, 0, stream>>>(lt, lr, mask, loss, n, c_hi, c_lo, w,
                                                            stats, nstats, T);
  else if (v == 3)
    is_stats_kernel<kMode, kW, 3><<<grid, 256, 0, stream>>>(lt, lr, mask, loss, n, c_hi, c_lo, w,
                                                            stats, nstats, T);
  else
    is_stats_kernel<kMode, kW, 4><<<grid, 256, 0, stream>>>(lt, lr, mask, loss, n, c_hi, c_lo, w,
                                                            stats, nstats, T);
}

void launch_is_stats(int32_t mode, bool with_w, int sms, cudaStream_t stream, const float* lt,
                     const float* lr, const uint8_t* mask, const float* loss, int64_t n,
                     float c_hi, float c_lo, float* w, double* stats, int nstats,
                     const fx::Exp2Table& T) {
  if (mode == FP8RL_IS_TRUNCATE) {
    if (with_w)
      launch_is_stats_v<0, true>(sms, stream, lt, lr, mask, loss, n, c_hi, c_lo, w, stats, nstats, T);
    else
      launch_is_stats_v<0, false>(sms, stream, lt, lr, mask, loss, n, c_hi, c_lo, w, stats, nstats, T);
  } else {
    if (with_w)
      launch_is_stats_v<1, true>(sms, stream, lt, lr, mask, loss, n, c_hi, c_lo, w, stats, nstats, T);
    else
      launch_is_stats_v<1, false>(sms, stream, lt, lr, mask, loss, n, c_hi, c_lo, w, stats, nstats, T);
  }
}

}  // namespace
}  // namespace fp8rl

using namespace fp8rl;

extern "C" fp8rl_status fp8rl_tis_weights(const float* logp_train, const float* logp_rollout,
                                          const uint8_t* mask, int64_t n, float c_hi, float c_lo,
                                          float* w, cudaStream_t stream) {
  if (!logp_train || !logp_rollout || !w) return fail(FP8RL_ERR_INVALID_ARG, "null pointer");
  if (n < 0) return fail(FP8RL_ERR_INVALID_ARG, "n must be >= 0");
  if (!(c_hi > 0.0f) || !std::isfinite(c_hi) || !(c_lo >= 0.0f) || !(c_lo <= c_hi))
    return fail(FP8RL_ERR_INVALID_ARG, "need 0 <= c_lo <= c_hi, c_hi finite and > 0");
  if (!aligned(logp_train, 16) || !aligned(logp_rollout, 16) || !aligned(w, 16) ||
      (mask && !aligned(mask, 4)))
    return fail(FP8RL_ERR_ALIGNMENT, "log-prob and weight arrays must be 16-byte aligned, mask 4-byte");
  DeviceState* ds = nullptr;
  fp8rl_status st = device_state(&ds);
  if (st != FP8RL_OK) return st;
  if (n == 0) return ok();
  static const fx::Exp2Table T = fx::make_exp_tables();
  static const int per_sm[3] = {resident_ctas_per_sm(tis_kernel<2>, 256),
                                resident_ctas_per_sm(tis_kernel<3>, 256),
                                resident_ctas_per_sm(tis_kernel<4>, 256)};
  const WaveFit f = fit_wave(n, ds->sm_count, per_sm);
  const unsigned grid = (unsigned)f.ctas;
  if (f.v == 2)
    tis_kernel<2><<<grid, 256, 0, stream>>>(logp_train, logp_rollout, mask, n, c_hi, c_lo, w, T);
  else if (f.v == 3)
    tis_kernel<3><<<grid, 256, 0, stream>>>(logp_train, logp_rollout, mask, n, c_hi, c_lo, w, T);
  else
    tis_kernel<4><<<grid, 256, 0, stream>>>(logp_train, logp_rollout, mask, n, c_hi, c_lo, w, T);
  st = cuda_check(cudaGetLastError(), "tis_kernel launch");
  return st == FP8RL_OK ? ok() : st;
}

namespace {
fp8rl_status is_stats_call(const float* logp_train, const float* logp_rollout, const uint8_t* mask,
                           const float* loss, int64_t n, float c_hi, float c_lo, int32_t mode,
                           float* w, double* stats, int nstats, cudaStream_t stream) {
  if (!stats || (n > 0 && (!logp_train || !logp_rollout)))
    return fail(FP8RL_ERR_INVALID_ARG, "null pointer");
  if (nstats == 6 && n > 0 && !loss) return fail(FP8RL_ERR_INVALID_ARG, "null loss");
  if (n < 0) return fail(FP8RL_ERR_INVALID_ARG, "n must be >= 0");
  if (mode != FP8RL_IS_TRUNCATE && mode != FP8RL_IS_MASK)
    return fail(FP8RL_ERR_INVALID_ARG, "mode must be FP8RL_IS_TRUNCATE or FP8RL_IS_MASK");
  if (!(c_hi > 0.0f) || !std::isfinite(c_hi) || !(c_lo >= 0.0f) || !(c_lo <= c_hi))
    return fail(FP8RL_ERR_INVALID_ARG, "need 0 <= c_lo <= c_hi, c_hi finite and > 0");
  if (!aligned(logp_train, 16) || !aligned(logp_rollout, 16) || (w && !aligned(w, 16)) ||
      (mask && !aligned(mask, 4)) || (loss && !aligned(loss, 16)) || !aligned(stats, 8))
    return fail(FP8RL_ERR_ALIGNMENT,
                "log-prob, loss and weight arrays must be 16-byte aligned, mask 4-byte, stats 8-byte");
  DeviceState* ds = nullptr;
  fp8rl_status st = device_state(&ds);
  if (st != FP8RL_OK) return st;
  st = cuda_check(cudaMemsetAsync(stats, 0, (size_t)nstats * sizeof(double), stream),
                  "cudaMemsetAsync(stats)");
  if (st != FP8RL_OK || n == 0) return st == FP8RL_OK ? ok() : st;
  static const fx::Exp2Table T = fx::make_exp_tables();
  launch_is_stats(mode, w != nullptr, ds->sm_count, stream, logp_train, logp_rollout, mask,
                  nstats == 6 ? loss : nullptr, n, c_hi, c_lo, w, stats, nstats, T);
  st = cuda_check(cudaGetLastError(), "is_stats_kernel launch");
  return st == FP8RL_OK ? ok() : st;
}
}  // namespace

extern "C" fp8rl_status fp8rl_is_weights_stats(const float* logp_train, const float* logp_rollout,
                                               const uint8_t* mask, int64_t n, float c_hi,
                                               float c_lo, int32_t mode, float* w, double* stats,
                                               cudaStream_t stream) {
  return is_stats_call(logp_train, logp_rollout, mask, nullptr, n, c_hi, c_lo, mode, w, stats, 5,
                       stream);
}

extern "C" fp8rl_status fp8rl_is_weights_stats_loss(const float* logp_train,
                                                    const float* logp_rollout, const uint8_t* mask,
                                                    const float* loss, int64_t n, float c_hi,
                                                    float c_lo, int32_t mode, float* w,
                                                    double* stats, cudaStream_t stream) {
  return is_stats_call(logp_train, logp_rollout, mask, loss, n, c_hi, c_lo, mode, w, stats, 6,
                       stream);
}
