// wquant.cu -- blockwise 128x128 weight re-quantization, one tensor or a
// whole model's tensors in one launch (FP8-RL summary, sections 3.4.1 and
// 3.4.2 Phase 2 step 2): per block scale = fl32(amax/448), codes
// E4M3_RNE_satfinite(fl32(x/scale)), the element map of quant_common.cuh.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "quant_common.cuh"

namespace fp8rl {
namespace {

// -------------------------------------------------- 128x128 weight blocks --
//
// Persistent: each CTA (256 threads, 2 per SM) walks blocks blockIdx.x,
// +gridDim.x, ... of all tensors of the launch.  Thread t holds rows t/16 +
// 16j (j < 8) and columns (t%16)*8 .. +8 of a block in registers, loaded with
// 16-byte non-allocating loads, so the block max and the codes need a single
// HBM read.  The next block's loads are issued before the current block is
// quantized: two blocks per CTA are in flight.  The block max is a bf16x2
// max over bit patterns, warp shuffles and one CTA barrier; codes go out as
// 8-byte stores.  Edge blocks load zeros outside the tensor (the max of the
// valid elements is unchanged) and mask their stores.  A CTA visits blocks in
// increasing order, so its tensor index only moves forward.

constexpr int kWQMaxDescs = 160;
constexpr int kWQThreads = 256;

struct WQDesc {
  const uint16_t* w;
  uint8_t* q;
  float* scales;
  int64_t ldw, ldq;
  int32_t n, k, kb, pad;
};

struct WQParams {
  WQDesc d[kWQMaxDescs];
  int32_t start[kWQMaxDescs + 1];   // first block id of each tensor; start[count] = total
  int32_t count;
  int32_t total;
  uint32_t* status;
};

__device__ __forceinline__ int wq_find(const WQParams& p, int b) {
  int lo = 0, hi = p.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.start[mid] <= b) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct WQBlock {
  int t, bi, bj;
};

// Block b of the launch; blocks are visited in increasing order by a CTA, so
// the tensor index only moves forward from the previous block's (t).
__device__ __forceinline__ WQBlock wq_block(const WQParams& p, int b, int t) {
  WQBlock x;
  while (t + 1 < p.count && p.start[t + 1] <= b) ++t;
  x.t = t;
  const int local = b - p.start[x.t];
  const int kb = p.d[x.t].kb;
  x.bi = local / kb;
  x.bj = local - x.bi * kb;
  return x;
}

// thread tid holds rows bi*128 + tid/16 + 16j (j < 8), columns bj*128 + (tid%16)*8 .. +8
__device__ __forceinline__ void wq_load(const WQParams& p, const WQBlock& x, int tid, uint4 (&v)[8]) {
  const WQDesc& d = p.d[x.t];
  const int col = x.bj * 128 + (tid & 15) * 8;
  const int r0 = x.bi * 128 + (tid >> 4);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = r0 + 16 * j;
    v[j] = (r < d.n && col < d.k) ? ld_stream(d.w + (int64_t)r * d.ldw + col) : make_uint4(0, 0, 0, 0);
  }
}

__global__ void __launch_bounds__(kWQThreads) wquant_kernel(const __grid_constant__ WQParams p) {
  __shared__ float red[2][8];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint4 cur[8], nxt[8];
  int b = blockIdx.x;
  WQBlock xc = {0, 0, 0}, xn = {0, 0, 0};
  if (b < p.total) {
    xc = wq_block(p, b, wq_find(p, b));
    wq_load(p, xc, tid, cur);
  }
  xn = xc;
  for (uint32_t i = 0; b < p.total; b += gridDim.x, ++i) {
    const int bn = b + gridDim.x;
    if (bn < p.total) {
      xn = wq_block(p, bn, xn.t);
      wq_load(p, xn, tid, nxt);
    }
    const WQDesc& d = p.d[xc.t];
    uint32_t m2 = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) m2 = absmax8(m2, cur[j]);
    float amax = warp_max(bf16x2_maxf(m2), 32);
    if (lane == 0) red[i & 1][warp] = amax;
    __syncthreads();
    amax = red[i & 1][0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[i & 1][w]);
    const float sc = fx::fdiv(amax, 448.0f);
    if (tid == 0) d.scales[(int64_t)xc.bi * d.kb + xc.bj] = sc;
    const ScaleDiv sd = make_scale_div(sc);
    const int col = xc.bj * 128 + (tid & 15) * 8;
    const int row0 = xc.bi * 128 + (tid >> 4);
    const bool full = (xc.bi * 128 + 128 <= d.n) && (xc.bj * 128 + 128 <= d.k);
    if (full && sd.mode == 1) {
      uint8_t* qp = d.q + (int64_t)row0 * d.ldq + col;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint2*>(qp + (int64_t)(16 * j) * d.ldq) =
            quant8_fast<false>(cur[j], sd.s, sd.y);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = row0 + 16 * j;
        if (r < d.n && col < d.k)
          *reinterpret_cast<uint2*>(d.q + (int64_t)r * d.ldq + col) = quant8<false>(cur[j], sd);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
    xc = xn;
  }
}

fp8rl_status check_wdesc(const fp8rl_wdesc& d, int idx) {
  if (!d.w || !d.q || !d.scales)
    return fail(FP8RL_ERR_INVALID_ARG, "weight tensor %d: null pointer", idx);
  if (d.n < 1 || d.k < 1 || d.ldw < d.k || d.ldq < d.k)
    return fail(FP8RL_ERR_INVALID_ARG,
                "weight tensor %d: need n, k >= 1, ldw >= k, ldq >= k (n=%lld k=%lld ldw=%lld ldq=%lld)",
                idx, (long long)d.n, (long long)d.k, (long long)d.ldw, (long long)d.ldq);
  if (d.k % 8 || d.ldw % 8 || d.ldq % 8)
    return fail(FP8RL_ERR_ALIGNMENT, "weight tensor %d: k, ldw and ldq must be multiples of 8", idx);
  if (!aligned(d.w, 16) || !aligned(d.q, 8) || !aligned(d.scales, 4))
    return fail(FP8RL_ERR_ALIGNMENT, "weight tensor %d: w must be 16-byte, q 8-byte aligned", idx);
  if (d.n > INT32_MAX / 2 || d.k > INT32_MAX / 2 || d.ldq > INT32_MAX)
    return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "weight tensor %d: dimension too large", idx);
  return FP8RL_OK;
}

}  // namespace
}  // namespace fp8rl

using namespace fp8rl;

extern "C" fp8rl_status fp8rl_quantize_weights_blockwise_multi(const fp8rl_wdesc* descs,
                                                               int32_t count,
                                                               cudaStream_t stream) {
  if (count < 0 || (count > 0 && !descs))
    return fail(FP8RL_ERR_INVALID_ARG, "descs must be a host array of count >= 0 descriptors");
  for (int i = 0; i < count; ++i) {
    fp8rl_status st = check_wdesc(descs[i], i);
    if (st != FP8RL_OK) return st;
  }
  if (count == 0) return ok();
  DeviceState* ds = nullptr;
  fp8rl_status st = device_state(&ds);
  if (st != FP8RL_OK) return st;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  static const int per_sm = resident_ctas_per_sm(wquant_kernel, kWQThreads);
  static WQParams p;   // ~10 KB of kernel parameters, filled per launch under the lock
  for (int base = 0; base < count; base += kWQMaxDescs) {
    const int c = std::min(kWQMaxDescs, count - base);
    std::memset(&p, 0, sizeof(p));
    p.count = c;
    p.status = ds->status;
    int64_t total = 0;
    for (int i = 0; i < c; ++i) {
      const fp8rl_wdesc& d = descs[base + i];
      const int64_t kb = (d.k + 127) / 128;
      p.start[i] = (int32_t)total;
      p.d[i].w = reinterpret_cast<const uint16_t*>(d.w);
      p.d[i].ldw = d.ldw;
      p.d[i].q = d.q;
      p.d[i].scales = d.scales;
      p.d[i].ldq = d.ldq;
      p.d[i].n = (int32_t)d.n;
      p.d[i].k = (int32_t)d.k;
      p.d[i].kb = (int32_t)kb;
      total += ((d.n + 127) / 128) * kb;
      if (total > INT32_MAX)
        return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "more than 2^31 blocks in one launch");
    }
    p.start[c] = (int32_t)total;
    p.total = (int32_t)total;
    const int grid = (int)std::min<int64_t>(total, (int64_t)ds->sm_count * per_sm);
    wquant_kernel<<<grid, kWQThreads, 0, stream>>>(p);
    st = cuda_check(cudaGetLastError(), "wquant_kernel launch");
    if (st != FP8RL_OK) return st;
  }
  return ok();
}

extern "C" fp8rl_status fp8rl_quantize_weights_blockwise(const void* w, int64_t n, int64_t k,
                                                         int64_t ldw, uint8_t* q, int64_t ldq,
                                                         float* scales, cudaStream_t stream) {
  fp8rl_wdesc d{w, q, scales, n, k, ldw, ldq};
  return fp8rl_quantize_weights_blockwise_multi(&d, 1, stream);
}
