// attention.cu -- decode attention over an FP8 E4M3 KV cache.
//
// FP8-RL summary, section 3.4.4: the KV cache stores K and V in E4M3 with
// per-head scales recalibrated every step, and the pipeline's attention reads
// that cache.  For every sequence s and query head hq (KV head
// h = hq / (Hq/Hkv), grouped-query attention):
//   s_t = sm_scale * <q, k_scale[h] * dec(K[t])>,  p = softmax(s over t < len),
//   o   = sum_t p_t * v_scale[h] * dec(V[t]),      out = BF16(o).
// Token t of sequence s lives in page block_table[s][t / page], slot t % page.
//
// One CTA per (sequence, KV head): a producer warp TMA-loads the head's
// 128-byte slice of 64 consecutive tokens of K and of V per stage (16 KB)
// into a 4-stage mbarrier ring, with the stage's valid-token mask; 4 consumer
// warps run 8 token streams of 16 lanes (lane j holds dimensions [8j, 8j+8)
// for all G query heads of the group, so each byte is used for the G heads),
// stream k taking the stage's tokens [8k, 8k+8).  Online softmax in the log2
// domain (q pre-multiplied by sm_scale * k_scale * log2 e), rescaled once per
// 8-token block; the 8 streams are combined through shared memory at the end.
// Codes are dequantized with the hardware e4m3x2 -> f16x2 conversion (exact:
// every E4M3 value is an FP16 value).  Every mbarrier wait is bounded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>
#include <numeric>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace fp8rl {
namespace {

using namespace ptx;

constexpr int kHeadDim = 128;
constexpr int kLanesPerToken = 16;
constexpr int kDimsPerLane = kHeadDim / kLanesPerToken;          // 8
constexpr int kConsumerWarps = 4;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;          // + producer warp
constexpr int kStreams = kConsumerWarps * 32 / kLanesPerToken;   // 8
constexpr int kBlk = 8;                                          // tokens per stream per stage
constexpr int kStageTokens = kStreams * kBlk;                    // 64
constexpr int kStages = 4;
constexpr int kHalfStage = kStageTokens * kHeadDim;              // K (or V) of a stage: 8 KB
constexpr int kStageBytes = 2 * kHalfStage;

struct AttnShared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t vmask[kStages];   // bit r: stage row r is a valid token
  uint32_t abort_flag;
};
constexpr size_t kAttnSmem = 1024 + (size_t)kStages * kStageBytes + sizeof(AttnShared);

// 2^x with the hardware approximation (relative error about 2^-22); the
// attention is compared with a tolerance, not bit for bit.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Four E4M3 codes (one 32-bit word) -> four floats, exactly.
__device__ __forceinline__ void dec4(uint32_t w, float* f) {
  uint32_t lo, hi;
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

struct AttnParams {
  const __nv_bfloat16* q;     // [S, Hq, 128]
  const float* k_scale;       // [Hkv]
  const float* v_scale;
  const int32_t* table;       // [S, max_pages] or null: page of (s, j) = s * max_pages + j
  const int32_t* lens;        // [S]
  __nv_bfloat16* out;         // [S, Hq, 128]
  int S, Hq, Hkv, page, max_pages, num_pages;
  int boxr;                   // rows per TMA box (divides page when paged; 64 if contiguous)
  float sm_scale_log2;        // sm_scale * log2(e)
  uint32_t* status;
};

// Pool row of token t of sequence s and whether it is valid (in range and
// on an existing page); invalid tokens map to row 0, which always exists.
__device__ __forceinline__ int token_row(const AttnParams& p, int s, int t, int len, bool& ok,
                                         bool& bad) {
  ok = t < len;
  bad = false;
  if (!ok) return 0;
  const int pi = t / p.page, slot = t - pi * p.page;
  const int pg = p.table ? __ldg(p.table + (size_t)s * p.max_pages + pi) : s * p.max_pages + pi;
  if (pg < 0 || pg >= p.num_pages) {
    ok = false;
    bad = true;
    return 0;
  }
  return pg * p.page + slot;
}

template <int G>
__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
    const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  AttnShared* sh = reinterpret_cast<AttnShared*>(smem + kStages * kStageBytes);
  volatile uint32_t* abort_flag = &sh->abort_flag;
  const int s = blockIdx.x / p.Hkv, h = blockIdx.x % p.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int len = __ldg(p.lens + s);
  const int cap = p.max_pages * p.page;
  if (len > cap) {
    if (tid == 0) atomicOr(p.status, kStatusBadIndex);
    len = cap;
  }
  const int nst = len > 0 ? (len + kStageTokens - 1) / kStageTokens : 0;
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&sh->full[i]), 1);
      mbar_init(smem_u32(&sh->empty[i]), kConsumerWarps);
    }
    sh->abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
  }
  __syncthreads();

  float m[G], l[G], o[G][kDimsPerLane];
  const int stream = (tid & 127) / kLanesPerToken;   // consumers: 0..7
  const int j = lane & (kLanesPerToken - 1);         // dimension slice
  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      uint32_t issued = 0;
      bool any_bad = false;
      for (int i = 0; i < nst; ++i) {
        const int st = i % kStages;
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        if (!mbar_wait(smem_u32(&sh->empty[st]), ph ^ 1u, abort_flag, p.status, 31)) break;
        uint64_t mask = 0;
        for (int r = 0; r < kStageTokens; r += p.boxr) {
          bool ok, bad;
          token_row(p, s, i * kStageTokens + r, len, ok, bad);
          any_bad |= bad;
          if (ok) {
            const int valid_rows = min(p.boxr, len - (i * kStageTokens + r));
            mask |= ((valid_rows >= 64 ? ~0ull : ((1ull << valid_rows) - 1ull)) << r);
          }
        }
        sh->vmask[st] = mask;
        const uint32_t fb = smem_u32(&sh->full[st]);
        mbar_expect_tx(fb, kStageBytes);   // arrives; the mask store above is released with it
        uint8_t* kdst = smem + st * kStageBytes;
        for (int r = 0; r < kStageTokens; r += p.boxr) {
          bool ok, bad;
          const int row = token_row(p, s, i * kStageTokens + r, len, ok, bad);
          tma_load_2d(smem_u32(kdst + r * kHeadDim), &tmK, fb, h * kHeadDim, row);
          tma_load_2d(smem_u32(kdst + kHalfStage + r * kHeadDim), &tmV, fb, h * kHeadDim, row);
        }
        ++issued;
      }
      if (any_bad) atomicOr(p.status, kStatusBadIndex);
      if (issued < (uint32_t)nst) {
        // gave up: let the stages still in flight land before the CTA moves on
        const uint32_t n = issued < (uint32_t)kStages ? issued : (uint32_t)kStages;
        for (uint32_t k = 1; k <= n; ++k) {
          const uint32_t i2 = issued - k;
          mbar_drain(smem_u32(&sh->full[i2 % kStages]), (i2 / kStages) & 1u, p.status, 33);
        }
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- consumers --
    const float kscale = __ldg(p.k_scale + h) * p.sm_scale_log2;
    float q[G][kDimsPerLane];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const uint4 raw = *reinterpret_cast<const uint4*>(
          p.q + ((size_t)s * p.Hq + h * G + g) * kHeadDim + j * kDimsPerLane);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b2[i]);
        q[g][2 * i] = f.x * kscale;
        q[g][2 * i + 1] = f.y * kscale;
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int i = 0; i < kDimsPerLane; ++i) o[g][i] = 0.f;
    }
    // every consumer lane runs all nst stages (a CTA-uniform count), so every
    // lane reaches every full-warp shuffle
    for (int i = 0; i < nst; ++i) {
      const int st = i % kStages;
      const uint32_t ph = (uint32_t)(i / kStages) & 1u;
      bool okw = mbar_wait(smem_u32(&sh->full[st]), ph, abort_flag, p.status, 32);
      okw = __all_sync(0xFFFFFFFFu, okw);
      if (!okw) break;
      const uint64_t vm = sh->vmask[st];
      const uint8_t* ks = smem + st * kStageBytes;
      uint2 kw[kBlk], vw[kBlk];
      bool val[kBlk];
#pragma unroll
      for (int u = 0; u < kBlk; ++u) {
        const int r = stream * kBlk + u;
        val[u] = (vm >> r) & 1ull;
        kw[u] = *reinterpret_cast<const uint2*>(ks + r * kHeadDim + j * kDimsPerLane);
        vw[u] = *reinterpret_cast<const uint2*>(ks + kHalfStage + r * kHeadDim + j * kDimsPerLane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh->empty[st]));
      float sc[kBlk][G];
#pragma unroll
      for (int u = 0; u < kBlk; ++u) {
        float kf[8];
        dec4(kw[u].x, kf);
        dec4(kw[u].y, kf + 4);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float a = 0.f;
#pragma unroll
          for (int d = 0; d < kDimsPerLane; ++d) a = fmaf(q[g][d], kf[d], a);
          sc[u][g] = a;
        }
      }
#pragma unroll
      for (int off2 = kLanesPerToken / 2; off2 > 0; off2 >>= 1) {
#pragma unroll
        for (int u = 0; u < kBlk; ++u)
#pragma unroll
          for (int g = 0; g < G; ++g) sc[u][g] += __shfl_xor_sync(0xFFFFFFFFu, sc[u][g], off2);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float bm = -INFINITY;
#pragma unroll
        for (int u = 0; u < kBlk; ++u)
          if (val[u]) bm = fmaxf(bm, sc[u][g]);
        if (bm == -INFINITY) continue;           // nothing valid for this stream here
        const float mn = fmaxf(m[g], bm);
        const float corr = ex2(m[g] - mn);       // 0 on the first block (m = -inf)
        l[g] *= corr;
#pragma unroll
        for (int d = 0; d < kDimsPerLane; ++d) o[g][d] *= corr;
        m[g] = mn;
      }
#pragma unroll
      for (int u = 0; u < kBlk; ++u) {
        if (!val[u]) continue;
        float vf[8];
        dec4(vw[u].x, vf);
        dec4(vw[u].y, vf + 4);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pr = ex2(sc[u][g] - m[g]);
          l[g] += pr;
#pragma unroll
          for (int d = 0; d < kDimsPerLane; ++d) o[g][d] = fmaf(pr, vf[d], o[g][d]);
        }
      }
    }
  }
  // ---------------------------------------------- combine the 8 streams --
  // (the stage buffers are idle now: every issued stage was consumed, or
  // drained by the producer after a timeout)
  __syncthreads();
  float* cm = reinterpret_cast<float*>(smem);            // [kStreams][G]
  float* cl = cm + kStreams * G;                         // [kStreams][G]
  float* co = cl + kStreams * G;                         // [kStreams][G][128]
  if (warp < kConsumerWarps) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (j == 0) {
        cm[stream * G + g] = m[g];
        cl[stream * G + g] = l[g];
      }
#pragma unroll
      for (int d = 0; d < kDimsPerLane; ++d)
        co[(stream * G + g) * kHeadDim + j * kDimsPerLane + d] = o[g][d];
    }
  }
  __syncthreads();
  const float vscale = __ldg(p.v_scale + h);
  for (int idx = tid; idx < G * kHeadDim; idx += kAttnThreads) {
    const int g = idx / kHeadDim, d = idx - g * kHeadDim;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kStreams; ++k) M = fmaxf(M, cm[k * G + g]);
    float L = 0.f, O = 0.f;
    if (M > -INFINITY) {
#pragma unroll
      for (int k = 0; k < kStreams; ++k) {
        const float w = ex2(cm[k * G + g] - M);
        L = fmaf(cl[k * G + g], w, L);
        O = fmaf(co[(k * G + g) * kHeadDim + d], w, O);
      }
    }
    const float r = L > 0.f ? O / L * vscale : 0.f;
    p.out[((size_t)s * p.Hq + h * G + g) * kHeadDim + d] = __float2bfloat16_rn(r);
  }
}

template <int G>
fp8rl_status set_attn_smem(const DeviceState* ds) {
  static bool done[64] = {false};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (ds->device < 64 && done[ds->device]) return FP8RL_OK;
  fp8rl_status st = cuda_check(cudaFuncSetAttribute(attn_decode_kernel<G>,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    (int)kAttnSmem),
                               "cudaFuncSetAttribute(attention)");
  if (st == FP8RL_OK && ds->device < 64) done[ds->device] = true;
  return st;
}

template <int G>
fp8rl_status launch_attn(const DeviceState* ds, const CUtensorMap& tk, const CUtensorMap& tv,
                         const AttnParams& p, cudaStream_t stream) {
  fp8rl_status st = set_attn_smem<G>(ds);
  if (st != FP8RL_OK) return st;
  attn_decode_kernel<G><<<(unsigned)(p.S * p.Hkv), kAttnThreads, kAttnSmem, stream>>>(tk, tv, p);
  return cuda_check(cudaGetLastError(), "attn_decode_kernel launch");
}

}  // namespace
}  // namespace fp8rl

using namespace fp8rl;

extern "C" fp8rl_status fp8rl_decode_attention_fp8kv(
    const void* q, const uint8_t* k_cache, const uint8_t* v_cache, const float* k_scale,
    const float* v_scale, const int32_t* block_table, const int32_t* seq_lens, int32_t num_seqs,
    int32_t q_heads, int32_t kv_heads, int32_t head_dim, int32_t page, int32_t max_pages,
    int32_t num_pages, float sm_scale, void* out, cudaStream_t stream) {
  if (num_seqs < 0 || q_heads < 1 || kv_heads < 1 || page < 1 || max_pages < 1 || num_pages < 0)
    return fail(FP8RL_ERR_INVALID_ARG, "need num_seqs >= 0 and positive heads, page, max_pages");
  if (num_seqs == 0) return ok();
  if (!q || !k_cache || !v_cache || !k_scale || !v_scale || !seq_lens || !out)
    return fail(FP8RL_ERR_INVALID_ARG, "null pointer");
  if (head_dim != kHeadDim) return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "head_dim must be 128");
  const int G = q_heads / kv_heads;
  if (q_heads % kv_heads || (G != 1 && G != 2 && G != 4 && G != 8))
    return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "q_heads / kv_heads must be 1, 2, 4 or 8");
  if (!(sm_scale > 0.0f) || !std::isfinite(sm_scale))
    return fail(FP8RL_ERR_INVALID_ARG, "sm_scale must be finite and > 0");
  if ((int64_t)page * max_pages > INT32_MAX || (int64_t)num_seqs * kv_heads > INT32_MAX)
    return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "sizes too large");
  if (block_table && num_pages < 1)
    return fail(FP8RL_ERR_INVALID_ARG, "a paged cache needs num_pages >= 1");
  const int64_t pool_rows = (int64_t)(block_table ? num_pages : (int64_t)num_seqs * max_pages) * page;
  if (pool_rows > (int64_t)UINT32_MAX) return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "cache too large");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 2) ||
      (block_table && !aligned(block_table, 4)))
    return fail(FP8RL_ERR_ALIGNMENT, "q and the caches must be 16-byte aligned");
  DeviceState* ds = nullptr;
  fp8rl_status st = device_state(&ds);
  if (st != FP8RL_OK) return st;
  AttnParams p;
  p.q = reinterpret_cast<const __nv_bfloat16*>(q);
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.table = block_table;
  p.lens = seq_lens;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.S = num_seqs;
  p.Hq = q_heads;
  p.Hkv = kv_heads;
  p.page = page;
  p.max_pages = max_pages;
  p.num_pages = block_table ? num_pages : num_seqs * max_pages;
  // a TMA box is boxr consecutive tokens; paged, it must stay inside a page
  p.boxr = block_table ? std::gcd(page, kStageTokens) : kStageTokens;
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  p.status = ds->status;
  // the pool as rows of kv_heads * 128 bytes; a box is one head's 128 bytes
  CUtensorMap tk, tv;
  const uint64_t row_bytes = (uint64_t)kv_heads * kHeadDim;
  if ((st = encode_tiled_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, k_cache, row_bytes,
                            (uint64_t)pool_rows, row_bytes, kHeadDim, (uint32_t)p.boxr,
                            CU_TENSOR_MAP_SWIZZLE_NONE, "K cache")) != FP8RL_OK)
    return st;
  if ((st = encode_tiled_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, v_cache, row_bytes,
                            (uint64_t)pool_rows, row_bytes, kHeadDim, (uint32_t)p.boxr,
                            CU_TENSOR_MAP_SWIZZLE_NONE, "V cache")) != FP8RL_OK)
    return st;
  switch (G) {
    case 1: st = launch_attn<1>(ds, tk, tv, p, stream); break;
    case 2: st = launch_attn<2>(ds, tk, tv, p, stream); break;
    case 4: st = launch_attn<4>(ds, tk, tv, p, stream); break;
    default: st = launch_attn<8>(ds, tk, tv, p, stream); break;
  }
  return st == FP8RL_OK ? ok() : st;
}
