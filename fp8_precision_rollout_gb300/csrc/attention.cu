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
// A cluster of C CTAs per (sequence, KV head) (C = 1 when the pairs already
// fill the GPU; up to 8 for small batches), rank r taking a contiguous range
// of the sequence's 64-token stages.  In each CTA a producer warp TMA-loads the head's
// 128-byte slice of 64 consecutive tokens of K and of V per stage (16 KB, in
// the 128-byte swizzled layout when the boxes allow it) into a 3-slot
// mbarrier ring, with the stage's valid-token mask; its lanes look up the
// pages of a stage's boxes together, one stage ahead.  Three consumer warps
// take whole stages in turn, warp w the stages i with i % 3 == w, so that a
// slot (i % 3) always has the same consumer, which waits on its barrier in
// order (a warp can never wait on a slot whose previous phase another warp
// has not consumed yet).  Both contractions of a stage run on the tensor cores as
// m16n8k16 FP16 MMAs with FP32 accumulation, the G <= 8 query heads of the
// group on the n = 8 side:
//   scores  S[16 tokens x 8 heads]   += K[16 tokens x 16 dims] * Q^T[16 dims x 8]
//   output  O^T[16 dims x 8 heads]   += V^T[16 dims x 16 tokens] * P^T[16 tokens x 8]
// The operands of the first product are exact: every E4M3 code is an FP16
// value (hardware e4m3x2 -> f16x2 conversion), and q is scaled per head by a
// power of two into [2^14, 2^15) before its FP16 conversion, the factor
// folded back into the score scale.  The probabilities, scaled by 2^15 so
// that FP16 keeps them normal down to 2^-29, are rounded to FP16 for the
// second product; the normaliser sums them in FP32.  The order of the
// dimensions inside a k-step, and of the output rows, are permutations chosen
// so that every lane reads whole 16-byte chunks; the score fragment becomes
// the second product's operand through an in-register transpose (movmatrix).
// Online softmax in the log2 domain, rescaled once per stage; the three warps
// are combined through shared memory, then the C ranks of a cluster through
// distributed shared memory (each rank writes a slice of the output).  Every
// mbarrier wait is bounded.
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
constexpr int kConsumerWarps = 3;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;          // + producer warp
constexpr int kStageTokens = 64;
constexpr int kMTiles = kStageTokens / 16;                       // 16-token MMA tiles per stage
// Three slots of 16 KB (one per consumer warp) and at most 128 registers a
// thread let four CTAs share an SM: 608 resident CTAs, so the 512 (sequence,
// head) pairs of a 64-sequence, 8-head batch run in one wave instead of 1.7
// waves of 304 (the second one too thin to keep HBM busy).  Bytes in flight
// per SM stay the same (4 x 48 KB against 2 x 96 KB).
constexpr int kStages = 3;
constexpr int kHalfStage = kStageTokens * kHeadDim;              // K (or V) of a stage: 8 KB
constexpr int kStageBytes = 2 * kHalfStage;
constexpr int kMaxG = 8;                                         // the MMA's n
constexpr float kPScale = 32768.0f;   // probabilities enter the FP16 product as p * 2^15
static_assert(kStages % kConsumerWarps == 0, "a ring slot must always have the same consumer warp");

struct AttnShared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t vmask[kStages];   // bit r: stage row r is a valid token
  uint32_t abort_flag;
};
constexpr size_t kAttnSmem = 1024 + (size_t)kStages * kStageBytes + sizeof(AttnShared);
static_assert((size_t)(kConsumerWarps + 1) * (2 + kHeadDim) * kMaxG * sizeof(float) <=
                  (size_t)kStages * kStageBytes,
              "the combine buffers must fit in the idle stages");
constexpr int kMaxCluster = 8;

// 2^x with the hardware approximation (relative error about 2^-22); the
// attention is compared with a tolerance, not bit for bit.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Four E4M3 codes (one 32-bit word, byte i = element i) -> two f16x2: lo
// holds elements (0, 1), hi holds (2, 3), the lower index in the lower half.
__device__ __forceinline__ void dec_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// D += A * B, m16n8k16, FP16 operands, FP32 accumulation.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of the warp's 8x8 matrix of 16-bit values (lane l holds row l/4,
// columns 2(l%4) and 2(l%4)+1).
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint4 lds128(const uint8_t* a) {
  return *reinterpret_cast<const uint4*>(a);
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

struct AttnParams {
  const __nv_bfloat16* q;     // [S, Hq, 128]
  const float* k_scale;       // [Hkv]
  const float* v_scale;
  const int32_t* table;       // [S, max_pages] or null: page of (s, j) = s * max_pages + j
  const int32_t* lens;        // [S]
  __nv_bfloat16* out;         // [S, Hq, 128]
  int S, Hq, Hkv, G, page, max_pages, num_pages;
  int boxr;                   // rows per TMA box (divides page when paged; 64 if contiguous)
  int csplit;                 // CTAs per (sequence, KV head): the cluster size
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

// kSwz: the stage rows are in the 128-byte swizzled layout (16-byte chunk j
// of row r stored at chunk j ^ (r % 8)); otherwise plain 128-byte rows.
template <bool kSwz>
__global__ void __launch_bounds__(kAttnThreads, 4) attn_decode_kernel(
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
    const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  AttnShared* sh = reinterpret_cast<AttnShared*>(smem + kStages * kStageBytes);
  volatile uint32_t* abort_flag = &sh->abort_flag;
  const int C = p.csplit;
  const uint32_t crank = C > 1 ? cluster_ctarank() : 0u;
  const int pair = (int)(blockIdx.x / (unsigned)C);
  const int s = pair / p.Hkv, h = pair % p.Hkv;
  const int G = p.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int len = __ldg(p.lens + s);
  const int cap = p.max_pages * p.page;
  if (len > cap) {
    if (tid == 0) atomicOr(p.status, kStatusBadIndex);
    len = cap;
  }
  const int nst_all = len > 0 ? (len + kStageTokens - 1) / kStageTokens : 0;
  // this rank's stages: [i0, i0 + nst); j = i - i0 numbers the ring's uses
  const int i0 = (int)(((int64_t)nst_all * crank) / C);
  const int nst = (int)(((int64_t)nst_all * (crank + 1)) / C) - i0;
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&sh->full[i]), 1);
      mbar_init(smem_u32(&sh->empty[i]), 1);
    }
    sh->abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
  }
  __syncthreads();

  // consumer lane (g, c) = (lane / 4, lane % 4) keeps the state of heads 2c, 2c+1
  const int g = lane >> 2, c = lane & 3;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  float o[8][4];
  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer --
    // lane l handles boxes l and l + 32 of a stage (64 / boxr boxes)
    const int nbox = kStageTokens / p.boxr;
    int row[2] = {0, 0}, vrows[2] = {0, 0};
    bool bad_seen = false;
    auto lookup = [&](int i) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int b = lane + 32 * u;
        row[u] = 0;
        vrows[u] = 0;
        if (b < nbox) {
          bool ok, bad;
          const int t = i * kStageTokens + b * p.boxr;
          row[u] = token_row(p, s, t, len, ok, bad);
          bad_seen |= bad;
          if (ok) vrows[u] = min(p.boxr, len - t);
        }
      }
    };
    if (nst > 0) lookup(i0);
    uint32_t issued = 0;
    for (int j = 0; j < nst; ++j) {
      const int st = j % kStages;
      const uint32_t ph = (uint32_t)(j / kStages) & 1u;
      bool okw = true;
      if (lane == 0) okw = mbar_wait(smem_u32(&sh->empty[st]), ph ^ 1u, abort_flag, p.status, 31);
      if (!__shfl_sync(0xFFFFFFFFu, okw ? 1 : 0, 0)) break;
      uint64_t mask = 0;
#pragma unroll
      for (int u = 0; u < 2; ++u)
        if (vrows[u] > 0)
          mask |= (vrows[u] >= 64 ? ~0ull : ((1ull << vrows[u]) - 1ull)) << ((lane + 32 * u) * p.boxr);
      const uint32_t mlo = __reduce_or_sync(0xFFFFFFFFu, (uint32_t)mask);
      const uint32_t mhi = __reduce_or_sync(0xFFFFFFFFu, (uint32_t)(mask >> 32));
      const uint32_t fb = smem_u32(&sh->full[st]);
      if (lane == 0) {
        sh->vmask[st] = ((uint64_t)mhi << 32) | mlo;
        mbar_expect_tx(fb, kStageBytes);   // arrives; the mask store above is released with it
      }
      __syncwarp();
      uint8_t* kdst = smem + st * kStageBytes;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int b = lane + 32 * u;
        if (b < nbox) {
          tma_load_2d(smem_u32(kdst + b * p.boxr * kHeadDim), &tmK, fb, h * kHeadDim, row[u]);
          tma_load_2d(smem_u32(kdst + kHalfStage + b * p.boxr * kHeadDim), &tmV, fb, h * kHeadDim,
                      row[u]);
        }
      }
      ++issued;
      if (j + 1 < nst) lookup(i0 + j + 1);   // the page-table loads overlap the next wait
    }
    if (__any_sync(0xFFFFFFFFu, bad_seen) && lane == 0) atomicOr(p.status, kStatusBadIndex);
    if (lane == 0 && issued < (uint32_t)nst) {
      // gave up: let the stages still in flight land before the CTA moves on
      const uint32_t n = issued < (uint32_t)kStages ? issued : (uint32_t)kStages;
      for (uint32_t k = 1; k <= n; ++k) {
        const uint32_t i2 = issued - k;
        mbar_drain(smem_u32(&sh->full[i2 % kStages]), (i2 / kStages) & 1u, p.status, 33);
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- consumers --
    // Q as the first product's B operand: lane (g, c) holds head g,
    // dimensions [32c, 32c + 32), k-step j taking [32c + 4j, 32c + 4j + 4)
    // (zero for g >= G).  Head g is scaled by 2^e_g, max |q| in [2^14, 2^15).
    uint32_t qb[8][2];
    int e = 0;
    {
      float qf[32];
      float amax = 0.f;
      const bool real = g < G;
      const __nv_bfloat16* qrow = p.q + ((size_t)s * p.Hq + h * G + (real ? g : 0)) * kHeadDim;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint4 raw = make_uint4(0u, 0u, 0u, 0u);
        if (real) raw = *reinterpret_cast<const uint4*>(qrow + 32 * c + 8 * u);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float2 f = __bfloat1622float2(b2[v]);
          qf[8 * u + 2 * v] = f.x;
          qf[8 * u + 2 * v + 1] = f.y;
          amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
      // e = 14 - floor(log2 max|q|), kept within [-100, 100]; zero heads: e = 0
      if (amax > 0.f) {
        const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
        e = min(max(14 - ex, -100), 100);
      }
      const float up = __int_as_float((uint32_t)(127 + e) << 23);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        qb[j][0] = pack_f16x2(qf[4 * j] * up, qf[4 * j + 1] * up);
        qb[j][1] = pack_f16x2(qf[4 * j + 2] * up, qf[4 * j + 3] * up);
      }
    }
    // score factor of head n: sm_scale * log2(e) * k_scale * 2^-e_n; lane
    // (g, c) needs heads 2c and 2c+1, whose exponents the lanes g = 2c, 2c+1 hold
    const float base = p.sm_scale_log2 * __ldg(p.k_scale + h);
    const int eA = __shfl_sync(0xFFFFFFFFu, e, (2 * c) * 4);
    const int eB = __shfl_sync(0xFFFFFFFFu, e, (2 * c + 1) * 4);
    const float fA = base * __int_as_float((uint32_t)(127 - eA) << 23);
    const float fB = base * __int_as_float((uint32_t)(127 - eB) << 23);

#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int r = 0; r < 4; ++r) o[i][r] = 0.f;

    // byte offsets of this lane's 16-byte chunks within a row; every MMA tile
    // starts at a multiple of 8 rows, so a row's swizzle term is known here
    const uint32_t kofs0 = (uint32_t)(((2 * c) ^ (kSwz ? g : 0)) << 4);       // K rows g, g+8
    const uint32_t kofs1 = (uint32_t)(((2 * c + 1) ^ (kSwz ? g : 0)) << 4);
    const uint32_t vofs0 = (uint32_t)((g ^ (kSwz ? 2 * c : 0)) << 4);         // V rows 2c, 2c+8
    const uint32_t vofs1 = (uint32_t)((g ^ (kSwz ? 2 * c + 1 : 0)) << 4);     // V rows 2c+1, 2c+9

    // warp w takes the rank's stages w, w+3, ...: a warp-uniform count, so every lane
    // reaches every full-warp shuffle, MMA and transpose
    for (int j = warp; j < nst; j += kConsumerWarps) {
      const int st = j % kStages;
      const uint32_t ph = (uint32_t)(j / kStages) & 1u;
      bool okw = mbar_wait(smem_u32(&sh->full[st]), ph, abort_flag, p.status, 32);
      okw = __all_sync(0xFFFFFFFFu, okw);
      if (!okw) break;
      const uint64_t vm = sh->vmask[st];
      const bool all_valid = vm == ~0ull;
      const uint8_t* ks = smem + st * kStageBytes;
      const uint8_t* vs = ks + kHalfStage;

      // scores of the stage's four 16-token tiles, in the log2 domain
      float sc[kMTiles][4];
#pragma unroll
      for (int mt = 0; mt < kMTiles; ++mt) {
        const uint8_t* r0 = ks + (mt * 16 + g) * kHeadDim;
        const uint8_t* r1 = r0 + 8 * kHeadDim;
        const uint4 ka0 = lds128(r0 + kofs0), ka1 = lds128(r0 + kofs1);
        const uint4 kb0 = lds128(r1 + kofs0), kb1 = lds128(r1 + kofs1);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t alo, ahi, blo, bhi;
          dec_f16x2(word(j < 4 ? ka0 : ka1, j & 3), alo, ahi);
          dec_f16x2(word(j < 4 ? kb0 : kb1, j & 3), blo, bhi);
          mma_f16(d, alo, blo, ahi, bhi, qb[j][0], qb[j][1]);
        }
        const bool v0 = all_valid || ((vm >> (mt * 16 + g)) & 1ull);
        const bool v1 = all_valid || ((vm >> (mt * 16 + g + 8)) & 1ull);
        sc[mt][0] = v0 ? d[0] * fA : -INFINITY;
        sc[mt][1] = v0 ? d[1] * fB : -INFINITY;
        sc[mt][2] = v1 ? d[2] * fA : -INFINITY;
        sc[mt][3] = v1 ? d[3] * fB : -INFINITY;
      }
      // stage maxima of heads 2c, 2c+1 (over the lanes with this c)
      float xA = -INFINITY, xB = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < kMTiles; ++mt) {
        xA = fmaxf(xA, fmaxf(sc[mt][0], sc[mt][2]));
        xB = fmaxf(xB, fmaxf(sc[mt][1], sc[mt][3]));
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        xA = fmaxf(xA, __shfl_xor_sync(0xFFFFFFFFu, xA, off));
        xB = fmaxf(xB, __shfl_xor_sync(0xFFFFFFFFu, xB, off));
      }
      const float nA = fmaxf(mA, xA), nB = fmaxf(mB, xB);
      const float uA = nA == -INFINITY ? 0.f : nA, uB = nB == -INFINITY ? 0.f : nB;
      const float cA = ex2(mA - uA), cB = ex2(mB - uB);   // 0 while nothing valid was seen
      mA = nA;
      mB = nB;
      lA *= cA;
      lB *= cB;
#pragma unroll
      for (int i2 = 0; i2 < 8; ++i2) {
        o[i2][0] *= cA;
        o[i2][1] *= cB;
        o[i2][2] *= cA;
        o[i2][3] *= cB;
      }
      // probabilities, then the B operands of the second product
      uint32_t pb[kMTiles][2];
#pragma unroll
      for (int mt = 0; mt < kMTiles; ++mt) {
        const float p0 = ex2(sc[mt][0] - uA), p1 = ex2(sc[mt][1] - uB);
        const float p2 = ex2(sc[mt][2] - uA), p3 = ex2(sc[mt][3] - uB);
        lA += p0 + p2;
        lB += p1 + p3;
        // x 2^15: p down to 2^-29 stays a normal FP16 number (undone at the end)
        pb[mt][0] = transpose8x8(pack_f16x2(p0 * kPScale, p1 * kPScale));   // tokens 2c, 2c+1, head g
        pb[mt][1] = transpose8x8(pack_f16x2(p2 * kPScale, p3 * kPScale));   // tokens 2c+8, 2c+9
      }
      // O^T += V^T P^T.  Row g of output tile i is dimension 16g + 2i, row
      // g+8 is 16g + 2i + 1; the k index is the tile's token order.
#pragma unroll
      for (int mt = 0; mt < kMTiles; ++mt) {
        const int t0 = mt * 16 + 2 * c;
        uint4 x0 = lds128(vs + t0 * kHeadDim + vofs0);
        uint4 x1 = lds128(vs + (t0 + 1) * kHeadDim + vofs1);
        uint4 x2 = lds128(vs + (t0 + 8) * kHeadDim + vofs0);
        uint4 x3 = lds128(vs + (t0 + 9) * kHeadDim + vofs1);
        if (!all_valid) {
          // an invalid row holds a copy of pool row 0; its p is 0, and its
          // codes are zeroed so that no NaN code can reach the sum
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          if (!((vm >> t0) & 1ull)) x0 = z;
          if (!((vm >> (t0 + 1)) & 1ull)) x1 = z;
          if (!((vm >> (t0 + 8)) & 1ull)) x2 = z;
          if (!((vm >> (t0 + 9)) & 1ull)) x3 = z;
        }
#pragma unroll
        for (int w = 0; w < 4; ++w) {
#pragma unroll
          for (int hs = 0; hs < 2; ++hs) {
            // bytes 2hs, 2hs+1 of word w: dimensions 16g + 4w + 2hs (+1)
            const uint32_t sel = hs ? 0x7362u : 0x5140u;
            uint32_t a0, a1, a2, a3;
            dec_f16x2(__byte_perm(word(x0, w), word(x1, w), sel), a0, a1);
            dec_f16x2(__byte_perm(word(x2, w), word(x3, w), sel), a2, a3);
            mma_f16(o[2 * w + hs], a0, a1, a2, a3, pb[mt][0], pb[mt][1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh->empty[st]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      lA += __shfl_xor_sync(0xFFFFFFFFu, lA, off);
      lB += __shfl_xor_sync(0xFFFFFFFFu, lB, off);
    }
  }
  // ------------------------------------------------ combine the 3 warps --
  // (the stage buffers are idle now: every issued stage was consumed, or
  // drained by the producer after a timeout)
  __syncthreads();
  float* cm = reinterpret_cast<float*>(smem);            // [kConsumerWarps][G]
  float* cl = cm + kConsumerWarps * G;                   // [kConsumerWarps][G]
  float* co = cl + kConsumerWarps * G;                   // [kConsumerWarps][G][128]
  if (warp < kConsumerWarps) {
    const int hA = 2 * c, hB = 2 * c + 1;
    if (g == 0) {
      if (hA < G) {
        cm[warp * G + hA] = mA;
        cl[warp * G + hA] = lA;
      }
      if (hB < G) {
        cm[warp * G + hB] = mB;
        cl[warp * G + hB] = lB;
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int d0 = 16 * g + 2 * i;
      const float un = 1.0f / kPScale;   // exact
      if (hA < G) {
        co[(warp * G + hA) * kHeadDim + d0] = o[i][0] * un;
        co[(warp * G + hA) * kHeadDim + d0 + 1] = o[i][2] * un;
      }
      if (hB < G) {
        co[(warp * G + hB) * kHeadDim + d0] = o[i][1] * un;
        co[(warp * G + hB) * kHeadDim + d0 + 1] = o[i][3] * un;
      }
    }
  }
  __syncthreads();
  const float vscale = __ldg(p.v_scale + h);
  // this CTA's state per head: max xm, sum xl, unnormalised xo (C > 1)
  float* xm = co + kConsumerWarps * G * kHeadDim;        // [G]
  float* xl = xm + kMaxG;                                // [G]
  float* xo = xl + kMaxG;                                // [G][128]
  for (int idx = tid; idx < G * kHeadDim; idx += kAttnThreads) {
    const int n = idx / kHeadDim, d = idx - n * kHeadDim;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kConsumerWarps; ++k) M = fmaxf(M, cm[k * G + n]);
    float L = 0.f, O = 0.f;
    if (M > -INFINITY) {
#pragma unroll
      for (int k = 0; k < kConsumerWarps; ++k) {
        const float w = ex2(cm[k * G + n] - M);
        L = fmaf(cl[k * G + n], w, L);
        O = fmaf(co[(k * G + n) * kHeadDim + d], w, O);
      }
    }
    if (C == 1) {
      const float r = L > 0.f ? O / L * vscale : 0.f;
      p.out[((size_t)s * p.Hq + h * G + n) * kHeadDim + d] = __float2bfloat16_rn(r);
    } else {
      xo[idx] = O;
      if (d == 0) {
        xm[n] = M;
        xl[n] = L;
      }
    }
  }
  if (C > 1) {
    // every rank's state is visible after this phase; rank r then writes the
    // output elements r, r + C*threads, ... reading all ranks' states
    cluster_arrive();
    cluster_wait();
    const uint32_t axm = smem_u32(xm), axl = smem_u32(xl), axo = smem_u32(xo);
    for (int idx = (int)crank * kAttnThreads + tid; idx < G * kHeadDim; idx += C * kAttnThreads) {
      const int n = idx / kHeadDim, d = idx - n * kHeadDim;
      float mr[8];
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        mr[r] = r < C ? ld_cluster_f32(mapa(axm + 4u * n, (uint32_t)r)) : -INFINITY;
        M = fmaxf(M, mr[r]);
      }
      float L = 0.f, O = 0.f;
      if (M > -INFINITY) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          if (r < C) {
            const float w = ex2(mr[r] - M);
            L = fmaf(ld_cluster_f32(mapa(axl + 4u * n, (uint32_t)r)), w, L);
            O = fmaf(ld_cluster_f32(mapa(axo + 4u * idx, (uint32_t)r)), w, O);
          }
        }
      }
      const float res = L > 0.f ? O / L * vscale : 0.f;
      p.out[((size_t)s * p.Hq + h * G + n) * kHeadDim + d] = __float2bfloat16_rn(res);
    }
    // no rank leaves while another may still read its shared memory
    cluster_arrive();
    cluster_wait();
  }
}

template <bool kSwz>
fp8rl_status set_attn_smem(const DeviceState* ds) {
  static bool done[64] = {false};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (ds->device < 64 && done[ds->device]) return FP8RL_OK;
  fp8rl_status st = cuda_check(cudaFuncSetAttribute(attn_decode_kernel<kSwz>,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    (int)kAttnSmem),
                               "cudaFuncSetAttribute(attention)");
  if (st == FP8RL_OK && ds->device < 64) done[ds->device] = true;
  return st;
}

// Clusters of c attention CTAs that can be resident at once (0 if none).
template <bool kSwz>
int attn_active_clusters(const DeviceState* ds, int c) {
  static int cache[64][kMaxCluster + 1] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  int* slot = ds->device < 64 ? &cache[ds->device][c] : nullptr;
  if (slot && *slot) return *slot > 0 ? *slot : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)c, 1, 1);
  cfg.blockDim = dim3(kAttnThreads, 1, 1);
  cfg.dynamicSmemBytes = kAttnSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, attn_decode_kernel<kSwz>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  if (slot) *slot = n > 0 ? n : -1;
  return n;
}

// Cluster size: double C while all pairs x C CTAs still fit in one resident
// wave and every rank keeps at least two stages per consumer warp.
template <bool kSwz>
int choose_csplit(const DeviceState* ds, int64_t pairs, int64_t nst_cap) {
  // resident CTAs per SM, queried once per device (not on every launch, so
  // that a launch under CUDA-graph capture makes no occupancy query)
  static int cache[64] = {};
  static std::mutex mu;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    int* slot = ds->device < 64 ? &cache[ds->device] : nullptr;
    if (slot && *slot) {
      per_sm = *slot;
    } else {
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_decode_kernel<kSwz>,
                                                        kAttnThreads, kAttnSmem) != cudaSuccess) {
        (void)cudaGetLastError();
        per_sm = 1;
      }
      per_sm = std::max(per_sm, 1);
      if (slot) *slot = per_sm;
    }
  }
  const int64_t slots = (int64_t)ds->sm_count * std::max(per_sm, 1);
  int c = 1;
  while (c < kMaxCluster && pairs * c * 2 <= slots && nst_cap / (c * 2) >= 2 * kConsumerWarps)
    c *= 2;
  while (c > 1 && attn_active_clusters<kSwz>(ds, c) <= 0) c /= 2;
  return c;
}

template <bool kSwz>
fp8rl_status launch_attn(const DeviceState* ds, const CUtensorMap& tk, const CUtensorMap& tv,
                         AttnParams p, cudaStream_t stream) {
  fp8rl_status st = set_attn_smem<kSwz>(ds);
  if (st != FP8RL_OK) return st;
  const int64_t pairs = (int64_t)p.S * p.Hkv;
  const int64_t nst_cap = ((int64_t)p.max_pages * p.page + kStageTokens - 1) / kStageTokens;
  p.csplit = choose_csplit<kSwz>(ds, pairs, nst_cap);
  if (p.csplit == 1) {
    attn_decode_kernel<kSwz><<<(unsigned)pairs, kAttnThreads, kAttnSmem, stream>>>(tk, tv, p);
    return cuda_check(cudaGetLastError(), "attn_decode_kernel launch");
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pairs * p.csplit), 1, 1);
  cfg.blockDim = dim3(kAttnThreads, 1, 1);
  cfg.dynamicSmemBytes = kAttnSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.csplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_check(cudaLaunchKernelEx(&cfg, attn_decode_kernel<kSwz>, tk, tv, p),
                    "attn_decode_kernel cluster launch");
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
  if ((int64_t)page * max_pages > INT32_MAX ||
      (int64_t)num_seqs * kv_heads * kMaxCluster > INT32_MAX)
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
  p.G = G;
  p.page = page;
  p.max_pages = max_pages;
  p.num_pages = block_table ? num_pages : num_seqs * max_pages;
  // a TMA box is boxr consecutive tokens; paged, it must stay inside a page
  p.boxr = block_table ? std::gcd(page, kStageTokens) : kStageTokens;
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  p.status = ds->status;
  p.csplit = 1;   // chosen at launch
  // the 128-byte swizzle wants every box to start on a 1024-byte boundary of
  // the stage: boxes of a multiple of 8 rows
  const bool swz = p.boxr % 8 == 0;
  const CUtensorMapSwizzle mode = swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  // the pool as rows of kv_heads * 128 bytes; a box is one head's 128 bytes
  CUtensorMap tk, tv;
  const uint64_t row_bytes = (uint64_t)kv_heads * kHeadDim;
  if ((st = encode_tiled_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, k_cache, row_bytes,
                            (uint64_t)pool_rows, row_bytes, kHeadDim, (uint32_t)p.boxr, mode,
                            "K cache")) != FP8RL_OK)
    return st;
  if ((st = encode_tiled_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, v_cache, row_bytes,
                            (uint64_t)pool_rows, row_bytes, kHeadDim, (uint32_t)p.boxr, mode,
                            "V cache")) != FP8RL_OK)
    return st;
  st = swz ? launch_attn<true>(ds, tk, tv, p, stream) : launch_attn<false>(ds, tk, tv, p, stream);
  return st == FP8RL_OK ? ok() : st;
}
