// gemm_decode.cu -- the decode-sized linear layer: 1x128 activation
// quantization fused with the blockwise W8A8 GEMM, stream-K over every SM.
//
// FP8-RL summary, section 3.4.2 Phase 3: every decode step quantizes the
// activations dynamically (1x128 groups, section 3.4.1) and multiplies them by
// the FP8 weights on FP8 tensor cores with FP32 accumulation and BF16 output.
// At decode batch sizes (M <= 256 tokens) the weights dominate the bytes and
// the output has few tiles, so this kernel:
//
//   * runs one persistent CTA per SM as a cooperative grid (all CTAs are
//     resident, so they may wait for one another);
//   * quantizes A first, every CTA its share of the 1x128 groups (the element
//     map of the activation quantizer, bit for bit), while its TMA producer
//     already streams its first weight tiles; a grid barrier then publishes
//     the codes and scales;
//   * treats the GEMM as U = (N/128) x (K/128) units (output tile of all M <=
//     256 rows x 128 columns, one 128-deep k-block) and gives CTA c the
//     contiguous units [c U / G, (c+1) U / G) in tile-major order, so every
//     SM gets the same number of k-blocks ("stream-K");
//   * per unit, two M=128 tcgen05 MMAs (rows 0-127 and 128-255) share the
//     weight tile in shared memory; k-block partials in TMEM are promoted by
//     sa * sw into FP32 registers as in the dense kernel;
//   * a CTA that owns a whole tile stores it as BF16; otherwise it writes its
//     FP32 partial to its slot of the caller's workspace and counts itself in
//     the tile's arrival counter.  After its main loop each CTA of a split
//     tile waits for the tile's partials, then adds them in k order (segment 0
//     first) for its share of the tile's rows and stores BF16, so the result
//     does not depend on arrival order and the reduction is spread over the
//     tile's CTAs.  The last CTA out returns the counters to zero.
//
// Shape: 11 warps.  Warp 0 lane 0: TMA producer (4 stages of 48 KB: A 256 x 128
// + W 128 x 128 bytes, 128-byte swizzle).  Warps 1-2 lane 0: MMA issuers,
// alternating units into the two TMEM buffers (2 x 256 columns).  Warps 3-10:
// epilogue, one output row each (128 FP32 accumulators per thread).  Warps
// 1-10 also do the fused quantization.  Every wait is bounded (1 s); on expiry
// the status word records it and the kernel returns.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "quant_common.cuh"
#include "sm100_ptx.cuh"

namespace fp8rl {
namespace {

using namespace ptx;

constexpr int DM = 256, DN = 128, DK = 128;
constexpr int kDStages = 4;
constexpr int kDAStage = DM * DK;                      // 32 KB
constexpr int kDBStage = DN * DK;                      // 16 KB
constexpr int kDStageBytes = kDAStage + kDBStage;      // 48 KB
constexpr int kDThreads = 352;
constexpr uint32_t kDTmemCols = 512;                   // 2 buffers x 2 row halves x 128
// tcgen05 instruction descriptor, kind::f8f6f4: D = F32, A = B = E4M3, both
// K-major, N = 128, M = 128.
constexpr uint32_t kDIdesc = (1u << 4) | ((uint32_t)(DN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
constexpr int kPartialFloats = DM * DN;                // one FP32 partial tile (128 KB)

struct DecodeTail {
  uint64_t full[kDStages];
  uint64_t empty[kDStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint32_t tmem_base;
  uint32_t abort_flag;
  uint32_t a_ready;
  uint32_t stop;
};
constexpr size_t kDTailPad = (sizeof(DecodeTail) + 1023) / 1024 * 1024;
constexpr size_t kDSmem = 1024 + (size_t)kDStages * kDStageBytes + kDTailPad;
static_assert(kDSmem <= 232448, "shared memory budget");

struct DecodeArgs {
  const uint16_t* a;     // BF16 [M, K], row stride lda; null: qa/sa are inputs
  int64_t lda;
  uint8_t* qa;           // E4M3 [M, K] dense
  float* sa;             // FP32 [KB, M] group-major
  const float* sw;       // FP32 [N/128, KB]
  __nv_bfloat16* y;
  int64_t ldy;
  int M, N, KB, n_tiles;
  float* partials;       // [2 G] slots of [32 chunks][256 rows][4 floats]
  uint32_t* arrive;      // [n_tiles] partials published per split tile (zero between calls)
  uint32_t* done;        // [n_tiles] CTAs done reducing per split tile (zero between calls)
  uint32_t* grid_bar;    // [0] arrivals, [1] generation
  uint32_t* status;
};

// Named barrier among `count` threads (id 0 is __syncthreads).
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Adds `bytes` to the transaction count of the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx_only(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void ffma2(float& acc0, float& acc1, uint32_t p0, uint32_t p1, float f) {
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %4};\n\t"
      "mov.b64 rc, {%0, %1};\n\t"
      "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rc;\n\t}"
      : "+f"(acc0), "+f"(acc1)
      : "r"(p0), "r"(p1), "f"(f));
}

// ---------------------------------------------------------- work split ----

// CTA holding unit x when U units are dealt contiguously to G CTAs
// (CTA c owns [floor(c U / G), floor((c+1) U / G))).
__device__ __forceinline__ int owner_of(int64_t x, int64_t U, int G) {
  return (int)(((x + 1) * (int64_t)G - 1) / U);
}
__device__ __forceinline__ int64_t first_unit(int c, int64_t U, int G) { return (int64_t)c * U / G; }
// Workspace slot of CTA c's partial of tile t: slot 2c if the tile is the
// first one of its range, 2c + 1 if the last (a CTA owns at most two partial
// tiles, those at the ends of its range).
__device__ __forceinline__ int slot_of(int c, int t, int64_t U, int G, int KB) {
  return first_unit(c, U, G) >= (int64_t)t * KB ? 2 * c : 2 * c + 1;
}

// ------------------------------------------------- fused quantization -----

// Warps 1-10 quantize this CTA's share of the M x KB groups, exactly as the
// activation quantizer does (4 lanes per 128-element group, 8 groups per warp
// task, scales group-major).
__device__ void quantize_share(const DecodeArgs& g, int c, int G, int qwarp, int lane) {
  const int64_t groups = (int64_t)g.M * g.KB;
  const int64_t f0 = groups * c / G, f1 = groups * (c + 1) / G;
  const int64_t n_tasks = (f1 - f0 + 7) / 8;
  const int slot = lane & 3;
  const int64_t K = (int64_t)g.KB * DK;
  for (int64_t task = qwarp; task < n_tasks; task += 10) {
    const int64_t f = f0 + task * 8 + (lane >> 2);
    const bool valid = f < f1;
    const int64_t r = valid ? f / g.KB : 0;
    const int gi = (int)(f - r * g.KB);
    const int64_t gcol = (int64_t)gi * 128;
    const uint16_t* arow = g.a + r * g.lda;
    uint4 v[4];
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t col = gcol + (slot + 4 * i) * 8;
      v[i] = valid ? ld_stream(arow + col) : make_uint4(0, 0, 0, 0);
      m2 = absmax8(m2, v[i]);
    }
    const float amax = warp_max(bf16x2_maxf(m2), 4);
    const float s = fx::fdiv(amax, 448.0f);
    if (slot == 0 && valid) g.sa[(int64_t)gi * g.M + r] = s;
    const ScaleDiv sd = make_scale_div(s);
    uint8_t* qrow = g.qa + r * K;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t col = gcol + (slot + 4 * i) * 8;
      if (valid) *reinterpret_cast<uint2*>(qrow + col) = quant8_any<false>(v[i], sd);
    }
  }
}

// Grid barrier of the cooperative launch (one thread per CTA).  The last CTA to
// arrive returns the arrival count to zero and advances the generation; the
// others wait (bounded) for the generation to move.  Returns false on timeout.
__device__ bool grid_barrier(uint32_t* bar, int G, uint32_t* status) {
  volatile uint32_t* gen = bar + 1;
  const uint32_t my_gen = *gen;
  __threadfence();
  const uint32_t old = atomicAdd(bar, 1u);
  if (old == (uint32_t)G - 1u) {
    atomicExch(bar, 0u);
    __threadfence();
    atomicAdd(bar + 1, 1u);
    return true;
  }
  const uint64_t t0 = gtimer();
  for (uint32_t i = 1;; ++i) {
    if (*gen != my_gen) {
      __threadfence();
      return true;
    }
    if ((i & 63u) == 0 && gtimer() - t0 > kWaitLimitNs) {
      atomicOr(status, kStatusTimeout);
      atomicExch(status + 1, 40u);
      return false;
    }
  }
}

// ----------------------------------------------------------------- kernel --

__global__ void __launch_bounds__(kDThreads, 1)
    gemm_decode_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const DecodeArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kDStages * kDAStage;
  DecodeTail* st = reinterpret_cast<DecodeTail*>(smem + kDStages * kDStageBytes);
  volatile uint32_t* abort_flag = &st->abort_flag;
  volatile uint32_t* a_ready = &st->a_ready;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = (int)gridDim.x, c = (int)blockIdx.x;
  const int KB = g.KB;
  const int64_t U = (int64_t)g.n_tiles * KB;
  const int64_t u0 = first_unit(c, U, G), u1 = first_unit(c + 1, U, G);
  const int n_units = (int)(u1 - u0);

  if (tid == 0) {
    for (int s = 0; s < kDStages; ++s) {
      mbar_init(smem_u32(&st->full[s]), 1);
      mbar_init(smem_u32(&st->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&st->tfull[b]), 1);
      mbar_init(smem_u32(&st->tempty[b]), 8);
    }
    st->abort_flag = 0;
    st->stop = 0;
    st->a_ready = g.a ? 0u : 1u;
    mbar_fence_init();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  if (warp == 1) tmem_alloc(smem_u32(&st->tmem_base), kDTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = st->tmem_base;

  if (warp == 0) {
    // --------------------------------------------------------- TMA producer --
    if (lane == 0) {
      // The weight tiles of the first stages do not depend on A: issue them
      // before the quantization finishes, then add A to the same stages.
      const int npre = min(kDStages, n_units);
      for (int i = 0; i < npre; ++i) {
        const int64_t u = u0 + i;
        const int t = (int)(u / KB), kb = (int)(u - (int64_t)t * KB);
        const uint32_t fb = smem_u32(&st->full[i]);
        mbar_expect_tx_only(fb, kDBStage);
        tma_load_2d(smem_u32(sB + i * kDBStage), &tmB, fb, kb * DK, t * DN);
      }
      bool alive = true;
      if (!*a_ready) {
        const uint64_t t0 = gtimer();
        for (uint32_t i = 1; !*a_ready; ++i) {
          if ((i & 63u) == 0 && (*abort_flag || gtimer() - t0 > kWaitLimitNs)) {
            alive = false;
            break;
          }
        }
      }
      if (!alive) {
        // no A will come: complete the preloaded stages' phases with their
        // weight bytes alone, so that the copies land before the CTA exits
        for (int i = 0; i < npre; ++i) mbar_arrive_expect_tx(smem_u32(&st->full[i]), 0);
        for (int i = 0; i < npre; ++i) mbar_drain(smem_u32(&st->full[i]), 0u, g.status, 41);
      } else {
        for (int i = 0; i < npre; ++i) {
          const int64_t u = u0 + i;
          const int kb = (int)(u % KB);
          const uint32_t fb = smem_u32(&st->full[i]);
          mbar_arrive_expect_tx(fb, kDAStage);
          tma_load_2d(smem_u32(sA + i * kDAStage), &tmA, fb, kb * DK, 0);
        }
        int it = npre;
        for (; it < n_units; ++it) {
          const int s = it % kDStages;
          const uint32_t ph = (uint32_t)(it / kDStages) & 1u;
          if (!mbar_wait(smem_u32(&st->empty[s]), ph ^ 1u, abort_flag, g.status, 42)) break;
          const int64_t u = u0 + it;
          const int t = (int)(u / KB), kb = (int)(u - (int64_t)t * KB);
          const uint32_t fb = smem_u32(&st->full[s]);
          mbar_arrive_expect_tx(fb, kDStageBytes);
          tma_load_2d(smem_u32(sB + s * kDBStage), &tmB, fb, kb * DK, t * DN);
          tma_load_2d(smem_u32(sA + s * kDAStage), &tmA, fb, kb * DK, 0);
        }
        if (it < n_units) {
          // aborted: let the copies already issued land before leaving
          const int n = min(it, kDStages);
          for (int j = 1; j <= n; ++j) {
            const int i2 = it - j;
            mbar_drain(smem_u32(&st->full[i2 % kDStages]), (uint32_t)(i2 / kDStages) & 1u, g.status, 43);
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------- fused quantization ------
    if (g.a) {
      quantize_share(g, c, G, warp - 1, lane);
      fence_proxy_async_global();   // the TMA loads of other CTAs read these codes
      __threadfence();
      named_bar(2, 320);
      if (tid == 32) {
        if (grid_barrier(g.grid_bar, G, g.status)) {
          fence_proxy_async_global();
          *a_ready = 1u;
        } else {
          *abort_flag = 1u;
        }
      }
      named_bar(2, 320);
    }
    if (warp <= 2) {
      // ------------------------------------------------------ MMA issuers --
      const uint32_t parity = (uint32_t)(warp - 1);
      if (lane == 0 && !*abort_flag) {
        int last = -1;
        for (int i = 0; i < n_units; ++i) {
          if (((uint32_t)i & 1u) != parity) continue;
          const int s = i % kDStages;
          const uint32_t ph = (uint32_t)(i / kDStages) & 1u;
          const int buf = (int)parity;
          const uint32_t use = (uint32_t)i >> 1;
          if (!mbar_wait(smem_u32(&st->tempty[buf]), (use & 1u) ^ 1u, abort_flag, g.status, 44) ||
              !mbar_wait(smem_u32(&st->full[s]), ph, abort_flag, g.status, 45))
            break;
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * kDAStage);
          const uint32_t b0 = smem_u32(sB + s * kDBStage);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t d = tmem_base + (uint32_t)(buf * 256 + h * 128);
#pragma unroll
            for (int kk = 0; kk < DK / 32; ++kk)
              mma_f8(d, sw128_desc(a0 + h * (128 * DK) + kk * 32), sw128_desc(b0 + kk * 32), kDIdesc,
                     kk > 0 ? 1u : 0u);
          }
          mma_commit(smem_u32(&st->empty[s]));
          mma_commit(smem_u32(&st->tfull[buf]));
          last = i;
        }
        if (last >= 0)
          mbar_drain(smem_u32(&st->empty[last % kDStages]), (uint32_t)(last / kDStages) & 1u, g.status,
                     46);
      }
      __syncwarp();
    } else {
      // ---------------------------------------------------------- epilogue --
      const int q = warp & 3;
      const int h = (warp - 3) >> 2;
      const int row = h * 128 + q * 32 + lane;
      const bool row_ok = row < g.M;
      const uint32_t lane_base = (uint32_t)(q * 32) << 16;
      bool alive = true;
      int i = 0;   // unit index within this CTA
      int64_t u = u0;
      int split[2];      // this CTA's split tiles (only the ends of its range can be)
      int n_split = 0;
      while (u < u1) {
        const int t = (int)(u / KB);
        const int ka = (int)(u - (int64_t)t * KB);
        const int64_t kz64 = (int64_t)ka + (u1 - u);
        const int kz = kz64 < KB ? (int)kz64 : KB;
        const float* swp = g.sw + (int64_t)t * KB;
        float acc[DN];
#pragma unroll
        for (int j = 0; j < DN; ++j) acc[j] = 0.0f;
        float sa_next = row_ok ? __ldcg(g.sa + (int64_t)ka * g.M + row) : 0.0f;
        float sw_next = __ldg(swp + ka);
        for (int kb = ka; kb < kz; ++kb, ++i) {
          const int buf = i & 1;
          const uint32_t use = (uint32_t)i >> 1;
          const float f = __fmul_rn(sa_next, sw_next);
          if (kb + 1 < kz) {
            sa_next = row_ok ? __ldcg(g.sa + (int64_t)(kb + 1) * g.M + row) : 0.0f;
            sw_next = __ldg(swp + kb + 1);
          }
          bool okw = mbar_wait(smem_u32(&st->tfull[buf]), use & 1u, abort_flag, g.status, 47);
          okw = __all_sync(0xFFFFFFFFu, okw);
          if (!okw) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem_base + lane_base + (uint32_t)(buf * 256 + h * 128);
          uint32_t p[16];
#pragma unroll
          for (int cc = 0; cc < DN / 16; ++cc) {
            tmem_ld16(taddr + cc * 16, p);
            tmem_wait_ld();
            if (cc == DN / 16 - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&st->tempty[buf]));
            }
#pragma unroll
            for (int j = 0; j < 16; j += 2) ffma2(acc[cc * 16 + j], acc[cc * 16 + j + 1], p[j], p[j + 1], f);
          }
        }
        // Leave together or not at all: a warp whose wait failed raises the
        // abort flag; after a barrier one thread reads it once and publishes
        // the decision, so all 8 warps take the same branch (the named
        // barriers below need all 256 threads).
        alive = __all_sync(0xFFFFFFFFu, alive);
        if (!alive && lane == 0) *abort_flag = 1u;
        named_bar(1, 256);
        if (tid == 96) st->stop = *abort_flag;
        named_bar(1, 256);
        if (st->stop) break;
        __nv_bfloat16* yrow = g.y + (int64_t)row * g.ldy + (int64_t)t * DN;
        if (ka == 0 && kz == KB) {
          if (row_ok) {
#pragma unroll
            for (int cc = 0; cc < DN / 8; ++cc) {
              uint4 v;
              __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[cc * 8 + 0], acc[cc * 8 + 1]);
              __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[cc * 8 + 2], acc[cc * 8 + 3]);
              __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[cc * 8 + 4], acc[cc * 8 + 5]);
              __nv_bfloat162 b3 = __floats2bfloat162_rn(acc[cc * 8 + 6], acc[cc * 8 + 7]);
              v.x = *reinterpret_cast<uint32_t*>(&b0);
              v.y = *reinterpret_cast<uint32_t*>(&b1);
              v.z = *reinterpret_cast<uint32_t*>(&b2);
              v.w = *reinterpret_cast<uint32_t*>(&b3);
              *reinterpret_cast<uint4*>(yrow + cc * 8) = v;
            }
          }
        } else {
          // partial tile: publish it and count this CTA in; the tile is
          // reduced after the main loop (below)
          float* mine = g.partials + (size_t)slot_of(c, t, U, G, KB) * kPartialFloats;
#pragma unroll
          for (int cc = 0; cc < DN / 4; ++cc)
            __stcg(reinterpret_cast<float4*>(mine + ((size_t)cc * DM + row) * 4),
                   make_float4(acc[cc * 4], acc[cc * 4 + 1], acc[cc * 4 + 2], acc[cc * 4 + 3]));
          // the barrier orders every thread's stores before thread 96's fence
          // and release (fences are cumulative), so one fence suffices
          named_bar(1, 256);
          if (tid == 96) {
            __threadfence();
            atomicAdd(g.arrive + t, 1u);
          }
          split[n_split++] = t;
        }
        u += kz - ka;
      }
      // ------------------------------------------------- split tiles ------
      // Every CTA publishes its partials during its main loop and waits for
      // nothing there, so each split tile's partials all arrive.  Here each
      // CTA of a split tile waits (bounded) for them, then sums its share of
      // the tile's rows over the tile's CTAs in k order (the result does not
      // depend on arrival order) and stores BF16.  All CTAs are resident
      // (cooperative launch), so the waits end.
      for (int p = 0; p < n_split && !st->stop; ++p) {
        const int t = split[p];
        const int cf = owner_of((int64_t)t * KB, U, G);
        const int nseg = owner_of((int64_t)t * KB + KB - 1, U, G) - cf + 1;
        const int myseg = c - cf;
        if (tid == 96) {
          volatile uint32_t* arr = g.arrive + t;
          const uint64_t t0 = gtimer();
          bool ok = true;
          for (uint32_t it = 1; *arr < (uint32_t)nseg; ++it) {
            if ((it & 63u) == 0 && (*abort_flag || gtimer() - t0 > kWaitLimitNs)) {
              if (!*abort_flag) {
                atomicOr(g.status, kStatusTimeout);
                atomicExch(g.status + 1, 48u);
                *abort_flag = 1u;
              }
              ok = false;
              break;
            }
          }
          __threadfence();
          st->stop = ok ? 0u : 1u;
        }
        named_bar(1, 256);
        if (st->stop) break;
        const int r0 = (DM * myseg) / nseg;
        const int r1 = min((DM * (myseg + 1)) / nseg, g.M);
        const int nrows = max(r1 - r0, 0);
        const int nel = nrows * (DN / 4);            // float4 elements of the share (<= 4096)
        const int et = tid - 96;
        constexpr int kEl = 16;                        // per thread; a partial's loads go out together
        float4 sum[kEl];
        for (int j = 0; j < nseg; ++j) {
          const float* pj = g.partials + (size_t)slot_of(cf + j, t, U, G, KB) * kPartialFloats;
          float4 v[kEl];
#pragma unroll
          for (int e = 0; e < kEl; ++e) {
            const int idx = et + e * 256;
            v[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (idx < nel) {
              const int cc = idx / nrows, r = r0 + idx % nrows;
              v[e] = __ldcg(reinterpret_cast<const float4*>(pj + ((size_t)cc * DM + r) * 4));
            }
          }
#pragma unroll
          for (int e = 0; e < kEl; ++e) {
            if (j == 0) {
              sum[e] = v[e];
            } else {
              sum[e].x = __fadd_rn(sum[e].x, v[e].x);
              sum[e].y = __fadd_rn(sum[e].y, v[e].y);
              sum[e].z = __fadd_rn(sum[e].z, v[e].z);
              sum[e].w = __fadd_rn(sum[e].w, v[e].w);
            }
          }
        }
#pragma unroll
        for (int e = 0; e < kEl; ++e) {
          const int idx = et + e * 256;
          if (idx < nel) {
            const int cc = idx / nrows, r = r0 + idx % nrows;
            __nv_bfloat162 b0 = __floats2bfloat162_rn(sum[e].x, sum[e].y);
            __nv_bfloat162 b1 = __floats2bfloat162_rn(sum[e].z, sum[e].w);
            uint2 o;
            o.x = *reinterpret_cast<uint32_t*>(&b0);
            o.y = *reinterpret_cast<uint32_t*>(&b1);
            *reinterpret_cast<uint2*>(g.y + (int64_t)r * g.ldy + (int64_t)t * DN + cc * 4) = o;
          }
        }
        named_bar(1, 256);
        if (tid == 96) {
          // the tile's last CTA out returns both counters to zero
          if (atomicAdd(g.done + t, 1u) == (uint32_t)nseg - 1u) {
            g.arrive[t] = 0u;
            g.done[t] = 0u;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kDTmemCols);
  }
}

// ------------------------------------------------------------------- host --

struct DecodeDevice {
  bool attr_set = false;
  int grid = 0;            // cooperative grid: co-resident CTAs (one per SM)
};
std::mutex g_dec_mu;
DecodeDevice g_dec[64];

fp8rl_status decode_device(const DeviceState* ds, DecodeDevice* out) {
  std::lock_guard<std::mutex> lock(g_dec_mu);
  DecodeDevice& d = g_dec[ds->device];
  if (!d.attr_set) {
    if ((size_t)ds->max_smem_optin < kDSmem)
      return fail(FP8RL_ERR_UNSUPPORTED_DEVICE, "decode GEMM needs %zu bytes of shared memory",
                  kDSmem);
    fp8rl_status st = cuda_check(cudaFuncSetAttribute(gemm_decode_kernel,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                      (int)kDSmem),
                                 "cudaFuncSetAttribute(decode gemm)");
    if (st != FP8RL_OK) return st;
    int per_sm = 0;
    st = cuda_check(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_decode_kernel,
                                                                  kDThreads, kDSmem),
                    "cudaOccupancyMaxActiveBlocksPerMultiprocessor(decode gemm)");
    if (st != FP8RL_OK) return st;
    if (per_sm < 1) return fail(FP8RL_ERR_UNSUPPORTED_DEVICE, "decode GEMM does not fit on an SM");
    d.grid = ds->sm_count;   // one CTA per SM
    d.attr_set = true;
  }
  *out = d;
  return FP8RL_OK;
}

size_t counters_bytes(int64_t n_tiles) { return (size_t)((4 * n_tiles + 255) / 256) * 256; }

size_t workspace_bytes_for(int grid, int64_t n_tiles) {
  const size_t ctl = 256 + 2 * counters_bytes(n_tiles);
  return ctl + (size_t)2 * grid * kPartialFloats * sizeof(float);
}

}  // namespace
}  // namespace fp8rl

using namespace fp8rl;

extern "C" size_t fp8rl_linear_w8a8_decode_workspace_bytes(int64_t n) {
  DeviceState* ds = nullptr;
  if (n < 0 || device_state(&ds) != FP8RL_OK) return 0;
  return workspace_bytes_for(ds->sm_count, (n + DN - 1) / DN);
}

extern "C" fp8rl_status fp8rl_linear_w8a8_decode(const void* a, int64_t lda, uint8_t* qa, float* sa,
                                                 const uint8_t* qw, const float* sw, int64_t m,
                                                 int64_t n, int64_t k, void* y, int64_t ldy,
                                                 void* workspace, size_t workspace_bytes,
                                                 cudaStream_t stream) {
  if (!qa || !sa || !qw || !sw || !y || !workspace) return fail(FP8RL_ERR_INVALID_ARG, "null pointer");
  if (m < 0 || m > DM) return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "need 0 <= m <= 256 (m=%lld)", (long long)m);
  if (n < DN || n % DN) return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "n must be a positive multiple of 128");
  if (k < DK || k % DK) return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "k must be a positive multiple of 128");
  if (n > INT32_MAX / 2 || k > INT32_MAX / 2) return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "n or k too large");
  if (ldy < n || ldy % 8) return fail(FP8RL_ERR_ALIGNMENT, "need ldy >= n and ldy % 8 == 0");
  if (a && (lda < k || lda % 8)) return fail(FP8RL_ERR_ALIGNMENT, "need lda >= k and lda % 8 == 0");
  if ((a && !aligned(a, 16)) || !aligned(qa, 16) || !aligned(qw, 16) || !aligned(y, 16) ||
      !aligned(sa, 4) || !aligned(sw, 4) || !aligned(workspace, 256))
    return fail(FP8RL_ERR_ALIGNMENT,
                "a, qa, qw and y must be 16-byte aligned and the workspace 256-byte aligned");
  if (m == 0) return ok();
  DeviceState* ds = nullptr;
  fp8rl_status st = device_state(&ds);
  if (st != FP8RL_OK) return st;
  DecodeDevice dd;
  if ((st = decode_device(ds, &dd)) != FP8RL_OK) return st;
  const int64_t n_tiles = n / DN;
  const size_t need = workspace_bytes_for(dd.grid, n_tiles);
  if (workspace_bytes < need)
    return fail(FP8RL_ERR_INVALID_ARG, "workspace holds %zu bytes; this call needs %zu", workspace_bytes,
                need);
  CUtensorMap tmA, tmB;
  if ((st = encode_tiled_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, qa, (uint64_t)k, (uint64_t)m, (uint64_t)k,
                            DK, DM, CU_TENSOR_MAP_SWIZZLE_128B, "decode A")) != FP8RL_OK)
    return st;
  if ((st = encode_tiled_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, qw, (uint64_t)k, (uint64_t)n, (uint64_t)k,
                            DK, DN, CU_TENSOR_MAP_SWIZZLE_128B, "decode W")) != FP8RL_OK)
    return st;
  DecodeArgs g;
  g.a = reinterpret_cast<const uint16_t*>(a);
  g.lda = lda;
  g.qa = qa;
  g.sa = sa;
  g.sw = sw;
  g.y = reinterpret_cast<__nv_bfloat16*>(y);
  g.ldy = ldy;
  g.M = (int)m;
  g.N = (int)n;
  g.KB = (int)(k / DK);
  g.n_tiles = (int)n_tiles;
  char* ws = static_cast<char*>(workspace);
  g.grid_bar = reinterpret_cast<uint32_t*>(ws);
  g.arrive = reinterpret_cast<uint32_t*>(ws + 256);
  g.done = reinterpret_cast<uint32_t*>(ws + 256 + counters_bytes(n_tiles));
  g.partials = reinterpret_cast<float*>(ws + 256 + 2 * counters_bytes(n_tiles));
  g.status = ds->status;
  // At most one CTA per unit, so that every CTA owns at least one: then the
  // CTAs from a tile's first owner to its last all hold part of it, and the
  // tile's arrival count is their number.
  const int grid = (int)std::min<int64_t>(dd.grid, n_tiles * (k / DK));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kDThreads, 1, 1);
  cfg.dynamicSmemBytes = kDSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // CTAs wait for one another at the grid barrier
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  st = cuda_check(cudaLaunchKernelEx(&cfg, gemm_decode_kernel, tmA, tmB, g), "gemm_decode_kernel launch");
  return st == FP8RL_OK ? ok() : st;
}
