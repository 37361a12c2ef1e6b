// gemm.cu -- blockwise-scaled FP8 W8A8 GEMM on sm_103a tensor cores.
//
// FP8-RL summary, section 3.4.2 Phase 3: the rollout's linear layers multiply
// dynamically quantized FP8 activations by the per-step re-quantized FP8
// weights on FP8 tensor cores, accumulate in FP32 and emit BF16; section
// 3.4.1 fixes the scale granularity (weights 128x128 blocks, activations
// 1x128 groups) and names the MoE expert layers (fc1/fc2) as the grouped case.
//
//   Y[i, j] = bf16( sum_kb  sa[kb, i] * sw[j/128, kb] * P_kb[i, j] ),
//   P_kb[i, j] = sum_{k in block kb} dec(qa[i, k]) * dec(qw[j, k]).
//
// The scales are arbitrary binary32 numbers (amax/448), so they cannot ride on
// the hardware's block-scaled MMA (power-of-two UE8M0 scales per 32 K).  Each
// 128-wide k-block is therefore one MMA group writing a fresh FP32 partial
// P_kb into tensor memory; epilogue warps read it back (tcgen05.ld, 16 columns at a time), multiply
// by sa*sw and add it into FP32 register accumulators (packed FP32x2 FMAs;
// the scales of k-block kb+1 are fetched while kb is promoted).
//
// Kernel shape (one CTA per SM, persistent over output tiles):
//   tile 128 (M) x 256 (N), k-block 128; TMA ring of 48 KB stages (A 128x128
//   + B 256x128 bytes, 128-byte swizzle), 3 stages plus 64 KB of output
//   staging.  The split-K flavour uses 128 x 128 tiles and 6 stages of 32 KB;
//   warp 0      TMA producer (lane 0),
//   warps 1, 2  MMA issuers (tcgen05.mma kind::f8f6f4, M=128 N=256 K=32, four
//               per k-block, lane 0): warp 1 issues the even k-blocks into
//               TMEM partial buffer 0, warp 2 the odd ones into buffer 1.
//               One thread alone spends longer issuing a k-block (barrier
//               waits, fence, four MMAs, two commits) than the tensor core
//               spends executing it; two alternating issuers keep it busy.
//               Each warp's commits track only its own MMAs.
//   warps 3-10  epilogue: warp w reads TMEM lanes 32*(w%4).. and column half
//               (w-3)/4, 128 FP32 accumulators per thread (64 in the split-K
//               flavour); a finished tile
//               is converted to BF16 into the warp's 8 KB staging buffer and
//               written by TMA tensor stores (plain stores for ragged rows).
//   TMEM: two partial buffers as wide as the tile (all 512 columns for the
//   256-wide tile), so the MMA of k-block kb+1 overlaps the promotion of kb.
// Mid-sized problems (fewer than two waves of 256-wide tiles) run the narrow
// flavour: 128 x 128 tiles and four TMEM partial buffers.  Decode-sized
// problems (256-wide tiles for at most half the SMs) run the split-K flavour:
// 128-wide tiles, so that twice as many CTAs share the work and each
// k-block's MMA and promotion take half as long, and a cluster of 2-4 CTAs
// per tile, each over a slice of the k-blocks (the narrow flavour, one CTA
// per tile, when no cluster of two fits).  Each split CTA stages its FP32
// partial tile in its own (by then idle) pipeline buffers; rank r then reads
// rows [r*128/S, (r+1)*128/S) of all S partials through distributed shared
// memory, sums them in rank order and stores them (reduce-scatter, no global
// scratch, deterministic).
// Every wait on an mbarrier is bounded (1 s); on expiry the kernel records it
// in the library's device status word, drains what it issued and returns.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace fp8rl {
namespace {

constexpr int BM = 128, BK = 128;
constexpr int kThreads = 352;            // 11 warps
constexpr int kAStage = BM * BK;                 // 16 KB
constexpr int kMaxExperts = 1024;
constexpr int kMGroup = 16;                      // m-tiles per raster band (L2 reuse)
constexpr int kMaxStages = 6;

// The tile flavours.
//   Wide (kWide; grouped GEMMs): 128 x 256 tiles, 3 stages of 48 KB, two TMEM
//     partial buffers, and 64 KB of output staging so the epilogue never waits
//     for its previous tile's stores.
//   Split-K (kSplitK; decode shapes): 128 x 128 tiles and 6 stages of 32 KB,
//     to keep more DRAM reads in flight; partials reduced across a cluster.
//   Narrow (kNarrow; dense GEMMs with many tiles): 128 x 128 tiles, 5 stages
//     of 32 KB, FOUR TMEM partial buffers and 32 KB of output staging.  With
//     two buffers, a buffer's promotion, the warps' skew and its release
//     take longer than the other buffer's MMAs, so the tensor pipe waits
//     every k-block; four buffers let the MMAs run three k-blocks ahead.
//     (Stages >= buffers: a stage's previous use is always a k-block whose
//     buffer the epilogue has released before its next wait can start.)
constexpr int kWide = 0, kSplitK = 1, kNarrow = 2;
template <int kF>
struct Flavour {
  static constexpr int kBN = kF == kWide ? 256 : 128;
  static constexpr int kStages = kF == kWide ? 3 : (kF == kSplitK ? 6 : 5);
  static constexpr int kBufs = kF == kNarrow ? 4 : 2;   // TMEM partial buffers
  static constexpr bool kStaged = kF != kSplitK;          // TMA output staging
  static constexpr int kBStage = kBN * BK;
  static constexpr int kStageBytes = kAStage + kBStage;
  static constexpr int kHalf = kBN / 2;             // columns per epilogue warp
  static constexpr int kBoxes = kHalf / 64;         // 32 x 64 output boxes per warp
  static constexpr uint32_t kTmemCols = kBufs * kBN;
  // tcgen05 instruction descriptor, kind::f8f6f4: D = F32 (bits 4-5 = 1),
  // A = B = E4M3 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0),
  // N >> 3 in bits 17-22, M >> 4 in bits 24-28.
  static constexpr uint32_t kIdesc =
      (1u << 4) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
};
static_assert(Flavour<kWide>::kStages <= kMaxStages && Flavour<kSplitK>::kStages <= kMaxStages &&
                  Flavour<kNarrow>::kStages <= kMaxStages && Flavour<kNarrow>::kStages >= Flavour<kNarrow>::kBufs,
              "");
static_assert(Flavour<kNarrow>::kTmemCols <= 512 && Flavour<kWide>::kTmemCols <= 512, "TMEM columns");

struct SharedTail {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[4];
  uint64_t tempty[4];
  uint32_t tmem_base;
  uint32_t abort_flag;
  int32_t total_tiles;
  int32_t pad;
  int32_t seg[kMaxExperts + 1];      // grouped: clamped row offsets
  int32_t tstart[kMaxExperts + 1];   // grouped: first tile of each expert
  int32_t wsum[8];
};

// Output staging (flavours without split): 8 KB per epilogue warp, its 32 rows
// x 128 columns as two 32 x 64 BF16 boxes in the 128-byte swizzled layout the
// Y tensor map describes; after the tail, 1 KB aligned.
constexpr int kYBox = 32, kYBoxCols = 64;
constexpr int kYBoxBytes = kYBox * kYBoxCols * 2;
constexpr size_t kTailPad = (sizeof(SharedTail) + 1023) / 1024 * 1024;
template <int kF>
constexpr size_t smem_bytes() {
  using F = Flavour<kF>;
  return 1024 + (size_t)F::kStages * F::kStageBytes + kTailPad +
         (F::kStaged ? 8 * (size_t)F::kBoxes * kYBoxBytes : 0);
}
static_assert(smem_bytes<kWide>() <= 232448 && smem_bytes<kSplitK>() <= 232448 &&
                  smem_bytes<kNarrow>() <= 232448,
              "shared memory budget");

// Split-K flavour: a cluster owns exactly one tile, so once its last MMA has
// completed the stage buffers are idle and hold the FP32 partial tile,
// [128 rows][kRedLd] (row pitch 528 B: 16-byte stores by consecutive rows
// and 16-byte loads along a row are both bank-conflict free).
constexpr int kRedLd = Flavour<kSplitK>::kBN + 4;
constexpr int kMaxSplit = 4;
constexpr int kRedBatch = 4;             // row chunks whose loads are in flight together
static_assert((size_t)BM * kRedLd * sizeof(float) <=
                  (size_t)Flavour<kSplitK>::kStages * Flavour<kSplitK>::kStageBytes,
              "the partial tile must fit in the stage buffers");

struct GemmArgs {
  const float* sa;         // [KB, M] group-major activation scales
  const float* sw;         // [E][NB][KB] weight block scales (E = 1 when dense)
  __nv_bfloat16* y;
  int64_t ldy;
  int M, N, KB, NB;        // M = rows of A (m or m_total)
  int num_m, num_n;        // num_m: dense only
  const int32_t* offsets;  // grouped: [E+1] device
  int E;                   // grouped: experts
  uint32_t* status;        // library status word
  int split;               // split-K cluster size (1 = no split)
};

using namespace ptx;

// acc0 += p0 * f, acc1 += p1 * f as one packed FP32x2 FMA (each lane an IEEE
// round-to-nearest FMA, the same result as two fmaf calls).
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

// ---------------------------------------------------------- tile schedule --

struct Tile {
  int m0;        // first A row
  int row_end;   // rows >= row_end are not part of this tile's problem
  int n0;        // first output column
  int brow;      // first B row (e * N + n0)
  int e;         // expert (0 when dense)
};

template <bool kGrouped, int kBN>
__device__ __forceinline__ Tile decode_tile(int t, const GemmArgs& g, const SharedTail* st) {
  Tile tl;
  if (!kGrouped) {
    const int per_band = kMGroup * g.num_n;
    const int band = t / per_band;
    const int first_m = band * kMGroup;
    const int gs = min(kMGroup, g.num_m - first_m);
    const int local = t - band * per_band;
    const int mt = first_m + local % gs;
    const int nt = local / gs;
    tl.m0 = mt * BM;
    tl.row_end = g.M;
    tl.n0 = nt * kBN;
    tl.brow = tl.n0;
    tl.e = 0;
  } else {
    int lo = 0, hi = g.E - 1;   // last expert whose first tile is <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (st->tstart[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int cnt = st->seg[e + 1] - st->seg[e];
    const int mtiles = (cnt + BM - 1) / BM;
    const int local = t - st->tstart[e];
    const int mt = local % mtiles;
    const int nt = local / mtiles;
    tl.m0 = st->seg[e] + mt * BM;
    tl.row_end = st->seg[e + 1];
    tl.n0 = nt * kBN;
    tl.brow = e * g.N + tl.n0;
    tl.e = e;
  }
  return tl;
}

// Grouped: copy the offsets (clamped to [0, M], made non-decreasing) and
// build the exclusive prefix of tiles per expert, all threads cooperating.
__device__ void build_expert_schedule(const GemmArgs& g, SharedTail* st) {
  const int tid = threadIdx.x;
  for (int i = tid; i <= g.E; i += kThreads) st->seg[i] = min(max(g.offsets[i], 0), g.M);
  __syncthreads();
  if (tid == 0) {
    for (int i = 1; i <= g.E; ++i) st->seg[i] = max(st->seg[i], st->seg[i - 1]);
  }
  __syncthreads();
  int loc[4];
  int sum = 0;
  if (tid < 256) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = tid * 4 + j;
      const int c = e < g.E ? st->seg[e + 1] - st->seg[e] : 0;
      loc[j] = sum;
      sum += ((c + BM - 1) / BM) * g.num_n;
    }
  }
  // inclusive warp scan of the per-thread sums, then across the 8 warps
  const int lane = tid & 31, warp = tid >> 5;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (warp < 8 && lane == 31) st->wsum[warp] = incl;
  __syncthreads();
  if (tid < 256) {
    int before = 0;
    for (int w = 0; w < warp; ++w) before += st->wsum[w];
    const int excl = before + incl - sum;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = tid * 4 + j;
      if (e < g.E) st->tstart[e] = excl + loc[j];
    }
    if (tid == 255) {
      int total = 0;
      for (int w = 0; w < 8; ++w) total += st->wsum[w];
      st->tstart[g.E] = total;
      st->total_tiles = total;
    }
  }
}

// ----------------------------------------------------------------- kernel --

// Split-K: rank r of S owns rows [128*r/S, 128*(r+1)/S) of the tile.  Its
// threads read those rows of every rank's staged partial (16-byte loads
// through distributed shared memory, all of a batch issued before any is
// used), sum them in rank order and store BF16.  Called by all kThreads
// threads (et = thread index) once every rank's partial is staged.
__device__ __forceinline__ void reduce_rows(uint32_t red, int crank, int nsplit, int m0,
                                            int row_end, int n0, const GemmArgs& g, int et) {
  const int lo = (BM * crank) / nsplit;
  const int hi = min((BM * (crank + 1)) / nsplit, row_end - m0);
  constexpr int kV = Flavour<kSplitK>::kBN / 4;   // 16-byte vectors per row
  const int tasks = (hi - lo) * kV;
  uint32_t base[kMaxSplit];
#pragma unroll
  for (int pr = 0; pr < kMaxSplit; ++pr) base[pr] = mapa(red, (uint32_t)(pr < nsplit ? pr : 0));
  for (int t0 = et; t0 < tasks; t0 += kRedBatch * kThreads) {
    float4 p[kRedBatch][kMaxSplit];
#pragma unroll
    for (int b = 0; b < kRedBatch; ++b) {
      const int t = t0 + b * kThreads;
      const int r = lo + t / kV, c4 = t % kV;
      const uint32_t off = (uint32_t)((r * kRedLd + c4 * 4) * (int)sizeof(float));
#pragma unroll
      for (int pr = 0; pr < kMaxSplit; ++pr)
        if (t < tasks && pr < nsplit) p[b][pr] = ld_cluster_v4(base[pr] + off);
    }
#pragma unroll
    for (int b = 0; b < kRedBatch; ++b) {
      const int t = t0 + b * kThreads;
      if (t >= tasks) break;
      const int r = lo + t / kV, c4 = t % kV;
      float4 v = p[b][0];
#pragma unroll
      for (int pr = 1; pr < kMaxSplit; ++pr) {
        if (pr < nsplit) {
          v.x = __fadd_rn(v.x, p[b][pr].x);
          v.y = __fadd_rn(v.y, p[b][pr].y);
          v.z = __fadd_rn(v.z, p[b][pr].z);
          v.w = __fadd_rn(v.w, p[b][pr].w);
        }
      }
      const int col = n0 + c4 * 4;
      if (col < g.N) {
        __nv_bfloat162 b0 = __floats2bfloat162_rn(v.x, v.y);
        __nv_bfloat162 b1 = __floats2bfloat162_rn(v.z, v.w);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&b0);
        o.y = *reinterpret_cast<uint32_t*>(&b1);
        *reinterpret_cast<uint2*>(g.y + (int64_t)(m0 + r) * g.ldy + col) = o;
      }
    }
  }
}

// kSplit: the CTAs of a thread-block cluster (g.split of them, launched with
// cluster dimension g.split along x) share one output tile; rank r
// accumulates k-blocks [r*KB/split, (r+1)*KB/split), then the partials are
// reduce-scattered over the ranks by rows (see reduce_rows).  Used when there
// are too few tiles to fill the GPU (decode-sized M); two cluster barrier
// phases order it: (A) every partial is staged, (B) no CTA reads a peer's
// shared memory any more (waited for only just before leaving).
template <bool kGrouped, int kF>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_w8a8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmY, const GemmArgs g) {
  using F = Flavour<kF>;
  constexpr bool kSplit = kF == kSplitK;
  constexpr int STAGES = F::kStages;
  constexpr int BUFS = F::kBufs;
  constexpr int kBN = F::kBN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * kAStage;
  SharedTail* st = reinterpret_cast<SharedTail*>(smem + STAGES * F::kStageBytes);
  float* red = reinterpret_cast<float*>(smem);   // split-K: aliases the idle stage buffers
  uint8_t* ystage = smem + STAGES * F::kStageBytes + kTailPad;   // staged flavours only
  volatile uint32_t* abort_flag = &st->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // cluster geometry (a plain launch is a "cluster" of one)
  const int nsplit = kSplit ? g.split : 1;
  const uint32_t crank = kSplit ? cluster_ctarank() : 0u;
  const int cid = kSplit ? (int)(blockIdx.x / nsplit) : (int)blockIdx.x;
  const int ncl = kSplit ? (int)(gridDim.x / nsplit) : (int)gridDim.x;
  const int kb_lo = kSplit ? (int)(((int64_t)g.KB * crank) / nsplit) : 0;
  const int kb_hi = kSplit ? (int)(((int64_t)g.KB * (crank + 1)) / nsplit) : g.KB;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&st->full[s]), 1);
      mbar_init(smem_u32(&st->empty[s]), 1);
    }
    for (int b = 0; b < BUFS; ++b) {
      mbar_init(smem_u32(&st->tfull[b]), 1);
      mbar_init(smem_u32(&st->tempty[b]), 8);
    }
    st->abort_flag = 0;
    if (!kGrouped) st->total_tiles = g.num_m * g.num_n;
    mbar_fence_init();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
    if (F::kStaged) tma_prefetch_map(&tmY);
  }
  // The launch allows programmatic serialization: the launch itself and the
  // set-up above (barriers, tensor-map prefetch) may overlap the tail of the
  // previous kernel in the stream.  Nothing touches global memory, and TMEM
  // is not allocated (a kernel still running on this SM may need it), before
  // that kernel has completed.
  grid_dependency_wait();
  if (warp == 1) {
    tmem_alloc(smem_u32(&st->tmem_base), F::kTmemCols);
  }
  if (kGrouped) build_expert_schedule(g, st);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = st->tmem_base;
  const int total_tiles = st->total_tiles;
  const int KB = g.KB;

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer --
    if (lane == 0) {
      uint32_t it = 0;
      bool alive = true;
      for (int t = cid; t < total_tiles && alive; t += ncl) {
        const Tile tl = decode_tile<kGrouped, kBN>(t, g, st);
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(smem_u32(&st->empty[s]), ph ^ 1u, abort_flag, g.status, 1)) {
            alive = false;
            break;
          }
          const uint32_t fb = smem_u32(&st->full[s]);
          mbar_expect_tx(fb, F::kStageBytes);
          tma_load_2d(smem_u32(sA + s * kAStage), &tmA, fb, kb * BK, tl.m0);
          tma_load_2d(smem_u32(sB + s * F::kBStage), &tmB, fb, kb * BK, tl.brow);
        }
      }
      if (!alive) {
        // let the copies already issued land before the CTA can exit
        const uint32_t n = it < (uint32_t)STAGES ? it : (uint32_t)STAGES;
        for (uint32_t j = 1; j <= n; ++j) {
          const uint32_t i2 = it - j;
          mbar_drain(smem_u32(&st->full[i2 % STAGES]), (i2 / STAGES) & 1u, g.status, 9);
        }
      }
    }
    __syncwarp();
  } else if (warp <= 2) {
    // ------------------------------------------------------- MMA issuers --
    // warp 1 takes the k-blocks with even global index, warp 2 the odd ones;
    // k-block it uses TMEM buffer it % BUFS (BUFS is even, so each buffer has
    // one issuer)
    const uint32_t parity = (uint32_t)(warp - 1);
    if (lane == 0) {
      uint32_t it = 0;        // global k-block index (all tiles of this CTA)
      uint32_t last = 0;
      bool any = false, alive = true;
      for (int t = cid; t < total_tiles && alive; t += ncl) {
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
          if ((it & 1u) != parity) continue;
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          const int buf = (int)(it % BUFS);
          const uint32_t u = it / BUFS;         // use count of this buffer
          if (!mbar_wait(smem_u32(&st->tempty[buf]), (u & 1u) ^ 1u, abort_flag, g.status, 2) ||
              !mbar_wait(smem_u32(&st->full[s]), ph, abort_flag, g.status, 3)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + (uint32_t)(buf * kBN);
          const uint32_t a0 = smem_u32(sA + s * kAStage);
          const uint32_t b0 = smem_u32(sB + s * F::kBStage);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk)
            mma_f8(d, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), F::kIdesc,
                   kk > 0 ? 1u : 0u);
          mma_commit(smem_u32(&st->empty[s]));
          mma_commit(smem_u32(&st->tfull[buf]));
          last = it;
          any = true;
        }
      }
      if (any) {
        // this warp's last stage release must have landed before the CTA exits
        mbar_drain(smem_u32(&st->empty[last % STAGES]), (last / STAGES) & 1u, g.status, 8);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int h = (warp - 3) >> 2;          // column half of the tile (F::kHalf columns)
    constexpr int kAcc = F::kHalf;          // FP32 accumulators per thread
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t kit = 0;
    bool alive = true;
    for (int t = cid; t < total_tiles && alive; t += ncl) {
      const Tile tl = decode_tile<kGrouped, kBN>(t, g, st);
      const int row = tl.m0 + q * 32 + lane;
      const bool row_ok = row < tl.row_end;
      // weight block of this column half (both halves of a 128-wide tile share one)
      const int nbi = (tl.n0 + h * kAcc) / 128;
      const float* swp = g.sw + ((int64_t)tl.e * g.NB + nbi) * KB;
      const bool nb_ok = nbi < g.NB;
      float acc[kAcc];
#pragma unroll
      for (int j = 0; j < kAcc; ++j) acc[j] = 0.0f;
      // scales of the next k-block are loaded one iteration ahead so their
      // latency hides behind the current promotion
      float sa_next = row_ok ? __ldg(g.sa + (int64_t)kb_lo * g.M + row) : 0.0f;
      float sw_next = nb_ok ? __ldg(swp + kb_lo) : 0.0f;
      for (int kb = kb_lo; kb < kb_hi; ++kb, ++kit) {
        const int buf = (int)(kit % BUFS);
        const uint32_t u = kit / BUFS;
        const float f = __fmul_rn(sa_next, sw_next);
        if (kb + 1 < kb_hi) {
          sa_next = row_ok ? __ldg(g.sa + (int64_t)(kb + 1) * g.M + row) : 0.0f;
          sw_next = nb_ok ? __ldg(swp + kb + 1) : 0.0f;
        }
        bool okw = mbar_wait(smem_u32(&st->tfull[buf]), u & 1u, abort_flag, g.status, 4);
        okw = __all_sync(0xFFFFFFFFu, okw);
        if (!okw) { alive = false; break; }
        tc_fence_after();
        const uint32_t taddr = tmem_base + lane_base + (uint32_t)(buf * kBN + h * kAcc);
        uint32_t p[16];
#pragma unroll
        for (int c = 0; c < kAcc / 16; ++c) {
          tmem_ld16(taddr + c * 16, p);
          tmem_wait_ld();
          if (c == kAcc / 16 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&st->tempty[buf]));
          }
#pragma unroll
          for (int j = 0; j < 16; j += 2)
            ffma2(acc[c * 16 + j], acc[c * 16 + j + 1], p[j], p[j + 1], f);
        }
      }
      if (!alive) break;
      if constexpr (kSplit) {
        // The last tfull wait above means every MMA of this CTA has completed:
        // the stage buffers are idle.  Stage this row of the partial there.
        float* mine = red + (size_t)(q * 32 + lane) * kRedLd + h * kAcc;
#pragma unroll
        for (int j = 0; j < kAcc; j += 4)
          *reinterpret_cast<float4*>(mine + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
      } else {
        const int row0 = tl.m0 + q * 32;
        if (row0 + kYBox <= tl.row_end) {
          // The warp's 32 rows all belong to this tile: stage them as two
          // 32 x 64 boxes and write them with TMA tensor stores (the tensor map
          // clips columns beyond N).  The buffer was last read by the stores of
          // this warp's previous tile, a whole tile of k-blocks ago.
          const uint32_t stg = smem_u32(ystage + (warp - 3) * (F::kBoxes * kYBoxBytes));
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int c = 0; c < F::kBoxes; ++c) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float* a8 = acc + c * 64 + j * 8;
              __nv_bfloat162 b0 = __floats2bfloat162_rn(a8[0], a8[1]);
              __nv_bfloat162 b1 = __floats2bfloat162_rn(a8[2], a8[3]);
              __nv_bfloat162 b2 = __floats2bfloat162_rn(a8[4], a8[5]);
              __nv_bfloat162 b3 = __floats2bfloat162_rn(a8[6], a8[7]);
              // 128-byte swizzle: 16-byte chunk j of row `lane` sits at j ^ (lane & 7)
              st_shared_v4(stg + (uint32_t)(c * kYBoxBytes + lane * 128 + ((j ^ (lane & 7)) * 16)),
                           *reinterpret_cast<uint32_t*>(&b0), *reinterpret_cast<uint32_t*>(&b1),
                           *reinterpret_cast<uint32_t*>(&b2), *reinterpret_cast<uint32_t*>(&b3));
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int c = 0; c < F::kBoxes; ++c) {
              const int col0 = tl.n0 + h * kAcc + c * kYBoxCols;
              if (col0 < g.N) tma_store_2d(&tmY, stg + (uint32_t)(c * kYBoxBytes), col0, row0);
            }
            bulk_commit();
          }
        } else if (row_ok) {
          // ragged rows (the last m-tile, or an expert segment's end): plain stores
          __nv_bfloat16* yrow = g.y + (int64_t)row * g.ldy;
#pragma unroll
          for (int c = 0; c < kAcc / 8; ++c) {
            const int col = tl.n0 + h * kAcc + c * 8;
            if (col < g.N) {
              uint4 v;
              __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[c * 8 + 0], acc[c * 8 + 1]);
              __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[c * 8 + 2], acc[c * 8 + 3]);
              __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[c * 8 + 4], acc[c * 8 + 5]);
              __nv_bfloat162 b3 = __floats2bfloat162_rn(acc[c * 8 + 6], acc[c * 8 + 7]);
              v.x = *reinterpret_cast<uint32_t*>(&b0);
              v.y = *reinterpret_cast<uint32_t*>(&b1);
              v.z = *reinterpret_cast<uint32_t*>(&b2);
              v.w = *reinterpret_cast<uint32_t*>(&b3);
              *reinterpret_cast<uint4*>(yrow + col) = v;
            }
          }
        }
      }
    }
    if (F::kStaged && lane == 0) bulk_wait_all();   // this warp's tensor stores are complete
  }

  if (kSplit) {
    // Every thread passes both phases exactly once, whatever path it took
    // (all waits before them are bounded, so every thread gets here).
    cluster_arrive();   // (A) this thread's part of the partial is staged
    cluster_wait();
    const Tile tl = decode_tile<kGrouped, kBN>(cid, g, st);
    reduce_rows(smem_u32(red), (int)crank, nsplit, tl.m0, tl.row_end, tl.n0, g, tid);
    cluster_arrive();   // (B) this thread reads no peer's shared memory any more
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, F::kTmemCols);
  }
  if (kSplit) cluster_wait();   // (B): no peer still reads this CTA's shared memory
}

// ------------------------------------------------------------------- host --

// 2-D uint8 map over a row-major [rows, inner] matrix, box [box_rows, 128],
// 128-byte swizzle (the layout the UMMA descriptors describe).
// BF16 output map over row-major Y [rows, n] (row stride ldy elements), box
// 64 columns x 32 rows, 128-byte swizzle (the epilogue's staging layout).
fp8rl_status make_out_map(CUtensorMap* m, void* y, uint64_t n, uint64_t rows, uint64_t ldy) {
  return encode_tiled_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, y, n, rows, ldy * 2, kYBoxCols, kYBox,
                         CU_TENSOR_MAP_SWIZZLE_128B, "Y");
}

fp8rl_status make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                      uint32_t box_rows, const char* what) {
  return encode_tiled_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, inner, rows, inner, BK, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_128B, what);
}

template <bool kGrouped, int kF>
fp8rl_status set_smem_attr(const DeviceState* ds) {
  static bool done[64] = {false};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (ds->device < 64 && done[ds->device]) return FP8RL_OK;
  const size_t bytes = smem_bytes<kF>();
  if ((size_t)ds->max_smem_optin < bytes)
    return fail(FP8RL_ERR_UNSUPPORTED_DEVICE, "GEMM needs %zu bytes of shared memory per block",
                bytes);
  fp8rl_status st = cuda_check(
      cudaFuncSetAttribute(gemm_w8a8_kernel<kGrouped, kF>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes),
      "cudaFuncSetAttribute(gemm)");
  if (st == FP8RL_OK && ds->device < 64) done[ds->device] = true;
  return st;
}

// Clusters of `s` split-K CTAs that can be resident at once (0 if unknown).
int max_active_clusters(const DeviceState* ds, int s) {
  static int cache[64][kMaxSplit + 1] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  int* c = ds->device < 64 ? &cache[ds->device][s] : nullptr;
  if (c && *c) return *c;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)s, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes<kSplitK>();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)s;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_w8a8_kernel<false, kSplitK>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  if (c) *c = n > 0 ? n : -1;
  return n;
}

// Cluster size S of the split-K flavour for `tiles` 128-wide output tiles:
// the largest S <= 4 (and <= the k-blocks) for which one cluster of S CTAs
// per tile fits in one wave, else 1.  The flavour runs only when the 256-wide
// tiles fill at most half of the SMs, so `tiles` never exceeds the SM count
// and S = 1 always fits.
int choose_split(const DeviceState* ds, int64_t tiles, int kb) {
  int s = (int)std::min<int64_t>(kMaxSplit, ds->sm_count / std::max<int64_t>(tiles, 1));
  for (s = std::min(s, kb); s >= 2; --s)
    if (max_active_clusters(ds, s) >= tiles) return s;
  return 1;
}

// Launches the kernel with programmatic stream serialization allowed (its
// prologue may overlap the previous kernel; see grid_dependency_wait) and,
// for the split-K flavour, a cluster of `cluster` CTAs along x.
template <bool kGrouped, int kF>
fp8rl_status launch_gemm(int grid, int cluster, cudaStream_t stream, const CUtensorMap& tmA,
                         const CUtensorMap& tmB, const CUtensorMap& tmY, const GemmArgs& g,
                         const char* what) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes<kF>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (kF == kSplitK) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cuda_check(cudaLaunchKernelEx(&cfg, gemm_w8a8_kernel<kGrouped, kF>, tmA, tmB, tmY, g),
                    what);
}

fp8rl_status check_common(const uint8_t* qa, const float* sa, const uint8_t* qw, const float* sw,
                          int64_t n, int64_t k, const void* y) {
  if (!qa || !sa || !qw || !sw || !y) return fail(FP8RL_ERR_INVALID_ARG, "null pointer");
  if (k < 128 || k % 128)
    return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "k must be a positive multiple of 128 (k=%lld)",
                (long long)k);
  if (n < 16 || n % 16)
    return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "n must be a positive multiple of 16 (n=%lld)",
                (long long)n);
  if (k > INT32_MAX / 2 || n > INT32_MAX / 2)
    return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "n or k too large");
  if (!aligned(qa, 16) || !aligned(qw, 16) || !aligned(y, 16) || !aligned(sa, 4) ||
      !aligned(sw, 4))
    return fail(FP8RL_ERR_ALIGNMENT, "qa, qw and y must be 16-byte aligned");
  return FP8RL_OK;
}

}  // namespace
}  // namespace fp8rl

using namespace fp8rl;

extern "C" fp8rl_status fp8rl_gemm_w8a8_blockwise(const uint8_t* qa, const float* sa,
                                                  const uint8_t* qw, const float* sw, int64_t m,
                                                  int64_t n, int64_t k, void* y, int64_t ldy,
                                                  cudaStream_t stream) {
  fp8rl_status st = check_common(qa, sa, qw, sw, n, k, y);
  if (st != FP8RL_OK) return st;
  if (m < 0 || m > INT32_MAX - BM) return fail(FP8RL_ERR_INVALID_ARG, "m out of range");
  if (ldy < n || ldy % 8) return fail(FP8RL_ERR_ALIGNMENT, "need ldy >= n and ldy % 8 == 0");
  if (m == 0) return ok();
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != FP8RL_OK) return st;
  // Flavour by the number of 256-wide tiles: at least two waves of them, the
  // wide flavour (its tile reads the fewest operand bytes per FLOP, and
  // operand intake from L2 bounds these shapes); fewer, the narrow flavour
  // (twice the tiles to spread, four TMEM buffers); at most half of the SMs,
  // the split-K flavour.
  const int64_t num_m = (m + BM - 1) / BM;
  const int64_t wide_tiles = num_m * ((n + Flavour<kWide>::kBN - 1) / Flavour<kWide>::kBN);
  const bool split = wide_tiles * 2 <= ds->sm_count;
  const bool wide = !split && wide_tiles >= 2 * (int64_t)ds->sm_count;
  const int bn = wide ? Flavour<kWide>::kBN : Flavour<kNarrow>::kBN;
  CUtensorMap tmA, tmB;
  if ((st = make_map(&tmA, qa, (uint64_t)k, (uint64_t)m, BM, "A")) != FP8RL_OK) return st;
  if ((st = make_map(&tmB, qw, (uint64_t)k, (uint64_t)n, (uint32_t)bn, "W")) != FP8RL_OK) return st;
  CUtensorMap tmY;
  if ((st = make_out_map(&tmY, y, (uint64_t)n, (uint64_t)m, (uint64_t)ldy)) != FP8RL_OK) return st;
  GemmArgs g;
  g.sa = sa;
  g.sw = sw;
  g.y = reinterpret_cast<__nv_bfloat16*>(y);
  g.ldy = ldy;
  g.M = (int)m;
  g.N = (int)n;
  g.KB = (int)(k / BK);
  g.NB = (int)((n + 127) / 128);
  g.num_m = (int)num_m;
  g.num_n = (int)((n + bn - 1) / bn);
  g.offsets = nullptr;
  g.E = 1;
  g.status = ds->status;
  const int64_t tiles = (int64_t)g.num_m * g.num_n;
  if (tiles > INT32_MAX) return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "too many tiles");
  if (!split) {
    g.split = 1;
    const int grid = (int)std::min<int64_t>(tiles, ds->sm_count);
    if (wide) {
      if ((st = set_smem_attr<false, kWide>(ds)) != FP8RL_OK) return st;
      st = launch_gemm<false, kWide>(grid, 1, stream, tmA, tmB, tmY, g, "gemm_w8a8_kernel launch");
    } else {
      if ((st = set_smem_attr<false, kNarrow>(ds)) != FP8RL_OK) return st;
      st = launch_gemm<false, kNarrow>(grid, 1, stream, tmA, tmB, tmY, g, "gemm_w8a8_kernel launch");
    }
    return st == FP8RL_OK ? ok() : st;
  }
  // few tiles: exactly one cluster of g.split CTAs per tile (the kernel's
  // reduction reuses the stage buffers, so a cluster never takes a second
  // tile), split along K; a cluster of one when no larger one fits
  // (the occupancy query behind choose_split needs the split flavour's
  // shared-memory attribute set first)
  if ((st = set_smem_attr<false, kSplitK>(ds)) != FP8RL_OK) return st;
  g.split = choose_split(ds, tiles, g.KB);
  if (g.split == 1) {
    // no split fits: one CTA per tile, so the narrow flavour (direct output
    // staging, four TMEM buffers) does the same work without the partial's
    // round trip through shared memory
    g.split = 1;
    if ((st = set_smem_attr<false, kNarrow>(ds)) != FP8RL_OK) return st;
    st = launch_gemm<false, kNarrow>((int)tiles, 1, stream, tmA, tmB, tmY, g, "gemm_w8a8_kernel launch");
    return st == FP8RL_OK ? ok() : st;
  }
  const int clusters = (int)tiles;
  st = launch_gemm<false, kSplitK>(clusters * g.split, g.split, stream, tmA, tmB, tmY, g,
                                   "split-K gemm_w8a8_kernel launch");
  return st == FP8RL_OK ? ok() : st;
}

extern "C" fp8rl_status fp8rl_grouped_gemm_w8a8_blockwise(const uint8_t* qa, const float* sa,
                                                          const uint8_t* qw, const float* sw,
                                                          const int32_t* offsets,
                                                          int32_t num_experts, int64_t m_total,
                                                          int64_t n, int64_t k, void* y,
                                                          cudaStream_t stream) {
  fp8rl_status st = check_common(qa, sa, qw, sw, n, k, y);
  if (st != FP8RL_OK) return st;
  if (!offsets) return fail(FP8RL_ERR_INVALID_ARG, "null offsets");
  if (!aligned(offsets, 4)) return fail(FP8RL_ERR_ALIGNMENT, "offsets must be 4-byte aligned");
  if (num_experts < 1 || num_experts > kMaxExperts)
    return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "need 1 <= num_experts <= %d", kMaxExperts);
  if (n % 128) return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "grouped GEMM needs n % 128 == 0");
  if (m_total < 0 || m_total > INT32_MAX - BM) return fail(FP8RL_ERR_INVALID_ARG, "m_total out of range");
  if ((int64_t)num_experts * n > INT32_MAX) return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "e*n too large");
  if (m_total == 0) return ok();
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != FP8RL_OK) return st;
  if ((st = set_smem_attr<true, kWide>(ds)) != FP8RL_OK) return st;
  CUtensorMap tmA, tmB;
  if ((st = make_map(&tmA, qa, (uint64_t)k, (uint64_t)m_total, BM, "A")) != FP8RL_OK) return st;
  if ((st = make_map(&tmB, qw, (uint64_t)k, (uint64_t)num_experts * n, Flavour<kWide>::kBN, "W")) !=
      FP8RL_OK)
    return st;
  CUtensorMap tmY;
  if ((st = make_out_map(&tmY, y, (uint64_t)n, (uint64_t)m_total, (uint64_t)n)) != FP8RL_OK)
    return st;
  GemmArgs g;
  g.sa = sa;
  g.sw = sw;
  g.y = reinterpret_cast<__nv_bfloat16*>(y);
  g.ldy = n;
  g.M = (int)m_total;
  g.N = (int)n;
  g.KB = (int)(k / BK);
  g.NB = (int)(n / 128);
  g.num_m = 0;
  g.num_n = (int)((n + Flavour<kWide>::kBN - 1) / Flavour<kWide>::kBN);
  g.offsets = offsets;
  g.E = num_experts;
  g.status = ds->status;
  const int64_t bound = ((m_total + BM - 1) / BM + num_experts) * (int64_t)g.num_n;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(bound, ds->sm_count));
  g.split = 1;
  st = launch_gemm<true, kWide>(grid, 1, stream, tmA, tmB, tmY, g, "grouped gemm_w8a8_kernel launch");
  return st == FP8RL_OK ? ok() : st;
}
