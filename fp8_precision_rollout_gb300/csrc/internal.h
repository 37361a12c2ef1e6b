// internal.h -- host-side plumbing shared by the fp8rl translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp8rl.h"

namespace fp8rl {

// Records a message for fp8rl_last_error() and returns `st`.
fp8rl_status fail(fp8rl_status st, const char* fmt, ...);
// Clears the thread's last error and returns FP8RL_OK.
fp8rl_status ok();
// Maps a CUDA error to FP8RL_ERR_CUDA with context; FP8RL_OK for cudaSuccess.
fp8rl_status cuda_check(cudaError_t e, const char* what);

// Per-device state, created on first use (current device).
struct DeviceState {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  int max_smem_optin = 0;
  // library workspace (device memory, zero-initialised at creation)
  uint32_t* status = nullptr;      // [0]: timeout flags, [1]: where the wait gave up
  uint32_t* kv_amax = nullptr;     // 256 calibration slots (float bits)
};

// Looks up (creating if needed) the state of the current device and checks
// that it is an sm_103 part.  On failure returns a status (message set).
fp8rl_status device_state(DeviceState** out);

// Builds the per-device lookup tables of the MoE glue (quant.cu); called once
// per device when its state is created, synchronously.
fp8rl_status init_glue_tables();

// Device status word bits.
enum : uint32_t {
  kStatusTimeout = 1u << 0,   // a pipelined kernel gave up on an mbarrier wait
  kStatusBadIndex = 1u << 1,  // a device-side index was out of range (ignored)
};

// Encodes a 2-D tiled TMA descriptor over a row-major [rows, inner] matrix of
// `dtype` elements with row pitch `row_bytes`; box [box_rows, box_inner].
fp8rl_status encode_tiled_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                             uint64_t inner, uint64_t rows, uint64_t row_bytes,
                             uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle,
                             const char* what);

inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// CTAs of `kernel` (launched with `threads` threads, no dynamic shared
// memory) that fit on one SM at once; streaming kernels size their grid to
// exactly one resident wave (SMs x this) and loop over the remaining work.
template <class K>
int resident_ctas_per_sm(K kernel, int threads) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1)
    n = 1;
  return n;
}

}  // namespace fp8rl
