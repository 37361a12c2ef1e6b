// runtime.cu -- error reporting, per-device state and workspace, status word.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <algorithm>
#include <cstdio>
#include <mutex>
#include <string>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace fp8rl {

namespace {
thread_local std::string g_last_error;
std::mutex g_mu;
constexpr int kMaxDevices = 64;
DeviceState g_states[kMaxDevices];
constexpr size_t kWorkspaceBytes = 4096;
}  // namespace

fp8rl_status fail(fp8rl_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

fp8rl_status ok() {
  g_last_error.clear();
  return FP8RL_OK;
}

fp8rl_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return FP8RL_OK;
  return fail(FP8RL_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

fp8rl_status device_state(DeviceState** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_check(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(FP8RL_ERR_UNSUPPORTED_DEVICE, "device %d", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_states[dev];
  if (st.device < 0) {
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return cuda_check(e, "cudaGetDeviceProperties");
    if (!(prop.major == 10 && prop.minor == 3))
      return fail(FP8RL_ERR_UNSUPPORTED_DEVICE,
                  "fp8rl is built for sm_103a (GB300); device %d is sm_%d%d (%s)", dev,
                  prop.major, prop.minor, prop.name);
    void* ws = nullptr;
    e = cudaMalloc(&ws, kWorkspaceBytes);
    if (e != cudaSuccess) return cuda_check(e, "cudaMalloc(workspace)");
    e = cudaMemset(ws, 0, kWorkspaceBytes);
    if (e != cudaSuccess) return cuda_check(e, "cudaMemset(workspace)");
    const fp8rl_status ts = init_glue_tables();
    if (ts != FP8RL_OK) {
      cudaFree(ws);
      return ts;
    }
    st.sm_count = prop.multiProcessorCount;
    st.cc_major = prop.major;
    st.cc_minor = prop.minor;
    st.max_smem_optin = (int)prop.sharedMemPerBlockOptin;
    st.status = reinterpret_cast<uint32_t*>(ws);
    st.kv_amax = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + 1024);
    st.device = dev;
  }
  *out = &st;
  return FP8RL_OK;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}
}  // namespace

fp8rl_status encode_tiled_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                             uint64_t inner, uint64_t rows, uint64_t row_bytes,
                             uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle,
                             const char* what) {
  auto fn = encode_fn();
  if (!fn) return fail(FP8RL_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(FP8RL_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", what, (int)r);
  return FP8RL_OK;
}

}  // namespace fp8rl

using namespace fp8rl;

extern "C" int32_t fp8rl_version(void) { return FP8RL_VERSION; }

extern "C" const char* fp8rl_last_error(void) { return g_last_error.c_str(); }

extern "C" fp8rl_status fp8rl_device_status(int32_t device, int32_t clear) {
  int prev = -1;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return cuda_check(e, "cudaGetDevice");
  if (device != prev) {
    e = cudaSetDevice(device);
    if (e != cudaSuccess) return cuda_check(e, "cudaSetDevice");
  }
  DeviceState* ds = nullptr;
  fp8rl_status st = device_state(&ds);
  uint32_t words[2] = {0, 0};
  if (st == FP8RL_OK) {
    e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(words, ds->status, sizeof(words), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && clear) e = cudaMemset(ds->status, 0, sizeof(words));
    st = cuda_check(e, "reading the device status word");
  }
  if (device != prev) cudaSetDevice(prev);
  if (st != FP8RL_OK) return st;
  if (words[0] & kStatusTimeout)
    return fail(FP8RL_ERR_TIMEOUT, "a kernel pipeline wait hit its time limit (site %u)", words[1]);
  if (words[0] & kStatusBadIndex)
    return fail(FP8RL_ERR_INVALID_ARG, "a device-side row index was out of range (row left zero)");
  return ok();
}

// ---------------------------------------------------------- error-path tests --

extern "C" fp8rl_status fp8rl_inject_device_status(int32_t device, uint32_t flags, uint32_t site) {
  if (flags & ~(uint32_t)(kStatusTimeout | kStatusBadIndex))
    return fail(FP8RL_ERR_INVALID_ARG, "unknown status flags 0x%x", flags);
  int prev = -1;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return cuda_check(e, "cudaGetDevice");
  if (device != prev) {
    e = cudaSetDevice(device);
    if (e != cudaSuccess) return cuda_check(e, "cudaSetDevice");
  }
  DeviceState* ds = nullptr;
  fp8rl_status st = device_state(&ds);
  if (st == FP8RL_OK) {
    const uint32_t words[2] = {flags, site};
    st = cuda_check(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
    if (st == FP8RL_OK)
      st = cuda_check(cudaMemcpy(ds->status, words, sizeof(words), cudaMemcpyHostToDevice),
                      "writing the device status word");
  }
  if (device != prev) cudaSetDevice(prev);
  return st == FP8RL_OK ? ok() : st;
}

namespace fp8rl {
namespace {
constexpr uint32_t kSelfTestSite = 90;

// One CTA of one warp: lane 0 waits on an mbarrier that nothing arrives on,
// through the pipelines' bounded wait with a short limit.  The wait gives up,
// records the timeout and the site in the status word, and the kernel returns
// normally; the context stays usable.
__global__ void bounded_wait_selftest_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    ptx::mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    (void)ptx::mbar_wait(ptx::smem_u32(&bar), 0u, &abort_flag, status, kSelfTestSite, limit_ns);
  __syncthreads();
}
}  // namespace
}  // namespace fp8rl

extern "C" fp8rl_status fp8rl_selftest_bounded_wait(int32_t limit_us, cudaStream_t stream) {
  if (limit_us < 1 || limit_us > 1000000)
    return fail(FP8RL_ERR_INVALID_ARG, "limit_us must be in [1, 1000000] (got %d)", limit_us);
  DeviceState* ds = nullptr;
  fp8rl_status st = device_state(&ds);
  if (st != FP8RL_OK) return st;
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(ds->status, (uint64_t)limit_us * 1000ull);
  st = cuda_check(cudaGetLastError(), "bounded_wait_selftest_kernel launch");
  return st == FP8RL_OK ? ok() : st;
}

// ------------------------------------------------ sharded weight sync plan --

extern "C" fp8rl_status fp8rl_weight_shard_rows(int64_t n, int32_t world, int32_t rank,
                                                int64_t* row_begin, int64_t* row_end) {
  if (!row_begin || !row_end) return fail(FP8RL_ERR_INVALID_ARG, "null pointer");
  if (n < 0 || world < 1 || rank < 0 || rank >= world)
    return fail(FP8RL_ERR_INVALID_ARG, "need n >= 0, world >= 1 and 0 <= rank < world");
  const int64_t blocks = (n + 127) / 128;
  const int64_t b0 = blocks * rank / world, b1 = blocks * (rank + 1) / world;
  *row_begin = std::min<int64_t>(b0 * 128, n);
  *row_end = std::min<int64_t>(b1 * 128, n);
  return ok();
}
