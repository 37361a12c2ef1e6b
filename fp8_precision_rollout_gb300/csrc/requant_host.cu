// requant_host.cu -- per-step weight re-quantization straight from and to
// host memory, copies overlapped with the quantization.
//
// FP8-RL summary, section 3.4.2, Phase 2: after every policy update the BF16
// weights are taken from the training side, quantized blockwise to E4M3 and
// loaded into the inference engine; the step is repeated thousands of times,
// so its latency matters.  When the BF16 weights and the FP8 destination live
// in host memory, the re-quantization is bound by the host link, not by the
// kernel; this runtime streams the tensors through a caller-provided device
// workspace split in two slots, so that the host-to-device copy of chunk c+1,
// the quantization of chunk c and the device-to-host copy of chunk c-1 run at
// the same time on internal streams ordered by events (one host-to-device
// and one device-to-host stream per slot, one compute stream).  Tensors larger
// than a slot are split at 128-row boundaries (whole blocks, so the pieces
// quantize independently); the kernel is the multi-tensor re-quantization.
#include <algorithm>
#include <mutex>
#include <vector>

#include "internal.h"

namespace fp8rl {
namespace {

struct HostPipe {
  bool ready = false;
  cudaStream_t h2d[2] = {nullptr, nullptr}, comp = nullptr, d2h[2] = {nullptr, nullptr};
  cudaEvent_t start = nullptr, end[2] = {nullptr, nullptr};
  cudaEvent_t h2d_done[2] = {nullptr, nullptr}, comp_done[2] = {nullptr, nullptr};
  cudaEvent_t slot_free[2] = {nullptr, nullptr};
  std::mutex mu;
};

HostPipe& host_pipe(int device) {
  static HostPipe pipes[64];
  return pipes[device & 63];
}

fp8rl_status pipe_init(HostPipe& hp) {
  if (hp.ready) return FP8RL_OK;
  fp8rl_status st = FP8RL_OK;
  auto stream = [&](cudaStream_t* s) {
    if (st == FP8RL_OK)
      st = cuda_check(cudaStreamCreateWithFlags(s, cudaStreamNonBlocking), "cudaStreamCreate");
  };
  auto event = [&](cudaEvent_t* e) {
    if (st == FP8RL_OK)
      st = cuda_check(cudaEventCreateWithFlags(e, cudaEventDisableTiming), "cudaEventCreate");
  };
  stream(&hp.comp);
  event(&hp.start);
  for (int i = 0; i < 2; ++i) {
    stream(&hp.h2d[i]);
    stream(&hp.d2h[i]);
    event(&hp.end[i]);
    event(&hp.h2d_done[i]);
    event(&hp.comp_done[i]);
    event(&hp.slot_free[i]);
  }
  if (st == FP8RL_OK) hp.ready = true;
  return st;
}

// One piece of a chunk: rows [r0, r1) of host tensor t, placed in a slot.
struct Piece {
  int t;
  int64_t r0, r1;
  size_t in_off, q_off, s_off;   // offsets inside the slot
};

constexpr size_t kAlign = 256;
inline size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

inline size_t piece_bytes(int64_t rows, int64_t k) {
  const int64_t kb = (k + 127) / 128, nb = (rows + 127) / 128;
  return round_up((size_t)rows * k * 2) + round_up((size_t)rows * k) + round_up((size_t)nb * kb * 4);
}

// 2-D copy (rows of `width` bytes) or a flat one when both pitches equal it.
cudaError_t copy_rows(void* dst, size_t dpitch, const void* src, size_t spitch, size_t width,
                      size_t rows, cudaMemcpyKind kind, cudaStream_t s) {
  if (dpitch == width && spitch == width)
    return cudaMemcpyAsync(dst, src, width * rows, kind, s);
  return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, s);
}

}  // namespace
}  // namespace fp8rl

using namespace fp8rl;

extern "C" fp8rl_status fp8rl_quantize_weights_blockwise_multi_host(const fp8rl_wdesc* descs,
                                                                    int32_t count, void* workspace,
                                                                    size_t workspace_bytes,
                                                                    cudaStream_t stream) {
  if (count < 0 || (count > 0 && !descs))
    return fail(FP8RL_ERR_INVALID_ARG, "descs must be a host array of count >= 0 descriptors");
  for (int i = 0; i < count; ++i) {
    const fp8rl_wdesc& d = descs[i];
    if (!d.w || !d.q || !d.scales)
      return fail(FP8RL_ERR_INVALID_ARG, "weight tensor %d: null pointer", i);
    if (d.n < 1 || d.k < 1 || d.ldw < d.k || d.ldq < d.k)
      return fail(FP8RL_ERR_INVALID_ARG, "weight tensor %d: need n, k >= 1, ldw >= k, ldq >= k", i);
    if (d.k % 8) return fail(FP8RL_ERR_ALIGNMENT, "weight tensor %d: k must be a multiple of 8", i);
    if (d.n > INT32_MAX / 2 || d.k > INT32_MAX / 2)
      return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "weight tensor %d: dimension too large", i);
  }
  if (count == 0) return ok();
  if (!workspace || !aligned(workspace, kAlign))
    return fail(FP8RL_ERR_ALIGNMENT, "workspace must be a 256-byte aligned device buffer");
  const size_t slot = workspace_bytes / 2 / kAlign * kAlign;
  for (int i = 0; i < count; ++i)
    if (piece_bytes(std::min<int64_t>(128, descs[i].n), descs[i].k) > slot)
      return fail(FP8RL_ERR_UNSUPPORTED_SHAPE,
                  "workspace too small: each half must hold 128 rows of tensor %d (%zu bytes)", i,
                  piece_bytes(std::min<int64_t>(128, descs[i].n), descs[i].k));
  DeviceState* ds = nullptr;
  fp8rl_status st = device_state(&ds);
  if (st != FP8RL_OK) return st;
  HostPipe& hp = host_pipe(ds->device);
  std::lock_guard<std::mutex> lock(hp.mu);
  if ((st = pipe_init(hp)) != FP8RL_OK) return st;

  // cut the tensors into chunks that fit one slot
  std::vector<std::vector<Piece>> chunks(1);
  size_t used = 0;
  for (int t = 0; t < count; ++t) {
    const fp8rl_wdesc& d = descs[t];
    int64_t r0 = 0;
    while (r0 < d.n) {
      int64_t rows = d.n - r0;
      if (used + piece_bytes(rows, d.k) > slot) {
        // the largest multiple of 128 rows that fits the rest of the slot
        int64_t lo = 0, hi = rows / 128;
        while (lo < hi) {
          const int64_t mid = (lo + hi + 1) / 2;
          if (used + piece_bytes(mid * 128, d.k) <= slot) lo = mid; else hi = mid - 1;
        }
        rows = lo * 128;
      }
      if (rows == 0) {
        // an empty slot holds 128 rows of every tensor (checked above)
        if (used == 0) return fail(FP8RL_ERR_UNSUPPORTED_SHAPE, "workspace too small");
        chunks.emplace_back();   // no room left in this slot: start a new chunk
        used = 0;
        continue;
      }
      const int64_t kb = (d.k + 127) / 128, nb = (rows + 127) / 128;
      Piece pc;
      pc.t = t;
      pc.r0 = r0;
      pc.r1 = r0 + rows;
      pc.in_off = used;
      pc.q_off = pc.in_off + round_up((size_t)rows * d.k * 2);
      pc.s_off = pc.q_off + round_up((size_t)rows * d.k);
      used = pc.s_off + round_up((size_t)nb * kb * 4);
      chunks.back().push_back(pc);
      r0 += rows;
    }
  }
  if (chunks.back().empty()) chunks.pop_back();

  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  auto cu = [&](cudaError_t e, const char* what) {
    if (st == FP8RL_OK) st = cuda_check(e, what);
  };
  cu(cudaEventRecord(hp.start, stream), "cudaEventRecord");
  for (int i = 0; i < 2; ++i) cu(cudaStreamWaitEvent(hp.h2d[i], hp.start, 0), "cudaStreamWaitEvent");
  std::vector<fp8rl_wdesc> dev;
  for (size_t c = 0; c < chunks.size() && st == FP8RL_OK; ++c) {
    const int sl = (int)(c & 1);
    uint8_t* base = ws + sl * slot;
    // each slot has its own copy streams, so consecutive chunks can use
    // different copy engines
    if (c >= 2) cu(cudaStreamWaitEvent(hp.h2d[sl], hp.slot_free[sl], 0), "cudaStreamWaitEvent");
    dev.clear();
    for (const Piece& pc : chunks[c]) {
      const fp8rl_wdesc& d = descs[pc.t];
      const int64_t rows = pc.r1 - pc.r0;
      cu(copy_rows(base + pc.in_off, (size_t)d.k * 2,
                   reinterpret_cast<const uint8_t*>(d.w) + (size_t)pc.r0 * d.ldw * 2,
                   (size_t)d.ldw * 2, (size_t)d.k * 2, (size_t)rows, cudaMemcpyHostToDevice,
                   hp.h2d[sl]),
         "host-to-device copy");
      fp8rl_wdesc w;
      w.w = base + pc.in_off;
      w.q = base + pc.q_off;
      w.scales = reinterpret_cast<float*>(base + pc.s_off);
      w.n = rows;
      w.k = d.k;
      w.ldw = d.k;
      w.ldq = d.k;
      dev.push_back(w);
    }
    cu(cudaEventRecord(hp.h2d_done[sl], hp.h2d[sl]), "cudaEventRecord");
    cu(cudaStreamWaitEvent(hp.comp, hp.h2d_done[sl], 0), "cudaStreamWaitEvent");
    if (st == FP8RL_OK) st = fp8rl_quantize_weights_blockwise_multi(dev.data(), (int32_t)dev.size(), hp.comp);
    cu(cudaEventRecord(hp.comp_done[sl], hp.comp), "cudaEventRecord");
    cu(cudaStreamWaitEvent(hp.d2h[sl], hp.comp_done[sl], 0), "cudaStreamWaitEvent");
    for (const Piece& pc : chunks[c]) {
      const fp8rl_wdesc& d = descs[pc.t];
      const int64_t rows = pc.r1 - pc.r0, kb = (d.k + 127) / 128;
      cu(copy_rows(d.q + (size_t)pc.r0 * d.ldq, (size_t)d.ldq, base + pc.q_off, (size_t)d.k,
                   (size_t)d.k, (size_t)rows, cudaMemcpyDeviceToHost, hp.d2h[sl]),
         "device-to-host copy (codes)");
      cu(cudaMemcpyAsync(d.scales + (size_t)(pc.r0 / 128) * kb, base + pc.s_off,
                         (size_t)((rows + 127) / 128) * kb * 4, cudaMemcpyDeviceToHost, hp.d2h[sl]),
         "device-to-host copy (scales)");
    }
    cu(cudaEventRecord(hp.slot_free[sl], hp.d2h[sl]), "cudaEventRecord");
  }
  for (int i = 0; i < 2; ++i) {
    cu(cudaEventRecord(hp.end[i], hp.d2h[i]), "cudaEventRecord");
    cu(cudaStreamWaitEvent(stream, hp.end[i], 0), "cudaStreamWaitEvent");
  }
  return st == FP8RL_OK ? ok() : st;
}
