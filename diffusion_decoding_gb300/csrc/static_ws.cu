// dllm_commit_threshold_static: the fused statistics + threshold-commit call for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point where they decode:
// a serving runtime that reserves all device memory up front in its own pool and forbids
// allocation while requests are in flight, a plugin whose host framework owns every device
// buffer, or code that must not take the device-wide synchronisation an allocation may imply.
// For them this entry point takes no workspace argument: its scratch (status word, slice
// partials) lives in one fixed-size array in device global memory that
// is part of the library image, so every GPU that loads the library holds it until the process
// exits.
//
// The array's host-side name is only a stand-in for the symbol; a kernel given that name would
// fault (or, on systems where the GPU can reach host memory, silently use the wrong memory).  The
// device address is therefore looked up with cudaGetSymbolAddress, once per device, with that
// device current, on the first call made on it.
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "internal.h"

namespace {

// 4 MiB: room for ~262,000 slice records of 16 bytes, B*L*ceil(V/1024) of them (for example
// B*L = 1024 rows at V up to ~262,000, or B*L = 2048 rows at V = 126464).
constexpr size_t kStaticWsBytes = DLLM_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

std::mutex g_setup_mutex;
void* g_static_ws_ptr[kMaxDevices] = {};

dllm_status fail(dllm_status s, const char* msg, cudaError_t e = cudaSuccess) {
  dllm::set_last_error(msg, e);
  return s;
}

// Device address of g_static_ws on the current device (looked up once per device).
dllm_status static_ws_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DLLM_ERR_CUDA, "cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return fail(DLLM_ERR_UNSUPPORTED, "device index too large");
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_static_ws_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess || !p)
      return fail(DLLM_ERR_CUDA, "cudaGetSymbolAddress(static workspace)", e);
    g_static_ws_ptr[dev] = p;
  }
  *out = g_static_ws_ptr[dev];
  return DLLM_OK;
}

// The call itself (wrapped below in an NVTX range named after the entry point).
dllm_status commit_static(const void* logits, const dllm_shape* shape, const dllm_stats* stats,
                          const dllm_block_state* state, float tau, int32_t eos_id,
                          dllm_stream_t stream) {
  const size_t need = dllm_workspace_bytes(shape);  // 0 when the shape is invalid
  if (need == 0) return fail(DLLM_ERR_INVALID_ARG, "invalid shape");
  if (need > kStaticWsBytes)
    return fail(DLLM_ERR_UNSUPPORTED,
                "shape needs more scratch than the 4 MiB static workspace holds; use "
                "dllm_commit_threshold with a caller-allocated workspace");
  if (!logits) return fail(DLLM_ERR_INVALID_ARG, "logits is null (the static variant always "
                                                 "computes the statistics itself)");
  void* ws = nullptr;
  dllm_status st = static_ws_address(&ws);
  if (st != DLLM_OK) return st;
  // The status word must start at zero: clear the header (no allocation).  The partials need no
  // clearing: every partial read is written by the call.
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, dllm::kWsHeader, s);
  if (e != cudaSuccess) return fail(DLLM_ERR_CUDA, "clearing the static workspace", e);
  return dllm_commit_threshold(logits, shape, stats, state, tau, eos_id, ws, stream);
}

}  // namespace

extern "C" {

dllm_status dllm_commit_threshold_static(const void* logits, const dllm_shape* shape,
                                         const dllm_stats* stats, const dllm_block_state* state,
                                         float tau, int32_t eos_id, dllm_stream_t stream) {
  nvtxRangePushA("dllm_commit_threshold_static");
  const dllm_status st = commit_static(logits, shape, stats, state, tau, eos_id, stream);
  nvtxRangePop();
  return st;
}

}  // extern "C"
