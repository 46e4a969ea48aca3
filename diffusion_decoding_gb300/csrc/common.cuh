// Device helpers shared by the decode-step kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dllm.h"

namespace dllm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned kFull = 0xffffffffu;

// Workspace header: the status word sits in the first 4 bytes of every workspace.
constexpr size_t kWsHeader = 256;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// 2^x on the special-function unit (one MUFU op; flushes subnormal results to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16-byte streaming load that bypasses L1 (every logit is read once per kernel).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float load_logit(const void* row, int dtype, int64_t v) {
  if (dtype == DLLM_F32) return static_cast<const float*>(row)[v];
  uint32_t h = static_cast<const uint16_t*>(row)[v];
  return __uint_as_float(h << 16);
}

// Running (max, rescaled sum, argmax) of one row slice.
struct RowAcc {
  float m;   // running maximum (-inf before any element)
  float s;   // sum of exp(z - m)
  int idx;   // lowest index attaining m (-1 before any element)
};

__device__ __forceinline__ RowAcc row_acc_empty() { return RowAcc{-INFINITY, 0.f, -1}; }

// Merge two partial accumulators: max, sum rescaled to the common max, lowest index on ties.
__device__ __forceinline__ RowAcc row_acc_merge(RowAcc a, RowAcc b) {
  bool b_wins = (b.m > a.m) || (b.m == a.m && b.idx >= 0 && (a.idx < 0 || b.idx < a.idx));
  if (b_wins) {
    RowAcc t = a;
    a = b;
    b = t;
  }
  // now a.m >= b.m
  float add = (b.m == -INFINITY) ? b.s : b.s * ex2((b.m - a.m) * kLog2e);
  return RowAcc{a.m, a.s + add, a.idx};
}

__device__ __forceinline__ RowAcc row_acc_shfl_xor(RowAcc a, int mask) {
  RowAcc o;
  o.m = __shfl_xor_sync(kFull, a.m, mask);
  o.s = __shfl_xor_sync(kFull, a.s, mask);
  o.idx = __shfl_xor_sync(kFull, a.idx, mask);
  return o;
}

__device__ __forceinline__ RowAcc row_acc_warp_reduce(RowAcc a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = row_acc_merge(a, row_acc_shfl_xor(a, o));
  return a;
}

// Record the first device-side fault in the workspace status word.
__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, DLLM_OK, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch.  A kernel launched with launch_dependent() may start while the
// previous kernel on its stream is still draining; it must execute pdl_wait() before it reads
// anything that kernel wrote (pdl_wait returns at once for a kernel launched plainly).  A kernel
// calls pdl_trigger() once its dependents may be scheduled (without it they start when it ends).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace dllm
