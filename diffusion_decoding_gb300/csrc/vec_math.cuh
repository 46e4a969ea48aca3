// Packed arithmetic on 16-byte vectors of logits, shared by the statistics kernels (sm_103a):
// bf16 pairs compared with max.bf16x2, fp32 pairs multiplied and added with the f32x2 pipes.
#pragma once

#include "common.cuh"

namespace dllm {

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Largest element of one 16-byte vector (8 bf16 or 4 fp32).
template <int DT>
__device__ __forceinline__ float vec_max(const uint4& q) {
  if constexpr (DT == DLLM_BF16) {
    const uint32_t m = bf16x2_max(bf16x2_max(q.x, q.y), bf16x2_max(q.z, q.w));
    return fmaxf(bf16lo(m), bf16hi(m));
  } else {
    return fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)),
                 fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
  }
}

// The elements of one 16-byte vector as fp32, in memory order (8 for bf16, 4 for fp32).
template <int DT>
__device__ __forceinline__ void unpack_vec(const uint4& q, float* x) {
  if constexpr (DT == DLLM_BF16) {
    x[0] = bf16lo(q.x); x[1] = bf16hi(q.x); x[2] = bf16lo(q.y); x[3] = bf16hi(q.y);
    x[4] = bf16lo(q.z); x[5] = bf16hi(q.z); x[6] = bf16lo(q.w); x[7] = bf16hi(q.w);
  } else {
    x[0] = __uint_as_float(q.x); x[1] = __uint_as_float(q.y);
    x[2] = __uint_as_float(q.z); x[3] = __uint_as_float(q.w);
  }
}

// fp32 pairs in one 64-bit register pair, for fma.rn.f32x2 / add.rn.f32x2
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

}  // namespace dllm
