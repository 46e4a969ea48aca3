// Single-read iteration smoothing: the statistics of the rows a step reads and their bf16
// probability rows P, from one read of the logits (dInfer explainer, diffusion-iteration
// manager: iteration smoothing feeds the undecided positions' whole distributions forward).
//
// P[j, v] = bf16(exp(z_{r_j, v} - lse_{r_j})) needs the row's log-sum-exp before the first
// probability can be written, so a row is held on chip while its statistics complete: a cluster
// of C CTAs shares one row, each CTA bringing its 64-element-aligned slice into shared memory
// with one bulk copy.  Each CTA reduces its slice to (max, sum of exp(z - max), lowest index of
// max); the C partials are exchanged through distributed shared memory and merged in rank order
// by every CTA (so all of them hold the same lse, bit for bit); rank 0 writes the row's
// statistics and every CTA writes its slice of P, K-slab-blocked, straight from shared memory.
// The logits cross HBM once instead of twice (statistics, then probabilities).
//
// P row j belongs to the j-th row read (the compaction of the block state taken before the
// commit); the GEMM maps P rows to the rows kept after the commit.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "mbarrier.cuh"

namespace dllm {
namespace {

constexpr int kSPThreads = 256;
constexpr int kSPWarps = kSPThreads / 32;
constexpr int kSPTargetBytes = 32768;       // slice of one CTA, aimed at
constexpr int kSPMaxSliceBytes = 192 * 1024;
constexpr int kCopyPiece = 16384;

struct SPParams {
  const char* logits;
  int64_t row_stride_bytes;
  int V;
  int C;               // CTAs per row (the cluster size)
  int slabs_per_cta;   // 64-element slabs per CTA
  const int32_t* rows;   // rows to read, ascending
  const int32_t* count;  // device: how many
  dllm_stats stats;
  uint16_t* P;           // K-slab-blocked [ceil(V/64)][R_pad][64]
  int R_pad;
  int32_t* status;
};

template <int DT>
struct Elem;
template <>
struct Elem<DLLM_BF16> {
  static constexpr int ES = 2, VEC = 8;
};
template <>
struct Elem<DLLM_F32> {
  static constexpr int ES = 4, VEC = 4;
};

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

template <int DT>
__device__ __forceinline__ float elem_at(uint32_t base, int k) {
  if constexpr (DT == DLLM_BF16) {
    uint16_t h;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(base + k * 2));
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  } else {
    float f;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(f) : "r"(base + k * 4));
    return f;
  }
}

__device__ __forceinline__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < kSPWarps; ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  return m;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kSPWarps; ++w) s += red[w];
  __syncthreads();
  return s;
}

__device__ __forceinline__ int block_min_int(int v, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(kFull, v, o));
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int m = red[0];
#pragma unroll
  for (int w = 1; w < kSPWarps; ++w) m = min(m, red[w]);
  __syncthreads();
  return m;
}

template <int DT>
__global__ void __launch_bounds__(kSPThreads, 4) stats_probs_kernel(const __grid_constant__ SPParams p) {
  using T = Elem<DT>;
  extern __shared__ __align__(128) uint8_t slice[];
  __shared__ uint64_t bar;
  __shared__ float redf[kSPWarps];
  __shared__ int redi[kSPWarps];
  __shared__ float part_m, part_s;
  __shared__ int part_i;
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const uint32_t rank = p.C > 1 ? cluster_ctarank() : 0u;
  const int c = static_cast<int>(blockIdx.x) / p.C;  // the same for every CTA of a cluster
  if (c >= *reinterpret_cast<const volatile int32_t*>(p.count)) return;  // whole cluster leaves
  const int r = p.rows[c];
  const int e0 = static_cast<int>(rank) * p.slabs_per_cta * 64;
  const int n = max(0, min(p.V, e0 + p.slabs_per_cta * 64) - e0);  // elements of this slice
  const uint32_t sbase = smem_u32(slice);

  // ---- the slice, by bulk copy (rounded up to 16 bytes: stays inside the row's stride)
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t bytes = static_cast<uint32_t>(align_up(static_cast<size_t>(n) * T::ES, 16));
  if (tid == 0) {
    mbar_expect_tx(smem_u32(&bar), bytes);
    const char* src = p.logits + static_cast<int64_t>(r) * p.row_stride_bytes +
                      static_cast<int64_t>(e0) * T::ES;
    for (uint32_t off = 0; off < bytes; off += kCopyPiece)
      bulk_g2s(sbase + off, src + off, min(static_cast<uint32_t>(kCopyPiece), bytes - off),
               smem_u32(&bar));
  }
  const bool ok = wait_bar(smem_u32(&bar), 0, &abort_flag, p.status);
  // (a failed wait still walks every barrier below, so the cluster never waits for this CTA)

  // ---- pass 1: slice maximum and the first vector holding it, per thread, then per CTA
  const int nvec = n * T::ES / 16;
  const int ntail = n - nvec * T::VEC;
  float tm = -INFINITY;
  int bu = -1;
  if (ok) {
    for (int v = tid; v < nvec; v += kSPThreads) {
      float x[T::VEC];
      unpack_vec<DT>(ld_shared_v4(sbase + v * 16), x);
      float vm = x[0];
#pragma unroll
      for (int k = 1; k < T::VEC; ++k) vm = fmaxf(vm, x[k]);
      if (vm > tm) {
        tm = vm;
        bu = v;
      }
    }
    if (tid < ntail) {
      const float x = elem_at<DT>(sbase, nvec * T::VEC + tid);
      if (x > tm) {
        tm = x;
        bu = nvec + tid;  // a tail element (index past the vectors)
      }
    }
  }
  const float mc = block_max(tm, redf);
  int idx = INT_MAX;
  if (ok && tm == mc && mc != -INFINITY) {
    if (bu >= nvec) {
      idx = nvec * T::VEC + (bu - nvec);
    } else {
      float x[T::VEC];
      unpack_vec<DT>(ld_shared_v4(sbase + bu * 16), x);
      for (int k = T::VEC - 1; k >= 0; --k)
        if (x[k] == mc) idx = bu * T::VEC + k;
    }
  }
  idx = block_min_int(idx, redi);

  // ---- pass 2: sum of exp(z - mc) over the slice
  float sum = 0.f;
  if (ok && mc != -INFINITY) {
    const float mb = mc * kLog2e;
    for (int v = tid; v < nvec; v += kSPThreads) {
      float x[T::VEC];
      unpack_vec<DT>(ld_shared_v4(sbase + v * 16), x);
#pragma unroll
      for (int k = 0; k < T::VEC; ++k) sum += ex2(fmaf(x[k], kLog2e, -mb));
    }
    if (tid < ntail) sum += ex2(fmaf(elem_at<DT>(sbase, nvec * T::VEC + tid), kLog2e, -mb));
  }
  const float sc = block_sum(sum, redf);

  // ---- merge the C partials in rank order (every CTA of the cluster gets the same result)
  float M = mc, S = sc;
  int I = (idx == INT_MAX) ? -1 : e0 + idx;
  if (p.C > 1) {
    if (tid == 0) {
      part_m = mc;
      part_s = sc;
      part_i = I;
    }
    cluster_sync();  // every CTA's partial is published
    M = -INFINITY;
    S = 0.f;
    I = -1;
    for (int k = 0; k < p.C; ++k) {
      const float mk = ld_shared_cluster_f32(map_to_rank(smem_u32(&part_m), k));
      M = fmaxf(M, mk);
    }
    for (int k = 0; k < p.C; ++k) {
      const float mk = ld_shared_cluster_f32(map_to_rank(smem_u32(&part_m), k));
      if (mk == -INFINITY) continue;
      const float sk = ld_shared_cluster_f32(map_to_rank(smem_u32(&part_s), k));
      S += sk * ex2((mk - M) * kLog2e);
      if (mk == M && I < 0) I = ld_shared_cluster_s32(map_to_rank(smem_u32(&part_i), k));
    }
  }
  const float lse = M + logf(S);
  if (rank == 0 && tid == 0) {
    p.stats.row_max[r] = M;
    p.stats.lse[r] = lse;
    p.stats.conf[r] = 1.f / S;
    p.stats.argmax[r] = I;
  }

  // ---- pass 3: this slice of P row c, from shared memory; zeros past V in the last slab
  const int vp = static_cast<int>(align_up(static_cast<size_t>(p.V), 64));
  const int e_end = min(vp, e0 + p.slabs_per_cta * 64);
  const float mb = lse * kLog2e;
  for (int g = tid; e0 + g * 8 < e_end; g += kSPThreads) {
    const int e = e0 + g * 8;  // 8 elements, one 16-byte store of P
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (ok && e < p.V) {
      float x[8];
      if constexpr (DT == DLLM_BF16) {
        unpack_vec<DT>(ld_shared_v4(sbase + (e - e0) * 2), x);
      } else {
        unpack_vec<DT>(ld_shared_v4(sbase + (e - e0) * 4), x);
        unpack_vec<DT>(ld_shared_v4(sbase + (e - e0) * 4 + 16), x + 4);
      }
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float lo = ex2(fmaf(x[2 * h], kLog2e, -mb));
        const float hi = ex2(fmaf(x[2 * h + 1], kLog2e, -mb));
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[h]) : "f"(hi), "f"(lo));
      }
      out = make_uint4(w[0], w[1], w[2], w[3]);
    }
    uint16_t* dst = p.P + ((static_cast<int64_t>(e >> 6) * p.R_pad + c) << 6) + (e & 63);
    *reinterpret_cast<uint4*>(dst) = out;
  }
  if (p.C > 1) cluster_sync();  // no CTA leaves while another may still read its partial
  if (!ok) drain_bar(smem_u32(&bar), 0);  // a copy that outlived the wait lands before exit
}

}  // namespace

bool stats_probs_split(int V, int dtype, int* C, int* slabs_per_cta) {
  const int es = dtype == DLLM_BF16 ? 2 : 4;
  const int slabs = (V + 63) / 64;
  const int target = std::max(1, kSPTargetBytes / (64 * es));
  int c = std::min(8, std::max(1, (slabs + target - 1) / target));
  const int per = (slabs + c - 1) / c;
  c = (slabs + per - 1) / per;  // every rank holds at least one slab
  *C = c;
  *slabs_per_cta = per;
  return static_cast<size_t>(per) * 64 * es <= kSPMaxSliceBytes;
}

cudaError_t launch_stats_probs(const void* logits, const dllm_shape& sh, const int32_t* rows,
                               const int32_t* count, const dllm_stats& stats, uint16_t* P,
                               int R_pad, int32_t* status, cudaStream_t stream) {
  SPParams p{};
  const int es = sh.dtype == DLLM_BF16 ? 2 : 4;
  p.logits = static_cast<const char*>(logits);
  p.row_stride_bytes = sh.row_stride * es;
  p.V = sh.V;
  if (!stats_probs_split(sh.V, sh.dtype, &p.C, &p.slabs_per_cta)) return cudaErrorInvalidValue;
  p.rows = rows;
  p.count = count;
  p.stats = stats;
  p.P = P;
  p.R_pad = R_pad;
  p.status = status;
  const size_t smem = static_cast<size_t>(p.slabs_per_cta) * 64 * es;
  auto kern = sh.dtype == DLLM_BF16 ? stats_probs_kernel<DLLM_BF16> : stats_probs_kernel<DLLM_F32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sh.B * sh.L * p.C));
  cfg.blockDim = dim3(kSPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace dllm
