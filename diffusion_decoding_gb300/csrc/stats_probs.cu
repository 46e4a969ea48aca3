// Single-read iteration smoothing: the statistics of the rows a step reads and their bf16
// probability rows P, from one read of the logits (dInfer explainer, diffusion-iteration
// manager: iteration smoothing feeds the undecided positions' whole distributions forward).
//
// P[j, v] = bf16(exp(z_{r_j, v} - lse_{r_j})) needs the row's log-sum-exp before the first
// probability can be written, so a row is held on chip while its statistics complete: a cluster
// of C CTAs shares one row, each CTA bringing its 64-element-aligned slice into shared memory
// with 16-byte cp.async copies from every thread.  Each CTA reduces its slice to (max, sum of exp(z - max), lowest index of
// max); the C partials are exchanged through distributed shared memory and merged in rank order
// by every CTA (so all of them hold the same lse, bit for bit); rank 0 writes the row's
// statistics and every CTA writes its slice of P, K-slab-blocked, straight from shared memory.
// The logits cross HBM once instead of twice (statistics, then probabilities).
//
// The clusters are persistent (as many as fit on the device, each looping over rows) and double
// buffered: the next row's slice streams in (16-byte cp.async from every thread) while the
// current one is reduced and written.  A one-shot form, one cluster per row, ran its phases
// (load ~2.5 us, two reduction passes, the cluster exchange, the P pass) back to back in every
// CTA and streamed at ~4.2 TB/s.
//
// P row j belongs to the j-th row read (the compaction of the block state taken before the
// commit); the GEMM maps P rows to the rows kept after the commit.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "mbarrier.cuh"
#include "vec_math.cuh"

namespace dllm {
namespace {

constexpr int kSPThreads = 256;
constexpr int kSPWarps = kSPThreads / 32;
constexpr int kSPTargetBytes = 32768;       // slice of one CTA, aimed at
constexpr int kSPMaxSliceBytes = 192 * 1024;

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
__global__ void __launch_bounds__(kSPThreads, 3) stats_probs_kernel(const __grid_constant__ SPParams p) {
  using T = Elem<DT>;
  extern __shared__ __align__(128) uint8_t slice[];  // two slice buffers (double buffering)
  __shared__ float redf[kSPWarps];
  __shared__ int redi[kSPWarps];
  __shared__ float part_m[2], part_s[2];  // this CTA's partial, by row parity
  __shared__ int part_i[2];
  __shared__ float red_M, red_S;
  __shared__ int red_I;

  const int tid = threadIdx.x;
  const uint32_t rank = p.C > 1 ? cluster_ctarank() : 0u;
  const int cl = static_cast<int>(blockIdx.x) / p.C;  // this cluster, the same in all its CTAs
  const int n_cl = static_cast<int>(gridDim.x) / p.C;
  pdl_wait();  // the row list comes from the kernel before this one
  pdl_trigger();
  const int count = *reinterpret_cast<const volatile int32_t*>(p.count);
  const int e0 = static_cast<int>(rank) * p.slabs_per_cta * 64;
  const int n = max(0, min(p.V, e0 + p.slabs_per_cta * 64) - e0);  // elements of this slice
  const uint32_t buf_bytes = static_cast<uint32_t>(p.slabs_per_cta) * 64 * T::ES;
  // rounded up to 16 bytes: stays inside the row's stride
  const int nchunks = static_cast<int>(align_up(static_cast<size_t>(n) * T::ES, 16) / 16);
  const uint32_t buf0 = smem_u32(slice);
  const int nvec = n * T::ES / 16;
  const int ntail = n - nvec * T::VEC;
  const int vp = static_cast<int>(align_up(static_cast<size_t>(p.V), 64));
  const int e_end = min(vp, e0 + p.slabs_per_cta * 64);
  const int ngroups = (e_end - e0) / 8;
  const int64_t slab_stride = static_cast<int64_t>(p.R_pad) << 6;  // P elements between slabs

  // 16-byte cp.async of this CTA's slice of P row c's logits, by every thread, one group
  auto load = [&](int c, uint32_t dst) {
    const char* src = p.logits + static_cast<int64_t>(p.rows[c]) * p.row_stride_bytes +
                      static_cast<int64_t>(e0) * T::ES;
#pragma unroll 4
    for (int i = tid; i < nchunks; i += kSPThreads) cp_async16(dst + i * 16, src + i * 16);
    cp_async_commit();
  };

  int c = cl;
  if (c < count) load(c, buf0);
  for (int it = 0; c < count; ++it, c += n_cl) {
    const uint32_t sbase = buf0 + (it & 1) * buf_bytes;
    // the next row's slice streams in while this one is reduced and written
    if (c + n_cl < count) {
      load(c + n_cl, buf0 + ((it + 1) & 1) * buf_bytes);
      cp_async_wait_group<1>();
    } else {
      cp_async_wait_group<0>();
    }
    __syncthreads();  // this row's slice is in shared memory, for every thread
    const int r = p.rows[c];

    // ---- pass 1: slice maximum and the first vector holding it
    float tm = -INFINITY;
    int bu = -1;
#pragma unroll 4
    for (int v = tid; v < nvec; v += kSPThreads) {
      const float vm = vec_max<DT>(ld_shared_v4(sbase + v * 16));
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
    const float mc = block_max(tm, redf);
    int idx = INT_MAX;
    if (tm == mc && mc != -INFINITY) {
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
    if (mc != -INFINITY) {
      const float mb = mc * kLog2e;
      const uint64_t k2 = pack2(kLog2e, kLog2e), nmb2 = pack2(-mb, -mb);
      uint64_t acc2 = pack2(0.f, 0.f);
#pragma unroll 4
      for (int v = tid; v < nvec; v += kSPThreads) {
        float x[T::VEC];
        unpack_vec<DT>(ld_shared_v4(sbase + v * 16), x);
#pragma unroll
        for (int k = 0; k < T::VEC; k += 2) {
          float t0, t1;
          unpack2(fma2(pack2(x[k], x[k + 1]), k2, nmb2), t0, t1);
          acc2 = add2(acc2, pack2(ex2(t0), ex2(t1)));
        }
      }
      float a0, a1;
      unpack2(acc2, a0, a1);
      sum = a0 + a1;
      if (tid < ntail) sum += ex2(fmaf(elem_at<DT>(sbase, nvec * T::VEC + tid), kLog2e, -mb));
    }
    const float sc = block_sum(sum, redf);

    // ---- merge the C partials in rank order (every CTA of the cluster gets the same result)
    float M = mc, S = sc;
    int I = (idx == INT_MAX) ? -1 : e0 + idx;
    if (p.C > 1) {
      const int slot = it & 1;
      if (tid == 0) {
        part_m[slot] = mc;
        part_s[slot] = sc;
        part_i[slot] = I;
      }
      cluster_sync();  // every CTA's partial of this row is published
      if (tid < 32) {  // one warp reads the C partials (lane k: rank k), merges in rank order
        const int k = tid;
        const bool has = k < p.C;
        const float mk =
            has ? ld_shared_cluster_f32(map_to_rank(smem_u32(&part_m[slot]), k)) : -INFINITY;
        const float sk = has ? ld_shared_cluster_f32(map_to_rank(smem_u32(&part_s[slot]), k)) : 0.f;
        const int ik = has ? ld_shared_cluster_s32(map_to_rank(smem_u32(&part_i[slot]), k)) : -1;
        float m = mk;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        float sum_all = 0.f;
        int first = -1;
        for (int j = 0; j < p.C; ++j) {
          const float mj = __shfl_sync(kFull, mk, j);
          const float sj = __shfl_sync(kFull, sk, j);
          const int ij = __shfl_sync(kFull, ik, j);
          if (mj == -INFINITY) continue;
          sum_all += sj * ex2((mj - m) * kLog2e);
          if (mj == m && first < 0) first = ij;
        }
        if (tid == 0) {
          red_M = m;
          red_S = sum_all;
          red_I = first;
        }
      }
      __syncthreads();
      M = red_M;
      S = red_S;
      I = red_I;
    }
    const float lse = M + logf(S);
    if (rank == 0 && tid == 0) {
      p.stats.row_max[r] = M;
      p.stats.lse[r] = lse;
      p.stats.conf[r] = 1.f / S;
      p.stats.argmax[r] = I;
    }

    // ---- pass 3: this slice of P row c, from shared memory; zeros past V in the last slab.
    // P element (c, e) at ((e / 64) * R_pad + c) * 64 + e % 64: 16-byte group g of the slice
    // (8 elements) lands in slab e0 / 64 + g / 8, at element (g % 8) * 8 of row c's run.
    const float mb = lse * kLog2e;
    const uint64_t k2 = pack2(kLog2e, kLog2e), nmb2 = pack2(-mb, -mb);
    uint16_t* const prow = p.P + ((static_cast<int64_t>(e0 >> 6) * p.R_pad + c) << 6);
#pragma unroll 4
    for (int g = tid; g < ngroups; g += kSPThreads) {
      const int e = e0 + g * 8;
      uint4 out = make_uint4(0u, 0u, 0u, 0u);
      if (e < p.V) {
        float x[8];
        if constexpr (DT == DLLM_BF16) {
          unpack_vec<DT>(ld_shared_v4(sbase + g * 16), x);
        } else {
          unpack_vec<DT>(ld_shared_v4(sbase + g * 32), x);
          unpack_vec<DT>(ld_shared_v4(sbase + g * 32 + 16), x + 4);
        }
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          float t0, t1;
          unpack2(fma2(pack2(x[2 * h], x[2 * h + 1]), k2, nmb2), t0, t1);
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[h]) : "f"(ex2(t1)), "f"(ex2(t0)));
        }
        out = make_uint4(w[0], w[1], w[2], w[3]);
      }
      *reinterpret_cast<uint4*>(prow + (g >> 3) * slab_stride + ((g & 7) << 3)) = out;
    }
    __syncthreads();  // every thread is done with this buffer before it is refilled
  }
  if (p.C > 1) cluster_sync();  // no CTA leaves while another may still read its partials
}

// Clusters of this kernel that fit on the device at once, queried once per configuration.
int resident_clusters(const void* kern, const cudaLaunchConfig_t& cfg, int dtype, int C,
                      size_t smem) {
  struct Entry {
    int dev, dtype, C;
    size_t smem;
    int n;
  };
  static std::mutex mu;
  static Entry cache[32];
  static int used = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].dtype == dtype && cache[i].C == C &&
        cache[i].smem == smem)
      return cache[i].n;
  cudaLaunchConfig_t q = cfg;
  q.gridDim = dim3(static_cast<unsigned>(C * 1024));
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess || n < 1) n = 1;
  if (used < 32) cache[used++] = Entry{dev, dtype, C, smem, n};
  return n;
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
  const size_t smem = 2 * static_cast<size_t>(p.slabs_per_cta) * 64 * es;  // double buffer
  auto kern = sh.dtype == DLLM_BF16 ? stats_probs_kernel<DLLM_BF16> : stats_probs_kernel<DLLM_F32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.C));
  cfg.blockDim = dim3(kSPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // persistent: as many clusters as can be resident at once, no more than there are rows
  const int n_cl = resident_clusters(reinterpret_cast<const void*>(kern), cfg, sh.dtype, p.C, smem);
  cfg.gridDim = dim3(static_cast<unsigned>(p.C * std::min(n_cl, sh.B * sh.L)));
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace dllm
