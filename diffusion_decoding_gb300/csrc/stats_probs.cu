// Single-read iteration smoothing: the statistics of the rows a step reads and their bf16
// probability rows P, from one read of the logits (dInfer explainer, diffusion-iteration
// manager: iteration smoothing feeds the undecided positions' whole distributions forward).
//
// P[j, v] = bf16(exp(z_{r_j, v} - lse_{r_j})) needs the row's log-sum-exp before the first
// probability can be written, so a row is held on chip while its statistics complete: a cluster
// of C CTAs shares one row, each CTA holding a 64-element-aligned slice of it.
//
// stats_probs_kernel (rows of up to 8 x 16384 elements).  The clusters are persistent (as many as
// fit on the device, each looping over rows).  Each CTA streams its slices through a ring of
// shared-memory stages: one thread issues one 1-D bulk copy (cp.async.bulk) per slice, completing
// on the stage's mbarrier, so two rows are in flight while one is reduced.  Every thread copies
// its 8-element groups of the slice into registers and the warp releases the stage at once.  The
// thread takes the maximum tm of its elements and keeps e = exp(z - tm) in fp32 registers (one
// ex2 per element); the warp merges (max, rescaled sum, lowest index of the maximum) by shuffles
// and pushes that partial into every CTA of the cluster with st.async, which completes on the
// receiving CTA's mbarrier.  Every warp then merges the 8*C partials itself in one fixed order
// (so every warp of the cluster holds the same lse, bit for bit) and writes its probabilities,
// P = bf16(e * exp(tm - lse)), K-slab-blocked, straight from registers.  No block-wide or
// cluster-wide barrier is taken per row: a warp waits only for its stage and for the partials.
//
// stats_probs_wide_kernel (longer rows): the same cluster split with the slice held in shared
// memory (16-byte cp.async from every thread, double buffered), block reductions and a cluster
// barrier per row, and a second exp per element when P is written.
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
__global__ void __launch_bounds__(kSPThreads, 3) stats_probs_wide_kernel(const __grid_constant__ SPParams p) {
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

// ------------------------------------------------------------------ register-resident form

constexpr int kRRThreads = 256;
constexpr int kRRWarps = kRRThreads / 32;
constexpr int kRRMaxC = 8;         // CTAs per row (portable cluster size)
constexpr int kRRMaxGroups = 8;    // 8-element groups per thread
constexpr int kRRMaxStages = 4;

struct RRParams {
  const char* logits;
  int64_t row_stride_bytes;
  int V;
  int C;                  // CTAs per row (the cluster size)
  int slabs_per_cta;      // 64-element slabs per CTA
  int stages;             // ring depth
  uint32_t stage_bytes;   // slabs_per_cta * 64 * element size
  const int32_t* rows;    // rows to read, ascending
  const int32_t* count;   // device: how many
  dllm_stats stats;
  uint16_t* P;            // K-slab-blocked [ceil(V/64)][R_pad][64]
  int R_pad;
  int32_t* status;
};

// 16-byte store into shared memory of CTA `rank` of the cluster (address and barrier already
// mapped there), completing 16 bytes of transaction count on that CTA's mbarrier.
__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, const uint4& v,
                                            uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, "
      "[%5];" ::"r"(remote_addr),
      "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
      : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// The 8 elements of group k of this thread, as fp32 (bf16: one 16-byte vector; fp32: two).
template <int DT>
__device__ __forceinline__ void unpack_group(const uint4 (&q)[2], float (&x)[8]) {
  if constexpr (DT == DLLM_BF16) {
    unpack_vec<DT>(q[0], x);
  } else {
    unpack_vec<DT>(q[0], x);
    unpack_vec<DT>(q[1], x + 4);
  }
}

template <int DT>
__device__ __forceinline__ float group_max(const uint4 (&q)[2]) {
  if constexpr (DT == DLLM_BF16) {
    return vec_max<DT>(q[0]);
  } else {
    return fmaxf(vec_max<DT>(q[0]), vec_max<DT>(q[1]));
  }
}

// Merge of the row's (max, sum of exp(z - max), lowest index of the max) partials, one per
// warp of every CTA (n of them, k = rank * 8 + warp), read from this CTA's copy; every warp
// computes it in the same order, so every warp of the cluster gets the same bits.
__device__ __forceinline__ RowAcc merge_partials(const uint4* part, int n) {
  const int lane = threadIdx.x & 31;
  const uint4 none = make_uint4(__float_as_uint(-INFINITY), 0u, 0xFFFFFFFFu, 0u);
  const uint4 a = lane < n ? part[lane] : none;
  const uint4 b = lane + 32 < n ? part[lane + 32] : none;
  const float ma = __uint_as_float(a.x), mb = __uint_as_float(b.x);
  float M = fmaxf(ma, mb);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  float S = 0.f;
  int I = INT_MAX;
  if (M != -INFINITY) {
    const float Mb = M * kLog2e;
    if (ma != -INFINITY) S = __uint_as_float(a.y) * ex2(fmaf(ma, kLog2e, -Mb));
    if (mb != -INFINITY) S += __uint_as_float(b.y) * ex2(fmaf(mb, kLog2e, -Mb));
    if (ma == M && static_cast<int>(a.z) >= 0) I = static_cast<int>(a.z);
    if (mb == M && static_cast<int>(b.z) >= 0) I = min(I, static_cast<int>(b.z));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    S += __shfl_xor_sync(kFull, S, o);
    I = min(I, __shfl_xor_sync(kFull, I, o));
  }
  return RowAcc{M, S, I == INT_MAX ? -1 : I};
}

template <int DT, int GPT>
__global__ void __launch_bounds__(kRRThreads, 2)
    stats_probs_kernel(const __grid_constant__ RRParams p) {
  using T = Elem<DT>;
  constexpr int VPG = DT == DLLM_BF16 ? 1 : 2;  // 16-byte vectors per 8-element group
  constexpr uint32_t kNegInf = DT == DLLM_BF16 ? 0xFF80FF80u : 0xFF800000u;  // -inf elements
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full_bar[kRRMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kRRMaxStages];
  __shared__ __align__(8) uint64_t part_bar[2];
  __shared__ __align__(16) uint4 part[2][kRRMaxC * kRRWarps];  // partials, by row parity
  __shared__ int abort_flag;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int cl = static_cast<int>(blockIdx.x) / p.C;  // this cluster, the same in all its CTAs
  const int n_cl = static_cast<int>(gridDim.x) / p.C;
  const int NS = p.stages;
  const uint32_t ring0 = smem_u32(ring);
  const uint32_t full0 = smem_u32(&full_bar[0]), empty0 = smem_u32(&empty_bar[0]);
  const uint32_t pbar0 = smem_u32(&part_bar[0]);
  volatile int* abort_v = &abort_flag;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);               // the producer's expect-tx arrival
      mbar_init(empty0 + 8 * s, kRRWarps);       // one arrival per warp that has read the stage
    }
    // per row: this CTA's expect-tx arrival (the other CTAs' partials) + one arrival per warp
    // after it stored its own partial here
    mbar_init(pbar0, 1 + kRRWarps);
    mbar_init(pbar0 + 8, 1 + kRRWarps);
    abort_flag = 0;
    fence_mbar_init();
  }
  cluster_sync();  // every CTA's barriers exist before anyone pushes a partial into it
  pdl_wait();      // the row list comes from the kernel before this one
  pdl_trigger();
  const int count = *reinterpret_cast<const volatile int32_t*>(p.count);
  const int nmine = cl < count ? (count - cl + n_cl - 1) / n_cl : 0;  // rows of this cluster

  const int e0 = static_cast<int>(rank) * p.slabs_per_cta * 64;
  const int n = max(0, min(p.V, e0 + p.slabs_per_cta * 64) - e0);  // elements of this slice
  const uint32_t copy_bytes = static_cast<uint32_t>(n) * T::ES;     // a multiple of 16
  const int ngv = n / 8;                                              // groups holding logits
  const int vp = static_cast<int>(align_up(static_cast<size_t>(p.V), 64));
  const int ngroups = (min(vp, e0 + p.slabs_per_cta * 64) - e0) / 8;  // groups of P to write
  const int64_t slab_stride = static_cast<int64_t>(p.R_pad) << 6;  // P elements between slabs
  const uint32_t part_bytes = static_cast<uint32_t>(16 * kRRWarps * (p.C - 1));  // remote

  // this CTA's slice of the j-th row of the cluster into stage j % NS (one thread)
  auto issue = [&](int j) {
    const int s = j % NS;
    const int r = p.rows[cl + j * n_cl];
    mbar_expect_tx(full0 + 8 * s, copy_bytes);
    bulk_g2s(ring0 + s * p.stage_bytes,
             p.logits + static_cast<int64_t>(r) * p.row_stride_bytes +
                 static_cast<int64_t>(e0) * T::ES,
             copy_bytes, full0 + 8 * s);
  };
  int issued = 0;  // rows whose copy this thread has issued (thread 0 only)
  if (tid == 0) {
    for (; issued < min(NS - 1, nmine); ++issued) issue(issued);
  }

  int it = 0;
  for (; it < nmine; ++it) {
    const int c = cl + it * n_cl;
    const int s = it % NS;
    bool ok = true;
    if (tid == 0) {
      // refill the stage row it - 1 used (every warp released it before it could finish that
      // row, since the row's merge needs every warp's partial), then expect this row's partials
      const int j = it + NS - 1;
      if (j < nmine) {
        if (j >= NS) ok = wait_bar(empty0 + 8 * (j % NS), ((j / NS) - 1) & 1, abort_v, p.status);
        if (ok) {
          issue(j);
          issued = j + 1;
        }
      }
      if (ok) {
        if (part_bytes) mbar_expect_tx(pbar0 + 8 * (it & 1), part_bytes);
        else mbar_arrive(pbar0 + 8 * (it & 1));
      }
    }
    if (!__all_sync(kFull, ok && wait_bar(full0 + 8 * s, (it / NS) & 1, abort_v, p.status)))
      break;

    // ---- this thread's groups g = tid + 256 k of the slice, into registers
    const uint32_t sb = ring0 + s * p.stage_bytes;
    uint4 q[GPT][2];
#pragma unroll
    for (int k = 0; k < GPT; ++k) {
      const int g = tid + k * kRRThreads;
#pragma unroll
      for (int h = 0; h < VPG; ++h) {
        q[k][h] = g < ngv ? ld_shared_v4(sb + (g * VPG + h) * 16)
                          : make_uint4(kNegInf, kNegInf, kNegInf, kNegInf);
      }
      if constexpr (VPG == 1) q[k][1] = q[k][0];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);  // the stage may be refilled

    // ---- thread maximum, the first group holding it, exp(z - tm) and their sum
    float tm = -INFINITY;
    int bk = 0;
#pragma unroll
    for (int k = 0; k < GPT; ++k) {
      const float gm = group_max<DT>(q[k]);
      if (gm > tm) {
        tm = gm;
        bk = k;
      }
    }
    int idx = INT_MAX;
    if (tm != -INFINITY) {
      uint4 best[2] = {q[0][0], q[0][1]};
#pragma unroll
      for (int k = 1; k < GPT; ++k)
        if (k == bk) {
          best[0] = q[k][0];
          best[1] = q[k][1];
        }
      float x[8];
      unpack_group<DT>(best, x);
#pragma unroll
      for (int j = 7; j >= 0; --j)
        if (x[j] == tm) idx = e0 + (tid + bk * kRRThreads) * 8 + j;
    }
    const float tmb = tm == -INFINITY ? 0.f : tm * kLog2e;
    const uint64_t k2 = pack2(kLog2e, kLog2e), ntm2 = pack2(-tmb, -tmb);
    uint64_t e2[GPT][4];
    uint64_t acc = pack2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < GPT; ++k) {
      float x[8];
      unpack_group<DT>(q[k], x);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float t0, t1;
        unpack2(fma2(pack2(x[2 * h], x[2 * h + 1]), k2, ntm2), t0, t1);
        e2[k][h] = pack2(ex2(t0), ex2(t1));
        acc = add2(acc, e2[k][h]);
      }
    }
    float a0, a1;
    unpack2(acc, a0, a1);
    const float st = a0 + a1;

    // ---- warp partial, stored here and pushed into every other CTA of the cluster (lane k ->
    // CTA k)
    float mw = tm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mw = fmaxf(mw, __shfl_xor_sync(kFull, mw, o));
    float sw = tm == -INFINITY ? 0.f : st * ex2(fmaf(tm, kLog2e, -mw * kLog2e));
    int iw = (tm == mw && tm != -INFINITY) ? idx : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sw += __shfl_xor_sync(kFull, sw, o);
      iw = min(iw, __shfl_xor_sync(kFull, iw, o));
    }
    if (lane < p.C) {
      const uint4 pw = make_uint4(__float_as_uint(mw), __float_as_uint(sw),
                                  static_cast<uint32_t>(iw == INT_MAX ? -1 : iw), 0u);
      const uint32_t slot = smem_u32(&part[it & 1][rank * kRRWarps + warp]);
      if (lane == static_cast<int>(rank)) {
        st_shared_v4(slot, pw);
        mbar_arrive(pbar0 + 8 * (it & 1));  // release: the store is seen by every waiter
      } else {
        st_async_v4(map_to_rank(slot, lane), pw, map_to_rank(pbar0 + 8 * (it & 1), lane));
      }
    }
    if (!__all_sync(kFull, wait_bar(pbar0 + 8 * (it & 1), (it >> 1) & 1, abort_v, p.status)))
      break;
    const RowAcc row = merge_partials(part[it & 1], kRRWarps * p.C);
    const float lse = row.m + logf(row.s);
    if (rank == 0 && tid == 0) {
      const int r = p.rows[c];
      p.stats.row_max[r] = row.m;
      p.stats.lse[r] = lse;
      p.stats.conf[r] = 1.f / row.s;
      p.stats.argmax[r] = row.idx;
    }

    // ---- P = bf16(e * exp(tm - lse)) from registers; zeros past V in the last slab.  P element
    // (c, v) sits at ((v / 64) * R_pad + c) * 64 + v % 64: group g of the slice (8 elements)
    // lands in slab e0 / 64 + g / 8, at element (g % 8) * 8 of row c's run of that slab.
    const float sc = (row.m == -INFINITY || tm == -INFINITY)
                         ? 0.f
                         : ex2(fmaf(tm, kLog2e, -lse * kLog2e));
    const uint64_t sc2 = pack2(sc, sc), zero2 = pack2(0.f, 0.f);
    uint16_t* const prow = p.P + ((static_cast<int64_t>(e0 >> 6) * p.R_pad + c) << 6);
#pragma unroll
    for (int k = 0; k < GPT; ++k) {
      const int g = tid + k * kRRThreads;
      if (g < ngroups) {
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          float lo, hi;
          unpack2(fma2(e2[k][h], sc2, zero2), lo, hi);
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[h]) : "f"(hi), "f"(lo));
        }
        const uint4 out = g < ngv ? make_uint4(w[0], w[1], w[2], w[3]) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(prow + (g >> 3) * slab_stride + ((g & 7) << 3)) = out;
      }
    }
  }
  if (it < nmine && tid == 0) {
    // gave up (a wait timed out): let the copies already issued land before the CTA leaves
    for (int j = it; j < issued; ++j) drain_bar(full0 + 8 * (j % NS), (j / NS) & 1);
  }
  cluster_sync();  // no CTA leaves while another may still push a partial into it
}

// Clusters of a kernel that fit on the device at once, queried once per configuration (kind
// tells the kernels apart).
int resident_clusters(const void* kern, const cudaLaunchConfig_t& cfg, int kind, int C,
                      size_t smem) {
  struct Entry {
    int dev, kind, C;
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
    if (cache[i].dev == dev && cache[i].kind == kind && cache[i].C == C &&
        cache[i].smem == smem)
      return cache[i].n;
  cudaLaunchConfig_t q = cfg;
  q.gridDim = dim3(static_cast<unsigned>(C * 1024));
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess || n < 1) n = 1;
  if (used < 32) cache[used++] = Entry{dev, kind, C, smem, n};
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

namespace {

template <int DT>
void* rr_kernel(int gpt) {
  switch (gpt) {
    case 1: return reinterpret_cast<void*>(stats_probs_kernel<DT, 1>);
    case 2: return reinterpret_cast<void*>(stats_probs_kernel<DT, 2>);
    case 4: return reinterpret_cast<void*>(stats_probs_kernel<DT, 4>);
    default: return reinterpret_cast<void*>(stats_probs_kernel<DT, 8>);
  }
}

cudaError_t launch_clustered(const void* kern, void* params, int C, int threads, size_t smem,
                             int kind, int rows, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(C));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // persistent: as many clusters as can be resident at once, no more than there are rows
  const int n_cl = resident_clusters(kern, cfg, kind, C, smem);
  cfg.gridDim = dim3(static_cast<unsigned>(C * std::min(n_cl, std::max(rows, 1))));
  void* args[] = {params};
  return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace

cudaError_t launch_stats_probs(const void* logits, const dllm_shape& sh, const int32_t* rows,
                               const int32_t* count, const dllm_stats& stats, uint16_t* P,
                               int R_pad, int32_t* status, cudaStream_t stream) {
  const int es = sh.dtype == DLLM_BF16 ? 2 : 4;
  int C = 0, per = 0;
  if (!stats_probs_split(sh.V, sh.dtype, &C, &per)) return cudaErrorInvalidValue;
  const int groups = per * 8;  // 8-element groups of one CTA's slice
  if (C <= kRRMaxC && groups <= kRRMaxGroups * kRRThreads) {
    RRParams p{};
    p.logits = static_cast<const char*>(logits);
    p.row_stride_bytes = sh.row_stride * es;
    p.V = sh.V;
    p.C = C;
    p.slabs_per_cta = per;
    p.stage_bytes = static_cast<uint32_t>(per) * 64 * es;
    // ring depth: three or four stages at two CTAs per SM when they fit, else one CTA per SM
    const size_t two_per_sm = 110 * 1024, one_per_sm = 220 * 1024;
    int ns = static_cast<int>(std::min<size_t>(kRRMaxStages, two_per_sm / p.stage_bytes));
    if (ns < 3) ns = static_cast<int>(std::min<size_t>(kRRMaxStages, one_per_sm / p.stage_bytes));
    p.stages = ns;
    p.rows = rows;
    p.count = count;
    p.stats = stats;
    p.P = P;
    p.R_pad = R_pad;
    p.status = status;
    const int gpt = groups <= kRRThreads ? 1 : groups <= 2 * kRRThreads ? 2
                    : groups <= 4 * kRRThreads ? 4 : 8;
    const void* kern = sh.dtype == DLLM_BF16 ? rr_kernel<DLLM_BF16>(gpt) : rr_kernel<DLLM_F32>(gpt);
    return launch_clustered(kern, &p, C, kRRThreads,
                            static_cast<size_t>(ns) * p.stage_bytes, sh.dtype * 16 + gpt,
                            sh.B * sh.L, stream);
  }
  SPParams p{};
  p.logits = static_cast<const char*>(logits);
  p.row_stride_bytes = sh.row_stride * es;
  p.V = sh.V;
  p.C = C;
  p.slabs_per_cta = per;
  p.rows = rows;
  p.count = count;
  p.stats = stats;
  p.P = P;
  p.R_pad = R_pad;
  p.status = status;
  const size_t smem = 2 * static_cast<size_t>(per) * 64 * es;  // double buffer
  const void* kern = reinterpret_cast<const void*>(
      sh.dtype == DLLM_BF16 ? stats_probs_wide_kernel<DLLM_BF16> : stats_probs_wide_kernel<DLLM_F32>);
  return launch_clustered(kern, &p, C, kSPThreads, smem, 100 + sh.dtype, sh.B * sh.L, stream);
}

}  // namespace dllm
