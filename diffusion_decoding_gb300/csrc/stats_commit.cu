// Softmax statistics + commit decision over one masked block (kernel "a": two launches).
//
// 1. stats_partials_kernel: every masked row of logits is streamed from HBM exactly once.  Rows
//    are cut into 4 KB slices; a warp reduces one slice at a time: it issues all of its 128-bit
//    loads up front (8 per lane), takes the slice maximum with warp shuffles, sums
//    exp(z - max) against that single maximum (no rescaling), finds the first index of the
//    maximum, and writes one partial (max, sum, argmax).  Small grids and blocks of more than
//    4096 rows launch one warp per slice; other blocks run a persistent grid whose CTAs first
//    list the rows read (one barrier-separated scan per CTA), so a nearly decided block does
//    not launch a CTA per 8 slices that are not read.  No atomic, no fence.  (Completing each
//    row inside this kernel, with an acquire/release atomic per slice on a row counter, cost
//    ~17 us at 1024 rows x V = 126464: every warp's release fence waited behind the loads in
//    flight.)
// 2. commit_only_kernel (one CTA per sequence, chained with programmatic dependent launch so it
//    is resident before the first kernel drains): merges the slice partials of its sequence's
//    rows into their statistics (eight threads per row, every load issued up front), then runs
//    the commit decision in shared memory (threshold, hierarchical or credit decoding; dInfer
//    explainer, decoding-strategy component, methods 1-3).  In statistics-only mode it only
//    merges.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "vec_math.cuh"

namespace dllm {
namespace {

constexpr int kThreads = 256;
constexpr int kStatsCtasPerSm = 4;  // resident statistics CTAs per SM (64 registers per thread)
constexpr int kCompactRows = 4096;  // largest block the persistent statistics grid lists

struct CommitCtx {
  int B, L;
  dllm_block_state state;
  CommitArgs ca;
};

struct FusedParams {
  const char* logits;
  int64_t row_stride_bytes;
  int V, S, chunk;
  int compact;             // persistent grid over the rows read (listed in shared memory)
  int pdl_from;            // CTAs from this index on let the dependent commit grid launch
  const uint8_t* masked;   // rows to read (state.masked when committing)
  const int32_t* eos_hit;  // null in statistics-only mode
  dllm_stats stats;
  StatsWs ws;
  CommitCtx c;
};

struct CommitOnlyParams {
  dllm_stats stats;
  CommitCtx c;
  int S;                  // slices per row (1: the statistics are complete, nothing to merge)
  const uint4* part;      // [R * S] slice partials {max, sum, argmax, 0}
  const uint8_t* masked;  // rows that were read (null: all rows; statistics-only mode)
  const int32_t* eos_hit; // null in statistics-only mode
};

// ------------------------------------------------------------------ slice reduction

constexpr int kVecs = 8;  // 16-byte vectors per lane: one warp slice = 4 KB

template <int DT>
struct SliceTraits;
template <>
struct SliceTraits<DLLM_BF16> {
  static constexpr int VEC = 8, ES = 2;
  static constexpr uint32_t kNegInf = 0xFF80FF80u;  // two bf16 -inf
};
template <>
struct SliceTraits<DLLM_F32> {
  static constexpr int VEC = 4, ES = 4;
  static constexpr uint32_t kNegInf = 0xFF800000u;  // fp32 -inf
};

// elements of one warp slice
template <int DT>
constexpr int slice_elems() {
  return 32 * kVecs * SliceTraits<DT>::VEC;
}

// One warp reduces elements [e0, e0 + n) of a row (n <= slice_elems) to (max, sum of
// exp(z - max), lowest index of max).  Pass 1 takes each lane's maximum and remembers the first
// of its vectors that holds it; the warp maximum follows by shuffles.  Pass 2 sums
// exp(z - max) against that single maximum (no rescaling).  Only lanes holding the maximum
// look for its index, by re-reading that one vector.  The result is valid in every lane.
template <int DT>
__device__ __forceinline__ RowAcc warp_reduce_slice(const char* row, int64_t e0, int n) {
  using T = SliceTraits<DT>;
  const int lane = threadIdx.x & 31;
  const int nvec = n * T::ES / 16;
  const int ntail = n - nvec * T::VEC;
  const char* base = row + e0 * T::ES;
  uint4 q[kVecs];
#pragma unroll
  for (int u = 0; u < kVecs; ++u) {
    const int vi = u * 32 + lane;
    q[u] = vi < nvec ? ld_stream_v4(base + static_cast<int64_t>(vi) * 16)
                     : make_uint4(T::kNegInf, T::kNegInf, T::kNegInf, T::kNegInf);
  }
  const float xt = lane < ntail ? load_logit(row, DT, e0 + nvec * T::VEC + lane) : -INFINITY;

  float tm = -INFINITY;
  int bu = -1;  // first vector of this lane holding tm (kVecs: the tail element)
#pragma unroll
  for (int u = 0; u < kVecs; ++u) {
    const float vm = vec_max<DT>(q[u]);
    if (vm > tm) {
      tm = vm;
      bu = u;
    }
  }
  if (xt > tm) {
    tm = xt;
    bu = kVecs;
  }
  float m = tm;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));

  const float mb = (m == -INFINITY) ? 0.f : m * kLog2e;
  // exp2(x*log2e - mb) summed with packed fp32x2 FMA / ADD: two elements per instruction
  const uint64_t k2 = pack2(kLog2e, kLog2e), nmb2 = pack2(-mb, -mb);
  uint64_t acc2[2] = {pack2(0.f, 0.f), pack2(0.f, 0.f)};
#pragma unroll
  for (int u = 0; u < kVecs; ++u) {
    float x[T::VEC];
    unpack_vec<DT>(q[u], x);
#pragma unroll
    for (int j = 0; j < T::VEC; j += 2) {
      float t0, t1;
      unpack2(fma2(pack2(x[j], x[j + 1]), k2, nmb2), t0, t1);
      acc2[(j >> 1) & 1] = add2(acc2[(j >> 1) & 1], pack2(ex2(t0), ex2(t1)));
    }
  }
  float a0, a1, a2, a3;
  unpack2(acc2[0], a0, a1);
  unpack2(acc2[1], a2, a3);
  float sum = ((a0 + a1) + (a2 + a3)) + ex2(fmaf(xt, kLog2e, -mb));
  int idx = INT_MAX;
  if (tm == m && m != -INFINITY) {  // rare: this lane holds the slice maximum
    if (bu == kVecs) {
      idx = nvec * T::VEC + lane;
    } else {
      const int vi = bu * 32 + lane;
      float x[T::VEC];
      unpack_vec<DT>(ld_stream_v4(base + static_cast<int64_t>(vi) * 16), x);
      for (int j = T::VEC - 1; j >= 0; --j)
        if (x[j] == m) idx = vi * T::VEC + j;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sum += __shfl_xor_sync(kFull, sum, o);
    idx = min(idx, __shfl_xor_sync(kFull, idx, o));
  }
  return RowAcc{m, sum, idx == INT_MAX ? -1 : static_cast<int>(e0) + idx};
}

// The same reduction for rows that are not 16-byte aligned (a row stride or a logits pointer
// that is only element-aligned): lane k reads elements k, k + 32, ... one at a time, keeping a
// running maximum, its first index and the sum of exp(z - maximum), rescaled whenever the
// maximum rises; the lanes are then merged by shuffles (lowest index on ties).
template <int DT>
__device__ __forceinline__ RowAcc warp_reduce_slice_scalar(const char* row, int64_t e0, int n) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY, s = 0.f;
  int idx = -1;
  for (int k = lane; k < n; k += 32) {
    const float x = load_logit(row, DT, e0 + k);
    if (x > m) {  // s * exp(m - x) + 1; exp(-inf) = 0 for the first element
      s = fmaf(s, ex2((m - x) * kLog2e), 1.f);
      m = x;
      idx = static_cast<int>(e0) + k;
    } else if (x != -INFINITY) {
      s += ex2((x - m) * kLog2e);
    }
  }
  return row_acc_warp_reduce(RowAcc{m, s, idx});
}

// ------------------------------------------------------------------ block helpers

constexpr int kBlockWarpsMax = 32;  // the block helpers below serve blocks of up to 1024 threads

// In-place inclusive max-scan of a[0..n) (values >= -1) with warp shuffles; ends synchronised.
__device__ void block_max_scan(int* a, int n) {
  __shared__ int warp_tot[kBlockWarpsMax];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nt = blockDim.x;
  const int ipt = (n + nt - 1) / nt;
  const int beg = tid * ipt, end = min(n, beg + ipt);
  int run = -1;
  for (int i = beg; i < end; ++i) {
    run = max(run, a[i]);
    a[i] = run;
  }
  int agg = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(kFull, agg, o);
    if (lane >= o) agg = max(agg, y);
  }
  int excl = __shfl_up_sync(kFull, agg, 1);
  if (lane == 0) excl = -1;
  if (lane == 31) warp_tot[warp] = agg;
  __syncthreads();
  int pre = excl;
  for (int w = 0; w < warp; ++w) pre = max(pre, warp_tot[w]);
  for (int i = beg; i < end; ++i) a[i] = max(a[i], pre);
  __syncthreads();
}

// Masked position of largest value, lowest index on ties (-1 if nothing is masked).
__device__ int block_masked_argmax(const float* val, const uint8_t* mask, int L) {
  __shared__ float wv[kBlockWarpsMax];
  __shared__ int wi[kBlockWarpsMax];
  __shared__ int result;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nt = blockDim.x, nw = nt >> 5;
  float best = -INFINITY;
  int bi = INT_MAX;
  for (int i = tid; i < L; i += nt) {
    if (mask[i] && (bi == INT_MAX || val[i] > best)) {
      best = val[i];
      bi = i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(kFull, best, o);
    int oi = __shfl_xor_sync(kFull, bi, o);
    if (oi != INT_MAX && (bi == INT_MAX || ov > best || (ov == best && oi < bi))) {
      best = ov;
      bi = oi;
    }
  }
  if (lane == 0) {
    wv[warp] = best;
    wi[warp] = bi;
  }
  __syncthreads();
  if (tid == 0) {
    float b = wv[0];
    int i0 = wi[0];
    for (int w = 1; w < nw; ++w) {
      if (wi[w] != INT_MAX && (i0 == INT_MAX || wv[w] > b || (wv[w] == b && wi[w] < i0))) {
        b = wv[w];
        i0 = wi[w];
      }
    }
    result = (i0 == INT_MAX) ? -1 : i0;
  }
  __syncthreads();
  return result;
}

struct EpiSmem {
  float* val;      // ranking value: confidence, or boosted score for credit decoding
  int* am;         // token committed if the position is chosen (the argmax, or the best
                   // tracked candidate for the tracked-credit variant)
  int* scan1;      // hierarchical: last unmasked index <= i
  int* scan2;      // hierarchical: same on the reversed block
  int* key;        // hierarchical: best (distance, index) key per leaf start
  int* keyi;       // hierarchical, a centre per level: same per internal node, at its cut
  uint8_t* mask;   // masked bits at the start of the step
  uint8_t* sel;    // positions committed in this step
};

__host__ __device__ inline size_t epi_smem_bytes(int L) { return static_cast<size_t>(L) * 26 + 64; }

__device__ EpiSmem carve(uint8_t* dyn, int L) {
  EpiSmem s;
  s.val = reinterpret_cast<float*>(dyn);
  s.am = reinterpret_cast<int*>(dyn + 4 * L);
  s.scan1 = reinterpret_cast<int*>(dyn + 8 * L);
  s.scan2 = reinterpret_cast<int*>(dyn + 12 * L);
  s.key = reinterpret_cast<int*>(dyn + 16 * L);
  s.keyi = reinterpret_cast<int*>(dyn + 20 * L);
  s.mask = dyn + 24 * L;
  s.sel = dyn + 25 * L;
  return s;
}

// Walk position i's path through the halving tree of its run, from the run down to its leaf,
// calling f(key_slot, key) at every node: internal nodes are identified by their cut (keyi),
// leaves by their start (key); key = distance to the node centre * 2048 + i.
template <typename F>
__device__ __forceinline__ void walk_levels(const EpiSmem& sm, int L, int min_width, int i,
                                            F f) {
  int s = sm.scan1[i] + 1;
  const int j = sm.scan2[L - 1 - i];
  int e = (j < 0) ? L : (L - 1 - j);
  for (;;) {
    const int k = abs(2 * i - (s + e - 1)) * 2048 + i;
    if (e - s >= 2 * min_width) {
      const int cut = s + (e - s) / 2;
      f(&sm.keyi[cut], k);
      if (i < cut) e = cut; else s = cut;
    } else {
      f(&sm.key[s], k);
      return;
    }
  }
}

// Probability of token id in row r (tracked-credit variant): exp(z_id - lse_r).
__device__ __forceinline__ float token_prob(const CommitArgs& ca, int64_t r, int id, float lse) {
  const char* row = ca.logits + r * ca.row_stride_bytes;
  const float z = load_logit(row, ca.dtype, id);
  return ex2((z - lse) * kLog2e);
}

// Leaf [s, e) of the recursive halving that contains masked position i (hierarchical decoding).
__device__ __forceinline__ void leaf_of(const EpiSmem& sm, int L, int min_width, int i, int* ls,
                                        int* le) {
  int s = sm.scan1[i] + 1;
  int j = sm.scan2[L - 1 - i];
  int e = (j < 0) ? L : (L - 1 - j);
  while (e - s >= 2 * min_width) {
    const int cut = s + (e - s) / 2;
    if (i < cut) e = cut; else s = cut;
  }
  *ls = s;
  *le = e;
}

// Commit decision for sequence b from sm.val / sm.am / sm.mask; all threads of the CTA.
__device__ void commit_sequence(const CommitCtx& c, int b, bool stopped, const EpiSmem& sm) {
  __shared__ int s_count;
  const int tid = threadIdx.x;
  const int nt = blockDim.x;
  const int L = c.L;
  const dllm_block_state& st = c.state;
  const int64_t r0 = static_cast<int64_t>(b) * L;
  if (stopped) {
    for (int i = tid; i < L; i += nt) st.committed_now[r0 + i] = 0;
    if (tid == 0) st.n_commit[b] = 0;
    return;
  }
  const int mode = c.ca.mode;
  if (mode == kCreditTracked) {
    const int K = c.ca.K;
    for (int i = tid; i < L; i += nt) {
      sm.sel[i] = 0;
      if (!sm.mask[i]) continue;
      const int64_t r = r0 + i;
      int32_t* ids = c.ca.cand_id + r * K;
      float* cr = c.ca.cand_credit + r * K;
      const int a = sm.am[i];
      const float pa = sm.val[i];
      const float lse = __ldcg(c.ca.lse + r);
      int id[kMaxK];
      float cc[kMaxK], pk[kMaxK];
      bool tracked = false;
      for (int k = 0; k < K; ++k) {
        id[k] = ids[k];
        cc[k] = cr[k] * c.ca.decay;
        pk[k] = 0.f;
        if (id[k] >= 0) {
          pk[k] = token_prob(c.ca, r, id[k], lse);
          cc[k] += pk[k];
        }
        if (id[k] == a) tracked = true;
      }
      if (!tracked) {
        int slot = -1;
        for (int k = 0; k < K && slot < 0; ++k)
          if (id[k] == -1) slot = k;
        if (slot < 0) {
          slot = 0;
          for (int k = 1; k < K; ++k)
            if (cc[k] < cc[slot]) slot = k;
        }
        id[slot] = a;
        cc[slot] = pa;
        pk[slot] = token_prob(c.ca, r, a, lse);
      }
      int best = -1;
      float best_s = 0.f;
      for (int k = 0; k < K; ++k) {
        ids[k] = id[k];
        cr[k] = cc[k];
        if (id[k] < 0) continue;
        const float sk = pk[k] * (1.f + c.ca.boost * log1pf(cc[k]));
        if (best < 0 || sk > best_s) {
          best = k;
          best_s = sk;
        }
      }
      sm.val[i] = best_s;
      sm.am[i] = id[best];
      sm.sel[i] = best_s > c.ca.tau ? 1 : 0;
    }
  } else if (mode == kHierarchicalLevels) {
    for (int i = tid; i < L; i += nt) {
      sm.scan1[i] = sm.mask[i] ? -1 : i;
      sm.scan2[i] = sm.mask[L - 1 - i] ? -1 : i;
      sm.key[i] = INT_MAX;
      sm.keyi[i] = INT_MAX;
    }
    __syncthreads();
    block_max_scan(sm.scan1, L);
    block_max_scan(sm.scan2, L);
    const int mw = c.ca.min_width;
    for (int i = tid; i < L; i += nt) {
      if (!sm.mask[i] || !(sm.val[i] >= c.ca.tau_low)) continue;
      walk_levels(sm, L, mw, i, [](int* slot, int k) { atomicMin(slot, k); });
    }
    __syncthreads();
    for (int i = tid; i < L; i += nt) {
      sm.sel[i] = 0;
      if (!sm.mask[i] || !(sm.val[i] >= c.ca.tau_low)) continue;
      int won = 0;
      walk_levels(sm, L, mw, i, [&won](int* slot, int k) { won |= (*slot == k); });
      sm.sel[i] = won ? 1 : 0;
    }
  } else if (mode == kThreshold) {
    for (int i = tid; i < L; i += nt) sm.sel[i] = (sm.mask[i] && sm.val[i] > c.ca.tau) ? 1 : 0;
  } else if (mode == kCredit) {
    const int K = c.ca.K;
    for (int i = tid; i < L; i += nt) {
      sm.sel[i] = 0;
      if (!sm.mask[i]) continue;
      int32_t* ids = c.ca.cand_id + (r0 + i) * K;
      float* cr = c.ca.cand_credit + (r0 + i) * K;
      const int a = sm.am[i];
      const float p = sm.val[i];
      int id[kMaxK];
      float cc[kMaxK];
      int slot = -1;
      for (int k = 0; k < K; ++k) {
        id[k] = ids[k];
        cc[k] = cr[k] * c.ca.decay;
        if (id[k] == a) slot = k;
      }
      if (slot >= 0) {
        cc[slot] += p;
      } else {
        for (int k = 0; k < K && slot < 0; ++k)
          if (id[k] == -1) slot = k;
        if (slot < 0) {
          slot = 0;
          for (int k = 1; k < K; ++k)
            if (cc[k] < cc[slot]) slot = k;
        }
        id[slot] = a;
        cc[slot] = p;
      }
      for (int k = 0; k < K; ++k) {
        ids[k] = id[k];
        cr[k] = cc[k];
      }
      const float score = p * (1.f + c.ca.boost * log1pf(cc[slot]));
      sm.val[i] = score;
      sm.sel[i] = score > c.ca.tau ? 1 : 0;
    }
  } else {  // hierarchical
    for (int i = tid; i < L; i += nt) {
      sm.scan1[i] = sm.mask[i] ? -1 : i;
      sm.scan2[i] = sm.mask[L - 1 - i] ? -1 : i;
      sm.key[i] = INT_MAX;
    }
    __syncthreads();
    block_max_scan(sm.scan1, L);
    block_max_scan(sm.scan2, L);
    const int mw = c.ca.min_width;
    for (int i = tid; i < L; i += nt) {
      if (!sm.mask[i] || !(sm.val[i] >= c.ca.tau_low)) continue;
      int s, e;
      leaf_of(sm, L, mw, i, &s, &e);
      atomicMin(&sm.key[s], abs(2 * i - (s + e - 1)) * 2048 + i);
    }
    __syncthreads();
    for (int i = tid; i < L; i += nt) {
      sm.sel[i] = 0;
      if (!sm.mask[i] || !(sm.val[i] >= c.ca.tau_low)) continue;
      int s, e;
      leaf_of(sm, L, mw, i, &s, &e);
      sm.sel[i] = (sm.key[s] == abs(2 * i - (s + e - 1)) * 2048 + i) ? 1 : 0;
    }
  }
  __syncthreads();
  int any = 0;
  for (int i = tid; i < L; i += nt) any |= sm.sel[i];
  any = __syncthreads_or(any);
  if (!any) {  // at least one commit per step: the best-ranked masked position
    const int best = block_masked_argmax(sm.val, sm.mask, L);
    if (tid == 0 && best >= 0) sm.sel[best] = 1;
    __syncthreads();
  }
  if (tid == 0) s_count = 0;
  __syncthreads();
  int cnt = 0, eos = 0;
  for (int i = tid; i < L; i += nt) {
    const uint8_t sel = sm.sel[i];
    st.committed_now[r0 + i] = sel;
    if (sel) {
      const int t = sm.am[i];
      st.tokens[r0 + i] = t;
      st.masked[r0 + i] = 0;
      ++cnt;
      if (c.ca.eos_id >= 0 && t == c.ca.eos_id) eos = 1;
    }
  }
  if (cnt) atomicAdd(&s_count, cnt);
  eos = __syncthreads_or(eos);
  if (tid == 0) {
    st.n_commit[b] = s_count;
    if (eos) st.eos_hit[b] = 1;
  }
}

// ------------------------------------------------------------------ kernels

__device__ __forceinline__ void write_row_stats(const dllm_stats& st, int64_t r, const RowAcc& a) {
  st.row_max[r] = a.m;
  st.lse[r] = a.m + logf(a.s);
  st.conf[r] = 1.f / a.s;
  st.argmax[r] = a.idx;
}

// One slice of row r (slice sl) reduced by the calling warp; lane 0 stores the result.
template <int DT, bool kScalar>
__device__ __forceinline__ void reduce_item(const FusedParams& p, int64_t r, int sl) {
  const int64_t e0 = static_cast<int64_t>(sl) * p.chunk;
  const int n = static_cast<int>(min(static_cast<int64_t>(p.V), e0 + p.chunk) - e0);
  const char* row = p.logits + r * p.row_stride_bytes;
  const RowAcc a = kScalar ? warp_reduce_slice_scalar<DT>(row, e0, n)
                           : warp_reduce_slice<DT>(row, e0, n);
  if ((threadIdx.x & 31) != 0) return;
  if (p.S == 1) {  // the slice is the whole row
    write_row_stats(p.stats, r, a);
  } else {         // merged by the commit kernel
    p.ws.part[r * p.S + sl] = make_uint4(__float_as_uint(a.m), __float_as_uint(a.s),
                                         static_cast<uint32_t>(a.idx), 0u);
  }
}

__device__ __forceinline__ void write_unread_stats(const dllm_stats& st, int64_t r) {
  st.row_max[r] = -INFINITY;  // rows not read report -inf, -inf, 0, -1
  st.lse[r] = -INFINITY;
  st.conf[r] = 0.f;
  st.argmax[r] = -1;
}

template <int DT, bool kScalar, bool kCompact>
__global__ void __launch_bounds__(kThreads, 4) stats_partials_kernel(FusedParams p) {
  // the block state comes from the kernel before this one (the previous step's commit)
  pdl_wait();
  // let the commit kernel's CTAs become resident while this grid's last waves run (earlier
  // CTAs count as triggered when they exit, so its CTAs do not hold SMs for the whole pass)
  if (static_cast<int>(blockIdx.x) >= p.pdl_from) pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S, L = p.c.L;
  const int64_t W = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
  const int64_t g = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + warp;
  if constexpr (kCompact) {
    extern __shared__ uint16_t act_rows[];  // the rows read, ascending
    __shared__ int warp_cnt[kThreads / 32];
    // Persistent grid over a block of at most kCompactRows rows: every CTA lists the rows read
    // (masked, sequence running) in shared memory, and warp g of the grid reduces slices
    // g, g + W, g + 2W, ... of the rows listed, so the work spreads evenly over the warps
    // however many rows are read (CTA c writes the -inf statistics of the unread rows
    // r = c mod grid).
    // Thread t owns rows [t * per, (t + 1) * per): all its mask bytes (and the stop flags of
    // the sequences they fall in) are loaded at once, then one block-wide scan of the counts
    // places its rows read in the list.
    const int R = p.c.B * L;
    const int per = (R + kThreads - 1) / kThreads;  // <= kCompactRows / kThreads = 16
    const int t0 = static_cast<int>(threadIdx.x) * per;
    uint32_t bits = 0;
#pragma unroll
    for (int k = 0; k < kCompactRows / kThreads; ++k) {
      const int r = t0 + k;
      if (k < per && r < R) {
        const bool a = (p.masked == nullptr || p.masked[r]) &&
                       !(p.eos_hit != nullptr && p.eos_hit[r / L]);
        if (a) bits |= 1u << k;
        else if (r % static_cast<int>(gridDim.x) == static_cast<int>(blockIdx.x))
          write_unread_stats(p.stats, r);
      }
    }
    const int cnt = __popc(bits);
    int incl = cnt;  // inclusive scan of the counts over the warp, then over the warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_cnt[warp] = incl;
    __syncthreads();
    int off = incl - cnt, n_act = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      off += w < warp ? warp_cnt[w] : 0;
      n_act += warp_cnt[w];
    }
    for (uint32_t b = bits; b != 0u; b &= b - 1u)
      act_rows[off++] = static_cast<uint16_t>(t0 + __ffs(b) - 1);
    __syncthreads();  // the list is complete
    const int64_t n_items = static_cast<int64_t>(n_act) * S;
    for (int64_t j = g; j < n_items; j += W) {
      const int64_t k = j / S;
      reduce_item<DT, kScalar>(p, act_rows[k], static_cast<int>(j - k * S));
    }
  } else {
    // One item (row, slice) per warp: the grid covers every item.
    (void)W;
    const int64_t n_items = static_cast<int64_t>(p.c.B) * L * S;
    if (g >= n_items) return;
    const int64_t r = g / S;
    const int sl = static_cast<int>(g - r * S);
    const bool active = (p.masked == nullptr || p.masked[r]) &&
                        !(p.eos_hit != nullptr && p.eos_hit[r / L]);
    if (!active) {  // written once, by slice 0's warp
      if (sl == 0 && lane == 0) write_unread_stats(p.stats, r);
      return;
    }
    reduce_item<DT, kScalar>(p, r, sl);
  }
}

constexpr int kCommitThreads = 512;

// Merge the S slice partials of every row of sequence b that was read into its statistics,
// leaving (mask, confidence, argmax) of each position in shared memory for the commit.  Eight
// threads per row; each loads its share of the row's partials together with the row's mask
// byte (partials of rows that turn out not to be read are loaded and ignored).  The row maximum
// M is taken first (max over the partial maxima, then over the 8 lanes); then every partial
// sum is rescaled once, s_j * exp(m_j - M), independently of the others, and the lowest index
// among the partials whose maximum equals M is the argmax.  Rows not read keep the -inf
// statistics the first kernel wrote.
__device__ void merge_sequence(const CommitOnlyParams& p, int b, const uint8_t* mask_ptr,
                               bool seq_read, const EpiSmem& sm) {
  constexpr int kGroup = 8, kBatch = 8;
  const int L = p.c.L, S = p.S;
  const int q = threadIdx.x & (kGroup - 1);
  for (int i0 = 0; i0 < L; i0 += kCommitThreads / kGroup) {  // uniform trip count: shuffles
    const int i = i0 + static_cast<int>(threadIdx.x) / kGroup;
    const bool in = i < L;
    const int64_t r = static_cast<int64_t>(b) * L + (in ? i : 0);
    const uint8_t mk = in ? (mask_ptr == nullptr ? 1 : mask_ptr[r]) : 0;
    const int64_t base = r * S;
    float M = -INFINITY, sum = 0.f;
    int idx = INT_MAX;
    // trip count uniform across the 8 lanes (the batch maximum is shuffled among them)
    for (int j0 = 0; j0 < S; j0 += kGroup * kBatch) {  // one pass whenever S <= 64
      float m[kBatch], sv[kBatch];
      int ix[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = j0 + q + u * kGroup;
        const bool ok = in && j < S;
        const uint4 v = ok ? __ldcg(p.part + base + j)
                           : make_uint4(__float_as_uint(-INFINITY), 0u, 0xFFFFFFFFu, 0u);
        m[u] = __uint_as_float(v.x);
        sv[u] = __uint_as_float(v.y);
        ix[u] = static_cast<int>(v.z);
      }
      float bm = -INFINITY;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) bm = fmaxf(bm, m[u]);
#pragma unroll
      for (int o = 1; o < kGroup; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, o));
      // fold this batch into the running (M, sum, idx)
      const float nM = fmaxf(M, bm);
      if (nM != -INFINITY) {
        if (nM > M) {  // the maximum rose: rescale the running sum; earlier indices lose
          sum = (M == -INFINITY) ? 0.f : sum * ex2((M - nM) * kLog2e);
          idx = INT_MAX;
        }
        const float nb = nM * kLog2e;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          if (m[u] != -INFINITY) sum = fmaf(sv[u], ex2(fmaf(m[u], kLog2e, -nb)), sum);
          if (m[u] == nM && ix[u] >= 0) idx = min(idx, ix[u]);
        }
        M = nM;
      }
    }
#pragma unroll
    for (int o = 1; o < kGroup; o <<= 1) {
      sum += __shfl_xor_sync(kFull, sum, o);
      idx = min(idx, __shfl_xor_sync(kFull, idx, o));
    }
    if (in && q == 0) {
      const bool read = seq_read && mk;
      const RowAcc t{M, sum, idx == INT_MAX ? -1 : idx};
      if (read) write_row_stats(p.stats, r, t);
      if (sm.val != nullptr) {
        sm.mask[i] = mk;
        sm.val[i] = read ? 1.f / t.s : 0.f;
        sm.am[i] = read ? t.idx : -1;
      }
    }
  }
}

__global__ void __launch_bounds__(kCommitThreads) commit_only_kernel(CommitOnlyParams p) {
  extern __shared__ __align__(1024) uint8_t dyn[];
  // launched after the statistics kernel as a programmatic dependent launch (or plainly):
  // wait until every partial, statistic and read of the block state there is complete
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  const int L = p.c.L;
  const int b = blockIdx.x;
  const bool commit = p.c.ca.mode != kStatsOnly;
  const int64_t r0 = static_cast<int64_t>(b) * L;
  const int32_t* eos_ptr = commit ? p.c.state.eos_hit : p.eos_hit;
  const uint8_t* mask_ptr = commit ? p.c.state.masked : p.masked;
  const bool seq_read = eos_ptr == nullptr || eos_ptr[b] == 0;
  EpiSmem sm = carve(dyn, L);
  if (!commit) sm.val = nullptr;  // statistics only: nothing to stage
  if (p.S > 1) {
    merge_sequence(p, b, mask_ptr, seq_read, sm);
  } else if (commit) {  // statistics already complete: mask and statistics in one round of loads
    for (int i = tid; i < L; i += kCommitThreads) {
      const uint8_t mk = mask_ptr[r0 + i];
      const float cf = __ldcg(p.stats.conf + r0 + i);
      const int am = __ldcg(p.stats.argmax + r0 + i);
      sm.mask[i] = mk;
      sm.val[i] = (mk && seq_read) ? cf : 0.f;
      sm.am[i] = am;
    }
  }
  if (!commit) return;
  int any_masked = 0;
  __syncthreads();
  for (int i = tid; i < L; i += kCommitThreads) any_masked |= sm.mask[i];
  any_masked = __syncthreads_or(any_masked);
  const bool stopped = !seq_read || !any_masked;
  commit_sequence(p.c, b, stopped, sm);
}

// Vocabulary-sharded statistics: one thread per row folds the n shards' (m, lse, argmax).
struct ShardParams {
  dllm_shard_stats sh[DLLM_MAX_SHARDS];
  int n;
  int64_t rows;
  dllm_stats out;
};

__global__ void __launch_bounds__(256) merge_shards_kernel(const __grid_constant__ ShardParams p) {
  pdl_wait();
  pdl_trigger();
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= p.rows) return;
  float m = -INFINITY;
  for (int k = 0; k < p.n; ++k) m = fmaxf(m, p.sh[k].stats.row_max[r]);
  if (m == -INFINITY) {
    p.out.row_max[r] = -INFINITY;
    p.out.lse[r] = -INFINITY;
    p.out.conf[r] = 0.f;
    p.out.argmax[r] = -1;
    return;
  }
  float s = 0.f;
  int64_t am = INT64_MAX;
  const float mb = m * kLog2e;
  for (int k = 0; k < p.n; ++k) {
    const float mk = p.sh[k].stats.row_max[r];
    if (mk == -INFINITY) continue;
    s += ex2(fmaf(p.sh[k].stats.lse[r], kLog2e, -mb));
    if (mk == m) am = min(am, p.sh[k].vocab_offset + p.sh[k].stats.argmax[r]);
  }
  p.out.row_max[r] = m;
  p.out.lse[r] = m + logf(s);
  p.out.conf[r] = 1.f / s;
  p.out.argmax[r] = static_cast<int32_t>(am);
}

// One 4 KB warp slice per item.
void choose_split(int V, int dtype, int* S_out, int* chunk_out) {
  const int chunk = dtype == DLLM_BF16 ? slice_elems<DLLM_BF16>() : slice_elems<DLLM_F32>();
  *S_out = (V + chunk - 1) / chunk;
  *chunk_out = chunk;
}

}  // namespace

// Upper bound of the slices per row over both dtypes (fp32 slices hold 1024 elements).
int max_splits(int V) { return std::max(1, (V + 1023) / 1024); }

size_t stats_ws_bytes(int B, int L, int V) {
  const size_t parts = static_cast<size_t>(B) * L * max_splits(V);
  return kWsHeader + align_up(16 * parts, 256);
}

StatsWs stats_ws_layout(void* ws, int B, int L, int V) {
  char* p = static_cast<char*>(ws);
  const size_t parts = static_cast<size_t>(B) * L * max_splits(V);
  StatsWs w;
  w.status = reinterpret_cast<int32_t*>(p);
  p += kWsHeader;
  w.part = reinterpret_cast<uint4*>(p);
  (void)parts;
  return w;
}

cudaError_t launch_stats_commit(const void* logits, const dllm_shape& sh, const uint8_t* masked,
                                const dllm_stats& stats, const dllm_block_state* state,
                                const CommitArgs& ca, const StatsWs& ws, int sm_count,
                                cudaStream_t stream) {
  FusedParams p{};
  const int R = sh.B * sh.L;
  const int es = sh.dtype == DLLM_BF16 ? 2 : 4;
  p.logits = static_cast<const char*>(logits);
  p.row_stride_bytes = sh.row_stride * es;
  p.V = sh.V;
  choose_split(sh.V, sh.dtype, &p.S, &p.chunk);
  p.stats = stats;
  p.ws = ws;
  p.c.B = sh.B;
  p.c.L = sh.L;
  p.c.ca = ca;
  p.c.ca.logits = static_cast<const char*>(logits);
  p.c.ca.row_stride_bytes = p.row_stride_bytes;
  p.c.ca.dtype = sh.dtype;
  p.c.ca.lse = stats.lse;
  if (ca.mode == kStatsOnly) {
    p.masked = masked;
    p.eos_hit = nullptr;
  } else {
    p.c.state = *state;
    p.masked = state->masked;
    p.eos_hit = state->eos_hit;
  }
  const int64_t items = static_cast<int64_t>(R) * p.S;
  const int64_t ctas = (items + kThreads / 32 - 1) / (kThreads / 32);
  // Blocks of up to kCompactRows rows that need more than two waves of CTAs run as a persistent
  // grid (as many CTAs as fit at once) over the rows actually read; otherwise one warp per item
  // (with two waves or fewer there are few CTAs to launch, and the list costs ~1 us).
  const int64_t resident = static_cast<int64_t>(kStatsCtasPerSm) * std::max(1, sm_count);
  p.compact = R <= kCompactRows && ctas > 2 * resident;
  const dim3 grid1(static_cast<unsigned>(p.compact ? resident : ctas));
  const size_t smem1 = p.compact ? sizeof(uint16_t) * static_cast<size_t>(R) : 0;
  p.pdl_from = std::max(0, static_cast<int>(grid1.x) - 2 * 4 * std::max(1, sm_count));
  // rows that are not all 16-byte aligned take the scalar-load reduction
  const bool scalar = (reinterpret_cast<uintptr_t>(logits) % 16) != 0 || p.row_stride_bytes % 16 != 0;
  cudaError_t e;
  const dim3 blk(kThreads);
  if (sh.dtype == DLLM_BF16) {
    if (p.compact)
      e = scalar ? launch_dependent(stats_partials_kernel<DLLM_BF16, true, true>, grid1, blk,
                                    smem1, stream, p)
                 : launch_dependent(stats_partials_kernel<DLLM_BF16, false, true>, grid1, blk,
                                    smem1, stream, p);
    else
      e = scalar ? launch_dependent(stats_partials_kernel<DLLM_BF16, true, false>, grid1, blk, 0,
                                    stream, p)
                 : launch_dependent(stats_partials_kernel<DLLM_BF16, false, false>, grid1, blk, 0,
                                    stream, p);
  } else {
    if (p.compact)
      e = scalar ? launch_dependent(stats_partials_kernel<DLLM_F32, true, true>, grid1, blk,
                                    smem1, stream, p)
                 : launch_dependent(stats_partials_kernel<DLLM_F32, false, true>, grid1, blk,
                                    smem1, stream, p);
    else
      e = scalar ? launch_dependent(stats_partials_kernel<DLLM_F32, true, false>, grid1, blk, 0,
                                    stream, p)
                 : launch_dependent(stats_partials_kernel<DLLM_F32, false, false>, grid1, blk, 0,
                                    stream, p);
  }
  if (e != cudaSuccess) return e;
  if (ca.mode == kStatsOnly && p.S == 1) return cudaSuccess;
  // the merge (+ commit) kernel, one CTA per sequence, as a programmatic dependent launch
  CommitOnlyParams cp{};
  cp.stats = stats;
  cp.c = p.c;
  cp.S = p.S;
  cp.part = ws.part;
  cp.masked = p.masked;
  cp.eos_hit = p.eos_hit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sh.B);
  cfg.blockDim = dim3(kCommitThreads);
  cfg.dynamicSmemBytes = epi_smem_bytes(sh.L);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, commit_only_kernel, cp);
}

cudaError_t launch_merge_shard_stats(const dllm_shard_stats* shards, int n, int64_t rows,
                                     const dllm_stats& out, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  ShardParams p{};
  for (int k = 0; k < n; ++k) p.sh[k] = shards[k];
  p.n = n;
  p.rows = rows;
  p.out = out;
  return launch_dependent(merge_shards_kernel, dim3(static_cast<unsigned>((rows + 255) / 256)),
                          dim3(256), 0, stream, p);
}

cudaError_t launch_commit_only(const dllm_shape& sh, const dllm_stats& stats,
                               const dllm_block_state& state, const CommitArgs& ca,
                               cudaStream_t stream) {
  CommitOnlyParams p{};
  p.stats = stats;
  p.c.B = sh.B;
  p.c.L = sh.L;
  p.c.state = state;
  p.c.ca = ca;
  p.S = 1;  // statistics already complete: commit only
  return launch_dependent(commit_only_kernel, dim3(sh.B), dim3(kCommitThreads),
                          epi_smem_bytes(sh.L), stream, p);
}

}  // namespace dllm
