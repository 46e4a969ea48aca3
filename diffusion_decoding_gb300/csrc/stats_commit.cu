// Fused softmax statistics + commit decision over one masked block (kernel "a").
//
// Every masked row of logits is streamed from HBM exactly once.  A row is cut into S vocabulary
// slices; each CTA reduces one slice to a partial (max, rescaled sum, argmax) with 128-bit loads
// and warp-shuffle merges, writes it to the workspace and bumps its sequence's counter.  The CTA
// that arrives last for a sequence merges the L*S partials of that sequence into the row
// statistics and runs the commit decision in shared memory (threshold, hierarchical or credit
// decoding; dInfer explainer, decoding-strategy component, methods 1-3), then re-arms the
// counter.  Nothing waits on another CTA: the last arriver is found with one atomic.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace dllm {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;

struct CommitCtx {
  int B, L;
  dllm_block_state state;
  CommitArgs ca;
};

struct FusedParams {
  const char* logits;
  int64_t row_stride_bytes;
  int V, S, chunk, vec;
  const uint8_t* masked;   // rows to read (state.masked when committing)
  const int32_t* eos_hit;  // null in statistics-only mode
  dllm_stats stats;
  StatsWs ws;
  CommitCtx c;
};

struct CommitOnlyParams {
  dllm_stats stats;
  CommitCtx c;
};

// ------------------------------------------------------------------ per-thread streaming

template <int N>
__device__ __forceinline__ void acc_elems(RowAcc& a, const float* x, int base) {
  float vm = x[0];
#pragma unroll
  for (int j = 1; j < N; ++j) vm = fmaxf(vm, x[j]);
  if (vm > a.m) {  // new running maximum: rescale the sum once, remember the first index
    int j0 = 0;
#pragma unroll
    for (int j = N - 1; j >= 0; --j)
      if (x[j] == vm) j0 = j;
    a.s = a.s * ex2((a.m - vm) * kLog2e);
    a.m = vm;
    a.idx = base + j0;
  }
  const float mb = (a.m == -INFINITY) ? 0.f : a.m * kLog2e;
#pragma unroll
  for (int j = 0; j < N; ++j) a.s += ex2(fmaf(x[j], kLog2e, -mb));
}

template <int DT>
__device__ __forceinline__ void unpack16(const uint4& q, float* x) {
  if constexpr (DT == DLLM_BF16) {
    x[0] = bf16lo(q.x); x[1] = bf16hi(q.x);
    x[2] = bf16lo(q.y); x[3] = bf16hi(q.y);
    x[4] = bf16lo(q.z); x[5] = bf16hi(q.z);
    x[6] = bf16lo(q.w); x[7] = bf16hi(q.w);
  } else {
    x[0] = __uint_as_float(q.x); x[1] = __uint_as_float(q.y);
    x[2] = __uint_as_float(q.z); x[3] = __uint_as_float(q.w);
  }
}

// Reduce elements [e0, e1) of one row into this thread's accumulator.  Each thread visits its
// elements in increasing index order, so a strict '>' keeps the lowest index of the maximum.
template <int DT>
__device__ __forceinline__ void stream_slice(const char* row, int64_t e0, int64_t e1, int vec,
                                             RowAcc& acc) {
  constexpr int VEC = DT == DLLM_BF16 ? 8 : 4;
  constexpr int ES = DT == DLLM_BF16 ? 2 : 4;
  const int tid = threadIdx.x;
  int64_t tail = e0;
  if (vec) {
    const int nvec = static_cast<int>((e1 - e0) / VEC);
    const char* base = row + e0 * ES;
    for (int v0 = 0; v0 < nvec; v0 += kThreads * kUnroll) {
      uint4 q[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int vi = v0 + u * kThreads + tid;
        if (vi < nvec) q[u] = ld_stream_v4(base + static_cast<int64_t>(vi) * 16);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int vi = v0 + u * kThreads + tid;
        if (vi < nvec) {
          float x[VEC];
          unpack16<DT>(q[u], x);
          acc_elems<VEC>(acc, x, static_cast<int>(e0) + vi * VEC);
        }
      }
    }
    tail = e0 + static_cast<int64_t>(nvec) * VEC;
  }
  for (int64_t e = tail + tid; e < e1; e += kThreads) {
    float x[1] = {load_logit(row, DT, e)};
    acc_elems<1>(acc, x, static_cast<int>(e));
  }
}

// ------------------------------------------------------------------ block helpers

// In-place inclusive max-scan of a[0..n) (values >= -1) with warp shuffles; ends synchronised.
__device__ void block_max_scan(int* a, int n) {
  __shared__ int warp_tot[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ipt = (n + kThreads - 1) / kThreads;
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
  __shared__ float wv[kWarps];
  __shared__ int wi[kWarps];
  __shared__ int result;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float best = -INFINITY;
  int bi = INT_MAX;
  for (int i = tid; i < L; i += kThreads) {
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
    for (int w = 1; w < kWarps; ++w) {
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
  int* am;         // argmax token of each position
  int* scan1;      // hierarchical: last unmasked index <= i
  int* scan2;      // hierarchical: same on the reversed block
  int* key;        // hierarchical: best (distance, index) key per leaf start
  uint8_t* mask;   // masked bits at the start of the step
  uint8_t* sel;    // positions committed in this step
};

__host__ __device__ inline size_t epi_smem_bytes(int L) { return static_cast<size_t>(L) * 22 + 64; }

__device__ EpiSmem carve(uint8_t* dyn, int L) {
  EpiSmem s;
  s.val = reinterpret_cast<float*>(dyn);
  s.am = reinterpret_cast<int*>(dyn + 4 * L);
  s.scan1 = reinterpret_cast<int*>(dyn + 8 * L);
  s.scan2 = reinterpret_cast<int*>(dyn + 12 * L);
  s.key = reinterpret_cast<int*>(dyn + 16 * L);
  s.mask = dyn + 20 * L;
  s.sel = dyn + 21 * L;
  return s;
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
  const int L = c.L;
  const dllm_block_state& st = c.state;
  const int64_t r0 = static_cast<int64_t>(b) * L;
  if (stopped) {
    for (int i = tid; i < L; i += kThreads) st.committed_now[r0 + i] = 0;
    if (tid == 0) st.n_commit[b] = 0;
    return;
  }
  const int mode = c.ca.mode;
  if (mode == kThreshold) {
    for (int i = tid; i < L; i += kThreads) sm.sel[i] = (sm.mask[i] && sm.val[i] > c.ca.tau) ? 1 : 0;
  } else if (mode == kCredit) {
    const int K = c.ca.K;
    for (int i = tid; i < L; i += kThreads) {
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
    for (int i = tid; i < L; i += kThreads) {
      sm.scan1[i] = sm.mask[i] ? -1 : i;
      sm.scan2[i] = sm.mask[L - 1 - i] ? -1 : i;
      sm.key[i] = INT_MAX;
    }
    __syncthreads();
    block_max_scan(sm.scan1, L);
    block_max_scan(sm.scan2, L);
    const int mw = c.ca.min_width;
    for (int i = tid; i < L; i += kThreads) {
      if (!sm.mask[i] || !(sm.val[i] >= c.ca.tau_low)) continue;
      int s, e;
      leaf_of(sm, L, mw, i, &s, &e);
      atomicMin(&sm.key[s], abs(2 * i - (s + e - 1)) * 2048 + i);
    }
    __syncthreads();
    for (int i = tid; i < L; i += kThreads) {
      sm.sel[i] = 0;
      if (!sm.mask[i] || !(sm.val[i] >= c.ca.tau_low)) continue;
      int s, e;
      leaf_of(sm, L, mw, i, &s, &e);
      sm.sel[i] = (sm.key[s] == abs(2 * i - (s + e - 1)) * 2048 + i) ? 1 : 0;
    }
  }
  __syncthreads();
  int any = 0;
  for (int i = tid; i < L; i += kThreads) any |= sm.sel[i];
  any = __syncthreads_or(any);
  if (!any) {  // at least one commit per step: the best-ranked masked position
    const int best = block_masked_argmax(sm.val, sm.mask, L);
    if (tid == 0 && best >= 0) sm.sel[best] = 1;
    __syncthreads();
  }
  if (tid == 0) s_count = 0;
  __syncthreads();
  int cnt = 0, eos = 0;
  for (int i = tid; i < L; i += kThreads) {
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

template <int DT>
__global__ void __launch_bounds__(kThreads) stats_commit_kernel(FusedParams p) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ RowAcc warp_acc[kWarps];
  __shared__ int s_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = p.c.L;
  const int r = blockIdx.x / p.S;
  const int split = blockIdx.x - r * p.S;
  const int b = r / L;

  const bool active = (p.masked == nullptr || p.masked[r]) &&
                      !(p.eos_hit != nullptr && p.eos_hit[b]);
  RowAcc acc = row_acc_empty();
  if (active) {
    const int64_t e0 = static_cast<int64_t>(split) * p.chunk;
    const int64_t e1 = min(static_cast<int64_t>(p.V), e0 + p.chunk);
    stream_slice<DT>(p.logits + static_cast<int64_t>(r) * p.row_stride_bytes, e0, e1, p.vec,
                     acc);
  }
  acc = row_acc_warp_reduce(acc);
  if (lane == 0) warp_acc[warp] = acc;
  __syncthreads();
  if (warp == 0) {
    RowAcc a = lane < kWarps ? warp_acc[lane] : row_acc_empty();
    a = row_acc_warp_reduce(a);
    if (lane == 0) {
      const int64_t pi = static_cast<int64_t>(r) * p.S + split;
      p.ws.part_m[pi] = a.m;
      p.ws.part_s[pi] = a.s;
      p.ws.part_i[pi] = a.idx;
      __threadfence();
      const int prev = atomicAdd(&p.ws.counters[b], 1);
      s_last = (prev == L * p.S - 1);
    }
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last CTA of sequence b: merge the partials, then decide the commits
  const EpiSmem sm = carve(dyn, L);
  const bool committing = p.c.ca.mode != kStatsOnly;
  int any_masked = 0;
  for (int i = tid; i < L; i += kThreads) {
    const uint8_t m = p.masked ? p.masked[static_cast<int64_t>(b) * L + i] : 1;
    sm.mask[i] = m;
    any_masked |= m;
  }
  any_masked = __syncthreads_or(any_masked);
  const bool stopped = committing && ((p.eos_hit && p.eos_hit[b]) || !any_masked);
  const int S = p.S;
  for (int i = warp; i < L; i += kWarps) {
    const int64_t row = static_cast<int64_t>(b) * L + i;
    const bool act = sm.mask[i] && !stopped;
    RowAcc a = row_acc_empty();
    if (act) {
      for (int j = lane; j < S; j += 32) {
        const int64_t pi = row * S + j;
        RowAcc q{__ldcg(p.ws.part_m + pi), __ldcg(p.ws.part_s + pi), __ldcg(p.ws.part_i + pi)};
        a = row_acc_merge(a, q);
      }
    }
    a = row_acc_warp_reduce(a);
    if (lane == 0) {
      float rm = -INFINITY, l = -INFINITY, cf = 0.f;
      int am = -1;
      if (act) {
        rm = a.m;
        l = a.m + logf(a.s);
        cf = 1.f / a.s;
        am = a.idx;
      }
      p.stats.row_max[row] = rm;
      p.stats.lse[row] = l;
      p.stats.conf[row] = cf;
      p.stats.argmax[row] = am;
      sm.val[i] = cf;
      sm.am[i] = am;
    }
  }
  __syncthreads();
  if (committing) commit_sequence(p.c, b, stopped, sm);
  if (tid == 0) p.ws.counters[b] = 0;  // re-arm for the next launch on this workspace
}

__global__ void __launch_bounds__(kThreads) commit_only_kernel(CommitOnlyParams p) {
  extern __shared__ __align__(16) uint8_t dyn[];
  const int tid = threadIdx.x;
  const int L = p.c.L;
  const int b = blockIdx.x;
  const EpiSmem sm = carve(dyn, L);
  const int64_t r0 = static_cast<int64_t>(b) * L;
  int any_masked = 0;
  for (int i = tid; i < L; i += kThreads) {
    const uint8_t m = p.c.state.masked[r0 + i];
    sm.mask[i] = m;
    any_masked |= m;
  }
  any_masked = __syncthreads_or(any_masked);
  const bool stopped = p.c.state.eos_hit[b] != 0 || !any_masked;
  for (int i = tid; i < L; i += kThreads) {
    sm.val[i] = (sm.mask[i] && !stopped) ? p.stats.conf[r0 + i] : 0.f;
    sm.am[i] = p.stats.argmax[r0 + i];
  }
  __syncthreads();
  commit_sequence(p.c, b, stopped, sm);
}

void choose_split(int R, int V, int dtype, int sm_count, int* S_out, int* chunk_out) {
  const int target = dtype == DLLM_BF16 ? 16384 : 8192;  // 32 KB per CTA
  const int smax = max_splits(V);
  int S = std::max(1, (V + target - 1) / target);
  // keep at least ~8 CTAs per SM in flight when there are few rows
  while (static_cast<int64_t>(R) * S < static_cast<int64_t>(sm_count) * 8 && S * 2 <= smax &&
         V / (S * 2) >= kMinChunk)
    S *= 2;
  S = std::min(S, smax);
  int chunk = static_cast<int>(align_up((V + S - 1) / S, 8));
  S = (V + chunk - 1) / chunk;
  *S_out = S;
  *chunk_out = chunk;
}

}  // namespace

int max_splits(int V) { return std::max(1, std::min(kMaxSplits, (V + kMinChunk - 1) / kMinChunk)); }

size_t stats_ws_bytes(int B, int L, int V) {
  const size_t R = static_cast<size_t>(B) * L;
  const size_t parts = R * max_splits(V);
  return kWsHeader + align_up(sizeof(int32_t) * B, 256) + 3 * align_up(4 * parts, 256);
}

StatsWs stats_ws_layout(void* ws, int B, int L, int V) {
  char* p = static_cast<char*>(ws);
  const size_t parts = static_cast<size_t>(B) * L * max_splits(V);
  StatsWs w;
  w.status = reinterpret_cast<int32_t*>(p);
  p += kWsHeader;
  w.counters = reinterpret_cast<int32_t*>(p);
  p += align_up(sizeof(int32_t) * B, 256);
  w.part_m = reinterpret_cast<float*>(p);
  p += align_up(4 * parts, 256);
  w.part_s = reinterpret_cast<float*>(p);
  p += align_up(4 * parts, 256);
  w.part_i = reinterpret_cast<int32_t*>(p);
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
  choose_split(R, sh.V, sh.dtype, sm_count, &p.S, &p.chunk);
  p.vec = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) && (p.row_stride_bytes % 16 == 0);
  p.stats = stats;
  p.ws = ws;
  p.c.B = sh.B;
  p.c.L = sh.L;
  p.c.ca = ca;
  if (ca.mode == kStatsOnly) {
    p.masked = masked;
    p.eos_hit = nullptr;
  } else {
    p.c.state = *state;
    p.masked = state->masked;
    p.eos_hit = state->eos_hit;
  }
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(R) * p.S));
  const size_t smem = epi_smem_bytes(sh.L);
  if (sh.dtype == DLLM_BF16)
    stats_commit_kernel<DLLM_BF16><<<grid, kThreads, smem, stream>>>(p);
  else
    stats_commit_kernel<DLLM_F32><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
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
  commit_only_kernel<<<sh.B, kThreads, epi_smem_bytes(sh.L), stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dllm
