// Warp-scan and block-state kernels (kernel "c"): compaction of the rows kept for iteration
// smoothing (and, for the single-read step, of the rows read before the commit and the map from
// them to the kept rows), the neighbourhood KV-refresh mask with its ascending index list, the
// reset of the decode state for a new block, and the device-side test that ends a decode loop
// captured as a CUDA graph.
//
// All are tiny (at most B*L flags, or P + L cache positions per sequence) and latency-bound; they
// use warp ballots and shuffle prefix sums, never a global barrier.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace dllm {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kRefreshThreads = 256;

// Exclusive prefix count of `flag` over the CTA (threads in order); returns this thread's
// offset and writes the CTA total to *total.  Ends synchronised.
template <int NT>
__device__ int block_exclusive_count(int flag, int* total) {
  __shared__ int warp_cnt[NT / 32];
  __shared__ int s_total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned bal = __ballot_sync(kFull, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) warp_cnt[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    int v = lane < NT / 32 ? warp_cnt[lane] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane < NT / 32) warp_cnt[lane] = incl - v;  // exclusive
    if (lane == 31) s_total = incl;
  }
  __syncthreads();
  const int off = warp_cnt[warp] + in_warp;
  *total = s_total;
  __syncthreads();
  return off;
}

__global__ void __launch_bounds__(kScanThreads) compact_rows_kernel(const uint8_t* masked,
                                                                    const int32_t* eos_hit,
                                                                    int B, int L, int32_t* row_ids,
                                                                    int32_t* M) {
  pdl_wait();
  pdl_trigger();
  const int R = B * L;
  int base = 0;
  for (int r0 = 0; r0 < R; r0 += kScanThreads) {
    const int r = r0 + threadIdx.x;
    const int keep = (r < R) && masked[r] && !eos_hit[r / L];
    int total;
    const int off = block_exclusive_count<kScanThreads>(keep, &total);
    if (keep) row_ids[base + off] = r;
    base += total;
  }
  for (int k = base + threadIdx.x; k < R; k += kScanThreads) row_ids[k] = -1;
  if (threadIdx.x == 0) *M = base;
}

// Rows a step reads (masked, sequence running), ascending: the single-read smoothing path's row
// list, taken before the commit.  Rows not read get the -inf, -inf, 0, -1 statistics here.
__global__ void __launch_bounds__(kScanThreads) read_rows_kernel(const uint8_t* masked,
                                                                 const int32_t* eos_hit, int B,
                                                                 int L, int32_t* rows,
                                                                 int32_t* count, dllm_stats st) {
  pdl_wait();
  pdl_trigger();
  const int R = B * L;
  int base = 0;
  for (int r0 = 0; r0 < R; r0 += kScanThreads) {
    const int r = r0 + threadIdx.x;
    const int read = (r < R) && masked[r] && !eos_hit[r / L];
    int total;
    const int off = block_exclusive_count<kScanThreads>(read, &total);
    if (read) {
      rows[base + off] = r;
    } else if (r < R) {
      st.row_max[r] = -INFINITY;
      st.lse[r] = -INFINITY;
      st.conf[r] = 0.f;
      st.argmax[r] = -1;
    }
    base += total;
  }
  if (threadIdx.x == 0) *count = base;
}

// After the commit: the rows kept for smoothing (row_ids, M, as compact_rows_kernel) and, for
// each row read this step (rows_read[0..count_read)), its index among the kept rows or -1 if it
// was just committed (map), through inv[r] = kept index of row r or -1.
__global__ void __launch_bounds__(kScanThreads) kept_rows_map_kernel(
    const uint8_t* masked, const int32_t* eos_hit, int B, int L, int32_t* row_ids, int32_t* M,
    const int32_t* rows_read, const int32_t* count_read, int32_t* inv, int32_t* map) {
  // The GEMM after this kernel reads only P and the row count (final once the commit kernel
  // before this one started: that kernel waits for the statistics grid before it lets this one
  // launch) until its epilogue, which waits for this grid; so it may launch at once and run its
  // mainloop while the commit kernel and this one finish.
  pdl_trigger();
  pdl_wait();  // the commit's block state
  const int R = B * L;
  int base = 0;
  for (int r0 = 0; r0 < R; r0 += kScanThreads) {
    const int r = r0 + threadIdx.x;
    const int keep = (r < R) && masked[r] && !eos_hit[r / L];
    int total;
    const int off = block_exclusive_count<kScanThreads>(keep, &total);
    if (keep) row_ids[base + off] = r;
    if (r < R) inv[r] = keep ? base + off : -1;
    base += total;
  }
  for (int k = base + threadIdx.x; k < R; k += kScanThreads) row_ids[k] = -1;
  if (threadIdx.x == 0) *M = base;
  __syncthreads();  // inv is complete (global writes of this CTA are visible to it)
  const int n = *count_read;
  for (int c = threadIdx.x; c < n; c += kScanThreads) map[c] = __ldcg(inv + rows_read[c]);
}

// One CTA per sequence.  cnt[x] = number of block positions < x committed in this step; cache
// position j is refreshed iff a committed block position lies in [j-P-w, j-P+w].
__global__ void __launch_bounds__(kRefreshThreads) kv_refresh_kernel(const uint8_t* committed_now,
                                                                     int L, int P, int w,
                                                                     uint8_t* refresh,
                                                                     int32_t* idx,
                                                                     int32_t* count) {
  extern __shared__ int cnt[];  // [L + 1]
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const int T = P + L;
  const uint8_t* com = committed_now + static_cast<int64_t>(b) * L;
  // inclusive prefix count of committed positions, chunk by chunk
  if (threadIdx.x == 0) cnt[0] = 0;
  int base = 0;
  for (int i0 = 0; i0 < L; i0 += kRefreshThreads) {
    const int i = i0 + threadIdx.x;
    const int f = (i < L) && com[i];
    int total;
    const int off = block_exclusive_count<kRefreshThreads>(f, &total);
    if (i < L) cnt[i + 1] = base + off + f;
    base += total;
  }
  __syncthreads();
  uint8_t* ref = refresh + static_cast<int64_t>(b) * T;
  int32_t* ix = idx + static_cast<int64_t>(b) * T;
  int out = 0;
  for (int j0 = 0; j0 < T; j0 += kRefreshThreads) {
    const int j = j0 + threadIdx.x;
    int hit = 0;
    if (j < T) {
      const int lo = max(0, j - P - w);
      const int hi = min(L - 1, j - P + w);
      hit = (lo <= hi) && (cnt[hi + 1] - cnt[lo] > 0);
      ref[j] = static_cast<uint8_t>(hit);
    }
    int total;
    const int off = block_exclusive_count<kRefreshThreads>(hit, &total);
    if (hit) ix[out + off] = j;
    out += total;
  }
  for (int k = out + threadIdx.x; k < T; k += kRefreshThreads) ix[k] = -1;
  if (threadIdx.x == 0) count[b] = out;
}

}  // namespace

cudaError_t launch_compact_rows(const dllm_block_state& state, int B, int L, int32_t* row_ids,
                                int32_t* M, cudaStream_t stream) {
  return launch_dependent(compact_rows_kernel, dim3(1), dim3(kScanThreads), 0, stream,
                          state.masked, state.eos_hit, B, L, row_ids, M);
}

cudaError_t launch_read_rows(const dllm_block_state& state, int B, int L, int32_t* rows,
                             int32_t* count, const dllm_stats& stats, cudaStream_t stream) {
  return launch_dependent(read_rows_kernel, dim3(1), dim3(kScanThreads), 0, stream, state.masked,
                          state.eos_hit, B, L, rows, count, stats);
}

cudaError_t launch_kept_rows_map(const dllm_block_state& state, int B, int L, int32_t* row_ids,
                                 int32_t* M, const int32_t* rows_read, const int32_t* count_read,
                                 int32_t* inv, int32_t* map, cudaStream_t stream) {
  return launch_dependent(kept_rows_map_kernel, dim3(1), dim3(kScanThreads), 0, stream,
                          state.masked, state.eos_hit, B, L, row_ids, M, rows_read, count_read,
                          inv, map);
}

// A new block: n = B*L positions masked with no token and nothing committed this step, B
// sequences with no commit counted and no stop; nk = B*L*K credit slots empty with zero credit.
__global__ void __launch_bounds__(256) block_state_reset_kernel(dllm_block_state st, int64_t n,
                                                                int B, int32_t* cand_id,
                                                                float* cand_credit, int64_t nk) {
  pdl_wait();  // the calls before this one may still read the state
  pdl_trigger();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t end = max(n, nk);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < end;
       i += stride) {
    if (i < n) {
      st.masked[i] = 1;
      st.tokens[i] = -1;
      st.committed_now[i] = 0;
    }
    if (i < B) {
      st.n_commit[i] = 0;
      st.eos_hit[i] = 0;
    }
    if (i < nk) {
      if (cand_id != nullptr) cand_id[i] = -1;
      if (cand_credit != nullptr) cand_credit[i] = 0.f;
    }
  }
}

cudaError_t launch_block_state_reset(const dllm_block_state& state, int64_t n, int B,
                                     int32_t* cand_id, float* cand_credit, int64_t nk,
                                     cudaStream_t stream) {
  const int64_t end = std::max(n, nk);
  const unsigned blocks = static_cast<unsigned>(std::min<int64_t>(1024, (end + 255) / 256));
  return launch_dependent(block_state_reset_kernel, dim3(std::max(1u, blocks)), dim3(256), 0,
                          stream, state, n, B, cand_id, cand_credit, nk);
}

// Whether the block still decodes: some sequence has a masked position and no EOS.  One CTA
// (the condition is set exactly once, by thread 0); 16 mask bytes per load where aligned.
__global__ void __launch_bounds__(1024) loop_continue_kernel(const uint8_t* masked,
                                                             const int32_t* eos_hit, int B, int L,
                                                             cudaGraphConditionalHandle handle) {
  pdl_wait();  // the commit before this one writes the state
  pdl_trigger();
  int running = 0;
  const bool vec = (L % 16) == 0 && (reinterpret_cast<uintptr_t>(masked) % 16) == 0;
  if (vec) {  // 16 positions of one sequence per load
    const int per = L / 16;
    const int64_t nv = static_cast<int64_t>(B) * per;
    const uint4* m4 = reinterpret_cast<const uint4*>(masked);
    for (int64_t v = threadIdx.x; v < nv && !running; v += blockDim.x) {
      const uint4 q = m4[v];
      if ((q.x | q.y | q.z | q.w) != 0u && eos_hit[v / per] == 0) running = 1;
    }
  } else {
    const int64_t n = static_cast<int64_t>(B) * L;
    for (int64_t i = threadIdx.x; i < n && !running; i += blockDim.x)
      if (masked[i] && eos_hit[i / L] == 0) running = 1;
  }
  running = __syncthreads_or(running);
  if (threadIdx.x == 0) cudaGraphSetConditional(handle, running ? 1u : 0u);
}

cudaError_t launch_loop_continue(const dllm_block_state& state, int B, int L,
                                 cudaGraphConditionalHandle handle, cudaStream_t stream) {
  return launch_dependent(loop_continue_kernel, dim3(1), dim3(1024), 0, stream, state.masked,
                          state.eos_hit, B, L, handle);
}

cudaError_t launch_kv_refresh(const dllm_block_state& state, int B, int L, int prefix_len,
                              int window, uint8_t* refresh, int32_t* idx, int32_t* count,
                              cudaStream_t stream) {
  const size_t smem = sizeof(int) * (static_cast<size_t>(L) + 1);
  return launch_dependent(kv_refresh_kernel, dim3(B), dim3(kRefreshThreads), smem, stream,
                          state.committed_now, L, prefix_len, window, refresh, idx, count);
}

}  // namespace dllm
