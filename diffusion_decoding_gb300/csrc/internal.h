// Host-side launch interfaces between the C ABI (abi.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dllm.h"

namespace dllm {

constexpr int kMaxL = 1024;
constexpr int kMaxK = 16;

enum CommitMode {
  kStatsOnly = 0,
  kThreshold = 1,
  kHierarchical = 2,
  kCredit = 3,
  kHierarchicalLevels = 4,  // variant: a centre per level of the halving tree
  kCreditTracked = 5,       // variant: every tracked candidate gains its own probability
};

struct CommitArgs {
  int mode;
  float tau;
  float tau_low;
  int min_width;
  int eos_id;
  int32_t* cand_id;
  float* cand_credit;
  int K;
  float decay;
  float boost;
  // kCreditTracked reads the logits of the tracked tokens (set by the launcher)
  const char* logits;
  int64_t row_stride_bytes;
  int dtype;
  const float* lse;
};

// Stats/commit workspace layout.
struct StatsWs {
  int32_t* status;
  uint4* part;        // [R * S_max] one {max, sum, argmax, 0} record (16 bytes) per slice
};

int max_splits(int V);
size_t stats_ws_bytes(int B, int L, int V);
StatsWs stats_ws_layout(void* ws, int B, int L, int V);

// Streaming statistics (slice partials), then one CTA per sequence that merges them and, unless
// in kStatsOnly mode, runs the commit.  masked may be null only in kStatsOnly mode (every row).
cudaError_t launch_stats_commit(const void* logits, const dllm_shape& sh, const uint8_t* masked,
                                const dllm_stats& stats, const dllm_block_state* state,
                                const CommitArgs& ca, const StatsWs& ws, int sm_count,
                                cudaStream_t stream);

// Commit only, from statistics already in memory (one CTA per sequence).
cudaError_t launch_commit_only(const dllm_shape& sh, const dllm_stats& stats,
                               const dllm_block_state& state, const CommitArgs& ca,
                               cudaStream_t stream);

// Rows kept for smoothing (masked after the commit, sequence running), compacted ascending.
cudaError_t launch_compact_rows(const dllm_block_state& state, int B, int L, int32_t* row_ids,
                                int32_t* M, cudaStream_t stream);

// Single-read smoothing: rows read this step (before the commit; -inf statistics for the
// others), the fused statistics + probability rows, and the kept-row map after the commit.
cudaError_t launch_read_rows(const dllm_block_state& state, int B, int L, int32_t* rows,
                             int32_t* count, const dllm_stats& stats, cudaStream_t stream);
bool stats_probs_split(int V, int dtype, int* C, int* slabs_per_cta);
cudaError_t launch_stats_probs(const void* logits, const dllm_shape& sh, const int32_t* rows,
                               const int32_t* count, const dllm_stats& stats, uint16_t* P,
                               int R_pad, int32_t* status, cudaStream_t stream);
cudaError_t launch_kept_rows_map(const dllm_block_state& state, int B, int L, int32_t* row_ids,
                                 int32_t* M, const int32_t* rows_read, const int32_t* count_read,
                                 int32_t* inv, int32_t* map, cudaStream_t stream);

// Fresh block state (every position masked); the credit slots too when given (nk > 0).
cudaError_t launch_block_state_reset(const dllm_block_state& state, int64_t n, int B,
                                     int32_t* cand_id, float* cand_credit, int64_t nk,
                                     cudaStream_t stream);

cudaError_t launch_kv_refresh(const dllm_block_state& state, int B, int L, int prefix_len,
                              int window, uint8_t* refresh, int32_t* idx, int32_t* count,
                              cudaStream_t stream);

// Sets a CUDA graph conditional handle to 1 while some sequence of the block still decodes
// (a masked position, no EOS), else 0.
cudaError_t launch_loop_continue(const dllm_block_state& state, int B, int L,
                                 cudaGraphConditionalHandle handle, cudaStream_t stream);

// Smoothing: workspace, probability rows and the tcgen05 GEMM.
struct SmoothPlan {
  int R;          // rows (upper bound of M)
  int V;
  int ldp;        // V rounded up to 64 (64-wide K slabs)
  int d;
  int m_tiles;    // 128-row tiles
  int n_tiles;    // column tiles
  int bn_max;     // widest column tile (multiple of 16, <= 256)
  int split_k;    // K splits of the main pairs (one tile over one split each)
  int kb_per_split;  // K blocks (64 wide) of each main split
  int tail_pairs; // pairs that each take tail_tiles tiles over the last K range [kb_tail0, V/64)
  int tail_tiles;
  int kb_tail0;
  int partials;   // K ranges summed per output element (>1: reduced by a second kernel)
  int stages;     // TMA/MMA pipeline depth
  int slabs_per_stage;  // 64-wide K slabs per ring stage (one TMA box of that depth per operand)
  size_t ws_bytes;
  size_t off_p;       // bf16 P, K-slab-blocked [ldp / 64][R_pad][64]
  size_t off_part;    // fp32 partials [partials, R_pad, d]
  size_t off_rows;    // single-read path: rows read [R], their count, kept index per row [R],
  size_t off_count;   // and kept index per row read [R]
  size_t off_inv;
  size_t off_map;
  size_t off_stats_ws;  // a statistics workspace, for the element-wise single-read fallback
};

SmoothPlan smooth_plan(int B, int L, int V, int d, int sm_count);

cudaError_t launch_prob_rows(const void* logits, const dllm_shape& sh, const float* lse,
                             const int32_t* row_ids, const int32_t* M, uint16_t* P, int R_pad,
                             int sm_count, cudaStream_t stream);

// out row of P row j: row_map[j] (-1: not written) when row_map is not null, else j.
// wait_late: P and M were written before the kernel launched just before this one, which only
// writes row_map (the single-read step): the GEMM's mainloop may overlap that kernel.
cudaError_t launch_smooth_gemm(const SmoothPlan& plan, const uint16_t* P, const uint16_t* Et,
                               int ldt, float* out, const int32_t* M, const int32_t* row_map,
                               bool wait_late, void* ws, cudaStream_t stream, const char** why);

cudaError_t launch_merge_shard_stats(const dllm_shard_stats* shards, int n, int64_t rows,
                                     const dllm_stats& out, cudaStream_t stream);

cudaError_t launch_wait_timeout_selftest(int32_t* status, uint64_t limit_ns,
                                         cudaStream_t stream);

// Record a message for dllm_last_error() on this thread (with a CUDA error string if e != 0).
void set_last_error(const char* msg, cudaError_t e);

cudaError_t launch_transpose_embedding(const uint16_t* E, int V, int d, uint16_t* Et, int Vp,
                                       cudaStream_t stream);

}  // namespace dllm
