// C ABI of the decode step: argument validation, workspace layout and kernel launches.
// Every entry point validates on the host first and launches nothing when it returns an error.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "internal.h"

namespace {

// One NVTX range per entry point, named after it, spanning the host-side work of the call
// (validation and kernel launches; the kernels themselves run later on the stream).  Free when
// no profiler is attached.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

thread_local char g_err[512];

dllm_status fail(dllm_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

dllm_status ok() {
  g_err[0] = '\0';
  return DLLM_OK;
}

dllm_status cuda_fail(cudaError_t e, const char* where) {
  return fail(DLLM_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

dllm_status check_shape(const dllm_shape* sh) {
  if (!sh) return fail(DLLM_ERR_INVALID_ARG, "shape is null");
  if (sh->B < 1 || sh->L < 1 || sh->V < 1)
    return fail(DLLM_ERR_INVALID_ARG, "B, L and V must be positive (B=%d L=%d V=%d)", sh->B,
                sh->L, sh->V);
  if (sh->dtype != DLLM_F32 && sh->dtype != DLLM_BF16)
    return fail(DLLM_ERR_UNSUPPORTED, "dtype %d is not fp32 (0) or bf16 (1)", sh->dtype);
  if (sh->L > dllm::kMaxL) return fail(DLLM_ERR_UNSUPPORTED, "L=%d exceeds %d", sh->L, dllm::kMaxL);
  if (static_cast<int64_t>(sh->B) * sh->L > (int64_t{1} << 20))
    return fail(DLLM_ERR_UNSUPPORTED, "B*L=%lld exceeds 2^20",
                static_cast<long long>(sh->B) * sh->L);
  if (sh->row_stride < sh->V)
    return fail(DLLM_ERR_INVALID_ARG, "row_stride %lld < V %d",
                static_cast<long long>(sh->row_stride), sh->V);
  return DLLM_OK;
}

dllm_status check_ws(const void* ws) {
  if (!ws) return fail(DLLM_ERR_INVALID_ARG, "workspace is null");
  if (!aligned(ws, 256)) return fail(DLLM_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  return DLLM_OK;
}

dllm_status check_stats(const dllm_stats* st) {
  if (!st || !st->row_max || !st->lse || !st->conf || !st->argmax)
    return fail(DLLM_ERR_INVALID_ARG, "stats or one of its arrays is null");
  return DLLM_OK;
}

dllm_status check_state(const dllm_block_state* s) {
  if (!s || !s->masked || !s->tokens || !s->committed_now || !s->n_commit || !s->eos_hit)
    return fail(DLLM_ERR_INVALID_ARG, "block state or one of its arrays is null");
  return DLLM_OK;
}

// Logits for the statistics and commit calls: aligned to their element size (rows that are
// not 16-byte aligned take the scalar-load path of the statistics kernel).
dllm_status check_logits(const void* logits, const dllm_shape* sh) {
  if (!aligned(logits, sh->dtype == DLLM_BF16 ? 2 : 4))
    return fail(DLLM_ERR_INVALID_ARG, "logits must be aligned to the element size");
  return DLLM_OK;
}

// Rows the single-read smoothing kernels can copy whole (16-byte aligned rows, V a multiple of
// 8); other layouts take the element-wise path.
bool rows_vector_aligned(const void* logits, const dllm_shape* sh) {
  const int es = sh->dtype == DLLM_BF16 ? 2 : 4;
  return aligned(logits, 16) && (sh->row_stride * es) % 16 == 0 && sh->V % 8 == 0;
}

dllm::CommitArgs threshold_args(float tau, int32_t eos_id) {
  dllm::CommitArgs ca{};
  ca.mode = dllm::kThreshold;
  ca.tau = tau;
  ca.eos_id = eos_id;
  return ca;
}

#define DLLM_TRY(x)                 \
  do {                              \
    dllm_status s_ = (x);           \
    if (s_ != DLLM_OK) return s_;   \
  } while (0)

// The graph `stream` is capturing (with its current capture dependencies when asked for);
// DLLM_ERR_INVALID_ARG when the stream is not capturing.
dllm_status capturing_graph(dllm_stream_t stream, cudaGraph_t* graph, const cudaGraphNode_t** deps,
                            size_t* n_deps, const char* name) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamGetCaptureInfo(reinterpret_cast<cudaStream_t>(stream), &cs, nullptr,
                                           graph, deps, nullptr, n_deps);
  if (e != cudaSuccess) return cuda_fail(e, name);
  if (cs != cudaStreamCaptureStatusActive)
    return fail(DLLM_ERR_INVALID_ARG, "%s: stream is not capturing a graph", name);
  return DLLM_OK;
}

// Shared body of the three commit entry points.
dllm_status commit_common(const void* logits, const dllm_shape* shape, const dllm_stats* stats,
                          const dllm_block_state* state, const dllm::CommitArgs& ca, void* ws,
                          dllm_stream_t stream, const char* name) {
  DLLM_TRY(check_shape(shape));
  DLLM_TRY(check_stats(stats));
  DLLM_TRY(check_state(state));
  cudaError_t e;
  if (logits) {
    DLLM_TRY(check_logits(logits, shape));
    DLLM_TRY(check_ws(ws));
    const dllm::StatsWs w = dllm::stats_ws_layout(ws, shape->B, shape->L, shape->V);
    e = dllm::launch_stats_commit(logits, *shape, nullptr, *stats, state, ca, w, sm_count(),
                                  reinterpret_cast<cudaStream_t>(stream));
  } else {
    e = dllm::launch_commit_only(*shape, *stats, *state, ca,
                                 reinterpret_cast<cudaStream_t>(stream));
  }
  if (e != cudaSuccess) return cuda_fail(e, name);
  return ok();
}

}  // namespace

namespace dllm {
void set_last_error(const char* msg, cudaError_t e) {
  if (e != cudaSuccess)
    snprintf(g_err, sizeof(g_err), "%s: %s", msg, cudaGetErrorString(e));
  else
    snprintf(g_err, sizeof(g_err), "%s", msg);
}
}  // namespace dllm

extern "C" {

const char* dllm_last_error(void) { return g_err; }

size_t dllm_workspace_bytes(const dllm_shape* shape) {
  if (check_shape(shape) != DLLM_OK) return 0;
  return dllm::stats_ws_bytes(shape->B, shape->L, shape->V);
}

dllm_status dllm_decode_stats(const void* logits, const dllm_shape* shape, const uint8_t* masked,
                              const dllm_stats* out, void* ws, dllm_stream_t stream) {
  CallRange range_("dllm_decode_stats");
  DLLM_TRY(check_shape(shape));
  if (!logits) return fail(DLLM_ERR_INVALID_ARG, "logits is null");
  DLLM_TRY(check_logits(logits, shape));
  DLLM_TRY(check_stats(out));
  DLLM_TRY(check_ws(ws));
  dllm::CommitArgs ca{};
  ca.mode = dllm::kStatsOnly;
  const dllm::StatsWs w = dllm::stats_ws_layout(ws, shape->B, shape->L, shape->V);
  cudaError_t e = dllm::launch_stats_commit(logits, *shape, masked, *out, nullptr, ca, w,
                                            sm_count(), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dllm_decode_stats");
  return ok();
}

dllm_status dllm_commit_threshold(const void* logits, const dllm_shape* shape,
                                  const dllm_stats* stats, const dllm_block_state* state,
                                  float tau, int32_t eos_id, void* ws, dllm_stream_t stream) {
  CallRange range_("dllm_commit_threshold");
  return commit_common(logits, shape, stats, state, threshold_args(tau, eos_id), ws, stream,
                       "dllm_commit_threshold");
}

dllm_status dllm_commit_hierarchical(const void* logits, const dllm_shape* shape,
                                     const dllm_stats* stats, const dllm_block_state* state,
                                     float tau_low, int32_t min_width, int32_t eos_id, void* ws,
                                     dllm_stream_t stream) {
  CallRange range_("dllm_commit_hierarchical");
  if (min_width < 1) return fail(DLLM_ERR_INVALID_ARG, "min_width must be >= 1");
  dllm::CommitArgs ca{};
  ca.mode = dllm::kHierarchical;
  ca.tau_low = tau_low;
  ca.min_width = min_width;
  ca.eos_id = eos_id;
  return commit_common(logits, shape, stats, state, ca, ws, stream, "dllm_commit_hierarchical");
}

dllm_status dllm_commit_credit(const void* logits, const dllm_shape* shape,
                               const dllm_stats* stats, const dllm_block_state* state,
                               int32_t* cand_id, float* cand_credit, int32_t K, float decay,
                               float boost, float tau, int32_t eos_id, void* ws,
                               dllm_stream_t stream) {
  CallRange range_("dllm_commit_credit");
  if (!cand_id || !cand_credit)
    return fail(DLLM_ERR_INVALID_ARG, "cand_id and cand_credit must not be null");
  if (K < 1 || K > dllm::kMaxK)
    return fail(K < 1 ? DLLM_ERR_INVALID_ARG : DLLM_ERR_UNSUPPORTED, "K=%d outside [1, %d]", K,
                dllm::kMaxK);
  dllm::CommitArgs ca{};
  ca.mode = dllm::kCredit;
  ca.tau = tau;
  ca.eos_id = eos_id;
  ca.cand_id = cand_id;
  ca.cand_credit = cand_credit;
  ca.K = K;
  ca.decay = decay;
  ca.boost = boost;
  return commit_common(logits, shape, stats, state, ca, ws, stream, "dllm_commit_credit");
}

dllm_status dllm_commit_hierarchical_levels(const void* logits, const dllm_shape* shape,
                                            const dllm_stats* stats,
                                            const dllm_block_state* state, float tau_low,
                                            int32_t min_width, int32_t eos_id, void* ws,
                                            dllm_stream_t stream) {
  CallRange range_("dllm_commit_hierarchical_levels");
  if (min_width < 1) return fail(DLLM_ERR_INVALID_ARG, "min_width must be >= 1");
  dllm::CommitArgs ca{};
  ca.mode = dllm::kHierarchicalLevels;
  ca.tau_low = tau_low;
  ca.min_width = min_width;
  ca.eos_id = eos_id;
  return commit_common(logits, shape, stats, state, ca, ws, stream,
                       "dllm_commit_hierarchical_levels");
}

dllm_status dllm_commit_credit_tracked(const void* logits, const dllm_shape* shape,
                                       const dllm_stats* stats, const dllm_block_state* state,
                                       int32_t* cand_id, float* cand_credit, int32_t K,
                                       float decay, float boost, float tau, int32_t eos_id,
                                       void* ws, dllm_stream_t stream) {
  CallRange range_("dllm_commit_credit_tracked");
  if (!logits)
    return fail(DLLM_ERR_INVALID_ARG,
                "logits is null (the tracked-credit variant reads every tracked token's logit)");
  if (!cand_id || !cand_credit)
    return fail(DLLM_ERR_INVALID_ARG, "cand_id and cand_credit must not be null");
  if (K < 1 || K > dllm::kMaxK)
    return fail(K < 1 ? DLLM_ERR_INVALID_ARG : DLLM_ERR_UNSUPPORTED, "K=%d outside [1, %d]", K,
                dllm::kMaxK);
  dllm::CommitArgs ca{};
  ca.mode = dllm::kCreditTracked;
  ca.tau = tau;
  ca.eos_id = eos_id;
  ca.cand_id = cand_id;
  ca.cand_credit = cand_credit;
  ca.K = K;
  ca.decay = decay;
  ca.boost = boost;
  return commit_common(logits, shape, stats, state, ca, ws, stream, "dllm_commit_credit_tracked");
}

size_t dllm_embedding_t_elems(int32_t V, int32_t d) {
  if (V < 1 || d < 1) return 0;
  return static_cast<size_t>(d) * dllm::align_up(static_cast<size_t>(V), 64);
}

dllm_status dllm_prepare_embedding(const uint16_t* E, int32_t V, int32_t d, uint16_t* Et,
                                   dllm_stream_t stream) {
  CallRange range_("dllm_prepare_embedding");
  if (!E || !Et) return fail(DLLM_ERR_INVALID_ARG, "E and Et must not be null");
  if (V < 1 || d < 1) return fail(DLLM_ERR_INVALID_ARG, "V and d must be positive");
  if (d % 16 != 0) return fail(DLLM_ERR_UNSUPPORTED, "d=%d is not a multiple of 16", d);
  if (!aligned(Et, 16)) return fail(DLLM_ERR_INVALID_ARG, "Et must be 16-byte aligned");
  const int Vp = static_cast<int>(dllm::align_up(static_cast<size_t>(V), 64));
  cudaError_t e = dllm::launch_transpose_embedding(E, V, d, Et, Vp,
                                                   reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dllm_prepare_embedding");
  return ok();
}

size_t dllm_smooth_workspace_bytes(const dllm_shape* shape, int32_t d) {
  if (check_shape(shape) != DLLM_OK || d < 16 || d % 16 != 0) return 0;
  return dllm::smooth_plan(shape->B, shape->L, shape->V, d, sm_count()).ws_bytes;
}

namespace {

dllm_status smooth_check(const dllm_shape* shape, int32_t d, void* ws, size_t ws_bytes,
                         dllm::SmoothPlan* pl) {
  DLLM_TRY(check_shape(shape));
  DLLM_TRY(check_ws(ws));
  if (d < 16 || d % 16 != 0 || d > 65536)
    return fail(DLLM_ERR_UNSUPPORTED, "d=%d must be a multiple of 16 in [16, 65536]", d);
  *pl = dllm::smooth_plan(shape->B, shape->L, shape->V, d, sm_count());
  if (ws_bytes < pl->ws_bytes)
    return fail(DLLM_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed",
                ws_bytes, pl->ws_bytes);
  return DLLM_OK;
}

}  // namespace

dllm_status dllm_smooth_plan_info(const dllm_shape* shape, int32_t d, int32_t* info) {
  CallRange range_("dllm_smooth_plan_info");
  DLLM_TRY(check_shape(shape));
  if (!info) return fail(DLLM_ERR_INVALID_ARG, "info is null");
  if (d < 16 || d % 16 != 0 || d > 65536)
    return fail(DLLM_ERR_UNSUPPORTED, "d=%d must be a multiple of 16 in [16, 65536]", d);
  const dllm::SmoothPlan pl = dllm::smooth_plan(shape->B, shape->L, shape->V, d, sm_count());
  info[0] = pl.m_tiles;
  info[1] = pl.n_tiles;
  info[2] = pl.bn_max;
  info[3] = pl.partials;
  info[4] = pl.stages;
  info[5] = 3 + (pl.partials > 1 ? 1 : 0);  // rows, probabilities, GEMM (+ partial-sum reduction)
  return ok();
}

dllm_status dllm_smooth_probs(const void* logits, const dllm_shape* shape, const dllm_stats* stats,
                              const dllm_block_state* state, int32_t d, int32_t* row_ids,
                              int32_t* M, void* ws, size_t ws_bytes, dllm_stream_t stream) {
  CallRange range_("dllm_smooth_probs");
  dllm::SmoothPlan pl;
  DLLM_TRY(smooth_check(shape, d, ws, ws_bytes, &pl));
  if (!logits) return fail(DLLM_ERR_INVALID_ARG, "logits is null");
  DLLM_TRY(check_logits(logits, shape));
  DLLM_TRY(check_stats(stats));
  DLLM_TRY(check_state(state));
  if (!row_ids || !M) return fail(DLLM_ERR_INVALID_ARG, "row_ids and M must not be null");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint16_t* P = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + pl.off_p);
  cudaError_t e = dllm::launch_compact_rows(*state, shape->B, shape->L, row_ids, M, st);
  if (e != cudaSuccess) return cuda_fail(e, "dllm_smooth_probs (rows)");
  e = dllm::launch_prob_rows(logits, *shape, stats->lse, row_ids, M, P, pl.m_tiles * 128,
                             sm_count(), st);
  if (e != cudaSuccess) return cuda_fail(e, "dllm_smooth_probs (probabilities)");
  return ok();
}

dllm_status dllm_smooth_gemm(const dllm_shape* shape, const uint16_t* Et, int32_t d, float* out,
                             const int32_t* M, void* ws, size_t ws_bytes, dllm_stream_t stream) {
  CallRange range_("dllm_smooth_gemm");
  dllm::SmoothPlan pl;
  DLLM_TRY(smooth_check(shape, d, ws, ws_bytes, &pl));
  if (!Et || !out || !M) return fail(DLLM_ERR_INVALID_ARG, "Et, out and M must not be null");
  if (!aligned(Et, 16) || !aligned(out, 16))
    return fail(DLLM_ERR_INVALID_ARG, "Et and out must be 16-byte aligned");
  const uint16_t* P =
      reinterpret_cast<const uint16_t*>(static_cast<const char*>(ws) + pl.off_p);
  const char* why = "launch failed";
  const int ldt = static_cast<int>(dllm::align_up(static_cast<size_t>(shape->V), 8));
  cudaError_t e = dllm::launch_smooth_gemm(pl, P, Et, ldt, out, M, nullptr, false, ws,
                                           reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess)
    return fail(DLLM_ERR_CUDA, "dllm_smooth_gemm: %s: %s", why, cudaGetErrorString(e));
  return ok();
}

dllm_status dllm_smooth_embed(const void* logits, const dllm_shape* shape, const dllm_stats* stats,
                              const dllm_block_state* state, const uint16_t* Et, int32_t d,
                              float* out, int32_t* row_ids, int32_t* M, void* ws,
                              size_t ws_bytes, dllm_stream_t stream) {
  CallRange range_("dllm_smooth_embed");
  if (!Et || !out) return fail(DLLM_ERR_INVALID_ARG, "Et and out must not be null");
  if (!aligned(Et, 16) || !aligned(out, 16))
    return fail(DLLM_ERR_INVALID_ARG, "Et and out must be 16-byte aligned");
  DLLM_TRY(dllm_smooth_probs(logits, shape, stats, state, d, row_ids, M, ws, ws_bytes, stream));
  return dllm_smooth_gemm(shape, Et, d, out, M, ws, ws_bytes, stream);
}

dllm_status dllm_commit_threshold_smooth(const void* logits, const dllm_shape* shape,
                                        const dllm_stats* stats, const dllm_block_state* state,
                                        float tau, int32_t eos_id, const uint16_t* Et, int32_t d,
                                        float* out, int32_t* row_ids, int32_t* M, void* ws,
                                        size_t ws_bytes, dllm_stream_t stream) {
  CallRange range_("dllm_commit_threshold_smooth");
  dllm::SmoothPlan pl;
  DLLM_TRY(smooth_check(shape, d, ws, ws_bytes, &pl));
  if (!logits) return fail(DLLM_ERR_INVALID_ARG, "logits is null");
  DLLM_TRY(check_logits(logits, shape));
  DLLM_TRY(check_stats(stats));
  DLLM_TRY(check_state(state));
  if (!Et || !out || !row_ids || !M)
    return fail(DLLM_ERR_INVALID_ARG, "Et, out, row_ids and M must not be null");
  if (!aligned(Et, 16) || !aligned(out, 16))
    return fail(DLLM_ERR_INVALID_ARG, "Et and out must be 16-byte aligned");
  int C = 0, per = 0;
  if (!rows_vector_aligned(logits, shape) ||
      !dllm::stats_probs_split(shape->V, shape->dtype, &C, &per)) {
    // rows the single-read kernels cannot copy whole (not 16-byte aligned, V not a multiple of
    // 8, or longer than 8 x 192 KB): the same results from the separate calls, which read such
    // rows element by element (the logits are read twice)
    DLLM_TRY(commit_common(logits, shape, stats, state, threshold_args(tau, eos_id),
                           static_cast<char*>(ws) + pl.off_stats_ws, stream,
                           "dllm_commit_threshold_smooth"));
    return dllm_smooth_embed(logits, shape, stats, state, Et, d, out, row_ids, M, ws, ws_bytes,
                             stream);
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  uint16_t* P = reinterpret_cast<uint16_t*>(w + pl.off_p);
  int32_t* rows = reinterpret_cast<int32_t*>(w + pl.off_rows);
  int32_t* count = reinterpret_cast<int32_t*>(w + pl.off_count);
  int32_t* inv = reinterpret_cast<int32_t*>(w + pl.off_inv);
  int32_t* map = reinterpret_cast<int32_t*>(w + pl.off_map);
  const int R_pad = pl.m_tiles * 128;
  cudaError_t e = dllm::launch_read_rows(*state, shape->B, shape->L, rows, count, *stats, st);
  if (e == cudaSuccess)
    e = dllm::launch_stats_probs(logits, *shape, rows, count, *stats, P, R_pad,
                                 static_cast<int32_t*>(ws), st);
  if (e != cudaSuccess) return cuda_fail(e, "dllm_commit_threshold_smooth (statistics)");
  dllm::CommitArgs ca{};
  ca.mode = dllm::kThreshold;
  ca.tau = tau;
  ca.eos_id = eos_id;
  e = dllm::launch_commit_only(*shape, *stats, *state, ca, st);
  if (e == cudaSuccess)
    e = dllm::launch_kept_rows_map(*state, shape->B, shape->L, row_ids, M, rows, count, inv, map,
                                   st);
  if (e != cudaSuccess) return cuda_fail(e, "dllm_commit_threshold_smooth (commit)");
  const char* why = "launch failed";
  const int ldt = static_cast<int>(dllm::align_up(static_cast<size_t>(shape->V), 8));
  // P (statistics kernel) and count (row list) predate the kept-row map, the only input the
  // kernel just before the GEMM writes: the GEMM's mainloop overlaps it
  e = dllm::launch_smooth_gemm(pl, P, Et, ldt, out, count, map, true, ws, st, &why);
  if (e != cudaSuccess)
    return fail(DLLM_ERR_CUDA, "dllm_commit_threshold_smooth: %s: %s", why,
                cudaGetErrorString(e));
  return ok();
}

dllm_status dllm_block_state_reset(const dllm_block_state* state, int32_t B, int32_t L,
                                   int32_t* cand_id, float* cand_credit, int32_t K,
                                   dllm_stream_t stream) {
  CallRange range_("dllm_block_state_reset");
  DLLM_TRY(check_state(state));
  if (B < 1 || L < 1) return fail(DLLM_ERR_INVALID_ARG, "need B, L >= 1 (B=%d L=%d)", B, L);
  if (L > dllm::kMaxL) return fail(DLLM_ERR_UNSUPPORTED, "L=%d exceeds %d", L, dllm::kMaxL);
  if (static_cast<int64_t>(B) * L > (int64_t{1} << 20))
    return fail(DLLM_ERR_UNSUPPORTED, "B*L=%lld exceeds 2^20",
                static_cast<long long>(B) * L);
  const bool credit = cand_id != nullptr || cand_credit != nullptr;
  if (credit && (K < 1 || K > dllm::kMaxK))
    return fail(DLLM_ERR_INVALID_ARG, "K=%d must be in [1, %d] with credit slots", K,
                dllm::kMaxK);
  const int64_t n = static_cast<int64_t>(B) * L;
  cudaError_t e = dllm::launch_block_state_reset(*state, n, B, cand_id, cand_credit,
                                                 credit ? n * K : 0,
                                                 reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dllm_block_state_reset");
  return ok();
}

dllm_status dllm_capture_condition(dllm_stream_t stream, uint32_t default_value,
                                   uint64_t* handle_out) {
  CallRange range_("dllm_capture_condition");
  if (!handle_out) return fail(DLLM_ERR_INVALID_ARG, "handle_out is null");
  cudaGraph_t graph = nullptr;
  DLLM_TRY(capturing_graph(stream, &graph, nullptr, nullptr, "dllm_capture_condition"));
  cudaGraphConditionalHandle h = 0;
  cudaError_t e = cudaGraphConditionalHandleCreate(&h, graph, default_value ? 1u : 0u,
                                                   cudaGraphCondAssignDefault);
  if (e != cudaSuccess) return cuda_fail(e, "dllm_capture_condition");
  *handle_out = static_cast<uint64_t>(h);
  return ok();
}

dllm_status dllm_capture_if_begin(dllm_stream_t stream, dllm_stream_t body_stream,
                                  uint64_t handle) {
  CallRange range_("dllm_capture_if_begin");
  if (stream == body_stream)
    return fail(DLLM_ERR_INVALID_ARG, "the conditional body needs a stream of its own");
  cudaGraph_t graph = nullptr;
  const cudaGraphNode_t* deps = nullptr;
  size_t n_deps = 0;
  DLLM_TRY(capturing_graph(stream, &graph, &deps, &n_deps, "dllm_capture_if_begin"));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t bs = reinterpret_cast<cudaStream_t>(body_stream);
  cudaStreamCaptureStatus bcs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(bs, &bcs);
  if (e != cudaSuccess) return cuda_fail(e, "dllm_capture_if_begin (body stream)");
  if (bcs != cudaStreamCaptureStatusNone)
    return fail(DLLM_ERR_INVALID_ARG, "body_stream is already capturing");
  cudaGraphNodeParams np = {};
  np.type = cudaGraphNodeTypeConditional;
  np.conditional.handle = static_cast<cudaGraphConditionalHandle>(handle);
  np.conditional.type = cudaGraphCondTypeIf;
  np.conditional.size = 1;
  cudaGraphNode_t node = nullptr;
  e = cudaGraphAddNode(&node, graph, deps, nullptr, n_deps, &np);
  if (e != cudaSuccess) return cuda_fail(e, "dllm_capture_if_begin (conditional node)");
  // later work on `stream` follows the node; the body is captured on body_stream
  e = cudaStreamUpdateCaptureDependencies(s, &node, nullptr, 1, cudaStreamSetCaptureDependencies);
  if (e != cudaSuccess) return cuda_fail(e, "dllm_capture_if_begin (dependencies)");
  e = cudaStreamBeginCaptureToGraph(bs, np.conditional.phGraph_out[0], nullptr, nullptr, 0,
                                    cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) return cuda_fail(e, "dllm_capture_if_begin (body capture)");
  return ok();
}

dllm_status dllm_capture_if_end(dllm_stream_t body_stream) {
  CallRange range_("dllm_capture_if_end");
  cudaGraph_t body = nullptr;  // owned by the conditional node
  cudaError_t e = cudaStreamEndCapture(reinterpret_cast<cudaStream_t>(body_stream), &body);
  if (e != cudaSuccess) return cuda_fail(e, "dllm_capture_if_end");
  return ok();
}

dllm_status dllm_loop_continue(const dllm_block_state* state, int32_t B, int32_t L,
                               uint64_t handle, dllm_stream_t stream) {
  CallRange range_("dllm_loop_continue");
  if (!state || !state->masked || !state->eos_hit)
    return fail(DLLM_ERR_INVALID_ARG, "state.masked and state.eos_hit must not be null");
  if (B < 1 || L < 1) return fail(DLLM_ERR_INVALID_ARG, "need B, L >= 1 (B=%d L=%d)", B, L);
  if (L > dllm::kMaxL) return fail(DLLM_ERR_UNSUPPORTED, "L=%d exceeds %d", L, dllm::kMaxL);
  if (static_cast<int64_t>(B) * L > (int64_t{1} << 20))
    return fail(DLLM_ERR_UNSUPPORTED, "B*L=%lld exceeds 2^20", static_cast<long long>(B) * L);
  cudaGraph_t graph = nullptr;  // the handle exists only inside its graph
  DLLM_TRY(capturing_graph(stream, &graph, nullptr, nullptr, "dllm_loop_continue"));
  cudaError_t e = dllm::launch_loop_continue(*state, B, L,
                                             static_cast<cudaGraphConditionalHandle>(handle),
                                             reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dllm_loop_continue");
  return ok();
}

dllm_status dllm_kv_refresh_mask(const dllm_block_state* state, int32_t B, int32_t L,
                                 int32_t prefix_len, int32_t window, uint8_t* refresh,
                                 int32_t* idx, int32_t* count, dllm_stream_t stream) {
  CallRange range_("dllm_kv_refresh_mask");
  if (!state || !state->committed_now)
    return fail(DLLM_ERR_INVALID_ARG, "state.committed_now is null");
  if (!refresh || !idx || !count)
    return fail(DLLM_ERR_INVALID_ARG, "refresh, idx and count must not be null");
  if (B < 1 || L < 1 || prefix_len < 0 || window < 0)
    return fail(DLLM_ERR_INVALID_ARG, "need B, L >= 1 and prefix_len, window >= 0");
  if (static_cast<int64_t>(prefix_len) + L > 65536)
    return fail(DLLM_ERR_UNSUPPORTED, "prefix_len + L exceeds 65536");
  if (L > dllm::kMaxL) return fail(DLLM_ERR_UNSUPPORTED, "L=%d exceeds %d", L, dllm::kMaxL);
  cudaError_t e = dllm::launch_kv_refresh(*state, B, L, prefix_len, window, refresh, idx, count,
                                          reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dllm_kv_refresh_mask");
  return ok();
}

dllm_status dllm_selftest_wait_timeout(void* ws, uint32_t limit_us, dllm_stream_t stream) {
  CallRange range_("dllm_selftest_wait_timeout");
  DLLM_TRY(check_ws(ws));
  if (limit_us < 1 || limit_us > 2000000)
    return fail(DLLM_ERR_INVALID_ARG, "limit_us must be in [1, 2000000]");
  cudaError_t e = dllm::launch_wait_timeout_selftest(static_cast<int32_t*>(ws),
                                                     static_cast<uint64_t>(limit_us) * 1000,
                                                     reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dllm_selftest_wait_timeout");
  return ok();
}

dllm_status dllm_merge_shard_stats(const dllm_shard_stats* shards, int32_t n, int64_t rows,
                                   const dllm_stats* out, dllm_stream_t stream) {
  CallRange range_("dllm_merge_shard_stats");
  if (!shards) return fail(DLLM_ERR_INVALID_ARG, "shards is null");
  if (n < 1 || n > DLLM_MAX_SHARDS)
    return fail(DLLM_ERR_INVALID_ARG, "n=%d must be in [1, %d]", n, DLLM_MAX_SHARDS);
  if (rows < 0 || rows > (int64_t{1} << 31))
    return fail(DLLM_ERR_INVALID_ARG, "rows=%lld out of range", static_cast<long long>(rows));
  DLLM_TRY(check_stats(out));
  for (int k = 0; k < n; ++k) {
    DLLM_TRY(check_stats(&shards[k].stats));
    if (shards[k].vocab_offset < 0 || shards[k].vocab_offset >= (int64_t{1} << 31))
      return fail(DLLM_ERR_INVALID_ARG, "shard %d: vocab_offset out of range", k);
    const dllm_stats& a = shards[k].stats;
    if (a.row_max == out->row_max || a.lse == out->lse || a.conf == out->conf ||
        a.argmax == out->argmax)
      return fail(DLLM_ERR_INVALID_ARG, "shard %d aliases the output", k);
  }
  cudaError_t e = dllm::launch_merge_shard_stats(shards, n, rows, *out,
                                                 reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dllm_merge_shard_stats");
  return ok();
}

dllm_status dllm_get_status(void* ws, dllm_stream_t stream, int32_t* out_host) {
  CallRange range_("dllm_get_status");
  DLLM_TRY(check_ws(ws));
  if (!out_host) return fail(DLLM_ERR_INVALID_ARG, "out_host is null");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "dllm_get_status");
  *out_host = v;
  if (v != DLLM_OK) {
    e = cudaMemsetAsync(ws, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "dllm_get_status (reset)");
  }
  return ok();
}

}  // extern "C"
