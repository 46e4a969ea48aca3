/*
 * dllm.h — C ABI of the parallel-decode step of a diffusion language model, for NVIDIA GB300
 * (sm_103a).
 *
 * One decode iteration of a masked-diffusion LM ends with the model's logits for a block of L
 * positions in each of B sequences.  The step turns them into decisions: which still-masked
 * positions to fix ("commit") now and with which token, what to feed back for the positions
 * left open, and which KV-cache entries must be recomputed.  Sources, cited by page and
 * section:
 *   [dInfer explainer]  the 91haoming.cn summary of the dInfer paper (arXiv 2510.08666): its
 *                       decoding-strategy component (threshold, hierarchical and credit
 *                       decoding), diffusion-iteration manager (iteration smoothing), KV-cache
 *                       manager (neighbourhood refresh) and engineering notes (early stop).
 *   [dInfer news]       the aibase.com article: the four modules (model access, KV-cache
 *                       manager, diffusion-iteration manager, decoding strategies).
 * The pages give no formulas; the exact definitions these functions compute are restated at
 * each declaration.
 *
 * Conventions shared by every function:
 *  - Every pointer argument is DEVICE memory owned by the caller, except the `const dllm_*`
 *    descriptor structs themselves, `out_host` of dllm_get_status and `handle_out` of
 *    dllm_capture_condition, which are host memory read (or written) before the function
 *    returns.  The library never allocates or frees
 *    device memory and never synchronises the stream, except dllm_get_status.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream) and runs
 *    asynchronously.  The functions hold no host state between calls, so a sequence of calls
 *    can be captured into a CUDA graph.
 *  - Return value: DLLM_OK when the work was enqueued.  DLLM_ERR_INVALID_ARG (a null pointer,
 *    a non-positive size, a misaligned pointer, a stride shorter than a row) and
 *    DLLM_ERR_UNSUPPORTED (a size beyond a documented limit) are returned before anything is
 *    launched.  DLLM_ERR_CUDA means a launch failed.  dllm_last_error() then describes the
 *    failure (thread-local, valid until the next call on the same thread).
 *  - Faults found while the kernels run (a wait that timed out inside the smoothing GEMM) are
 *    recorded in the status word at the start of the workspace; dllm_get_status reads it.
 *  - Workspace: `ws` points to at least dllm_workspace_bytes(shape) bytes (or
 *    dllm_smooth_workspace_bytes for dllm_smooth_embed), 256-byte aligned, zero-filled ONCE
 *    before its first use (its first 4 bytes are the status word).  The same workspace serves
 *    any number of later calls on one stream.  Calls that run at the same time must use
 *    different workspaces.
 *
 * Data layout (row r = b*L + i is position i of sequence b):
 *  - logits: B*L rows of V elements, row r starting at element r*row_stride; row_stride >= V.
 *    fp32 or bf16 (dllm_shape.dtype).  The pointer is aligned to the element size.  Rows that
 *    all start on 16-byte boundaries (pointer and row_stride * element size multiples of 16)
 *    are read with 16-byte vector loads; any other layout (and, for the smoothing calls, V not
 *    a multiple of 8) is read element by element by the same kernels (slower, same results).
 *  - block state (dllm_block_state), all [B, L] or [B] row-major:
 *      masked[B*L]        uint8, 1 = position still undecided;
 *      tokens[B*L]        int32, committed token id, -1 while masked;
 *      committed_now[B*L] uint8, written by every commit call: 1 = committed in this call;
 *      n_commit[B]        int32, written by every commit call: number committed in this call;
 *      eos_hit[B]         int32, set to 1 when a committed token equals eos_id; a sequence
 *                         with eos_hit set, or with nothing masked, is stopped: later calls do
 *                         not read its logits, commit nothing and leave its state untouched.
 *  - statistics (dllm_stats), [B*L] each: row_max (fp32), lse (fp32, natural log-sum-exp),
 *    conf (fp32, top-1 probability) and argmax (int32, lowest index of the maximum).  Rows not
 *    computed hold -inf, -inf, 0 and -1.
 */
#ifndef DLLM_H_
#define DLLM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* dllm_stream_t; /* same type as cudaStream_t */

typedef enum {
  DLLM_OK = 0,
  DLLM_ERR_INVALID_ARG = 1,
  DLLM_ERR_UNSUPPORTED = 2,
  DLLM_ERR_CUDA = 3,
  DLLM_ERR_TIMEOUT = 4
} dllm_status;

typedef enum { DLLM_F32 = 0, DLLM_BF16 = 1 } dllm_dtype;

/* Shape of one block of logits.  Limits: B >= 1, 1 <= L <= 1024, 2 <= V < 2^31,
 * B*L <= 2^20, row_stride >= V. */
typedef struct {
  int32_t B;
  int32_t L;
  int32_t V;
  int32_t dtype;      /* dllm_dtype */
  int64_t row_stride; /* elements between the starts of consecutive rows */
} dllm_shape;

typedef struct {
  uint8_t* masked;
  int32_t* tokens;
  uint8_t* committed_now;
  int32_t* n_commit;
  int32_t* eos_hit;
} dllm_block_state;

typedef struct {
  float* row_max;
  float* lse;
  float* conf;
  int32_t* argmax;
} dllm_stats;

/* Description of the last error on this thread ("" if none). */
const char* dllm_last_error(void);

/*
 * Start a new block (dInfer explainer, diffusion-iteration manager: a block starts with every
 * position masked and is decoded over iterations until filled or stopped): one kernel sets
 *   masked[B*L] = 1, tokens[B*L] = -1, committed_now[B*L] = 0, n_commit[B] = 0, eos_hit[B] = 0
 * and, when cand_id / cand_credit are not NULL (the credit-decoding state, [B*L, K] each),
 * cand_id = -1 (empty slot) and cand_credit = 0.  1 <= K <= 16 when either is given.
 * B >= 1, 1 <= L <= 1024, B*L <= 2^20.  Same stream rules as every call: it is ordered after
 * the calls before it on `stream`, so a decode loop with its reset can be captured whole.
 */
dllm_status dllm_block_state_reset(const dllm_block_state* state, int32_t B, int32_t L,
                                   int32_t* cand_id, float* cand_credit, int32_t K,
                                   dllm_stream_t stream);

/* Bytes of workspace the stats and commit calls need for `shape` (0 if shape is invalid). */
size_t dllm_workspace_bytes(const dllm_shape* shape);

/*
 * Softmax statistics of every row (dInfer explainer, decoding strategies: each strategy ranks
 * the undecided positions by the model's confidence in its top token).  For a computed row z:
 *   row_max = max_v z_v;  s = sum_v exp(z_v - row_max);  lse = row_max + ln s;
 *   conf = 1/s (the top-1 probability);  argmax = lowest v with z_v = row_max.
 * masked: [B*L] uint8 or NULL.  With a mask, only rows with masked[r] = 1 are read and
 * computed; with NULL every row is.  Each logit crosses HBM once.
 */
dllm_status dllm_decode_stats(const void* logits, const dllm_shape* shape, const uint8_t* masked,
                              const dllm_stats* out, void* ws, dllm_stream_t stream);

/*
 * Threshold decoding (dInfer explainer, decoding strategies, method 1: fix a position at once
 * when the model is confident in it).  Per sequence that is not stopped:
 *   C = { masked i : conf_i > tau };  if C is empty, C = { the masked i of largest conf,
 *   lowest i on ties };  for i in C: tokens[i] = argmax_i, masked[i] = 0, committed_now[i] = 1.
 * With logits != NULL the statistics are computed in the same pass (only the masked rows of
 * running sequences are read) and written to *stats; with logits == NULL, *stats must hold
 * the statistics of this step (conf and argmax are read) and the call only commits.
 * eos_id >= 0 enables the early stop; -1 disables it.
 */
dllm_status dllm_commit_threshold(const void* logits, const dllm_shape* shape,
                                  const dllm_stats* stats, const dllm_block_state* state,
                                  float tau, int32_t eos_id, void* ws, dllm_stream_t stream);

/*
 * Hierarchical decoding (dInfer explainer, decoding strategies, method 2: split the region
 * still to be filled recursively and decide the centre of each sub-region first).  Per
 * sequence that is not stopped, on the mask as it stands at the call:
 *   maximal runs [s, e) of masked positions are halved at s + floor(w/2) while their width
 *   w >= 2*min_width; in each resulting leaf the position with conf >= tau_low that is closest
 *   to the leaf centre (smallest |2i - (s+e-1)|, lowest i on ties) is committed; a sequence
 *   that commits nothing commits its masked position of largest conf (lowest i on ties).
 * min_width >= 1.  logits, stats, state and eos_id as in dllm_commit_threshold.
 */
dllm_status dllm_commit_hierarchical(const void* logits, const dllm_shape* shape,
                                     const dllm_stats* stats, const dllm_block_state* state,
                                     float tau_low, int32_t min_width, int32_t eos_id, void* ws,
                                     dllm_stream_t stream);

/*
 * Credit decoding (dInfer explainer, decoding strategies, method 3: each candidate token of
 * each position keeps a credit recording how often and how confidently it was chosen across
 * iterations; stable candidates are favoured).  Per masked position of a running sequence,
 * with top token a and confidence p:
 *   every slot decays, c_k <- decay*c_k;  a's slot gains p (a takes the first empty slot, or
 *   evicts the slot of least credit, lowest slot on ties, starting at p);
 *   score = p * (1 + boost * ln(1 + c_a));
 *   C = { i : score_i > tau }, or the masked i of largest score (lowest i) if C is empty.
 * cand_id: [B*L, K] int32 (-1 = empty slot), cand_credit: [B*L, K] fp32, both read and
 * updated; initialise to -1 / 0 for a fresh block.  Positions not masked keep their slots.
 * 1 <= K <= 16.
 */
dllm_status dllm_commit_credit(const void* logits, const dllm_shape* shape,
                               const dllm_stats* stats, const dllm_block_state* state,
                               int32_t* cand_id, float* cand_credit, int32_t K, float decay,
                               float boost, float tau, int32_t eos_id, void* ws,
                               dllm_stream_t stream);

/*
 * Hierarchical decoding, a centre per level (variant of dllm_commit_hierarchical; the pages'
 * "decide the centre of each sub-region first" read as deciding every level's centre).  Same
 * halving tree; every node [s, e), internal or leaf, selects its position with
 * conf >= tau_low closest to the node centre (smallest |2i - (s+e-1)|, lowest i on ties) and
 * the union of the selections is committed; fallback, arguments and errors as
 * dllm_commit_hierarchical.
 */
dllm_status dllm_commit_hierarchical_levels(const void* logits, const dllm_shape* shape,
                                            const dllm_stats* stats,
                                            const dllm_block_state* state, float tau_low,
                                            int32_t min_width, int32_t eos_id, void* ws,
                                            dllm_stream_t stream);

/*
 * Credit decoding, every tracked candidate credited (variant of dllm_commit_credit; dInfer
 * explainer, decoding strategies, method 3).  Per masked position of a running sequence, with
 * p_v = exp(z_v - lse), top token a and p_a = conf:
 *   every slot decays, c_k <- decay*c_k;  every occupied slot gains its own token's probability,
 *   c_k <- c_k + p_{id_k};  if a is not tracked it takes the first empty slot, or evicts the
 *   slot of least credit (after the gains; lowest slot on ties), starting at p_a;
 *   s_k = p_{id_k} * (1 + boost * ln(1 + c_k)) over occupied slots; the best slot (lowest slot on
 *   ties) is the position's candidate: score = s_k, token = id_k (may differ from a);
 *   C = { i : score_i > tau }, or the masked i of largest score (lowest i); commits the
 *   candidate tokens.
 * logits must not be NULL (the tracked tokens' logits are read after the statistics).  Other
 * arguments and errors as dllm_commit_credit.
 */
dllm_status dllm_commit_credit_tracked(const void* logits, const dllm_shape* shape,
                                       const dllm_stats* stats, const dllm_block_state* state,
                                       int32_t* cand_id, float* cand_credit, int32_t K,
                                       float decay, float boost, float tau, int32_t eos_id,
                                       void* ws, dllm_stream_t stream);

/*
 * Re-lay the embedding table once for the smoothing GEMM: E [V, d] bf16 row-major (the usual
 * table) -> Et, the transpose stored K-slab-blocked: Et[(v / 64) * d + c][v % 64] = E[v][c], so
 * that each 64-wide slab of the vocabulary is contiguous for every column c; slab entries with
 * v >= V are zero.  dllm_embedding_t_elems(V, d) = d * (V rounded up to 64) elements.  Bit
 * patterns are copied unchanged.  d % 16 == 0.  Et must be 16-byte aligned.
 */
size_t dllm_embedding_t_elems(int32_t V, int32_t d);
dllm_status dllm_prepare_embedding(const uint16_t* E, int32_t V, int32_t d, uint16_t* Et,
                                   dllm_stream_t stream);

/* Bytes of workspace dllm_smooth_embed needs (status word, bf16 probability rows, partials). */
size_t dllm_smooth_workspace_bytes(const dllm_shape* shape, int32_t d);

/*
 * How dllm_smooth_gemm will run on the current device (host query, launches nothing):
 * info[0] row tiles, info[1] column tiles, info[2] widest column tile, info[3] K ranges summed
 * per output element (1: the GEMM writes the output itself; more: split-K partial sums added by
 * a second kernel),
 * info[4] pipeline stages, info[5] kernels launched by one dllm_smooth_embed call.
 */
dllm_status dllm_smooth_plan_info(const dllm_shape* shape, int32_t d, int32_t* info);

/*
 * Iteration smoothing (dInfer explainer, diffusion-iteration manager: positions that stay
 * undecided keep their whole distribution for the next round instead of dropping it).  After
 * this step's commit, the rows still masked in sequences that are not stopped are listed in
 * ascending order, row_ids[0..M), and for each
 *   P[j, v] = bf16_round_nearest_even( exp(z_{row_ids[j], v} - lse_{row_ids[j]}) ),
 *   out[j, :] = sum_v P[j, v] * E[v, :]       (fp32 accumulation, tensor cores)
 * logits/shape: the step's logits (bf16 or fp32); stats: its statistics (lse is read);
 * state: the block state after the commit (masked, eos_hit read);
 * Et: the table from dllm_prepare_embedding; d % 16 == 0, d <= 65536;
 * out: [B*L, d] fp32, rows >= M untouched; row_ids: [B*L] int32, entries >= M set to -1;
 * M: one int32.  M is produced on the device; nothing is read back to the host.
 * ws: dllm_smooth_workspace_bytes(shape, d) bytes.  Logits rows that are not 16-byte aligned,
 * or V not a multiple of 8, are read element by element (same results).
 */
dllm_status dllm_smooth_embed(const void* logits, const dllm_shape* shape, const dllm_stats* stats,
                              const dllm_block_state* state, const uint16_t* Et, int32_t d,
                              float* out, int32_t* row_ids, int32_t* M, void* ws,
                              size_t ws_bytes, dllm_stream_t stream);

/*
 * The two halves of dllm_smooth_embed, for callers that schedule them separately (same
 * arguments and results; call them in this order on one stream with the same workspace):
 *   dllm_smooth_probs: rows kept (row_ids, M) and the bf16 probability rows P, written to the
 *                      workspace;
 *   dllm_smooth_gemm:  out[0..M) = P x E on the tensor cores.
 */
dllm_status dllm_smooth_probs(const void* logits, const dllm_shape* shape, const dllm_stats* stats,
                              const dllm_block_state* state, int32_t d, int32_t* row_ids,
                              int32_t* M, void* ws, size_t ws_bytes, dllm_stream_t stream);
dllm_status dllm_smooth_gemm(const dllm_shape* shape, const uint16_t* Et, int32_t d, float* out,
                             const int32_t* M, void* ws, size_t ws_bytes, dllm_stream_t stream);

/*
 * Statistics of rows whose vocabulary is split over n tensor-parallel shards (dInfer explainer,
 * system optimisations: tensor parallelism splits the output layer, so each GPU holds the logits
 * of one contiguous vocabulary range).  Shard k covers ids [vocab_offset, vocab_offset + V_k)
 * and its `stats` are dllm_decode_stats of those columns (local argmax).  Per row:
 *   row_max = max_k m_k;  s = sum_k exp(lse_k - row_max);  lse = row_max + ln s;  conf = 1/s;
 *   argmax = lowest vocab_offset_k + argmax_k over the shards with m_k = row_max.
 * A row that no shard read (all m_k = -inf) gets -inf, -inf, 0, -1.  Exchanging the shards'
 * statistics (R x 16 bytes each, an all-gather) is the caller's: `shards` is a host array of n
 * descriptors whose arrays are device memory on this GPU (this rank's own, or received).
 * n in [1, DLLM_MAX_SHARDS]; rows >= 0; out may not alias a shard's arrays.  Asynchronous on
 * `stream`; nothing is allocated.
 */
#define DLLM_MAX_SHARDS 64
typedef struct {
  dllm_stats stats;
  int64_t vocab_offset;
} dllm_shard_stats;
dllm_status dllm_merge_shard_stats(const dllm_shard_stats* shards, int32_t n, int64_t rows,
                                   const dllm_stats* out, dllm_stream_t stream);

/*
 * Threshold commit and iteration smoothing in one call, reading each logit from HBM once
 * (single-read smoothing).  Results are those of dllm_commit_threshold followed by
 * dllm_smooth_embed on the same arguments: the statistics of the rows read, the commit, and
 * out[0..M) = P x E for the rows kept (row_ids ascending, M on the device), within the same
 * tolerances.  The rows read are held on chip (a cluster of up to 8 CTAs per row, up to 192 KB
 * per CTA) while their log-sum-exp completes, so their probabilities are written without a
 * second read; the GEMM then covers the rows read (rows committed in this step included) and
 * writes only the kept ones.
 * ws: dllm_smooth_workspace_bytes(shape, d) bytes; Et prepared by dllm_prepare_embedding.
 * Rows the single-read kernels cannot hold whole (not 16-byte aligned, V not a multiple of 8, or
 * longer than 8 x 192 KB) give the same results through the separate calls (dllm_commit_threshold
 * then dllm_smooth_embed, which read rows that are not aligned element by element); the logits
 * are then read twice.
 */
dllm_status dllm_commit_threshold_smooth(const void* logits, const dllm_shape* shape,
                                        const dllm_stats* stats, const dllm_block_state* state,
                                        float tau, int32_t eos_id, const uint16_t* Et, int32_t d,
                                        float* out, int32_t* row_ids, int32_t* M, void* ws,
                                        size_t ws_bytes, dllm_stream_t stream);

/*
 * Neighbourhood KV refresh (dInfer explainer, KV-cache manager: when a region of the sequence
 * changes, its cache entries and those of its neighbours are recomputed).  The cache row of
 * sequence b is [prefix 0..prefix_len) followed by the block, T = prefix_len + L entries:
 *   refresh[b, j] = 1 iff some i with committed_now[b, i] = 1 has |j - (prefix_len + i)| <= window;
 *   idx[b, 0..count[b]) = the refreshed j ascending, idx[b, k] = -1 for k >= count[b].
 * refresh: [B, T] uint8; idx: [B, T] int32; count: [B] int32.  T <= 65536.
 */
dllm_status dllm_kv_refresh_mask(const dllm_block_state* state, int32_t B, int32_t L,
                                 int32_t prefix_len, int32_t window, uint8_t* refresh,
                                 int32_t* idx, int32_t* count, dllm_stream_t stream);

/*
 * Device-side early stop for decode loops captured as CUDA graphs (dInfer explainer, system
 * optimisations: the iterations run back to back on the GPU without waiting on the host, and
 * decoding stops as soon as the end token is produced instead of running the remaining
 * iterations).  A caller that captures its whole loop as one graph tests the block every k
 * iterations and captures the rest of the loop inside a conditional section on that test,
 * each section nested in the one before:
 *
 *   on S0 (capturing):  reset; iterations 0 .. k-1;
 *                       dllm_capture_condition(S0, 0, &h1); dllm_loop_continue(state, B, L, h1, S0);
 *                       dllm_capture_if_begin(S0, S1, h1);
 *     on S1:              iterations k .. 2k-1; the same test and a section on S2; ...
 *   innermost first:    dllm_capture_if_end(S_n); ... dllm_capture_if_end(S1);
 *
 * Once every sequence has stopped, the next test skips everything after it.  A conditional
 * section costs several microseconds of graph scheduling whether it runs or not (on a GB300:
 * ~8 us when taken, ~5 us when not, against ~1.4 us per plain kernel node), so a test every
 * few iterations, not every iteration, pays for itself.
 *
 * dllm_capture_condition: `stream` is capturing a CUDA graph (cudaStreamBeginCapture, directly
 * or through a framework).  Creates a condition handle in that graph with `default_value` (0 or
 * non-zero -> 1), assigned again at every launch of the graph.  *handle_out receives it.
 *
 * dllm_capture_if_begin: adds to the graph `stream` is capturing a conditional IF node on
 * `handle` (created by dllm_capture_condition on the same capture) that depends on everything
 * captured on `stream` so far, makes the node `stream`'s only capture dependency (later work
 * captured on `stream` runs after it) and starts capturing body_stream, another stream that is
 * not capturing, into the node's body: work enqueued on body_stream until dllm_capture_if_end
 * runs only when the handle is non-zero when the node is reached.  Sections nest: `stream` may
 * itself be a body stream.
 *
 * dllm_capture_if_end: ends the capture of a body begun by dllm_capture_if_begin (the body graph
 * belongs to the conditional node).
 *
 * dllm_loop_continue: captured in the graph that owns `handle` (at any depth of its conditional
 * sections); when the graph runs, sets the handle to 1 if some sequence b of the block still
 * decodes (eos_hit[b] = 0 and a masked position), else 0.  One CTA, ordered after the calls
 * before it on `stream`.  B >= 1, 1 <= L <= 1024, B*L <= 2^20.
 *
 * Errors: DLLM_ERR_INVALID_ARG (a null pointer, stream == body_stream, a stream that must be
 * capturing and is not, a body_stream already capturing); DLLM_ERR_CUDA (the driver refused the
 * handle or node, or the body capture was invalidated).  A handle that belongs to another graph
 * is not detected and must not be passed.
 */
dllm_status dllm_capture_condition(dllm_stream_t stream, uint32_t default_value,
                                   uint64_t* handle_out);
dllm_status dllm_capture_if_begin(dllm_stream_t stream, dllm_stream_t body_stream,
                                  uint64_t handle);
dllm_status dllm_capture_if_end(dllm_stream_t body_stream);
dllm_status dllm_loop_continue(const dllm_block_state* state, int32_t B, int32_t L,
                               uint64_t handle, dllm_stream_t stream);

/*
 * Self-test of failure detection (no counterpart in the pages): runs the bounded wait the
 * smoothing GEMM uses on a barrier that nothing ever completes.  After limit_us microseconds
 * (1 .. 2,000,000) the wait gives up and records DLLM_ERR_TIMEOUT in the status word of `ws`
 * (any workspace, or 256 zeroed bytes); read it with dllm_get_status.  Nothing faults or hangs.
 */
dllm_status dllm_selftest_wait_timeout(void* ws, uint32_t limit_us, dllm_stream_t stream);

/*
 * dllm_commit_threshold without a workspace argument, for callers that cannot allocate device
 * memory where they decode (a serving runtime that reserves all memory up front and forbids
 * allocation while requests are in flight, a plugin whose host framework owns every device
 * buffer).  The pages have no counterpart to this call; it exists for those callers only.
 * Same arguments (minus ws), same results and same errors as dllm_commit_threshold with
 * logits != NULL, computed by the same kernel.  Its scratch is one static array of
 * DLLM_STATIC_WORKSPACE_BYTES in device memory, part of the library image: every GPU that loads
 * the library holds it until the process exits.
 *  - Shapes whose dllm_workspace_bytes exceeds DLLM_STATIC_WORKSPACE_BYTES are rejected with
 *    DLLM_ERR_UNSUPPORTED (4 MiB: e.g. B*L up to 2048 rows at V = 126464).
 *  - The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 *    that device current; make that first call before any stream capture.
 *  - Each call clears the array's status word on `stream`; nothing is allocated or freed.
 *    All calls share the one array and it keeps the last call's contents, so calls that
 *    overlap on the GPU (different streams, or concurrent graphs) race: serialise them.
 *  - dllm_get_status cannot be used on this scratch; a fault inside the kernel still surfaces
 *    as wrong results only, as for any call whose status word is never read.
 */
#define DLLM_STATIC_WORKSPACE_BYTES ((size_t)4 << 20)
dllm_status dllm_commit_threshold_static(const void* logits, const dllm_shape* shape,
                                         const dllm_stats* stats, const dllm_block_state* state,
                                         float tau, int32_t eos_id, dllm_stream_t stream);

/*
 * Read the device status word of a workspace (its first 4 bytes; synchronises `stream`).
 * *out_host receives DLLM_OK or the first fault a kernel recorded there (DLLM_ERR_TIMEOUT);
 * the word is then reset to DLLM_OK.  Works for both kinds of workspace.
 */
dllm_status dllm_get_status(void* ws, dllm_stream_t stream, int32_t* out_host);

#ifdef __cplusplus
}
#endif

#endif /* DLLM_H_ */
