// Oracle for the parallel-decode step over one masked block.
//
// TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded CPU statement of what
// the decode step computes.  Only the test suite, the smoke check and the benchmark's CPU-baseline
// leg may load it; the product path never does.  It shares no code, header or constant with the
// CUDA library: every formula below is written out directly from its definition, in double.
//
// Sources, cited by page title and section:
//   dInfer explainer  = the 91haoming.cn summary of the dInfer paper (arXiv 2510.08666), with its
//                       four components: model; diffusion-iteration manager (iteration smoothing);
//                       decoding strategies (threshold, hierarchical, credit); KV-cache manager
//                       (neighbourhood refresh); plus its engineering notes (early stop at EOS).
// The pages describe each strategy in words only.  The exact formulas used here, and every
// reading taken where the pages are silent, are stated at each function.
//
// Parity status: every function is pinned by the not-gpu tests (closed forms, hand-worked
// examples, brute force, an independent second formulation, textbook GEMM).  Fidelity to the
// dInfer code base itself is unpinned: the pages print no formula.

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <limits>
#include <vector>

namespace {

const double kNegInf = -std::numeric_limits<double>::infinity();

// Exact value of element i of a logits row: dtype 0 = fp32, 1 = bf16 (upper half of an fp32).
double load_logit(const void* row, int dtype, int64_t i) {
  if (dtype == 0) {
    float f;
    std::memcpy(&f, static_cast<const char*>(row) + 4 * i, 4);
    return static_cast<double>(f);
  }
  uint16_t h;
  std::memcpy(&h, static_cast<const char*>(row) + 2 * i, 2);
  uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

double bf16_bits_to_double(uint16_t h) {
  uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// Round a non-negative finite double to the nearest bf16 value (ties to even), returned as a
// double.  bf16 keeps 8 significant bits; normal exponents reach down to 2^-126, subnormals are
// spaced 2^-133 apart.  Computed from the real value directly (no intermediate fp32 rounding).
double round_to_bf16(double x) {
  if (x == 0.0) return 0.0;
  const double min_normal = std::ldexp(1.0, -126);
  if (x < min_normal) {
    return std::nearbyint(std::ldexp(x, 133)) * std::ldexp(1.0, -133);
  }
  int e;
  double f = std::frexp(x, &e);          // x = f * 2^e, f in [0.5, 1)
  double q = std::nearbyint(std::ldexp(f, 8));  // 8 significant bits, ties to even
  return std::ldexp(q, e - 8);
}

// Index of the largest value among the masked positions, lowest index on ties; -1 if none.
int masked_argmax(int L, const uint8_t* masked, const double* value) {
  int best = -1;
  for (int i = 0; i < L; ++i) {
    if (!masked[i]) continue;
    if (best < 0 || value[i] > value[best]) best = i;
  }
  return best;
}

// Apply a commit set: token <- argmax, mask cleared, committed_now set, EOS recorded.
void apply_commits(int L, const std::vector<int>& commit, const int32_t* argmax, uint8_t* masked,
                   int32_t* tokens, uint8_t* committed_now, int32_t* n_commit, int32_t* eos_hit,
                   int eos_id) {
  for (int i = 0; i < L; ++i) committed_now[i] = 0;
  int n = 0;
  for (int i : commit) {
    tokens[i] = argmax[i];
    masked[i] = 0;
    committed_now[i] = 1;
    ++n;
    if (eos_id >= 0 && argmax[i] == eos_id) *eos_hit = 1;
  }
  *n_commit = n;
}

bool sequence_stopped(int L, const uint8_t* masked, const int32_t* eos_hit_b) {
  if (eos_hit_b && *eos_hit_b) return true;
  for (int i = 0; i < L; ++i)
    if (masked[i]) return false;
  return true;
}

// Hierarchical decoding: leaves of the recursive halving of one run [s, e).
void halve(int s, int e, int min_width, std::vector<int>* leaves) {
  int w = e - s;
  if (w >= 2 * min_width) {
    int c = s + w / 2;
    halve(s, c, min_width, leaves);
    halve(c, e, min_width, leaves);
  } else {
    leaves->push_back(s);
    leaves->push_back(e);
  }
}

// Node selections of the halving tree of run [s, e) (see orc_commit_hierarchical_levels).
void select_levels(int s, int e, int min_width, const double* cf, double tau_low,
                   std::vector<uint8_t>* sel) {
  int best = -1, best_dist = 0;
  for (int j = s; j < e; ++j) {
    if (!(cf[j] >= tau_low)) continue;
    const int dist = std::abs(2 * j - (s + e - 1));
    if (best < 0 || dist < best_dist) {
      best = j;
      best_dist = dist;
    }
  }
  if (best >= 0) (*sel)[best] = 1;
  const int w = e - s;
  if (w >= 2 * min_width) {
    const int c = s + w / 2;
    select_levels(s, c, min_width, cf, tau_low, sel);
    select_levels(c, e, min_width, cf, tau_low, sel);
  }
}

}  // namespace

extern "C" {

// Softmax statistics of each row (dInfer explainer, decoding strategies: every strategy ranks
// positions by the model's confidence in its top token).
//   m = max_v z_v, s = sum_v exp(z_v - m), lse = m + ln s, conf = 1/s = exp(m - lse),
//   argmax = lowest v attaining m.
// Rows with active[r] == 0 are not read and report -inf, -inf, 0, -1.  active may be null.
// logits: R rows of V elements, row r at element offset r * row_stride.
int orc_stats(const void* logits, int dtype, int64_t R, int64_t V, int64_t row_stride,
              const uint8_t* active, double* row_max, double* lse, double* conf,
              int32_t* argmax) {
  if (!logits || R < 0 || V <= 0 || row_stride < V || (dtype != 0 && dtype != 1)) return 1;
  const int64_t esize = dtype == 0 ? 4 : 2;
  for (int64_t r = 0; r < R; ++r) {
    if (active && !active[r]) {
      row_max[r] = kNegInf;
      lse[r] = kNegInf;
      conf[r] = 0.0;
      argmax[r] = -1;
      continue;
    }
    const void* row = static_cast<const char*>(logits) + r * row_stride * esize;
    double m = kNegInf;
    int64_t am = -1;
    for (int64_t v = 0; v < V; ++v) {
      double z = load_logit(row, dtype, v);
      if (am < 0 || z > m) {
        m = z;
        am = v;
      }
    }
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) s += std::exp(load_logit(row, dtype, v) - m);
    row_max[r] = m;
    lse[r] = m + std::log(s);
    conf[r] = 1.0 / s;
    argmax[r] = static_cast<int32_t>(am);
  }
  return 0;
}

// Which rows a commit step reads: masked positions of sequences that have not stopped
// (stopped = EOS already hit, or nothing masked; dInfer explainer, engineering notes: early stop).
int orc_active_rows(int B, int L, const uint8_t* masked, const int32_t* eos_hit, uint8_t* active) {
  for (int b = 0; b < B; ++b) {
    bool stopped = eos_hit && eos_hit[b];
    for (int i = 0; i < L; ++i) active[b * L + i] = (!stopped && masked[b * L + i]) ? 1 : 0;
  }
  return 0;
}

// Threshold decoding (dInfer explainer, decoding strategies, method 1: a position is fixed at
// once when the model is confident enough in it).  Reading: commit every masked position whose
// confidence exceeds tau (strictly); if none does, commit the single most confident masked
// position (lowest index on ties) so that every step makes progress.
int orc_commit_threshold(int B, int L, const double* conf, const int32_t* argmax, uint8_t* masked,
                         int32_t* tokens, uint8_t* committed_now, int32_t* n_commit,
                         int32_t* eos_hit, double tau, int eos_id) {
  for (int b = 0; b < B; ++b) {
    const double* cf = conf + b * L;
    uint8_t* mk = masked + b * L;
    std::vector<int> commit;
    if (!sequence_stopped(L, mk, eos_hit + b)) {
      for (int i = 0; i < L; ++i)
        if (mk[i] && cf[i] > tau) commit.push_back(i);
      if (commit.empty()) commit.push_back(masked_argmax(L, mk, cf));
    }
    apply_commits(L, commit, argmax + b * L, mk, tokens + b * L, committed_now + b * L,
                  n_commit + b, eos_hit + b, eos_id);
  }
  return 0;
}

// Hierarchical decoding (dInfer explainer, decoding strategies, method 2: split the region still
// to be filled recursively into smaller sub-regions and decide the centre of each first).
// Reading: maximal masked runs are halved (cut at s + floor(w/2)) while w >= 2*min_width; in each
// leaf the masked position closest to the leaf centre (|2i - (s+e-1)| smallest, lowest i on
// ties) among those with conf >= tau_low is committed; a sequence that commits nothing falls
// back to its most confident masked position.
int orc_commit_hierarchical(int B, int L, const double* conf, const int32_t* argmax,
                            uint8_t* masked, int32_t* tokens, uint8_t* committed_now,
                            int32_t* n_commit, int32_t* eos_hit, double tau_low, int min_width,
                            int eos_id) {
  if (min_width < 1) return 1;
  for (int b = 0; b < B; ++b) {
    const double* cf = conf + b * L;
    uint8_t* mk = masked + b * L;
    std::vector<int> commit;
    if (!sequence_stopped(L, mk, eos_hit + b)) {
      std::vector<int> leaves;  // pairs (s, e)
      int i = 0;
      while (i < L) {
        if (!mk[i]) {
          ++i;
          continue;
        }
        int s = i;
        while (i < L && mk[i]) ++i;
        halve(s, i, min_width, &leaves);
      }
      for (size_t k = 0; k < leaves.size(); k += 2) {
        int s = leaves[k], e = leaves[k + 1];
        int best = -1, best_dist = 0;
        for (int j = s; j < e; ++j) {
          if (!(cf[j] >= tau_low)) continue;
          int dist = std::abs(2 * j - (s + e - 1));
          if (best < 0 || dist < best_dist) {
            best = j;
            best_dist = dist;
          }
        }
        if (best >= 0) commit.push_back(best);
      }
      if (commit.empty()) commit.push_back(masked_argmax(L, mk, cf));
    }
    apply_commits(L, commit, argmax + b * L, mk, tokens + b * L, committed_now + b * L,
                  n_commit + b, eos_hit + b, eos_id);
  }
  return 0;
}

// Credit decoding (dInfer explainer, decoding strategies, method 3: every candidate token of every
// position carries a credit that records how often and how confidently it was chosen over the
// iterations; candidates that stay stable are boosted).  Exact rule used here, per masked
// position with top token a and confidence p:
//   c_k <- decay * c_k for every slot; c_a <- c_a + p (a takes the first empty slot, else evicts
//   the slot of least credit, lowest slot on ties, and starts at p);
//   score = p * (1 + boost * ln(1 + c_a));  commit if score > tau; fallback: largest score.
// cand_id / cand_credit: [B, L, K]; score (nullable) receives the boosted score of active rows.
int orc_commit_credit(int B, int L, const double* conf, const int32_t* argmax, uint8_t* masked,
                      int32_t* tokens, uint8_t* committed_now, int32_t* n_commit,
                      int32_t* eos_hit, int32_t* cand_id, double* cand_credit, int K,
                      double decay, double boost, double tau, int eos_id, double* score_out) {
  if (K < 1) return 1;
  std::vector<double> score(L);
  for (int b = 0; b < B; ++b) {
    const double* cf = conf + b * L;
    uint8_t* mk = masked + b * L;
    std::vector<int> commit;
    if (!sequence_stopped(L, mk, eos_hit + b)) {
      for (int i = 0; i < L; ++i) {
        score[i] = 0.0;
        if (!mk[i]) continue;
        int32_t* ids = cand_id + (static_cast<int64_t>(b) * L + i) * K;
        double* cr = cand_credit + (static_cast<int64_t>(b) * L + i) * K;
        const int32_t a = argmax[b * L + i];
        const double p = cf[i];
        for (int k = 0; k < K; ++k) cr[k] = decay * cr[k];
        int slot = -1;
        for (int k = 0; k < K; ++k)
          if (ids[k] == a) slot = k;
        if (slot >= 0) {
          cr[slot] += p;
        } else {
          for (int k = 0; k < K && slot < 0; ++k)
            if (ids[k] == -1) slot = k;
          if (slot < 0) {
            slot = 0;
            for (int k = 1; k < K; ++k)
              if (cr[k] < cr[slot]) slot = k;
          }
          ids[slot] = a;
          cr[slot] = p;
        }
        score[i] = p * (1.0 + boost * std::log1p(cr[slot]));
      }
      for (int i = 0; i < L; ++i)
        if (mk[i] && score[i] > tau) commit.push_back(i);
      if (commit.empty()) commit.push_back(masked_argmax(L, mk, score.data()));
      if (score_out)
        for (int i = 0; i < L; ++i) score_out[b * L + i] = mk[i] ? score[i] : 0.0;
    } else if (score_out) {
      for (int i = 0; i < L; ++i) score_out[b * L + i] = 0.0;
    }
    apply_commits(L, commit, argmax + b * L, mk, tokens + b * L, committed_now + b * L,
                  n_commit + b, eos_hit + b, eos_id);
  }
  return 0;
}

// Hierarchical decoding, a centre per level (variant of the function above; dInfer explainer,
// decoding strategies, method 2, "decide each centre first" read as: every level's centre is
// decided).  Every node [s, e) of the halving tree of each maximal masked run, internal or leaf,
// selects its eligible position (conf >= tau_low) nearest its centre, |2j - (s + e - 1)|
// smallest, lowest j on ties; the union of the selections is committed; fallback as above.
// Written as a recursive walk over the tree's nodes.
int orc_commit_hierarchical_levels(int B, int L, const double* conf, const int32_t* argmax,
                                   uint8_t* masked, int32_t* tokens, uint8_t* committed_now,
                                   int32_t* n_commit, int32_t* eos_hit, double tau_low,
                                   int min_width, int eos_id) {
  if (min_width < 1) return 1;
  for (int b = 0; b < B; ++b) {
    const double* cf = conf + b * L;
    uint8_t* mk = masked + b * L;
    std::vector<int> commit;
    if (!sequence_stopped(L, mk, eos_hit + b)) {
      std::vector<uint8_t> sel(L, 0);
      int i = 0;
      while (i < L) {
        if (!mk[i]) {
          ++i;
          continue;
        }
        const int s = i;
        while (i < L && mk[i]) ++i;
        select_levels(s, i, min_width, cf, tau_low, &sel);
      }
      for (int j = 0; j < L; ++j)
        if (sel[j]) commit.push_back(j);
      if (commit.empty()) commit.push_back(masked_argmax(L, mk, cf));
    }
    apply_commits(L, commit, argmax + b * L, mk, tokens + b * L, committed_now + b * L,
                  n_commit + b, eos_hit + b, eos_id);
  }
  return 0;
}

// Credit decoding, every tracked candidate credited (variant of orc_commit_credit; dInfer
// explainer, decoding strategies, method 3).  Per masked position with probabilities
// p_v = exp(z_v - lse) (z read from the logits, lse from orc_stats), top token a, p_a = conf:
//   c_k <- decay * c_k for every slot; c_k <- c_k + p_{id_k} for every occupied slot;
//   a not tracked: first empty slot, else evict the least credit (after the gains; lowest slot
//   on ties), starting at p_a;
//   s_k = p_{id_k} * (1 + boost * ln(1 + c_k)) over occupied slots; the best slot (lowest slot
//   on ties) gives the position's score and token; commit if score > tau; fallback: best score.
// token_out (nullable) receives the candidate token of every active row (-1 elsewhere).
int orc_commit_credit_tracked(int B, int L, const void* logits, int dtype, int64_t V,
                              int64_t row_stride, const double* lse, const double* conf,
                              const int32_t* argmax, uint8_t* masked, int32_t* tokens,
                              uint8_t* committed_now, int32_t* n_commit, int32_t* eos_hit,
                              int32_t* cand_id, double* cand_credit, int K, double decay,
                              double boost, double tau, int eos_id, double* score_out,
                              int32_t* token_out) {
  if (K < 1 || !logits || V <= 0 || row_stride < V) return 1;
  const int64_t esize = dtype == 0 ? 4 : 2;
  std::vector<double> score(L);
  std::vector<int32_t> token(L);
  for (int b = 0; b < B; ++b) {
    const double* cf = conf + b * L;
    uint8_t* mk = masked + b * L;
    std::vector<int> commit;
    const bool stopped = sequence_stopped(L, mk, eos_hit + b);
    for (int i = 0; i < L; ++i) {
      score[i] = 0.0;
      token[i] = -1;
      if (stopped || !mk[i]) continue;
      const int64_t r = static_cast<int64_t>(b) * L + i;
      const void* row = static_cast<const char*>(logits) + r * row_stride * esize;
      int32_t* ids = cand_id + r * K;
      double* cr = cand_credit + r * K;
      const int32_t a = argmax[r];
      for (int k = 0; k < K; ++k) {
        cr[k] = decay * cr[k];
        if (ids[k] >= 0) cr[k] += std::exp(load_logit(row, dtype, ids[k]) - lse[r]);
      }
      bool tracked = false;
      for (int k = 0; k < K; ++k)
        if (ids[k] == a) tracked = true;
      if (!tracked) {
        int slot = -1;
        for (int k = 0; k < K && slot < 0; ++k)
          if (ids[k] == -1) slot = k;
        if (slot < 0) {
          slot = 0;
          for (int k = 1; k < K; ++k)
            if (cr[k] < cr[slot]) slot = k;
        }
        ids[slot] = a;
        cr[slot] = cf[i];
      }
      int best = -1;
      double best_s = 0.0;
      for (int k = 0; k < K; ++k) {
        if (ids[k] < 0) continue;
        const double p = std::exp(load_logit(row, dtype, ids[k]) - lse[r]);
        const double sk = p * (1.0 + boost * std::log1p(cr[k]));
        if (best < 0 || sk > best_s) {
          best = k;
          best_s = sk;
        }
      }
      score[i] = best_s;
      token[i] = ids[best];
    }
    if (!stopped) {
      for (int i = 0; i < L; ++i)
        if (mk[i] && score[i] > tau) commit.push_back(i);
      if (commit.empty()) commit.push_back(masked_argmax(L, mk, score.data()));
    }
    if (score_out)
      for (int i = 0; i < L; ++i) score_out[b * L + i] = score[i];
    if (token_out)
      for (int i = 0; i < L; ++i) token_out[b * L + i] = token[i];
    apply_commits(L, commit, token.data(), mk, tokens + b * L, committed_now + b * L,
                  n_commit + b, eos_hit + b, eos_id);
  }
  return 0;
}

// Rows that iteration smoothing carries into the next round: still masked after the commit, in
// sequences that have not stopped, listed in ascending row order (dInfer explainer, diffusion-
// iteration manager: undecided positions keep their distribution instead of dropping it).
int orc_smooth_rows(int B, int L, const uint8_t* masked, const int32_t* eos_hit, int32_t* row_ids,
                    int32_t* M) {
  int n = 0;
  for (int b = 0; b < B; ++b) {
    if (eos_hit && eos_hit[b]) continue;
    for (int i = 0; i < L; ++i)
      if (masked[b * L + i]) row_ids[n++] = b * L + i;
  }
  *M = n;
  return 0;
}

// Soft input embedding of one smoothed row (dInfer explainer, diffusion-iteration manager,
// iteration smoothing): the row's probabilities, each rounded to bf16 (nearest even), weight the
// rows of the embedding table.  S[j, c] = sum_v bf16(exp(z_v - lse)) * E[v, c].
// E: bf16 bit patterns [V, d] row-major.  out: [M, d].
int orc_smooth_embed(const void* logits, int dtype, int64_t V, int64_t row_stride,
                     const double* lse, const int32_t* row_ids, int64_t M, const uint16_t* E,
                     int64_t d, double* out) {
  const int64_t esize = dtype == 0 ? 4 : 2;
  std::vector<double> acc(d);
  for (int64_t j = 0; j < M; ++j) {
    const int64_t r = row_ids[j];
    const void* row = static_cast<const char*>(logits) + r * row_stride * esize;
    for (int64_t c = 0; c < d; ++c) acc[c] = 0.0;
    for (int64_t v = 0; v < V; ++v) {
      double p = round_to_bf16(std::exp(load_logit(row, dtype, v) - lse[r]));
      if (p == 0.0) continue;
      const uint16_t* e = E + v * d;
      for (int64_t c = 0; c < d; ++c) acc[c] += p * bf16_bits_to_double(e[c]);
    }
    for (int64_t c = 0; c < d; ++c) out[j * d + c] = acc[c];
  }
  return 0;
}

// The bf16 probability row itself (for checking the materialised operand).
int orc_prob_row_bf16(const void* logits, int dtype, int64_t V, int64_t row_stride, int64_t r,
                      double lse_r, double* p) {
  const int64_t esize = dtype == 0 ? 4 : 2;
  const void* row = static_cast<const char*>(logits) + r * row_stride * esize;
  for (int64_t v = 0; v < V; ++v) p[v] = round_to_bf16(std::exp(load_logit(row, dtype, v) - lse_r));
  return 0;
}

int orc_round_to_bf16(const double* x, int64_t n, double* y) {
  for (int64_t i = 0; i < n; ++i) y[i] = round_to_bf16(x[i]);
  return 0;
}

// Statistics of rows whose vocabulary is split into n contiguous shards, from each shard's own
// statistics (dInfer explainer, system optimisations: tensor parallelism splits the output layer,
// so each GPU holds the logits of one vocabulary range).  Shard k covers ids
// [offset[k], offset[k] + V_k) and reports, per row r, m_k = row_max[k*R + r],
// lse_k = lse[k*R + r] and its local argmax a_k = argmax[k*R + r] (orc_stats of its columns).
// Each shard's sum is s_k = exp(lse_k - m_k) against its own maximum, so over the whole row
//   m = max_k m_k,   s = sum_k s_k exp(m_k - m) = sum_k exp(lse_k - m),
//   lse = m + ln s,  conf = 1/s,  argmax = lowest offset[k] + a_k over the shards with m_k = m.
// Shards reporting m_k = -inf (row not read) contribute nothing; a row no shard read reports
// -inf, -inf, 0, -1.
int orc_merge_shard_stats(int n, int64_t R, const double* row_max, const double* lse,
                          const int32_t* argmax, const int64_t* offset, double* out_max,
                          double* out_lse, double* out_conf, int32_t* out_argmax) {
  if (n < 1 || R < 0) return 1;
  for (int64_t r = 0; r < R; ++r) {
    double m = kNegInf;
    for (int k = 0; k < n; ++k) m = std::fmax(m, row_max[k * R + r]);
    if (m == kNegInf) {
      out_max[r] = kNegInf;
      out_lse[r] = kNegInf;
      out_conf[r] = 0.0;
      out_argmax[r] = -1;
      continue;
    }
    double s = 0.0;
    int64_t am = -1;
    for (int k = 0; k < n; ++k) {
      const double mk = row_max[k * R + r];
      if (mk == kNegInf) continue;
      s += std::exp(lse[k * R + r] - m);
      if (mk == m) {
        const int64_t g = offset[k] + argmax[k * R + r];
        if (am < 0 || g < am) am = g;
      }
    }
    out_max[r] = m;
    out_lse[r] = m + std::log(s);
    out_conf[r] = 1.0 / s;
    out_argmax[r] = static_cast<int32_t>(am);
  }
  return 0;
}

// Neighbourhood KV refresh (dInfer explainer, KV-cache manager: when a region changes, its cache
// entries and those of its neighbours are recomputed).  Cache row = [prefix 0..P)[block P..P+L);
// refresh[j] = 1 iff a position i committed in this step has |j - (P + i)| <= window.
// idx lists the refreshed j ascending, then -1; count = number refreshed.
int orc_kv_refresh(int B, int L, const uint8_t* committed_now, int prefix_len, int window,
                   uint8_t* refresh, int32_t* idx, int32_t* count) {
  if (prefix_len < 0 || window < 0) return 1;
  const int T = prefix_len + L;
  for (int b = 0; b < B; ++b) {
    int n = 0;
    for (int j = 0; j < T; ++j) {
      uint8_t hit = 0;
      for (int i = 0; i < L; ++i) {
        if (!committed_now[b * L + i]) continue;
        if (std::abs(j - (prefix_len + i)) <= window) hit = 1;
      }
      refresh[static_cast<int64_t>(b) * T + j] = hit;
      if (hit) idx[static_cast<int64_t>(b) * T + n++] = j;
    }
    for (int k = n; k < T; ++k) idx[static_cast<int64_t>(b) * T + k] = -1;
    count[b] = n;
  }
  return 0;
}

}  // extern "C"
