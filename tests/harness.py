"""Shared test machinery: seeded inputs with the decision-margin guard, GPU/oracle runners.

The guard keeps every decision at least 1e-3 away from its threshold (absolute) and from a tie
(relative), so that fp32 on the GPU and double in the oracle decide alike: confidences (or
boosted scores) vs tau, the top-2 gap of a fallback, and the least-credit gap of an eviction.  A draw that violates it
is redrawn with the next attempt number.  Only the oracle is consulted.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth

MARGIN = 1e-3
# Credits carry state across steps, so redrawing one step cannot move a near-tie between two
# stored credits; the eviction guard uses 1e-4 relative, 20x the worst-case fp32 drift of a
# credit over 24 decay-and-add updates (~5e-6 relative).
EVICT_MARGIN = 1e-4
RTOL = 2e-3


def _gap_ok(values: np.ndarray) -> bool:
    """Largest value ahead of the runner-up by MARGIN relative (the fallback pick)."""
    if values.size < 2:
        return True
    top2 = np.sort(values)[-2:]
    return top2[1] - top2[0] >= MARGIN * top2[1]


def _tracked_margins_ok(w, st: oracle.BlockState, lg: np.ndarray, s) -> bool:
    """Tracked-credit variant: the slot to evict (credits after the gains) and the best tracked
    candidate (per-slot boosted scores) must both be separated from the runner-up."""
    B, L, K = st.B, st.L, st.K
    V = lg.shape[-1]
    rows = lg.reshape(B * L, V)
    decay, boost = float(np.float32(w.decay)), float(np.float32(w.boost))
    trial = st.copy()
    oracle.commit_credit_tracked(trial, lg, s, decay, boost, float(np.float32(w.tau)))
    for b in range(B):
        if st.eos_hit[b] or not st.masked[b].any():
            continue
        for i in np.nonzero(st.masked[b])[0]:
            r = b * L + i
            if rows.dtype == np.uint16:  # bf16 bit patterns
                row = (rows[r].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            else:
                row = rows[r].astype(np.float64)
            ids = st.cand_id[b, i]
            p_of = lambda v: float(np.exp(row[v] - s.lse[r]))
            a = int(s.argmax[r])
            if a not in ids and not (ids == -1).any():
                gained = [decay * st.cand_credit[b, i, k] + p_of(ids[k]) for k in range(K)]
                g = np.sort(gained)
                if g.size > 1 and g[1] - g[0] < EVICT_MARGIN * max(g[1], 1e-30):
                    return False
            tid, tc = trial.cand_id[b, i], trial.cand_credit[b, i]
            sc = np.sort([p_of(tid[k]) * (1 + boost * np.log1p(tc[k]))
                          for k in range(K) if tid[k] >= 0])
            if len(sc) > 1 and sc[-1] - sc[-2] < EVICT_MARGIN * sc[-1]:
                return False
    return True


def margins_ok(w, st: oracle.BlockState, conf: np.ndarray, argmax: np.ndarray,
               lg: np.ndarray | None = None, s=None) -> bool:
    """Check the guard for one step of workload w from oracle state st (not mutated)."""
    B, L = st.B, st.L
    conf = conf.reshape(B, L)
    argmax = argmax.reshape(B, L)
    scores = None
    if w.strategy == "credit":
        trial = st.copy()
        scores = oracle.commit_credit(trial, conf, argmax, float(np.float32(w.decay)),
                                      float(np.float32(w.boost)), float(np.float32(w.tau)))
    elif w.strategy == "credit_tracked":
        if not _tracked_margins_ok(w, st, lg, s):
            return False
        trial = st.copy()
        scores, _ = oracle.commit_credit_tracked(trial, lg, s, float(np.float32(w.decay)),
                                                 float(np.float32(w.boost)),
                                                 float(np.float32(w.tau)))
    for b in range(B):
        m = (st.masked[b] == 1) & (st.eos_hit[b] == 0)
        if not m.any():
            continue
        c = conf[b][m]
        if w.strategy in ("threshold", "smooth"):
            if np.any(np.abs(c - float(np.float32(w.tau))) < MARGIN):
                return False
            if not np.any(c > w.tau) and not _gap_ok(c):
                return False
        elif w.strategy in ("hierarchical", "hierarchical_levels"):
            tl = float(np.float32(w.tau_low))
            if np.any(np.abs(c - tl) < MARGIN):
                return False
            # an eligible position always commits in its leaf, so the fallback runs only when
            # no masked position is eligible
            if not np.any(c >= tl) and not _gap_ok(c):
                return False
        elif w.strategy in ("credit", "credit_tracked"):
            s = scores[b][m]
            if np.any(np.abs(s - float(np.float32(w.tau))) < MARGIN):
                return False
            if not np.any(s > w.tau) and not _gap_ok(s):
                return False
            for i in np.nonzero(m)[0] if w.strategy == "credit" else []:
                ids = st.cand_id[b, i]
                if argmax[b, i] in ids or (ids == -1).any():
                    continue
                cr = np.sort(st.cand_credit[b, i])
                if cr.size > 1 and cr[1] - cr[0] < EVICT_MARGIN * max(cr[1], 1e-30):
                    return False
    return True


def oracle_step(w, st: oracle.BlockState, lg: np.ndarray, s=None):
    """One oracle step in place (s: this step's stats if already computed)."""
    if s is None:
        s = oracle.stats(lg, oracle.active_rows(st.masked, st.eos_hit))
    conf = s.conf.reshape(st.B, st.L)
    am = s.argmax.reshape(st.B, st.L)
    scores = None
    if w.strategy in ("threshold", "smooth"):
        oracle.commit_threshold(st, conf, am, float(np.float32(w.tau)), w.eos_id)
    elif w.strategy == "hierarchical":
        oracle.commit_hierarchical(st, conf, am, float(np.float32(w.tau_low)), w.min_width,
                                   w.eos_id)
    elif w.strategy == "hierarchical_levels":
        oracle.commit_hierarchical_levels(st, conf, am, float(np.float32(w.tau_low)),
                                          w.min_width, w.eos_id)
    elif w.strategy == "credit_tracked":
        scores, _ = oracle.commit_credit_tracked(st, lg, s, float(np.float32(w.decay)),
                                                 float(np.float32(w.boost)),
                                                 float(np.float32(w.tau)), w.eos_id)
    else:
        scores = oracle.commit_credit(st, conf, am, float(np.float32(w.decay)),
                                      float(np.float32(w.boost)), float(np.float32(w.tau)),
                                      w.eos_id)
    return s, scores


def guarded_logits(w, seed: int, it: int, st: oracle.BlockState, calibrated: bool = False,
                   max_attempts: int = 50):
    """Logits for step `it` that satisfy the margin guard from oracle state st."""
    for attempt in range(max_attempts):
        lg = synth.logits(w, seed, it, attempt, calibrated)
        act = oracle.active_rows(st.masked, st.eos_hit)
        s = oracle.stats(lg, act)
        if margins_ok(w, st, s.conf, s.argmax, lg, s):
            return lg, attempt, s
    raise RuntimeError(f"no draw satisfied the margin guard after {max_attempts} attempts")


def close(gpu: np.ndarray, ref: np.ndarray, rtol: float = RTOL) -> bool:
    """Relative agreement, with -inf matching -inf."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    inf = np.isinf(ref)
    if not np.array_equal(np.isinf(gpu), inf) or not np.array_equal(gpu[inf], ref[inf]):
        return False
    g, r = gpu[~inf], ref[~inf]
    return bool(np.all(np.abs(g - r) <= rtol * np.abs(r) + 1e-30))
