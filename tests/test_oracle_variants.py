"""Pins for the two strategy variants: hierarchical decoding with a centre per level, and credit
decoding where every tracked candidate gains its own probability."""
import itertools
import math

import numpy as np
import pytest

import oracle


# ------------------------------------------------------------------ hierarchical, every level

def _levels_by_enumeration(mask, conf, tau_low, min_width):
    """Independent formulation: list every node of every run's halving tree with an explicit
    work queue, let each node pick its eligible position nearest its centre by sorting
    (distance, index), take the union; fallback to the best masked confidence."""
    L = len(mask)
    nodes, i = [], 0
    while i < L:
        if not mask[i]:
            i += 1
            continue
        s = i
        while i < L and mask[i]:
            i += 1
        queue = [(s, i)]
        while queue:
            a, b = queue.pop()
            nodes.append((a, b))
            if b - a >= 2 * min_width:
                c = a + (b - a) // 2
                queue += [(a, c), (c, b)]
    chosen = set()
    for a, b in nodes:
        cands = sorted((abs(2 * j - (a + b - 1)), j) for j in range(a, b) if conf[j] >= tau_low)
        if cands:
            chosen.add(cands[0][1])
    if not chosen and any(mask):
        best = max((conf[j], -j) for j in range(L) if mask[j])
        chosen = {-best[1]}
    return sorted(chosen)


def _run_levels(mask, conf, tau_low=0.6, min_width=2):
    L = len(mask)
    st = oracle.BlockState(1, L)
    st.masked[0] = np.array(mask, np.uint8)
    oracle.commit_hierarchical_levels(st, np.array([conf], np.float64),
                                      np.arange(L, dtype=np.int32)[None], tau_low, min_width)
    return sorted(np.flatnonzero(st.committed_now[0]).tolist()), st


def test_levels_hand_example_fills_eight_positions_in_two_steps():
    # root [0,8) -> 3; [0,4) -> 1, [4,8) -> 5; leaves [0,2) -> 0, [2,4) -> 2, [4,6) -> 4,
    # [6,8) -> 6 (every distance tie to the lower index); then the lone position 7
    got, st = _run_levels([1] * 8, [0.7] * 8)
    assert got == [0, 1, 2, 3, 4, 5, 6]
    oracle.commit_hierarchical_levels(st, np.full((1, 8), 0.7), np.arange(8, dtype=np.int32)[None],
                                      0.6, 2)
    assert np.flatnonzero(st.committed_now[0]).tolist() == [7]


@pytest.mark.parametrize("L", [1, 2, 3, 5, 7])
def test_levels_brute_force_against_node_enumeration(L):
    for mask in itertools.product([0, 1], repeat=L):
        if not any(mask):
            continue
        for elig in itertools.product([0, 1], repeat=L):
            conf = [0.61 + 0.01 * j if e else 0.2 + 0.01 * j for j, e in enumerate(elig)]
            got, _ = _run_levels(list(mask), conf)
            assert got == _levels_by_enumeration(mask, conf, 0.6, 2), (mask, elig)


def test_levels_commit_a_superset_of_the_leaves():
    rng = np.random.default_rng(0)
    for _ in range(200):
        L = int(rng.integers(1, 40))
        mask = (rng.random(L) < 0.7).astype(np.uint8)
        if not mask.any():
            continue
        conf = rng.random(L)
        lv, _ = _run_levels(mask, conf)
        st = oracle.BlockState(1, L)
        st.masked[0] = mask
        oracle.commit_hierarchical(st, conf[None], np.arange(L, dtype=np.int32)[None], 0.6, 2)
        leaves = set(np.flatnonzero(st.committed_now[0]).tolist())
        if (conf[mask.astype(bool)] >= 0.6).any():
            assert leaves <= set(lv)


# ------------------------------------------------------------------ credit, every tracked candidate

def _logits_with_probs(V, probs):
    """fp32 row with given probabilities for the listed ids (dict id -> p), the rest shared
    equally by the other ids."""
    rest = (1.0 - sum(probs.values())) / (V - len(probs))
    row = np.full(V, math.log(rest), np.float32)
    for v, p in probs.items():
        row[v] = math.log(p)
    return row


def _credit_run(rows_per_iter, K=4, decay=0.7, boost=0.3, tau=100.0):
    """rows_per_iter: list over iterations of [L, V] fp32 logits; position 0 is the one watched,
    the others are decoys whose boosted scores stay higher so the fallback commits one decoy per
    iteration and position 0 stays masked.  Returns per-iteration (score_0, token_0, ids, c)."""
    L = rows_per_iter[0].shape[0]
    st = oracle.BlockState(1, L, K)
    trace = []
    for lg in rows_per_iter:
        s = oracle.stats(lg, st.masked.reshape(-1))
        score, token = oracle.commit_credit_tracked(st, lg[None], s, decay, boost, tau)
        assert st.masked[0, 0] == 1, "the watched position must stay masked"
        trace.append((score[0, 0], token[0, 0], st.cand_id[0, 0].copy(),
                      st.cand_credit[0, 0].copy()))
    return trace


def _decoys(T, V):
    # decoy rows: one dominant id (conf ~ 0.999), boosted score ~1 > any watched score below
    return [_logits_with_probs(V, {7: 0.999}) for _ in range(T)]


def test_tracked_credit_closed_form_two_candidates():
    V, T, d, b = 32, 6, 0.7, 0.3
    pA, pB, pB1 = 0.30, 0.20, 0.40
    A, B = 3, 5
    iters = []
    for t in range(1, T + 1):
        watched = (_logits_with_probs(V, {B: pB1, A: 0.05}) if t == 1
                   else _logits_with_probs(V, {A: pA, B: pB}))
        iters.append(np.stack([watched] + _decoys(T, V)))
    trace = _credit_run(iters, decay=d, boost=b)
    for t, (score, token, ids, c) in enumerate(trace, start=1):
        cB = d ** (t - 1) * pB1 + pB * (1 - d ** (t - 1)) / (1 - d)   # B tracked from t = 1
        cA = pA * (1 - d ** (t - 1)) / (1 - d) if t >= 2 else None    # A inserted at t = 2
        got = dict(zip(ids.tolist(), c.tolist()))
        assert abs(got[B] - cB) < 1e-6 * max(1.0, cB)
        if t == 1:
            assert A not in got
            sB = pB1 * (1 + b * math.log1p(cB))
            assert token == B and abs(score - sB) < 1e-6
        else:
            assert abs(got[A] - cA) < 1e-6
            sA = pA * (1 + b * math.log1p(cA))
            sB = pB * (1 + b * math.log1p(cB))
            want_tok, want_s = (A, sA) if sA >= sB else (B, sB)
            assert token == want_tok and abs(score - want_s) < 1e-6


def test_tracked_credit_reduces_to_base_when_one_candidate_is_tracked():
    # the same id is top-1 at every iteration and nothing else is ever inserted: the variant's
    # trajectory (credits, scores, commits) must equal the base rule's
    rng = np.random.default_rng(4)
    B_, L, V, K = 1, 6, 64, 8
    st_a = oracle.BlockState(B_, L, K)
    st_b = oracle.BlockState(B_, L, K)
    for it in range(5):
        lg = rng.normal(0, 1, size=(L, V)).astype(np.float32)
        lg[np.arange(L), np.arange(L) + 10] = 4.0 + rng.random(L).astype(np.float32)
        s_a = oracle.stats(lg, st_a.masked.reshape(-1))
        s_b = oracle.stats(lg, st_b.masked.reshape(-1))
        sc_a, _ = oracle.commit_credit_tracked(st_a, lg[None], s_a, 0.7, 0.3, 0.9)
        sc_b = oracle.commit_credit(st_b, s_b.conf.reshape(B_, L), s_b.argmax.reshape(B_, L),
                                    0.7, 0.3, 0.9)
        assert np.array_equal(st_a.masked, st_b.masked)
        assert np.array_equal(st_a.tokens, st_b.tokens)
        assert np.array_equal(st_a.cand_id, st_b.cand_id)
        assert np.allclose(st_a.cand_credit, st_b.cand_credit, rtol=1e-12, atol=0)
        assert np.allclose(sc_a, sc_b, rtol=1e-12, atol=0)


# ------------------------------------------------------------------ eviction, hand-worked

def _two_logit_row(V, top, second):
    """fp32 row whose only finite logits are ln(p) of two tokens (p summing to 1): every other
    token has probability exactly 0."""
    row = np.full(V, -np.inf, np.float32)
    for tok, p in (top, second):
        row[tok] = np.float32(math.log(p))
    return row


def _pair(field):
    tok, p = field.split(":")
    return int(tok), float(p)


def test_tracked_credit_eviction_hand_traces():
    # tests/golden/credit_tracked_eviction_hand.txt: K = 2 slots and three candidates, so every
    # new top-1 token evicts.  Trace 1 is built so that the slot evicted on the credits after
    # the gains differs from the one evicted on the credits before them (or before the decay);
    # trace 2 gives exact credit ties (decay 1, untouched tokens gain exactly 0), which must
    # evict the lowest slot.  The last line of trace 1 commits to a tracked token that is not
    # the top-1.
    import golden_io
    traces = {}
    for f in golden_io.rows("credit_tracked_eviction_hand.txt"):
        traces.setdefault(int(f[0]), []).append(f)
    assert sorted(traces) == [1, 2]
    V = 16
    for tid, lines in traces.items():
        K, decay, boost = int(lines[0][1]), float(lines[0][2]), float(lines[0][3])
        rows = []
        for f in lines:
            watched = _two_logit_row(V, _pair(f[4]), _pair(f[5]))
            rows.append(np.stack([watched] + _decoys(len(lines), V)))
        trace = _credit_run(rows, K=K, decay=decay, boost=boost)
        for it, (f, (score, token, ids, c)) in enumerate(zip(lines, trace), start=1):
            want_ids = golden_io.ints(f[6])
            want_c = golden_io.floats(f[7])
            assert ids.tolist() == want_ids, (tid, it, ids, want_ids)
            assert np.allclose(c, want_c, rtol=0, atol=1e-6), (tid, it, c, want_c)
            assert token == int(f[8]), (tid, it, token)
            assert abs(score - float(f[9])) < 2e-6, (tid, it, score)
