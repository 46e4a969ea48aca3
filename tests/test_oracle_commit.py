"""Pins for the oracle's commit rules: hand-worked fixtures, brute force, invariants."""
import itertools
import math

import numpy as np
import pytest

import oracle
from golden_io import bits, floats, ints, rows


def _state(mask):
    st = oracle.BlockState(1, len(mask), K=8)
    st.masked[0, :] = mask
    return st


def _argmax_ids(L):
    return (np.arange(L, dtype=np.int32) + 100).reshape(1, L)


# ------------------------------------------------------------------ threshold

@pytest.mark.parametrize("row", list(rows("threshold_hand.txt")))
def test_threshold_hand_worked(row):
    tau, mask, conf, expect = float(row[0]), bits(row[1]), floats(row[2]), ints(row[3])
    st = _state(mask)
    am = _argmax_ids(len(mask))
    oracle.commit_threshold(st, np.array([conf]), am, tau)
    got = list(np.nonzero(st.committed_now[0])[0])
    assert got == expect
    for i in expect:
        assert st.tokens[0, i] == am[0, i] and st.masked[0, i] == 0
    assert st.n_commit[0] == len(expect)


def _threshold_properties(mask, conf, tau, committed):
    """The commit set is fixed by these properties alone (uniqueness argument in the test)."""
    masked = [i for i in range(len(mask)) if mask[i]]
    above = [i for i in masked if conf[i] > tau]
    if not masked:
        return committed == []
    if above:
        return committed == above
    best = max(conf[i] for i in masked)
    return committed == [min(i for i in masked if conf[i] == best)]


@pytest.mark.parametrize("L", [1, 2, 5, 8])
def test_threshold_brute_force_patterns(L):
    rng = np.random.default_rng(L)
    tau = 0.9
    for mask in itertools.product([0, 1], repeat=L):
        for above in itertools.product([0, 1], repeat=L):
            conf = np.where(np.array(above) == 1, rng.uniform(0.901, 1.0, L),
                            rng.uniform(0.0, 0.899, L))
            st = _state(mask)
            oracle.commit_threshold(st, conf[None, :], _argmax_ids(L), tau)
            got = list(np.nonzero(st.committed_now[0])[0])
            assert _threshold_properties(mask, conf, tau, got), (mask, conf, got)
            # committed positions are exactly those that left the mask
            assert all(st.masked[0, i] == (mask[i] and i not in got) for i in range(L))


def test_threshold_end_to_end_from_logits():
    # logits rows built to reach given confidences: one entry a, V-1 zeros,
    # conf = e^a/(e^a+V-1)  =>  a = ln(conf (V-1)/(1-conf))
    V = 4096
    target = [0.95, 0.50, 0.92, 0.30]
    lg = np.zeros((4, V), np.float32)
    ids = [17, 4000, 5, 123]
    for r, (c, k) in enumerate(zip(target, ids)):
        lg[r, k] = math.log(c * (V - 1) / (1 - c))
    s = oracle.stats(lg)
    assert np.allclose(s.conf, target, rtol=1e-6)
    st = oracle.BlockState(1, 4)
    oracle.commit_threshold(st, s.conf[None, :], s.argmax[None, :], 0.9)
    assert st.committed_now[0].tolist() == [1, 0, 1, 0]
    assert st.tokens[0].tolist() == [17, -1, 5, -1]


def test_stopped_sequences_do_nothing():
    st = oracle.BlockState(2, 3)
    st.eos_hit[1] = 1
    st.masked[0, :] = 0
    oracle.commit_threshold(st, np.full((2, 3), 0.99), np.zeros((2, 3), np.int32), 0.9)
    assert st.n_commit.tolist() == [0, 0]
    assert st.masked[1].tolist() == [1, 1, 1]


def test_eos_is_recorded_only_for_the_committed_eos_token():
    st = oracle.BlockState(2, 3)
    conf = np.array([[0.95, 0.2, 0.3], [0.1, 0.2, 0.95]])
    am = np.array([[2, 2, 2], [7, 2, 9]], np.int32)
    oracle.commit_threshold(st, conf, am, 0.9, eos_id=2)
    assert st.eos_hit.tolist() == [1, 0]
    assert st.tokens.tolist() == [[2, -1, -1], [-1, -1, 9]]


# ------------------------------------------------------------------ hierarchical

@pytest.mark.parametrize("row", list(rows("hierarchical_hand.txt")))
def test_hierarchical_hand_worked(row):
    tau_low, min_width = row[0].split()
    mask, conf, expect = bits(row[1]), floats(row[2]), ints(row[3])
    st = _state(mask)
    oracle.commit_hierarchical(st, np.array([conf]), _argmax_ids(len(mask)), float(tau_low),
                               int(min_width))
    assert list(np.nonzero(st.committed_now[0])[0]) == expect


def _leaves_by_enumeration(mask, min_width):
    """Second formulation: an explicit work list of intervals instead of recursion."""
    L = len(mask)
    runs, i = [], 0
    while i < L:
        if mask[i]:
            j = i
            while j < L and mask[j]:
                j += 1
            runs.append((i, j))
            i = j
        else:
            i += 1
    leaves, work = [], list(runs)
    while work:
        s, e = work.pop()
        if e - s >= 2 * min_width:
            c = s + (e - s) // 2
            work += [(s, c), (c, e)]
        else:
            leaves.append((s, e))
    return sorted(leaves)


def _hier_expect(mask, conf, tau_low, min_width):
    out = []
    for s, e in _leaves_by_enumeration(mask, min_width):
        el = [i for i in range(s, e) if conf[i] >= tau_low]
        if el:
            out.append(min(el, key=lambda i: (abs(2 * i - (s + e - 1)), i)))
    masked = [i for i in range(len(mask)) if mask[i]]
    if not out and masked:
        best = max(conf[i] for i in masked)
        out = [min(i for i in masked if conf[i] == best)]
    return sorted(out)


@pytest.mark.parametrize("L,min_width", [(6, 2), (9, 2), (10, 1), (10, 3), (12, 2)])
def test_hierarchical_brute_force_against_enumeration(L, min_width):
    rng = np.random.default_rng(L * 10 + min_width)
    for mask in itertools.product([0, 1], repeat=L):
        elig = rng.integers(0, 2, size=L)
        conf = np.where(elig == 1, rng.uniform(0.6, 1.0, L), rng.uniform(0.0, 0.599, L))
        st = _state(mask)
        oracle.commit_hierarchical(st, conf[None, :], _argmax_ids(L), 0.6, min_width)
        got = list(np.nonzero(st.committed_now[0])[0])
        assert got == _hier_expect(mask, conf, 0.6, min_width), (mask, conf)


def test_hierarchical_leaves_cover_runs_with_expected_widths():
    for L in range(1, 40):
        for mw in (1, 2, 3):
            leaves = _leaves_by_enumeration([1] * L, mw)
            assert sum(e - s for s, e in leaves) == L
            assert all(1 <= e - s < 2 * mw for s, e in leaves)


def test_hierarchical_fills_block_in_two_steps_at_uniform_confidence():
    st = oracle.BlockState(1, 8)
    conf = np.full((1, 8), 0.7)
    am = _argmax_ids(8)
    oracle.commit_hierarchical(st, conf, am, 0.6, 2)
    assert st.committed_now[0].tolist() == [1, 0, 1, 0, 1, 0, 1, 0]
    oracle.commit_hierarchical(st, conf, am, 0.6, 2)
    assert st.committed_now[0].tolist() == [0, 1, 0, 1, 0, 1, 0, 1]
    assert st.masked.sum() == 0


# ------------------------------------------------------------------ credit

def _credit_run(p_seq, ids_seq, K=8, decay=0.7, boost=0.3, tau=0.9, decoys=0, decoy_p=None):
    """One tracked position (the last row) behind `decoys` positions of lower index.

    The decoys hold one constant candidate at confidence decoy_p (default: the tracked
    position's first confidence), so their scores are at least the tracked one's and the
    per-step fallback (largest score, lowest index) takes a decoy, not the tracked position.
    """
    L = 1 + decoys
    t = decoys
    dp = p_seq[0] if decoy_p is None else decoy_p
    st = oracle.BlockState(1, L, K=K)
    scores = []
    for p, a in zip(p_seq, ids_seq):
        conf = np.array([[dp] * decoys + [p]])
        am = np.array([[999] * decoys + [a]], np.int32)
        sc = oracle.commit_credit(st, conf, am, decay, boost, tau)
        scores.append(sc[0, t])
        if not st.masked[0, t]:
            break
    return st, scores, t


@pytest.mark.parametrize("p", [0.3, 0.5, 0.7])
def test_credit_closed_form_constant_candidate(p):
    # c_t = p (1 - 0.7^t) / 0.3 and s*_t = p (1 + 0.3 ln(1 + c_t)) for a stable candidate
    d, b = float(np.float32(0.7)), float(np.float32(0.3))
    n = 6
    st, scores, r = _credit_run([p] * n, [42] * n, decay=d, boost=b, tau=0.999, decoys=n)
    assert len(scores) == n
    for t, s in enumerate(scores, start=1):
        c = p * (1 - d ** t) / (1 - d)
        assert s == pytest.approx(p * (1 + b * math.log1p(c)), rel=1e-14)
    assert st.cand_credit[0, r, 0] == pytest.approx(p * (1 - d ** n) / (1 - d), rel=1e-14)
    assert st.cand_id[0, r].tolist() == [42] + [-1] * 7


def test_credit_hand_values_first_commit():
    # p = 0.7: boosted 0.811432, 0.864619, 0.895175, 0.914193 -> commits at step 4 (tau 0.9)
    # (three decoys of equal score and lower index take the fallback of steps 1-3)
    st, scores, r = _credit_run([0.7] * 6, [5] * 6, decoys=3)
    assert [round(s, 6) for s in scores] == [0.811432, 0.864619, 0.895175, 0.914193]
    assert st.masked[0, r] == 0 and st.tokens[0, r] == 5
    assert st.masked[0, :r].sum() == 0
    # p = 0.8 commits at once: 0.8 (1 + 0.3 ln 1.8) = 0.941069
    st, scores, r = _credit_run([0.8], [9], decoys=0)
    assert round(scores[0], 6) == 0.941069 and st.masked[0, r] == 0
    # p = 0.5 stays below 0.9: 0.560820, 0.592278, 0.610933, ...
    st, scores, r = _credit_run([0.5] * 3, [1] * 3, decoys=3)
    assert [round(s, 6) for s in scores] == [0.560820, 0.592278, 0.610933]


def test_credit_eviction_of_least_credit_slot():
    # nine different candidates at equal confidence: the ninth evicts slot 0, whose credit
    # (first inserted, most decayed) is the smallest
    p = 0.2
    st, _, r = _credit_run([p] * 9, list(range(10, 19)), tau=0.999, decoys=9)
    assert st.masked[0, r] == 1
    assert st.cand_id[0, r].tolist() == [18, 11, 12, 13, 14, 15, 16, 17]
    d = 0.7
    expect = [p] + [p * d ** (8 - k) for k in range(1, 8)]
    assert np.allclose(st.cand_credit[0, r], expect, rtol=1e-14)


def test_credit_switching_candidate_resets_to_its_own_credit():
    st, scores, r = _credit_run([0.6, 0.6, 0.6], [1, 2, 1], tau=0.999, decoys=3)
    d = 0.7
    # id 1: 0.6 at step 1, decayed twice plus 0.6 at step 3; id 2 starts over at 0.6
    c1 = 0.6 * d * d + 0.6
    assert scores[1] == pytest.approx(0.6 * (1 + 0.3 * math.log1p(0.6)), rel=1e-14)
    assert scores[2] == pytest.approx(0.6 * (1 + 0.3 * math.log1p(c1)), rel=1e-14)
    assert st.cand_id[0, r, :2].tolist() == [1, 2]


def test_credit_bounds_and_fallback():
    rng = np.random.default_rng(5)
    B, L, K = 4, 16, 8
    st = oracle.BlockState(B, L, K=K)
    for _ in range(10):
        conf = rng.uniform(0, 1, (B, L))
        am = rng.integers(0, 5, (B, L)).astype(np.int32)
        before = st.masked.copy()
        sc = oracle.commit_credit(st, conf, am, 0.7, 0.3, 0.9)
        assert (st.cand_credit >= 0).all() and (st.cand_credit <= 1 / 0.3 + 1e-12).all()
        assert (sc <= conf * (1 + 0.3 * math.log(1 + 1 / 0.3)) + 1e-12).all()
        for b in range(B):
            if before[b].any():
                assert st.n_commit[b] >= 1
                com = np.nonzero(st.committed_now[b])[0]
                if not (sc[b][before[b] == 1] > 0.9).any():
                    best = np.max(sc[b][before[b] == 1])
                    assert list(com) == [int(np.nonzero((sc[b] == best) & (before[b] == 1))[0][0])]
