"""Pins for iteration smoothing and the neighbourhood KV refresh, plus loop invariants."""
import itertools

import numpy as np
import pytest

import oracle
import synth
from golden_io import ints, rows


def _table(V, d, seed=11):
    return synth.embedding_table(seed, V, d)


def test_one_hot_rows_give_embedding_rows_exactly():
    V, d = 300, 24
    E = _table(V, d)
    lg = np.full((3, V), -200.0, np.float32)
    hot = [0, 123, 299]
    for r, k in enumerate(hot):
        lg[r, k] = 200.0
    st = oracle.stats(lg)
    S = oracle.smooth_embed(lg, st.lse, np.arange(3, dtype=np.int32), E)
    Ef = synth.bf16_bits_to_f32(E).astype(np.float64)
    for r, k in enumerate(hot):
        assert np.array_equal(S[r], Ef[k])


def test_uniform_rows_give_column_mean():
    V, d = 256, 16  # 1/256 is exact in bf16
    E = _table(V, d)
    lg = np.full((2, V), 0.75, np.float32)
    st = oracle.stats(lg)
    S = oracle.smooth_embed(lg, st.lse, np.array([1], np.int32), E)
    Ef = synth.bf16_bits_to_f32(E).astype(np.float64)
    assert np.allclose(S[0], Ef.mean(axis=0), rtol=1e-13, atol=1e-16)


def test_smoothing_is_the_textbook_product_of_bf16_probabilities_and_table():
    w = synth.WORKLOADS["smooth_step"].scaled(B=2, L=4, V=1000, d=40)
    lg = synth.logits(w, seed=3)
    E = _table(w.V, w.d)
    st = oracle.stats(lg)
    ids = np.array([0, 3, 5, 6], np.int32)
    S = oracle.smooth_embed(lg, st.lse, ids, E)
    Ef = synth.bf16_bits_to_f32(E).astype(np.float64)
    z = synth.bf16_bits_to_f32(lg).reshape(-1, w.V).astype(np.float64)
    for j, r in enumerate(ids):
        p = oracle.prob_row_bf16(lg, r, st.lse[r])
        # each probability is the bf16 neighbour of exp(z - lse): bf16 keeps 8 significant bits,
        # so the rounding error is at most half an ulp, 2^-8 relative
        exact = np.exp(z[r] - st.lse[r])
        assert (np.abs(p - exact) <= exact * 2.0 ** -8 * (1 + 1e-12)).all()
        assert abs(p.sum() - 1.0) <= 2.0 ** -8
        assert np.allclose(S[j], p @ Ef, rtol=1e-12, atol=1e-15)


def test_smooth_rows_select_masked_rows_of_running_sequences():
    masked = np.array([[1, 0, 1], [1, 1, 1], [0, 0, 1]], np.uint8)
    eos = np.array([0, 1, 0], np.int32)
    assert oracle.smooth_rows(masked, eos).tolist() == [0, 2, 8]


@pytest.mark.parametrize("row", list(rows("kv_refresh_hand.txt")))
def test_kv_refresh_hand_worked(row):
    P, w, L = ints(row[0])
    com = np.zeros((1, L), np.uint8)
    com[0, ints(row[1])] = 1
    refresh, idx, count = oracle.kv_refresh(com, P, w)
    expect = ints(row[2])
    assert count[0] == len(expect)
    assert idx[0, : count[0]].tolist() == expect
    assert (idx[0, count[0]:] == -1).all()
    assert list(np.nonzero(refresh[0])[0]) == expect


@pytest.mark.parametrize("L,P,w", [(4, 0, 0), (5, 3, 1), (8, 16, 4), (16, 2, 3), (16, 16, 6)])
def test_kv_refresh_brute_force_interval_union(L, P, w):
    T = P + L
    patterns = itertools.product([0, 1], repeat=L) if L <= 8 else (
        np.random.default_rng(L).integers(0, 2, size=(300, L)))
    for pat in patterns:
        com = np.array([pat], np.uint8)
        refresh, idx, count = oracle.kv_refresh(com, P, w)
        cover = set()
        for i in np.nonzero(com[0])[0]:
            cover.update(range(max(0, P + i - w), min(T, P + i + w + 1)))
        assert sorted(cover) == idx[0, : count[0]].tolist()
        assert refresh[0].sum() == len(cover)


def test_threshold_loop_invariants():
    w = synth.WORKLOADS["threshold_loop"].scaled(B=3, L=16, V=2003)
    st = oracle.BlockState(w.B, w.L)
    prev_tokens = st.tokens.copy()
    for it in range(w.max_iters):
        lg = synth.logits(w, seed=21, it=it, calibrated=True)
        act = oracle.active_rows(st.masked, st.eos_hit)
        s = oracle.stats(lg, act)
        before = st.masked.copy()
        running = (before.sum(1) > 0) & (st.eos_hit == 0)
        oracle.commit_threshold(st, s.conf.reshape(w.B, w.L), s.argmax.reshape(w.B, w.L), w.tau,
                                w.eos_id)
        assert ((st.masked <= before)).all()
        done = before == 0
        assert np.array_equal(st.tokens[done], prev_tokens[done])
        assert (st.n_commit[running] >= 1).all() and (st.n_commit[~running] == 0).all()
        prev_tokens = st.tokens.copy()
        if not running.any():
            break
    assert ((st.masked.sum(1) == 0) | (st.eos_hit == 1)).all()
