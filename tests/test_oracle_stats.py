"""Pins for the oracle's softmax statistics: closed forms, brute force, invariants."""
import itertools
import math

import mpmath
import numpy as np
import pytest

import oracle
import synth


def _bf16(x):
    return synth.to_bf16_bits(np.asarray(x, np.float32))


@pytest.mark.parametrize("V", [1, 2, 7, 4096, 126464])
@pytest.mark.parametrize("c", [0.0, -3.5, 1000.0])
def test_constant_rows_closed_form(V, c):
    # z == c everywhere: lse = c + ln V, conf = 1/V, argmax = 0 (lowest of V tied maxima)
    lg = np.full((2, V), c, np.float32)
    st = oracle.stats(lg)
    assert np.allclose(st.lse, c + math.log(V), rtol=0, atol=1e-9 * max(1.0, abs(c)))
    assert np.allclose(st.conf, 1.0 / V, rtol=1e-12, atol=0)
    assert (st.argmax == 0).all()
    assert (st.row_max == c).all()


@pytest.mark.parametrize("V", [2, 16, 4096, 126464])
@pytest.mark.parametrize("a", [-5.0, 0.5, 3.0, 12.0, 30.0])
def test_two_valued_rows_closed_form(V, a):
    # one entry a (bf16-exact), the rest 0: conf = e^a/(e^a + V - 1) when a > 0
    k = V // 3
    lg = np.zeros((1, V), np.float32)
    lg[0, k] = a
    st = oracle.stats(_bf16(lg))
    if a > 0:
        expect_conf = math.exp(a) / (math.exp(a) + V - 1)
        expect_lse = math.log(math.exp(a) + V - 1)
        assert st.argmax[0] == k
        assert st.row_max[0] == a
    else:
        expect_conf = 1.0 / (V - 1 + math.exp(a))
        expect_lse = math.log(V - 1 + math.exp(a))
        assert st.argmax[0] == (0 if k != 0 else 1)
        assert st.row_max[0] == 0.0
    assert st.conf[0] == pytest.approx(expect_conf, rel=1e-11)
    assert st.lse[0] == pytest.approx(expect_lse, rel=1e-11, abs=1e-12)


def _brute(row):
    mpmath.mp.dps = 40
    m = max(row)
    am = min(i for i, z in enumerate(row) if z == m)
    s = mpmath.fsum(mpmath.exp(mpmath.mpf(z) - m) for z in row)
    return m, float(m + mpmath.log(s)), float(1 / s), am


@pytest.mark.parametrize("V", [1, 2, 3, 4, 5])
def test_brute_force_small_grids(V):
    grid = [-2.0, -0.5, 0.0, 1.0, 2.5]  # all exactly representable in bf16
    rows = np.array(list(itertools.product(grid, repeat=V)), np.float32)
    for dt in ("f32", "bf16"):
        lg = rows if dt == "f32" else _bf16(rows)
        st = oracle.stats(lg)
        for r, row in enumerate(rows.tolist()):
            m, lse, conf, am = _brute(row)
            assert st.row_max[r] == m
            assert st.argmax[r] == am, (row, st.argmax[r], am)
            assert st.lse[r] == pytest.approx(lse, rel=1e-14, abs=1e-14)
            assert st.conf[r] == pytest.approx(conf, rel=1e-13)


def test_probabilities_sum_to_one_and_conf_is_top_probability():
    w = synth.WORKLOADS["threshold_loop"].scaled(V=3001)
    lg = synth.logits(w, seed=7)
    st = oracle.stats(lg)
    z = synth.bf16_bits_to_f32(lg).astype(np.float64).reshape(-1, w.V)
    for r in range(z.shape[0]):
        p = np.exp(z[r] - st.lse[r])
        assert abs(p.sum() - 1.0) < 1e-12
        assert p.max() == pytest.approx(st.conf[r], rel=1e-12)
        assert p.argmax() == st.argmax[r]


def test_inactive_rows_are_not_read():
    lg = np.random.default_rng(0).normal(size=(4, 9)).astype(np.float32)
    act = np.array([1, 0, 1, 0], np.uint8)
    st = oracle.stats(lg, act)
    assert np.isneginf(st.lse[[1, 3]]).all() and np.isneginf(st.row_max[[1, 3]]).all()
    assert (st.conf[[1, 3]] == 0).all() and (st.argmax[[1, 3]] == -1).all()
    full = oracle.stats(lg)
    assert np.array_equal(st.lse[[0, 2]], full.lse[[0, 2]])


def test_negative_infinity_entries_contribute_zero():
    lg = np.array([[0.0, -np.inf, 0.0, -np.inf]], np.float32)
    st = oracle.stats(lg)
    assert st.conf[0] == pytest.approx(0.5, rel=1e-15)
    assert st.lse[0] == pytest.approx(math.log(2.0), rel=1e-15)


def test_bf16_decoding_of_bit_patterns():
    # bit patterns with known values: 1.0, -2.0, the largest finite bf16, 2^-133 (min subnormal)
    pats = np.array([[0x3F80, 0xC000, 0x7F7F, 0x0001]], np.uint16)
    st = oracle.stats(pats)
    big = (2 - 2 ** -7) * 2.0 ** 127
    assert st.row_max[0] == big and st.argmax[0] == 2


def test_round_to_bf16_matches_library_conversion_and_ties_to_even():
    import torch
    rng = np.random.default_rng(3)
    x = np.abs(rng.normal(size=20000)).astype(np.float32).astype(np.float64)
    x = np.concatenate([x, np.exp(-rng.uniform(0, 80, size=5000)).astype(np.float32)])
    lib = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_to_bf16(x), lib)
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 2 ** -130 * 1.5, 0.0])
    assert oracle.round_to_bf16(ties).tolist() == [1.0, 1 + 2 ** -6, 2 ** -130 * 1.5, 0.0]
