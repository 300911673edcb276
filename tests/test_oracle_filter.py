"""Pins for the oracle's filters (temperature, top-k, top-p) and argmax.

Each check reduces to something other than the oracle itself: scipy's
softmax, numpy's stable sort and argmax, exact properties of the filtered
distribution (support size, prefix and minimality of the top-p set,
probability ratios), and bf16/fp32 equivalence of the same values.
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
import synth


def _rows(seed, n, V, ties=False):
    rng = np.random.default_rng(seed)
    if ties:
        return rng.integers(-3, 4, size=(n, V)).astype(np.float32)
    return (rng.standard_normal((n, V)) * 2).astype(np.float32)


def _order(x):
    """(value desc, index asc) by numpy's stable sort."""
    return np.argsort(-x.astype(np.float64), kind="stable")


@pytest.mark.parametrize("T", [0.3, 0.6, 1.0, 2.5])
def test_unfiltered_is_softmax(T):
    for x in _rows(1, 40, 7):
        p = oracle.filter_row(x, T, 0, 1.0)
        assert np.allclose(p, softmax(x.astype(np.float64) / T), rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("k", [1, 2, 3, 5, 7])
def test_top_k_support_and_ratios(k, ties):
    V = 8
    for x in _rows(2 + k, 60, V, ties):
        T = 0.8
        p = oracle.filter_row(x, T, k, 1.0)
        keep = _order(x)[:k]
        assert set(np.nonzero(p)[0]) == set(keep)
        assert abs(p.sum() - 1.0) < 1e-12
        # inside the kept set the probabilities follow exp(x / T)
        xs = x[keep].astype(np.float64)
        assert np.allclose(p[keep], softmax(xs / T), rtol=1e-12, atol=1e-15)
        idx, prob = oracle.filter_row_sparse(x, T, k, 1.0)
        assert np.array_equal(idx, keep)
        assert np.allclose(prob, p[keep], rtol=0, atol=0)


def test_top_k_one_is_argmax():
    for x in _rows(3, 100, 8, ties=True):
        p = oracle.filter_row(x, 1.0, 1, 1.0)
        assert p[np.argmax(x)] == 1.0 and p.sum() == 1.0


@pytest.mark.parametrize("top_p", [0.05, 0.3, 0.5, 0.8, 0.95, 0.999])
@pytest.mark.parametrize("k", [0, 4, 8])
def test_top_p_is_minimal_prefix(top_p, k):
    V = 8
    for x in _rows(4, 80, V, ties=False):
        T = 1.3
        p = oracle.filter_row(x, T, k, top_p)
        order = _order(x)
        kk = V if k <= 0 else k
        pi = softmax(x[order[:kk]].astype(np.float64) / T)   # mass after top-k
        kept = np.nonzero(p)[0]
        n = len(kept)
        assert set(kept) == set(order[:n]), "kept set is a prefix of the order"
        before_last = pi[: n - 1].sum()
        including_last = pi[:n].sum()
        assert before_last < top_p + 1e-7
        assert n == kk or including_last >= top_p - 1e-7
        assert np.allclose(p[order[:n]], pi[:n] / pi[:n].sum(), rtol=1e-12, atol=1e-15)


def test_top_p_exact_boundary():
    # equal logits with -inf padding give exactly dyadic masses, so the mass
    # before a token can equal top_p exactly: that token is dropped (the kept
    # set is the shortest prefix whose mass reaches top_p)
    x = np.array([0.0, 0.0, -np.inf, -np.inf], np.float32)
    p = oracle.filter_row(x, 1.0, 0, 0.5)
    assert np.array_equal(p, [1.0, 0.0, 0.0, 0.0])
    x = np.array([1.0, 1.0, 1.0, 1.0], np.float32)
    p = oracle.filter_row(x, 1.0, 0, 0.75)
    assert np.array_equal(p, [1 / 3, 1 / 3, 1 / 3, 0.0])
    p = oracle.filter_row(x, 1.0, 0, 0.7500001)
    assert np.array_equal(p, [0.25] * 4)


def test_top_p_keeps_at_least_one_token():
    x = np.array([5.0, 0.0, 0.0, 0.0], np.float32)
    p = oracle.filter_row(x, 1.0, 0, 1e-6)
    assert p[0] == 1.0 and p[1:].sum() == 0.0


def test_bf16_rows_equal_their_fp32_values():
    x = _rows(5, 30, 64)
    xb = synth.f32_to_bf16_bits(x)
    xf = synth.bf16_bits_to_f32(xb)
    for a, b in zip(xb, xf):
        for k, tp in ((20, 0.95), (0, 1.0), (5, 0.5)):
            assert np.array_equal(oracle.filter_row(a, 0.7, k, tp), oracle.filter_row(b, 0.7, k, tp))
        assert oracle.argmax_row(a) == oracle.argmax_row(b)


def test_shift_invariance():
    x = np.round(_rows(6, 20, 16) * 8) / 8   # exactly representable after a shift
    for r in x:
        p0 = oracle.filter_row(r, 1.0, 5, 0.9)
        p1 = oracle.filter_row((r + np.float32(64.0)).astype(np.float32), 1.0, 5, 0.9)
        assert np.allclose(p0, p1, rtol=0, atol=1e-12)


def test_temperature_sharpens():
    x = _rows(7, 1, 16)[0]
    top = np.argmax(x)
    prev = 0.0
    for T in (4.0, 2.0, 1.0, 0.5, 0.25, 0.05):
        p = oracle.filter_row(x, T, 0, 1.0)
        assert p[top] >= prev - 1e-15
        prev = p[top]
    assert prev > 0.99


def test_argmax_matches_numpy_first_max():
    for x in _rows(8, 200, 33, ties=True):
        j, st = oracle.argmax_row(x)
        assert j == int(np.argmax(x)) and st == 0
    # -0 and +0 are the same value: the lower index wins
    x = np.array([-1.0, -0.0, 0.0, -2.0], np.float32)
    assert oracle.argmax_row(x)[0] == 1


def test_bad_rows_are_flagged():
    x = np.zeros(8, np.float32)
    x[3] = np.nan
    assert oracle.argmax_row(x)[1] == oracle.STATUS_BAD_ROW
    assert oracle.filter_row(x, 1.0, 3, 0.9) is None
    x = np.full(8, -np.inf, np.float32)
    assert oracle.argmax_row(x)[1] == oracle.STATUS_BAD_ROW
    x = np.zeros(8, np.float32)
    x[5] = np.inf
    assert oracle.argmax_row(x)[1] == oracle.STATUS_BAD_ROW
    # -inf entries inside a finite row are fine and get probability 0
    x = np.array([1.0, -np.inf, 0.5, -np.inf], np.float32)
    p = oracle.filter_row(x, 1.0, 3, 1.0)
    assert p[1] == 0.0 and p[3] == 0.0 and abs(p.sum() - 1) < 1e-12
