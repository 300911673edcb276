"""Pins of the oracle's LM-head product (logits = h W^T from bf16 values)."""
from fractions import Fraction

import numpy as np

import oracle
import synth


def _bits(x):
    return synth.f32_to_bf16_bits(np.asarray(x, np.float32))


def test_small_worked_product():
    # h = [[1, 2]], W = [[3, 4], [5, 6]]: logits are the rows' dot products 11 and 17
    got = oracle.lmhead_logits(_bits([[1, 2]]), _bits([[3, 4], [5, 6]]))
    assert got.tolist() == [[11.0, 17.0]]


def test_identity_projection_returns_the_hidden_states():
    rng = np.random.default_rng(0)
    h = _bits(rng.standard_normal((5, 8)))
    eye = _bits(np.eye(8))
    got = oracle.lmhead_logits(h, eye)
    assert np.array_equal(got, synth.bf16_bits_to_f32(h).astype(np.float64))


def test_matches_exact_rational_sums():
    rng = np.random.default_rng(1)
    h = _bits(rng.standard_normal((3, 64)))
    w = _bits(rng.standard_normal((4, 64)))
    got = oracle.lmhead_logits(h, w)
    hf = synth.bf16_bits_to_f32(h).astype(np.float64)
    wf = synth.bf16_bits_to_f32(w).astype(np.float64)
    for m in range(3):
        for n in range(4):
            exact = sum(Fraction(float(hf[m, k])) * Fraction(float(wf[n, k])) for k in range(64))
            scale = float(oracle.lmhead_abs(h, w)[m, n])
            assert abs(Fraction(got[m, n]) - exact) <= Fraction(2.0 ** -50) * Fraction(scale)


def test_transposition_and_row_order():
    # W's rows are the vocabulary: swapping two rows of W swaps two logit columns
    rng = np.random.default_rng(2)
    h = _bits(rng.standard_normal((2, 16)))
    w = _bits(rng.standard_normal((3, 16)))
    a = oracle.lmhead_logits(h, w)
    b = oracle.lmhead_logits(h, w[[2, 1, 0]])
    assert np.array_equal(a[:, [2, 1, 0]], b)
    assert a.shape == (2, 3)
