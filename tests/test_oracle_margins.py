"""Pins for the oracle's decision margins, reported apart.

The cut margin is the smallest relative gap |before - top_p| / top_p over
the top-p decisions of every row a request filters. Because the mass before
a token only grows along the sorted order, that gap sits at the cut. With
equal logits every probability is dyadic and every mass-before is exact, so
the margin has a closed form. The accept margin, once reported apart, holds
the accept tests alone: with q = p every ratio is 1, every draft is
accepted, and the margin is min_i (1 - u_i) over the request's uniforms.
Without the split, the accept margin is the smaller of the two, as before.
"""
import numpy as np
import pytest

import oracle


def _rows(B, gamma, V, value=0.25):
    X = np.full((B, gamma + 1, V), value, np.float32)
    return X, np.ascontiguousarray(X[:, :gamma])


@pytest.mark.parametrize("V,top_p", [(4, 0.6), (4, 0.5), (8, 0.3), (4, 0.9), (16, 0.95)])
def test_cut_margin_closed_form(V, top_p):
    B, gamma = 3, 2
    X, Y = _rows(B, gamma, V)
    d = np.zeros((B, gamma), np.int32)
    T = np.ones(B, np.float32)
    tp = float(np.float32(top_p))
    # equal logits: p = 1/V each; the cut keeps tokens while before = t/V < top_p
    befores = [t / V for t in range(V)]
    checked = []
    for b in befores:
        checked.append(abs(b - tp) / tp)
        if not (np.float32(b) < np.float32(top_p)):
            break
    want = min(checked)
    for fn in ("verify", "verify_det"):
        if fn == "verify":
            _, ln, (m_acc, m_cut, m_draw), st = oracle.verify(X, Y, d, T, 0, top_p, 5, cut_margin=True)
        else:
            _, ln, (m_acc, m_cut, m_draw), st = oracle.verify_det(X, d, T, 0, top_p, 5, cut_margin=True)
        assert st == 0
        assert np.allclose(m_cut, want, rtol=0, atol=1e-15), (fn, m_cut, want)


def test_accept_margin_alone_is_the_uniforms_gap():
    B, gamma, V = 5, 3, 6
    X, Y = _rows(B, gamma, V)
    d = np.zeros((B, gamma), np.int32)
    T = np.ones(B, np.float32)
    _, ln, (m_acc, m_cut, _), st = oracle.verify(X, Y, d, T, 0, 0.95, 11, cut_margin=True)
    assert st == 0 and np.all(ln == gamma + 1)   # q = p: ratio 1, always accepted
    for b in range(B):
        u = [oracle.uniforms(11, b, i)[0] for i in range(gamma)]
        assert m_acc[b] == pytest.approx(min(1.0 - x for x in u), rel=0, abs=1e-15)
        assert m_acc[b] != m_cut[b]


@pytest.mark.parametrize("top_k,top_p", [(20, 0.95), (0, 0.8), (5, 0.9), (0, 1.0)])
def test_merged_margin_is_the_smaller_of_the_two(top_k, top_p):
    rng = np.random.default_rng(top_k * 7 + 1)
    B, gamma, V = 12, 4, 50
    X = (rng.standard_normal((B, gamma + 1, V)) * 1.5).astype(np.float32)
    Y = (X[:, :gamma] + rng.standard_normal((B, gamma, V)) * 0.7).astype(np.float32)
    T = np.array([1.0, 0.0, 0.7, 1.3] * 3, np.float32)
    d = np.argmax(Y, axis=-1).astype(np.int32)
    t1, l1, (acc, draw), s1 = oracle.verify(X, Y, d, T, top_k, top_p, 3, split_margins=True)
    t2, l2, (acc2, cut, draw2), s2 = oracle.verify(X, Y, d, T, top_k, top_p, 3, cut_margin=True)
    assert np.array_equal(t1, t2) and np.array_equal(l1, l2) and s1 == s2
    assert np.array_equal(acc, np.minimum(acc2, cut)) and np.array_equal(draw, draw2)
    if top_p >= 1.0:
        assert np.all(cut == np.finfo(np.float64).max)   # no top-p decision was taken
    t3, l3, (a3, d3), _ = oracle.verify_det(X, d, T, top_k, top_p, 3, split_margins=True)
    t4, l4, (a4, c4, d4), _ = oracle.verify_det(X, d, T, top_k, top_p, 3, cut_margin=True)
    assert np.array_equal(t3, t4) and np.array_equal(a3, np.minimum(a4, c4)) and np.array_equal(d3, d4)


@pytest.mark.parametrize("V", [4, 8, 16])
def test_draw_margin_is_absolute_closed_form(V):
    """The draw's margin is the absolute gap between u * total and the
    cumulative weights on either side of the chosen token. With equal logits
    and q = p every draft is accepted and the bonus token is drawn from the
    uniform p_gamma: the total is 1, the cumulative weights are (j + 1) / V,
    the token is j = floor(V u), and the margin is min(u - j / V, (j + 1) / V - u)
    (the lower side only when j > 0), in probability units."""
    B, gamma = 6, 2
    X, Y = _rows(B, gamma, V)
    d = np.zeros((B, gamma), np.int32)
    T = np.ones(B, np.float32)
    tok, ln, (m_acc, m_cut, m_draw), st = oracle.verify(X, Y, d, T, 0, 1.0, 21, cut_margin=True)
    assert st == 0 and np.all(ln == gamma + 1)
    for b in range(B):
        u = oracle.uniforms(21, b, gamma)[1]
        j = int(np.floor(V * u))
        assert tok[b, gamma] == j
        want = (j + 1) / V - u
        if j > 0:
            want = min(want, u - j / V)
        assert m_draw[b] == pytest.approx(want, rel=0, abs=1e-15)
