"""Pins for the oracle's verification of deterministic drafts.

A greedy drafter (bml.asia, the speculative-decoding listing) or a path
selector (rytg.cn, the lightweight-selector paragraph) proposes d_i with
certainty, so its distribution is the point mass q_i = delta_{d_i}. The
general accept rule with that q accepts d_i with probability p_i(d_i) and, at
the first rejection, draws from max(0, p_i - delta_{d_i}), which is p_i with
d_i taken out. Checked here against things the oracle's own code does not
restate:
  * the general verification, fed draft logits whose filtered distribution is
    exactly delta_{d_i}, gives the same tokens and lengths on the same seeds;
  * the accept-length law P(len >= i + 1) = prod_{j < i} p_j(d_j), the
    correction token's law (p_i without d_i, renormalised) and the bonus
    token's law (p_gamma), by chi-square over many requests;
  * the target distribution is kept: the first emitted token follows p_0
    whatever d_0 is (rytg.cn, the lossless paragraph);
  * special cases: a draft outside the kept set is always rejected, a draft
    with p = 1 always accepted, and greedy requests are the argmax prefix.
"""
import numpy as np
import pytest

import oracle
from test_oracle_verify import _chi2_ok


def _one_hot_logits(d, V, dtype=np.float32):
    """Draft logits whose filtered distribution is delta_d for any
    temperature <= 2 and any top-k / top-p: exp(-1e4 / T) underflows to 0."""
    B, gamma = d.shape
    Y = np.full((B, gamma, V), -1.0e4, dtype)
    bi, ii = np.meshgrid(np.arange(B), np.arange(gamma), indexing="ij")
    Y[bi, ii, d] = 0.0
    return Y


@pytest.mark.parametrize("top_k,top_p", [(20, 0.95), (0, 1.0), (5, 0.8), (1, 1.0)])
def test_det_equals_general_rule_with_point_mass_drafts(top_k, top_p):
    rng = np.random.default_rng(7 + top_k)
    B, gamma, V = 96, 5, 40
    X = (rng.standard_normal((B, gamma + 1, V)) * 2.0).astype(np.float32)
    # drafts: half the target row's argmax (often accepted), half uniform
    am = np.argmax(X[:, :gamma], axis=-1)
    d = np.where(rng.random((B, gamma)) < 0.5, am, rng.integers(0, V, (B, gamma))).astype(np.int32)
    T = rng.choice(np.array([0.0, 0.6, 1.0, 1.7], np.float32), B)
    Y = _one_hot_logits(d, V)
    for seed in (1, 99, 2024):
        t1, l1, _, s1 = oracle.verify(X, Y, d, T, top_k, top_p, seed)
        t2, l2, _, s2 = oracle.verify_det(X, d, T, top_k, top_p, seed)
        assert s1 == 0 and s2 == 0
        assert np.array_equal(l1, l2)
        assert np.array_equal(t1, t2)
    # the comparison covered both outcomes
    assert 1 < l2.mean() < gamma + 1


def _det_law_run(X, d, T, top_k, top_p, n, seed):
    gamma1, V = X.shape
    gamma = gamma1 - 1
    Xb = np.broadcast_to(X, (n, gamma + 1, V))
    db = np.broadcast_to(d, (n, gamma))
    tok, ln, _, st = oracle.verify_det(Xb, db, np.full(n, T, np.float32), top_k, top_p, seed)
    assert st == 0
    return tok, ln


DET_LAW_CASES = [
    # V, gamma, T, top_k, top_p
    (6, 3, 1.0, 0, 1.0),
    (8, 3, 0.7, 5, 1.0),
    (8, 2, 1.3, 0, 0.8),
    (7, 4, 1.0, 4, 0.9),
]


@pytest.mark.parametrize("V,gamma,T,top_k,top_p", DET_LAW_CASES)
def test_det_accept_length_and_token_laws(V, gamma, T, top_k, top_p):
    rng = np.random.default_rng(V * 17 + gamma)
    X = (rng.standard_normal((gamma + 1, V)) * 1.2).astype(np.float32)
    p = np.stack([oracle.filter_row(X[i], T, top_k, top_p) for i in range(gamma + 1)])
    # each draft is a kept token of its row, not always the most likely one
    d = np.array([np.argsort(-p[i])[i % 2] for i in range(gamma)], np.int32)
    pd = p[np.arange(gamma), d]
    assert 0.15 < pd.min() and pd.max() < 0.95, "case should accept and reject"
    n = 60000
    tok, ln = _det_law_run(X, d, T, top_k, top_p, n, seed=5 + V)
    surv = np.concatenate([[1.0], np.cumprod(pd)])
    pmf = np.append(surv[:-1] - surv[1:], surv[-1])
    assert _chi2_ok(np.bincount(ln - 1, minlength=gamma + 1), pmf)
    assert abs(ln.mean() - surv.sum()) < 4 * ln.std() / np.sqrt(n)
    # lossless: position 0 emits a sample of p_0
    assert _chi2_ok(np.bincount(tok[:, 0], minlength=V), p[0])
    # a rejection at position i draws from p_i with d_i removed
    for i in range(gamma):
        sel = ln == i + 1
        r = p[i].copy()
        r[d[i]] = 0.0
        assert np.all(tok[sel, i] != d[i])
        assert _chi2_ok(np.bincount(tok[sel, i], minlength=V), r / r.sum())
    # all accepted: the bonus token follows p_gamma
    full = ln == gamma + 1
    assert full.sum() > 300
    assert _chi2_ok(np.bincount(tok[full, gamma], minlength=V), p[gamma])
    # accepted prefix is the drafts, padding is -1
    for b in range(300):
        L = ln[b]
        assert np.array_equal(tok[b, : L - 1], d[: L - 1])
        assert np.all(tok[b, L:] == -1)


def test_det_draft_outside_kept_set_is_always_rejected():
    rng = np.random.default_rng(3)
    V, gamma, n = 12, 3, 20000
    X = (rng.standard_normal((gamma + 1, V)) * 1.5).astype(np.float32)
    p0 = oracle.filter_row(X[0], 1.0, 4, 1.0)
    out = int(np.flatnonzero(p0 == 0)[0])
    d = np.array([out, 0, 0], np.int32)
    tok, ln = _det_law_run(X, d, 1.0, 4, 1.0, n, seed=8)
    assert np.all(ln == 1)
    # removing a token of zero probability leaves p_0 itself
    assert _chi2_ok(np.bincount(tok[:, 0], minlength=V), p0)


def test_det_certain_draft_is_always_accepted():
    rng = np.random.default_rng(4)
    V, gamma, n = 10, 4, 5000
    X = (rng.standard_normal((gamma + 1, V)) * 1.5).astype(np.float32)
    d = np.argmax(X[:gamma], axis=-1).astype(np.int32)
    # top-k 1 keeps only the argmax: p(d) = 1
    tok, ln = _det_law_run(X, d, 1.0, 1, 1.0, n, seed=9)
    assert np.all(ln == gamma + 1)
    assert np.all(tok[:, gamma] == np.argmax(X[gamma]))


def test_det_greedy_requests_are_the_argmax_prefix():
    rng = np.random.default_rng(5)
    B, gamma, V = 64, 6, 33
    X = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    am = np.argmax(X, axis=-1)
    d = am[:, :gamma].copy().astype(np.int32)
    cut = rng.integers(0, gamma + 1, B)
    for b in range(B):
        if cut[b] < gamma:
            d[b, cut[b]] = (am[b, cut[b]] + 1) % V
    tok, ln, _, st = oracle.verify_det(X, d, np.zeros(B, np.float32), 20, 0.95, 1)
    tg, lg, sg = oracle.verify_greedy(X, d)
    assert st == 0 and sg == 0
    assert np.array_equal(ln, np.minimum(cut, gamma) + 1)
    assert np.array_equal(tok, tg) and np.array_equal(ln, lg)


def test_det_status_bits():
    rng = np.random.default_rng(6)
    B, gamma, V = 4, 3, 16
    X = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    d = rng.integers(0, V, (B, gamma)).astype(np.int32)
    T = np.ones(B, np.float32)
    _, _, _, st = oracle.verify_det(X, d, T, 20, 0.95, 1)
    assert st == 0
    d_bad = d.copy()
    d_bad[2, 1] = V
    _, ln, _, st = oracle.verify_det(X, d_bad, T, 20, 0.95, 1)
    assert st & oracle.STATUS_BAD_TOKEN
    assert np.all((ln >= 1) & (ln <= gamma + 1))
    X_bad = X.copy()
    X_bad[1, 2, 5] = np.nan
    _, _, _, st = oracle.verify_det(X_bad, d, T, 20, 0.95, 1)
    assert st & oracle.STATUS_BAD_ROW
