"""Pins for the oracle's verification step.

What the pages fix, checked here:
  * greedy output is the target's own greedy decoding, token for token
    ("greedy output matches the target model exactly", rytg.cn, lossless
    paragraph);
  * sampling keeps the target distribution (bml.asia: rejection sampling
    keeps the output distribution identical; rytg.cn "无损的数学保障"): on tiny
    vocabularies the emitted token at every position follows the filtered
    target distribution p, and acceptance at position i happens with
    probability sum(min(p_i, q_i)), so the accept length has a closed-form law;
  * a bad draft only shortens the accept length (rytg.cn FAQ), and the accept
    length lies in [1, block size].
Sampling laws are checked with chi-square tests over many requests, each with
its own Philox uniforms and its own draft tokens drawn from q by numpy.
"""
import json
import os

import numpy as np
import pytest
from scipy import stats

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_settings.json")


def _chi2_ok(counts, probs, alpha=1e-3):
    counts = np.asarray(counts, np.float64)
    probs = np.asarray(probs, np.float64)
    n = counts.sum()
    assert abs(probs.sum() - 1.0) < 1e-9, "probabilities do not sum to one"
    assert counts[probs == 0].sum() == 0, "an impossible outcome occurred"
    keep = probs > 0
    exp = probs[keep] * n
    obs = counts[keep]
    # merge sparse cells so every expected count is >= 5
    order = np.argsort(exp)
    e_m, o_m, acc_e, acc_o = [], [], 0.0, 0.0
    for i in order:
        acc_e += exp[i]
        acc_o += obs[i]
        if acc_e >= 5:
            e_m.append(acc_e)
            o_m.append(acc_o)
            acc_e = acc_o = 0.0
    if acc_e > 0 and e_m:
        e_m[-1] += acc_e
        o_m[-1] += acc_o
    if len(e_m) < 2:
        return True
    return stats.chisquare(o_m, e_m).pvalue > alpha


def _case(seed, V, gamma, spread):
    rng = np.random.default_rng(seed)
    X = (rng.standard_normal((gamma + 1, V)) * 1.5).astype(np.float32)
    Y = (X[:gamma] + rng.standard_normal((gamma, V)) * spread).astype(np.float32)
    return X, Y


def _law_run(X, Y, T, top_k, top_p, n, seed):
    """n requests sharing the logits, each with its own drafts d ~ q."""
    gamma, V = Y.shape
    p = np.stack([oracle.filter_row(X[i], T, top_k, top_p) for i in range(gamma + 1)])
    q = np.stack([oracle.filter_row(Y[i], T, top_k, top_p) for i in range(gamma)])
    rng = np.random.default_rng(seed + 99)
    d = np.stack([np.searchsorted(np.cumsum(q[i]), rng.random(n) * q[i].sum(), side="right")
                  for i in range(gamma)], 1).astype(np.int32)
    d = np.minimum(d, V - 1)
    Xb = np.broadcast_to(X, (n, gamma + 1, V))
    Yb = np.broadcast_to(Y, (n, gamma, V))
    tok, ln, _, st = oracle.verify(Xb, Yb, d, np.full(n, T, np.float32), top_k, top_p, seed)
    assert st == 0
    return p, q, d, tok, ln


LAW_CASES = [
    # V, gamma, T, top_k, top_p, draft spread
    (6, 3, 1.0, 0, 1.0, 1.5),
    (8, 3, 0.7, 5, 1.0, 1.0),
    (8, 2, 1.3, 0, 0.8, 1.2),
    (7, 3, 1.0, 4, 0.9, 2.0),
]


@pytest.mark.parametrize("V,gamma,T,top_k,top_p,spread", LAW_CASES)
def test_sampling_law_closed_form(V, gamma, T, top_k, top_p, spread):
    X, Y = _case(V * 31 + gamma, V, gamma, spread)
    n = 60000
    p, q, d, tok, ln = _law_run(X, Y, T, top_k, top_p, n, seed=11 + V)
    alpha = np.minimum(p[:gamma], q).sum(1)
    assert 0.2 < alpha.min() and alpha.max() < 0.999, "case should reject often"
    # accept-length law: P(len >= i + 1) = prod_{j < i} alpha_j
    surv = np.concatenate([[1.0], np.cumprod(alpha)])
    pmf = surv[:-1] - surv[1:]
    pmf = np.append(pmf, surv[-1])            # len = gamma + 1: all accepted
    counts = np.bincount(ln - 1, minlength=gamma + 1)
    assert _chi2_ok(counts, pmf)
    se = ln.std() / np.sqrt(n)
    assert abs(ln.mean() - surv.sum()) < 4 * se
    # the token emitted at position 0 follows p_0 (lossless)
    assert _chi2_ok(np.bincount(tok[:, 0], minlength=V), p[0])
    # given position 0 was accepted, the token at position 1 follows p_1
    sel = ln >= 2
    assert _chi2_ok(np.bincount(tok[sel, 1], minlength=V), p[1])
    # the correction token at a rejection follows the normalised residual
    rej0 = ln == 1
    r = np.maximum(p[0] - q[0], 0)
    assert _chi2_ok(np.bincount(tok[rej0, 0], minlength=V), r / r.sum())
    # the bonus token (all accepted) follows p_gamma
    full = ln == gamma + 1
    if full.sum() > 200:
        assert _chi2_ok(np.bincount(tok[full, gamma], minlength=V), p[gamma])
    # accepted tokens are the drafts; padding is -1
    for b in range(200):
        L = ln[b]
        assert np.array_equal(tok[b, : L - 1], d[b, : L - 1])
        assert np.all(tok[b, L:] == -1)


def test_identical_draft_is_always_accepted():
    V, gamma = 8, 4
    X, _ = _case(5, V, gamma, 1.0)
    n = 20000
    p, q, d, tok, ln = _law_run(X, X[:gamma].copy(), 1.0, 5, 0.9, n, seed=3)
    assert np.all(ln == gamma + 1)
    assert _chi2_ok(np.bincount(tok[:, gamma], minlength=V), p[gamma])


def test_draft_outside_target_support_is_rejected():
    V, gamma = 8, 2
    X, Y = _case(6, V, gamma, 0.3)
    p0 = oracle.filter_row(X[0], 1.0, 2, 1.0)
    outside = int(np.nonzero(p0 == 0)[0][0])
    n = 500
    d = np.full((n, gamma), outside, np.int32)
    tok, ln, _, st = oracle.verify(np.broadcast_to(X, (n, gamma + 1, V)),
                                   np.broadcast_to(Y, (n, gamma, V)), d,
                                   np.ones(n, np.float32), 2, 1.0, 17)
    assert np.all(ln == 1)
    assert np.all(p0[tok[:, 0]] > 0)


def _greedy_expected_ok(X, d, tok, ln):
    """Every emitted token is the target argmax at its position; the accept
    length counts the leading drafts that equal it, plus one."""
    am = np.argmax(X, axis=-1)       # numpy: first maximum
    B, g1 = am.shape
    for b in range(B):
        n = 0
        while n < g1 - 1 and d[b, n] == am[b, n]:
            n += 1
        assert ln[b] == n + 1
        assert np.array_equal(tok[b, : n + 1], am[b, : n + 1])
        assert np.all(tok[b, n + 1:] == -1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_greedy_is_target_argmax_decoding(dtype):
    rng = np.random.default_rng(9)
    B, gamma, V = 64, 7, 50
    X = rng.integers(-4, 5, size=(B, gamma + 1, V)).astype(np.float32)   # many ties
    am = np.argmax(X, -1)
    d = np.where(rng.random((B, gamma)) < 0.8, am[:, :gamma], rng.integers(0, V, (B, gamma)))
    d = d.astype(np.int32)
    Xin = synth.f32_to_bf16_bits(X) if dtype == "bf16" else X
    tok, ln, st = oracle.verify_greedy(Xin, d)
    assert st == 0
    _greedy_expected_ok(X, d, tok, ln)
    # the sampling entry with temperature 0 is the same greedy step
    Y = np.zeros((B, gamma, V), Xin.dtype)
    tok2, ln2, _, st2 = oracle.verify(Xin, Y, d, np.zeros(B, np.float32), 20, 0.95, 5)
    assert st2 == 0 and np.array_equal(tok, tok2) and np.array_equal(ln, ln2)


def test_top_k_one_sampling_equals_greedy_for_any_seed():
    rng = np.random.default_rng(10)
    B, gamma, V = 40, 5, 30
    X = (rng.standard_normal((B, gamma + 1, V)) * 2).astype(np.float32)
    Y = (X[:, :gamma] + rng.standard_normal((B, gamma, V))).astype(np.float32)
    d = np.argmax(Y, -1).astype(np.int32)     # the only token q gives mass to
    g_tok, g_len, _ = oracle.verify_greedy(X, d)
    for seed in (0, 1, 77, 2**40 + 3):
        tok, ln, _, st = oracle.verify(X, Y, d, np.ones(B, np.float32), 1, 0.95, seed)
        assert st == 0 and np.array_equal(tok, g_tok) and np.array_equal(ln, g_len)


def test_status_bits_and_bad_inputs():
    rng = np.random.default_rng(12)
    B, gamma, V = 3, 3, 16
    X = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    Y = rng.standard_normal((B, gamma, V)).astype(np.float32)
    d = rng.integers(0, V, (B, gamma)).astype(np.int32)
    T = np.ones(B, np.float32)
    d_bad = d.copy()
    d_bad[1, 0] = V
    d_bad[2, 1] = -1
    tok, ln, _, st = oracle.verify(X, Y, d_bad, T, 5, 0.9, 0)
    assert st == oracle.STATUS_BAD_TOKEN
    assert ln[1] == 1                     # an out-of-range draft is never accepted
    assert np.all((tok >= -1) & (tok < V))
    Xn = X.copy()
    Xn[0, 2, 4] = np.nan
    _, _, _, st = oracle.verify(Xn, Y, d, T, 5, 0.9, 0)
    assert st & oracle.STATUS_BAD_ROW
    _, _, _, st = oracle.verify(X, Y, d, np.array([1.0, -1.0, np.nan], np.float32), 5, 0.9, 0)
    assert st == oracle.STATUS_BAD_TEMPERATURE
    # draft rows of greedy requests are not read
    Yn = Y.copy()
    Yn[0, 0, 0] = np.nan
    _, _, _, st = oracle.verify(X, Yn, d, np.array([0.0, 1.0, 1.0], np.float32), 5, 0.9, 0)
    assert st == 0


def test_page_settings_bound_the_accept_length():
    g = json.load(open(GOLDEN))
    block = g["block_size"]["value"]
    gamma = g["draft_tokens_verified_per_step"]["value"]
    assert gamma == block - 1
    # every acceptance length the pages report fits the definition's range
    for table in ("acceptance_length_dflash2", "acceptance_length_mtp"):
        for v in g[table]["value"].values():
            assert 1.0 <= v <= block
    w = synth.WORKLOADS["b32_mixed_v248320"]
    assert (w["gamma"], w["top_k"], w["top_p"]) == (gamma, g["top_k"]["value"],
                                                    g["top_p"]["value"])
    assert w["V"] > g["mask_token_id"]["value"]
    inp = synth.make_workload("tiny_v1024", data_seed=3)
    B, gm, V = inp.shape
    assert gm == gamma
    lens = []
    for seed in range(40):
        d, _, _ = oracle.sample_rows(inp.draft.reshape(B * gm, V),
                                     synth.draft_sampling_temperatures(inp.temperature, gm),
                                     g["top_k"]["value"], g["top_p"]["value"], seed)
        _, ln, _, st = oracle.verify(inp.target, inp.draft, d.reshape(B, gm), inp.temperature,
                                     g["top_k"]["value"], g["top_p"]["value"], seed)
        assert st == 0
        lens.append(int(ln[0]))
    assert min(lens) >= 1 and max(lens) <= block


def test_tiny_workload_mean_accept_length_matches_closed_form():
    inp = synth.make_workload("tiny_v1024", data_seed=0)
    B, gamma, V = inp.shape
    T, k, tp = float(inp.temperature[0]), inp.top_k, inp.top_p
    # the closed form the benchmark reports (oracle.accept_rates, expected_accept_len)
    alpha = oracle.accept_rates(inp.target, inp.draft, inp.temperature, k, tp)
    expected = float(oracle.expected_accept_len(alpha)[0])
    assert 1.0 <= expected <= gamma + 1
    n = 20000
    rows = np.broadcast_to(inp.draft[0], (n, gamma, V)).reshape(n * gamma, V)
    d, _, _ = oracle.sample_rows(rows, np.full(n * gamma, T, np.float32), k, tp, 1234)
    # each request r uses rows r*gamma .. r*gamma+gamma-1 of the sampler: independent drafts
    d = d.reshape(n, gamma)
    _, ln, _, st = oracle.verify(np.broadcast_to(inp.target, (n, gamma + 1, V)),
                                 np.broadcast_to(inp.draft, (n, gamma, V)), d,
                                 np.full(n, T, np.float32), k, tp, 4321)
    assert st == 0
    assert abs(ln.mean() - expected) < 4 * ln.std() / np.sqrt(n)


def test_sampler_follows_filtered_distribution():
    rng = np.random.default_rng(13)
    V = 8
    x = (rng.standard_normal(V) * 1.5).astype(np.float32)
    n = 40000
    for k, tp, T in ((0, 1.0, 1.0), (5, 0.9, 0.8)):
        p = oracle.filter_row(x, T, k, tp)
        tok, _, st = oracle.sample_rows(np.broadcast_to(x, (n, V)), np.full(n, T, np.float32),
                                        k, tp, 5)
        assert st == 0
        assert _chi2_ok(np.bincount(tok, minlength=V), p)
    tok, _, _ = oracle.sample_rows(np.broadcast_to(x, (10, V)), np.zeros(10, np.float32), 20,
                                   0.95, 5)
    assert np.all(tok == np.argmax(x))


def test_split_margins_recombine():
    """The accept/draw margins are a split of the single margin: same outputs,
    and their minimum is the combined margin (greedy requests keep both open)."""
    inp = synth.make_workload("tiny_v1024", data_seed=3)
    B = 6
    X = np.broadcast_to(inp.target, (B,) + inp.target.shape[1:])
    Y = np.broadcast_to(inp.draft, (B,) + inp.draft.shape[1:])
    gamma, V = inp.shape[1], inp.shape[2]
    # drafts: each request's row argmax for some positions, a random token for others
    rng = np.random.default_rng(5)
    d = np.where(rng.random((B, gamma)) < 0.5, np.argmax(inp.draft[0], axis=-1)[None, :],
                 rng.integers(0, V, (B, gamma))).astype(np.int32)
    T = np.array([1.0, 0.0, 0.7, 1.0, 0.0, 1.3], np.float32)
    for k, tp in ((20, 0.95), (0, 1.0)):
        t1, l1, m, s1 = oracle.verify(X, Y, d, T, k, tp, 11)
        t2, l2, (ma, md), s2 = oracle.verify(X, Y, d, T, k, tp, 11, split_margins=True)
        assert np.array_equal(t1, t2) and np.array_equal(l1, l2) and s1 == s2
        assert np.array_equal(m, np.minimum(ma, md))
        greedy = T == 0
        assert np.all(ma[greedy] > 1e300) and np.all(md[greedy] > 1e300)
        assert np.all(md[~greedy] < 1e300)  # every sampling request draws once


def test_accept_rates_special_cases():
    """alpha = sum min(p, q): 1 for a draft row equal to the target row, 0 when
    the filtered supports are disjoint, NaN for greedy requests; the closed
    form is gamma + 1 when every alpha is 1 and 1 when the first is 0."""
    V, gamma = 64, 3
    rng = np.random.default_rng(4)
    X = (rng.standard_normal((3, gamma + 1, V)) * 2).astype(np.float32)
    Y = X[:, :gamma].copy()
    # request 1: each draft row's top tokens are far below the target's top-5 set
    order = np.argsort(-X[1, :gamma], axis=-1)
    for i in range(gamma):
        Y[1, i] = -10.0
        Y[1, i, order[i, 10:15]] = 5.0
    T = np.array([1.0, 1.0, 0.0], np.float32)
    a = oracle.accept_rates(X, Y, T, 5, 1.0)
    assert np.allclose(a[0], 1.0, atol=1e-12)
    assert np.allclose(a[1], 0.0, atol=1e-12)
    assert np.all(np.isnan(a[2]))
    e = oracle.expected_accept_len(np.array([[1.0, 1.0, 1.0], [0.0, 0.5, 0.5], [0.5, 0.5, 0.5]]))
    assert np.allclose(e, [4.0, 1.0, 1.0 + 0.5 + 0.25 + 0.125])
