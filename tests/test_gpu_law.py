"""The lossless sampling law, checked on the GPU path itself.

The pages' guarantee is that speculative sampling leaves the output
distribution unchanged: the token emitted at every position follows the
target's own filtered distribution ("DFlash2 用投机解码给 Qwen 提速",
bml.asia: rejection sampling keeps the output distribution identical;
"无损加速是真的吗？Qwen3.8-27B-DFlash2如何保证输出与目标模型完全一致",
rytg.cn, "无损的数学保障"). On vocabularies of at most 8 tokens the laws have
closed forms, computed here from the oracle's fp64 filtered distributions
p_i, q_i:
  * position i is reached with probability prod_{j<i} alpha_j, alpha_j =
    sum_v min(p_j(v), q_j(v)): the accept-length law and its mean;
  * the token emitted at position 0 follows p_0; given position 0 accepted,
    the token at position 1 follows p_1;
  * after a rejection at position 0 the token follows max(0, p_0 - q_0)
    normalised;
  * when every draft is accepted, the bonus token follows p_gamma.
Each case runs 10^5 requests through dflash_verify (B = 2048 per call, every
request with its own uniforms and its own drafts d ~ q drawn by numpy), and
each law is a chi-square goodness-of-fit test at level 1e-3.
"""
import numpy as np
import pytest
from scipy import stats

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"
N = 100_000
CALL = 2048


@pytest.fixture(scope="module")
def dv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_83_gb300 as m

    m.build()
    m.load()
    return m


def _chi2_ok(counts, probs, alpha=1e-3):
    """Pearson chi-square of observed counts against probabilities, cells
    merged (smallest expected first) until every expected count is >= 5; an
    outcome of probability 0 must never occur."""
    counts = np.asarray(counts, np.float64)
    probs = np.asarray(probs, np.float64)
    probs = probs / probs.sum()
    assert counts[probs == 0].sum() == 0, "an impossible outcome occurred"
    keep = probs > 0
    exp, obs = probs[keep] * counts.sum(), counts[keep]
    e_m, o_m, acc_e, acc_o = [], [], 0.0, 0.0
    for i in np.argsort(exp):
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


CASES = [
    # V, gamma, T, top_k, top_p, draft spread, dtype
    (6, 3, 1.0, 0, 1.0, 1.5, "f32"),     # full-vocabulary softmax
    (8, 3, 0.7, 5, 1.0, 1.0, "f32"),     # top-k
    (7, 3, 1.0, 4, 0.9, 2.0, "bf16"),    # top-k and top-p
    (8, 2, 1.3, 7, 0.8, 1.2, "f32"),     # top-p with a top-k that drops one token
    (8, 3, 1.0, 0, 0.85, 1.0, "f32"),    # top-p over the full vocabulary (top-k off)
    (7, 3, 0.9, 0, 0.7, 1.5, "bf16"),
]


def _logits(seed, V, gamma, spread, dtype):
    rng = np.random.default_rng(seed)
    X = (rng.standard_normal((gamma + 1, V)) * 1.5).astype(np.float32)
    Y = (X[:gamma] + rng.standard_normal((gamma, V)) * spread).astype(np.float32)
    if dtype == "bf16":
        X, Y = synth.f32_to_bf16_bits(X), synth.f32_to_bf16_bits(Y)
    return X, Y


@pytest.mark.parametrize("V,gamma,T,top_k,top_p,spread,dtype", CASES)
def test_gpu_sampling_law(dv, V, gamma, T, top_k, top_p, spread, dtype):
    X, Y = _logits(V * 131 + gamma, V, gamma, spread, dtype)
    p = np.stack([oracle.filter_row(X[i], T, top_k, top_p) for i in range(gamma + 1)])
    q = np.stack([oracle.filter_row(Y[i], T, top_k, top_p) for i in range(gamma)])
    alpha = np.minimum(p[:gamma], q).sum(1)
    assert 0.2 < alpha.min() and alpha.max() < 0.999, "the case should reject often"
    rng = np.random.default_rng(V + 7)
    Xd = synth.to_torch(np.ascontiguousarray(np.broadcast_to(X, (CALL, gamma + 1, V))), DEV)
    Yd = synth.to_torch(np.ascontiguousarray(np.broadcast_to(Y, (CALL, gamma, V))), DEV)
    Td = torch.full((CALL,), T, dtype=torch.float32, device=DEV)
    toks, lens = [], []
    for call in range((N + CALL - 1) // CALL):
        d = np.stack([np.minimum(np.searchsorted(np.cumsum(q[i]), rng.random(CALL) * q[i].sum(), side="right"),
                                 V - 1) for i in range(gamma)], 1).astype(np.int32)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        tok, ln = dv.verify(Xd, Yd, torch.from_numpy(d).to(DEV), Td, top_k, top_p, 1000 + call, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        toks.append(tok.cpu().numpy())
        lens.append(ln.cpu().numpy())
    tok, ln = np.concatenate(toks)[:N], np.concatenate(lens)[:N]
    assert ln.min() >= 1 and ln.max() <= gamma + 1
    # accept-length law P(len >= i + 1) = prod_{j<i} alpha_j, and its mean
    surv = np.concatenate([[1.0], np.cumprod(alpha)])
    pmf = np.append(surv[:-1] - surv[1:], surv[-1])
    assert _chi2_ok(np.bincount(ln - 1, minlength=gamma + 1), pmf)
    assert abs(ln.mean() - surv.sum()) < 4 * ln.std() / np.sqrt(N)
    # the token at position 0 follows p_0 (lossless), position 1 given position 0 accepted follows p_1
    assert _chi2_ok(np.bincount(tok[:, 0], minlength=V), p[0])
    sel = ln >= 2
    assert _chi2_ok(np.bincount(tok[sel, 1], minlength=V), p[1])
    # the correction token after a rejection at position 0
    r = np.maximum(p[0] - q[0], 0.0)
    assert _chi2_ok(np.bincount(tok[ln == 1, 0], minlength=V), r)
    # the bonus token when every draft is accepted
    full = ln == gamma + 1
    if full.sum() > 500:
        assert _chi2_ok(np.bincount(tok[full, gamma], minlength=V), p[gamma])


def test_gpu_sampling_law_deterministic_drafts(dv):
    """With deterministic drafts (q = the point mass at d) the output still
    follows p whatever the drafts: the token at position 0 follows p_0, the
    draft is accepted with probability p_0(d_0), and after its rejection the
    token follows p_0 without d_0."""
    V, gamma, T = 8, 3, 1.0
    X, _ = _logits(99, V, gamma, 1.0, "f32")
    p = np.stack([oracle.filter_row(X[i], T, 0, 1.0) for i in range(gamma + 1)])
    d_fixed = np.argsort(-p[:gamma], axis=1)[:, 1].astype(np.int32)  # each position's second choice
    Xd = synth.to_torch(np.ascontiguousarray(np.broadcast_to(X, (CALL, gamma + 1, V))), DEV)
    Td = torch.full((CALL,), T, dtype=torch.float32, device=DEV)
    dd = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(d_fixed, (CALL, gamma)))).to(DEV)
    toks, lens = [], []
    for call in range((N + CALL - 1) // CALL):
        tok, ln = dv.verify_det(Xd, dd, Td, 0, 1.0, 5000 + call)
        torch.cuda.synchronize()
        toks.append(tok.cpu().numpy())
        lens.append(ln.cpu().numpy())
    tok, ln = np.concatenate(toks)[:N], np.concatenate(lens)[:N]
    assert _chi2_ok(np.bincount(tok[:, 0], minlength=V), p[0])
    acc0 = (ln >= 2).mean()
    assert abs(acc0 - p[0, d_fixed[0]]) < 4 * np.sqrt(p[0, d_fixed[0]] * (1 - p[0, d_fixed[0]]) / N)
    rej = ln == 1
    r = p[0].copy()
    r[d_fixed[0]] = 0.0
    assert np.all(tok[rej, 0] != d_fixed[0])
    assert _chi2_ok(np.bincount(tok[rej, 0], minlength=V), r)
