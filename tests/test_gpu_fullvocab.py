"""GPU parity of the full-vocabulary mode (top-k off, top-p 1) against the oracle.

With no top-k, the filtered distributions are the softmax over all V tokens.
The residual max(0, p - q) and the bonus draw then span the whole vocabulary.
At V = 248320 neighbouring cumulative weights are a few parts per million
apart, so the draw is compared at fp32 resolution.

Bars:
- Greedy requests and status words are bit-exact.
- A sampling request must match the oracle exactly (tokens and accept length)
  unless the oracle's margins put a decision within the GPU's rounding
  (parity_bounds: the accept test on the stream's fp32 normalisers, relative
  FV_ACCEPT_REL; the float-float draw, absolute FV_DRAW_ABS = 2^-22).
- Such near-boundary mismatches stay under 0.01% of requests.
"""
import numpy as np
import pytest

import oracle
import synth
from parity_bounds import FV_DRAW_ABS, ROW_BAR, compare_rows, excused_fullvocab

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def dv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_83_gb300 as m

    m.build()
    m.load()
    return m


def _t(a):
    return synth.to_torch(a, DEV)


def _draft_tokens(Y, T, seed):
    """Drafts sampled from the full-vocabulary draft distributions (oracle
    sampler; greedy requests take the draft row's argmax)."""
    B, gamma, V = Y.shape
    d, _, _ = oracle.sample_rows(Y.reshape(B * gamma, V), synth.draft_sampling_temperatures(T, gamma),
                                 0, 1.0, seed)
    return d.reshape(B, gamma)


def _run(dv, X, Y, d, T, seed, ws=None, Xd=None, Yd=None):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok, ln = dv.verify(_t(X) if Xd is None else Xd, _t(Y) if Yd is None else Yd,
                        torch.from_numpy(np.ascontiguousarray(d)).to(DEV),
                        torch.from_numpy(np.ascontiguousarray(T, np.float32)).to(DEV), 0, 1.0, seed,
                        status=st, workspace=ws)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), ln.cpu().numpy(), int(st.item())


def _check(dv, X, Y, d, T, seed, **kw):
    """Returns (mismatches, requests); asserts every mismatch is near a boundary."""
    want_tok, want_len, (m_acc, m_draw), want_st = oracle.verify(X, Y, d, T, 0, 1.0, seed,
                                                                 split_margins=True)
    tok, ln, st = _run(dv, X, Y, d, T, seed, **kw)
    assert st == want_st
    g = T == 0
    assert np.array_equal(tok[g], want_tok[g]) and np.array_equal(ln[g], want_len[g])
    n_bad = compare_rows(tok, ln, want_tok, want_len, lambda b: excused_fullvocab(m_acc[b], m_draw[b]))
    return n_bad, len(ln)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V,gamma", [(1024, 7), (777, 7), (20000, 15), (4097, 3), (1, 2), (33, 32)])
def test_fullvocab_small(dv, dtype, V, gamma):
    n_bad = total = 0
    for data_seed in range(3):
        X, Y, _ = synth.make_logits(9, gamma, V, dtype, data_seed=data_seed, sigma_d=0.5)
        T = np.array([1.0, 0.0, 0.6, 1.0, 1.5, 0.0, 0.8, 1.0, 2.0], np.float32)
        d = _draft_tokens(Y, T, 50 + data_seed)
        for seed in (data_seed, 777 + data_seed):
            nb, nt = _check(dv, X, Y, d, T, seed)
            n_bad += nb
            total += nt
    assert n_bad <= ROW_BAR * total


def test_fullvocab_identical_drafts_take_the_bonus(dv):
    """Y == X accepts every draft (p/q = 1); the bonus draw spans the vocabulary."""
    X, _, _ = synth.make_logits(16, 7, 50000, "f32", data_seed=21)
    Y = np.ascontiguousarray(X[:, :7, :])
    T = np.full(16, 1.0, np.float32)
    d = _draft_tokens(Y, T, 3)
    tok, ln, st = _run(dv, X, Y, d, T, 99)
    assert st == 0 and np.all(ln == 8)
    want_tok, want_len, (m_acc, m_draw), _ = oracle.verify(X, Y, d, T, 0, 1.0, 99, split_margins=True)
    assert np.array_equal(want_len, ln)
    diff = np.nonzero(np.any(tok != want_tok, axis=1))[0]
    assert all(m_draw[b] < FV_DRAW_ABS for b in diff) and len(diff) <= ROW_BAR * len(ln)


def test_fullvocab_temperatures_and_misaligned_rows(dv):
    """Rows off a 16-byte boundary (the stream's head and tail logits) and
    temperatures other than 1 (the float-float 1/T)."""
    B, gamma, V = 6, 5, 30001
    for dtype in ("f32", "bf16"):
        X, Y, _ = synth.make_logits(B, gamma, V, dtype, data_seed=31, sigma_d=0.7)
        T = np.array([0.3, 1.7, 0.0, 0.9, 1.1, 2.5], np.float32)
        d = _draft_tokens(Y, T, 9)
        # the same values, one element later in the allocation
        fx = _t(np.concatenate([X.reshape(-1)[:1], X.reshape(-1)]))
        fy = _t(np.concatenate([Y.reshape(-1)[:1], Y.reshape(-1)]))
        Xd, Yd = fx[1:].view(B, gamma + 1, V), fy[1:].view(B, gamma, V)
        assert Xd.data_ptr() % 16 != 0
        n_bad, total = _check(dv, X, Y, d, T, 5, Xd=Xd, Yd=Yd)
        assert n_bad <= ROW_BAR * total


def test_fullvocab_status_bits(dv):
    B, gamma, V = 5, 4, 6007
    X, Y, _ = synth.make_logits(B, gamma, V, "f32", data_seed=41)
    T = np.array([1.0, 1.0, 1.0, -2.0, 1.0], np.float32)
    d = _draft_tokens(Y, np.abs(T), 2)
    d[0, 1] = V          # a token outside the vocabulary is never accepted
    X = X.copy()
    X[1, 3, 100] = np.nan  # a bad row
    Y = Y.copy()
    Y[4, 0, :] = -np.inf   # a draft row with no finite logit
    want_tok, want_len, _, want_st = oracle.verify(X, Y, d, T, 0, 1.0, 6)
    tok, ln, st = _run(dv, X, Y, d, T, 6)
    assert st == want_st == (oracle.STATUS_BAD_TOKEN | oracle.STATUS_BAD_ROW
                             | oracle.STATUS_BAD_TEMPERATURE)
    assert np.all((tok >= -1) & (tok < V)) and np.all((ln >= 1) & (ln <= gamma + 1))
    # a request whose loop stops before its bad row, and the greedy one, agree
    for b in (0, 2, 3):
        assert np.array_equal(tok[b], want_tok[b]) and ln[b] == want_len[b]


def test_fullvocab_workspace_shared_with_top_k_calls(dv):
    """One workspace serves full-vocabulary and top-k calls in turn."""
    B, gamma, V = 4, 7, 9000
    X, Y, _ = synth.make_logits(B, gamma, V, "bf16", data_seed=51)
    T = np.array([1.0, 0.6, 0.0, 1.0], np.float32)
    d = _draft_tokens(Y, T, 4)
    ws = dv.Workspace(max(dv.workspace_bytes(B, gamma, V, dv.DFLASH_BF16, 0, 1.0),
                          dv.workspace_bytes(B, gamma, V, dv.DFLASH_BF16, 20, 0.95)), DEV)
    first = _run(dv, X, Y, d, T, 8, ws=ws)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dv.verify(_t(X), _t(Y), torch.from_numpy(d).to(DEV), torch.from_numpy(T).to(DEV), 20, 0.95, 8,
              status=st, workspace=ws)
    again = _run(dv, X, Y, d, T, 8, ws=ws)
    assert np.array_equal(first[0], again[0]) and np.array_equal(first[1], again[1])
    n_bad, total = _check(dv, X, Y, d, T, 8, ws=ws)
    assert n_bad <= ROW_BAR * total


def test_fullvocab_full_size_workload(dv):
    """Block 16, V = 248320, fp32, top-k off, top-p 1, B = 128: every request
    against the oracle."""
    inp = synth.make_workload("b128_g15_fullvocab_f32", data_seed=0, seed=0)
    d = _draft_tokens(inp.draft, inp.temperature, 100)
    n_bad, total = _check(dv, inp.target, inp.draft, d, inp.temperature, inp.seed)
    assert n_bad <= ROW_BAR * total, n_bad


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sampler_full_vocab_matches_oracle(dv, dtype):
    """dflash_sample with top-k off and top-p 1: one token per row from the
    whole softmax (T = 0 rows: the argmax), uniforms of the sampler's stream.
    More than 2048 rows cross the launches the rows go in."""
    for R, V in ((2100, 300), (24, 30011)):
        X, _, _ = synth.make_logits(R, 0, V, dtype, data_seed=R + V)
        L = X.reshape(R, V)
        T = np.array([1.0, 0.0, 0.7, 1.3, -1.0], np.float32)[np.arange(R) % 5]
        for seed in (0, 31):
            want, margin, want_st = oracle.sample_rows(L, T, 0, 1.0, seed)
            st = torch.zeros(1, dtype=torch.int32, device=DEV)
            got = dv.sample_rows(_t(L), torch.from_numpy(T).to(DEV), 0, 1.0, seed, status=st)
            torch.cuda.synchronize()
            got = got.cpu().numpy()
            assert int(st.item()) == want_st == oracle.STATUS_BAD_TEMPERATURE
            greedy = T <= 0
            assert np.array_equal(got[greedy], want[greedy])
            diff = np.nonzero(got != want)[0]
            assert all(margin[r] < FV_DRAW_ABS for r in diff), [(int(r), margin[r]) for r in diff[:5]]
            assert len(diff) <= ROW_BAR * R
