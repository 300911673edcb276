"""GPU parity of the verification of deterministic drafts (q = point mass at d).

The CUDA path (dflash_verify_det through the C ABI) against the oracle's
verify_det, with the bars of the general verification: greedy requests and
status words bit-exact, sampled tokens and accept lengths equal on every
request unless the oracle's margins put a decision within the GPU's rounding
(parity_bounds), and differing rows under 0.01%. Drafts come from a
greedy drafter (the argmax of each draft row, as the drafter of the
speculative-decoding listing on bml.asia does), mixed with uniform tokens that
often fall outside the kept set.
"""
import numpy as np
import pytest

import oracle
import synth
from parity_bounds import ROW_BAR, compare_rows, excused_fullvocab, excused_topk

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


def _greedy_drafts(inp, mix_seed=None, frac_random=0.25):
    d = np.argmax(synth.to_float(inp.draft), axis=-1).astype(np.int32)
    if mix_seed is not None:
        rng = np.random.default_rng(mix_seed)
        V = inp.shape[2]
        d = np.where(rng.random(d.shape) < frac_random, rng.integers(0, V, d.shape), d).astype(np.int32)
    return d


def _run_det(dv, X, d, T, top_k, top_p, seed, workspace=None):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok, ln = dv.verify_det(_t(X), torch.from_numpy(np.ascontiguousarray(d)).to(DEV),
                            torch.from_numpy(np.ascontiguousarray(T, np.float32)).to(DEV), top_k,
                            top_p, seed, status=st, workspace=workspace)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), ln.cpu().numpy(), int(st.item())


def _compare(tok, ln, want_tok, want_len, margins):
    """margins: (accept, cut, draw) from the oracle with cut_margin=True."""
    m_acc, m_cut, m_draw = margins
    return compare_rows(tok, ln, want_tok, want_len, lambda b: excused_topk(m_acc[b], m_cut[b], m_draw[b]))


@pytest.mark.parametrize("V", [1024, 777, 20000])
def test_det_small_many_seeds(dv, V):
    n_bad = total = 0
    for data_seed in range(5):
        inp = synth.make_workload("tiny_v1024", data_seed=data_seed, B=9, V=V)
        T = np.array([1.0, 0.0, 0.6, 1.0, 1.5, 0.0, 0.8, 1.0, 2.0], np.float32)
        d = _greedy_drafts(inp, mix_seed=data_seed)
        for seed in (data_seed, 1000 + data_seed):
            want_tok, want_len, margins, want_st = oracle.verify_det(inp.target, d, T, inp.top_k,
                                                                     inp.top_p, seed, cut_margin=True)
            tok, ln, st = _run_det(dv, inp.target, d, T, inp.top_k, inp.top_p, seed)
            assert st == want_st
            n_bad += _compare(tok, ln, want_tok, want_len, margins)
            total += len(ln)
    assert n_bad <= ROW_BAR * total


@pytest.mark.parametrize("gamma", [1, 2, 15, 32])
def test_det_gamma_range(dv, gamma):
    inp = synth.make_workload("b8_v248320", data_seed=gamma, B=4, V=4099, gamma=gamma)
    T = np.array([1.0, 0.0, 0.7, 1.0], np.float32)
    d = _greedy_drafts(inp, mix_seed=gamma, frac_random=0.1)
    want_tok, want_len, margins, _ = oracle.verify_det(inp.target, d, T, inp.top_k, inp.top_p, 3,
                                                       cut_margin=True)
    tok, ln, _ = _run_det(dv, inp.target, d, T, inp.top_k, inp.top_p, 3)
    assert _compare(tok, ln, want_tok, want_len, margins) == 0


@pytest.mark.parametrize("filt", [(20, 0.95), (5, 0.9), (1, 1.0), (32, 1.0)])
def test_det_filters(dv, filt):
    top_k, top_p = filt
    inp = synth.make_workload("tiny_v1024", data_seed=11, B=12, V=5003)
    T = synth.cycle_temperatures(12)
    d = _greedy_drafts(inp, mix_seed=4)
    for seed in (1, 2):
        want_tok, want_len, margins, want_st = oracle.verify_det(inp.target, d, T, top_k, top_p, seed,
                                                                 cut_margin=True)
        tok, ln, st = _run_det(dv, inp.target, d, T, top_k, top_p, seed)
        assert st == want_st
        assert _compare(tok, ln, want_tok, want_len, margins) == 0


def test_det_full_size_b32_mixed(dv):
    """The B=32 mixed bf16 workload (block 8, V=248320) with greedy-drafter
    drafts, every request against the oracle."""
    inp = synth.make_workload("b32_mixed_v248320", data_seed=0, seed=0)
    d = _greedy_drafts(inp, mix_seed=1, frac_random=0.1)
    want_tok, want_len, margins, want_st = oracle.verify_det(inp.target, d, inp.temperature,
                                                             inp.top_k, inp.top_p, inp.seed, cut_margin=True)
    tok, ln, st = _run_det(dv, inp.target, d, inp.temperature, inp.top_k, inp.top_p, inp.seed)
    assert st == want_st == 0
    n_bad = _compare(tok, ln, want_tok, want_len, margins)
    assert n_bad <= ROW_BAR * len(ln)
    g = inp.temperature == 0
    assert np.array_equal(tok[g], want_tok[g]) and np.array_equal(ln[g], want_len[g])
    # the drafts were accepted at some positions and rejected at others
    assert 1 < ln[~g].mean() < inp.shape[1] + 1


def test_det_equals_general_path_on_point_mass_drafts(dv):
    """On the GPU, the general verification fed draft logits whose filtered
    distribution is exactly the point mass at d (d at 0, the rest at -1e4)
    takes the same decisions as the deterministic-draft path, bit for bit:
    q(d) = 1, so p/q = p(d), and max(0, p - q) is p without d."""
    B, gamma, V = 16, 7, 30011
    X, _, _ = synth.make_logits(B, gamma, V, "f32", data_seed=21)
    rng = np.random.default_rng(8)
    am = np.argmax(X[:, :gamma], axis=-1)
    d = np.where(rng.random((B, gamma)) < 0.6, am, rng.integers(0, V, (B, gamma))).astype(np.int32)
    Y = np.full((B, gamma, V), -1.0e4, np.float32)
    bi, ii = np.meshgrid(np.arange(B), np.arange(gamma), indexing="ij")
    Y[bi, ii, d] = 0.0
    T = synth.cycle_temperatures(B)
    for seed in (5, 6, 7):
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        t1, l1 = dv.verify(_t(X), _t(Y), torch.from_numpy(d).to(DEV), torch.from_numpy(T).to(DEV), 20,
                           0.95, seed, status=st)
        t2, l2, st2 = _run_det(dv, X, d, T, 20, 0.95, seed)
        assert int(st.item()) == st2 == 0
        assert np.array_equal(t1.cpu().numpy(), t2) and np.array_equal(l1.cpu().numpy(), l2)


def test_det_status_bits_and_rejected_filters(dv):
    inp = synth.make_workload("tiny_v1024", data_seed=2, B=4, V=3001)
    T = np.array([1.0, 1.0, -1.0, np.nan], np.float32)
    d = _greedy_drafts(inp)
    d[0, 0] = 3001
    d[1, 3] = -5
    X = inp.target.copy()
    X[1, 6, 17] = np.nan
    want_tok, want_len, _, want_st = oracle.verify_det(X, d, T, inp.top_k, inp.top_p, 1)
    tok, ln, st = _run_det(dv, X, d, T, inp.top_k, inp.top_p, 1)
    assert st == want_st == (oracle.STATUS_BAD_TOKEN | oracle.STATUS_BAD_ROW
                             | oracle.STATUS_BAD_TEMPERATURE)
    assert np.all((tok >= -1) & (tok < 3001)) and np.all((ln >= 1) & (ln <= 8))
    for b in (0, 2, 3):
        assert np.array_equal(tok[b], want_tok[b]) and ln[b] == want_len[b]
    # top-k beyond 32, with or without top-p, is refused by the entry point
    # itself, before any launch
    ws = dv.Workspace(dv.workspace_bytes(4, 7, 3001, dv.DFLASH_F32, 0, 1.0), DEV)
    Xd, dd = _t(X), torch.from_numpy(d).to(DEV)
    Td = torch.ones(4, dtype=torch.float32, device=DEV)
    out_t = torch.full((4, 8), -7, dtype=torch.int32, device=DEV)
    out_l = torch.zeros(4, dtype=torch.int32, device=DEV)
    lib = dv.load()
    for k, tp in ((40, 0.9), (64, 0.95)):
        rc = lib.dflash_verify_det(Xd.data_ptr(), dd.data_ptr(), 4, 7, 3001, dv.DFLASH_F32, Td.data_ptr(),
                                   k, tp, 1, out_t.data_ptr(), out_l.data_ptr(), ws.ptr, ws.nbytes, None,
                                   torch.cuda.current_stream().cuda_stream)
        assert rc == 2, lib.dflash_last_error()
        assert b"deterministic drafts" in lib.dflash_last_error()
    torch.cuda.synchronize()
    assert int((out_t != -7).sum().item()) == 0 and int(out_l.sum().item()) == 0


def test_det_workspace_left_zero_across_modes(dv):
    """Deterministic-draft calls and general calls of other shapes take turns
    on one workspace; each agrees with the oracle and leaves it at zero."""
    ws = dv.Workspace(48 << 20, DEV)
    for V, dtype, det in [(1024, "f32", True), (20000, "f32", False), (5003, "bf16", True),
                          (777, "f32", False), (20000, "f32", True)]:
        B, gamma = 6, 5
        X, Y, _ = synth.make_logits(B, gamma, V, dtype, data_seed=V + det)
        T = np.array([1.0, 0.0, 0.6, 1.0, 1.5, 0.0], np.float32)
        dd, _, _ = oracle.sample_rows(Y.reshape(B * gamma, V), synth.draft_sampling_temperatures(T, gamma),
                                      20, 0.95, 3)
        dd = dd.reshape(B, gamma)
        if det:
            tok, ln, st = _run_det(dv, X, dd, T, 20, 0.95, 9, workspace=ws)
            want_tok, want_len, margins, want_st = oracle.verify_det(X, dd, T, 20, 0.95, 9, cut_margin=True)
        else:
            s = torch.zeros(1, dtype=torch.int32, device=DEV)
            t_, l_ = dv.verify(_t(X), _t(Y), torch.from_numpy(dd).to(DEV), torch.from_numpy(T).to(DEV), 20,
                               0.95, 9, status=s, workspace=ws)
            torch.cuda.synchronize()
            tok, ln, st = t_.cpu().numpy(), l_.cpu().numpy(), int(s.item())
            want_tok, want_len, margins, want_st = oracle.verify(X, Y, dd, T, 20, 0.95, 9, cut_margin=True)
        assert st == want_st
        assert _compare(tok, ln, want_tok, want_len, margins) == 0
        assert int(torch.count_nonzero(ws.buf).item()) == 0, f"workspace not left at zero after V={V}"


# ---------------------------------------------------------------- full vocabulary
# Top-k off and top_p = 1: p is the softmax over all V tokens; a rejected
# deterministic draft's residual is p without d, drawn over the whole
# vocabulary in float-float like the general full-vocabulary draw. The bars
# are that mode's (parity_bounds: the accept test on the stream's fp32
# normalisers, the draw in float-float).


def _check_det_fv(dv, X, d, T, seed, ws=None):
    want_tok, want_len, (m_acc, m_draw), want_st = oracle.verify_det(X, d, T, 0, 1.0, seed, split_margins=True)
    tok, ln, st = _run_det(dv, X, d, T, 0, 1.0, seed, workspace=ws)
    assert st == want_st
    g = ~((T > 0) & np.isfinite(T))
    assert np.array_equal(tok[g], want_tok[g]) and np.array_equal(ln[g], want_len[g])
    n_bad = compare_rows(tok, ln, want_tok, want_len, lambda b: excused_fullvocab(m_acc[b], m_draw[b]))
    return n_bad, tok, ln


def _mixed_drafts(Y, seed, frac_random=0.3):
    d = np.argmax(synth.to_float(Y), axis=-1).astype(np.int32)
    rng = np.random.default_rng(seed)
    V = Y.shape[2]
    return np.where(rng.random(d.shape) < frac_random, rng.integers(0, V, d.shape), d).astype(np.int32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V,gamma", [(1024, 7), (777, 7), (20000, 15), (4097, 3), (1, 2), (33, 32)])
def test_det_fullvocab_small(dv, dtype, V, gamma):
    n_bad = 0
    for data_seed in range(3):
        X, Y, _ = synth.make_logits(9, gamma, V, dtype, data_seed=data_seed, sigma_d=0.5)
        T = np.array([1.0, 0.0, 0.6, 1.0, 1.5, 0.0, 0.8, 1.0, 2.0], np.float32)
        d = _mixed_drafts(Y, 60 + data_seed)
        for seed in (data_seed, 555 + data_seed):
            nb, _, _ = _check_det_fv(dv, X, d, T, seed)
            n_bad += nb
    assert n_bad == 0


def test_det_fullvocab_full_size(dv):
    """Block 16, V = 248320, fp32, top-k off, top-p 1, 16 requests with
    greedy-drafter drafts (a tenth replaced by uniform tokens)."""
    X, Y, _ = synth.make_logits(16, 15, 248320, "f32", data_seed=7, sigma_d=0.5)
    T = np.ones(16, np.float32)
    d = _mixed_drafts(Y, 8, frac_random=0.1)
    n_bad, tok, ln = _check_det_fv(dv, X, d, T, 3)
    assert n_bad <= ROW_BAR * len(ln)
    # a rejected draft is never the token drawn in its place
    for b in range(16):
        n = ln[b] - 1
        if n < 15:
            assert tok[b, n] != d[b, n]


def test_det_fullvocab_status_and_workspace(dv):
    """Bad rows, tokens and temperatures set the same status bits as the
    oracle, and full-vocabulary and top-k calls share one workspace, which
    each leaves at zero."""
    B, gamma, V = 5, 4, 6007
    X, Y, _ = synth.make_logits(B, gamma, V, "f32", data_seed=41)
    X = X.copy()
    T = np.array([1.0, 1.0, 1.0, -2.0, 1.0], np.float32)
    d = _mixed_drafts(Y, 2)
    d[0, 1] = V
    X[1, 3, 100] = np.nan
    want_tok, want_len, (m_acc, m_draw), want_st = oracle.verify_det(X, d, T, 0, 1.0, 6, split_margins=True)
    ws = dv.Workspace(48 << 20, DEV)
    tok, ln, st = _run_det(dv, X, d, T, 0, 1.0, 6, workspace=ws)
    assert st == want_st == (oracle.STATUS_BAD_TOKEN | oracle.STATUS_BAD_ROW
                             | oracle.STATUS_BAD_TEMPERATURE)
    assert np.all((tok >= -1) & (tok < V)) and np.all((ln >= 1) & (ln <= gamma + 1))
    # the greedy request (bad temperature) exactly; request 2 (no bad input)
    # within the draw's bars
    assert np.array_equal(tok[3], want_tok[3]) and ln[3] == want_len[3]
    assert (np.array_equal(tok[2], want_tok[2]) and ln[2] == want_len[2]) or excused_fullvocab(m_acc[2], m_draw[2])
    assert int(torch.count_nonzero(ws.buf).item()) == 0
    X2, Y2, _ = synth.make_logits(B, gamma, V, "f32", data_seed=42)
    T2 = np.array([1.0, 0.0, 0.6, 1.0, 1.5], np.float32)
    d2 = _mixed_drafts(Y2, 3)
    for top_k, top_p in ((20, 0.95), (0, 1.0)):
        if top_k:
            _run_det(dv, X2, d2, T2, top_k, top_p, 1, workspace=ws)
        else:
            _check_det_fv(dv, X2, d2, T2, 1, ws=ws)
        assert int(torch.count_nonzero(ws.buf).item()) == 0
