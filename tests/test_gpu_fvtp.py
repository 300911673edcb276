"""GPU parity of top-p over the full vocabulary (top-k off, 0 < top_p < 1).

The filter keeps, in the order logit descending / token index ascending, every
token whose preceding mass is below top_p, then renormalises; with no top-k
the kept set can hold most of a 248320-token vocabulary. The CUDA path finds
the cut by a mass-weighted radix selection on exact fixed-point sums
(dflash_fvtp.cu) and draws over the kept sets in float-float.

Bars (parity_bounds):
- greedy requests and status words are bit-exact;
- a sampling request matches the oracle exactly (tokens, accept length)
  unless one of the oracle's margins puts a decision within the GPU's
  rounding: the accept test (ACCEPT_REL), the top-p cut (fvtp_cut_rel), the
  draw (FV_DRAW_ABS); differing requests stay under 0.01%;
- the audited p(d), q(d) are within fvtp_prob_rel of the oracle's fp64 values
  on requests whose cuts are clear of the bound;
- every call leaves the workspace at zero.
"""
import numpy as np
import pytest

import oracle
import synth
from parity_bounds import (FV_DRAW_ABS, ROW_BAR, compare_rows, excused_fullvocab, excused_fvtp,
                           excused_topk, fvtp_cut_rel, fvtp_prob_rel)

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


def _drafts(Y, T, top_p, seed):
    """Drafts from the draft rows' own top-p distributions (oracle sampler)."""
    B, gamma, V = Y.shape
    d, _, _ = oracle.sample_rows(Y.reshape(B * gamma, V), synth.draft_sampling_temperatures(T, gamma),
                                 0, top_p, seed)
    return d.reshape(B, gamma)


def _run(dv, X, Y, d, T, top_p, seed, ws=None):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok, ln = dv.verify(_t(X), _t(Y), torch.from_numpy(np.ascontiguousarray(d)).to(DEV),
                        torch.from_numpy(np.ascontiguousarray(T, np.float32)).to(DEV), 0, top_p, seed,
                        status=st, workspace=ws)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), ln.cpu().numpy(), int(st.item())


def _check(dv, X, Y, d, T, top_p, seed, ws=None):
    """Returns (differing requests, requests); asserts each difference is excused."""
    V = X.shape[2]
    want_tok, want_len, (m_acc, m_cut, m_draw), want_st = oracle.verify(X, Y, d, T, 0, top_p, seed,
                                                                        cut_margin=True)
    tok, ln, st = _run(dv, X, Y, d, T, top_p, seed, ws=ws)
    assert st == want_st
    g = T == 0
    assert np.array_equal(tok[g], want_tok[g]) and np.array_equal(ln[g], want_len[g])
    n_bad = compare_rows(tok, ln, want_tok, want_len,
                         lambda b: excused_fvtp(V, top_p, m_acc[b], m_cut[b], m_draw[b]), "top-p")
    return n_bad, len(ln)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V,gamma", [(1024, 7), (777, 7), (20000, 15), (4097, 3), (1, 2), (33, 32),
                                     (12289, 5)])
def test_fvtp_small(dv, dtype, V, gamma):
    n_bad = total = 0
    for data_seed, top_p in ((0, 0.95), (1, 0.6), (2, 0.2)):
        X, Y, _ = synth.make_logits(9, gamma, V, dtype, data_seed=data_seed, sigma_d=0.5)
        T = np.array([1.0, 0.0, 0.6, 1.0, 1.5, 0.0, 0.8, 1.0, 2.0], np.float32)
        d = _drafts(Y, T, top_p, 50 + data_seed)
        for seed in (data_seed, 777 + data_seed):
            nb, nt = _check(dv, X, Y, d, T, top_p, seed)
            n_bad += nb
            total += nt
    assert n_bad <= ROW_BAR * total


def _tied_logits(B, rows, V, levels, seed, dtype):
    """Logits on a few levels (exact in bf16), so the cut falls inside a group
    of equal logits spread over every 4096-token slice of the row."""
    rng = np.random.default_rng(seed)
    x = (-0.5 * rng.integers(0, levels, size=(B, rows, V))).astype(np.float32)
    return synth.f32_to_bf16_bits(x) if dtype == "bf16" else x


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fvtp_ties_at_the_cut(dv, dtype):
    """The last kept token sits inside a group of equal logits: only the ones
    of lower index are kept (the order's tie rule), found by the per-slice
    counts and the scan of one slice."""
    B, gamma, V = 6, 4, 50000
    X = _tied_logits(B, gamma + 1, V, 6, 7, dtype)
    Y = _tied_logits(B, gamma, V, 6, 8, dtype)
    T = np.array([1.0, 0.7, 1.0, 1.3, 0.0, 1.0], np.float32)
    n_bad = total = 0
    for top_p in (0.5, 0.83, 0.97):
        d = _drafts(Y, T, top_p, 3)
        for seed in (1, 2):
            nb, nt = _check(dv, X, Y, d, T, top_p, seed)
            n_bad += nb
            total += nt
    assert n_bad <= ROW_BAR * total


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fvtp_keeps_exactly_the_oracles_set(dv, dtype):
    """With identical target and draft rows every draft is accepted and the
    audit returns p(d) = q(d) for any token d: positive exactly on the kept
    set. Drafts picked around the cut inside a tie group (the last kept and
    the first dropped of equal logits) must fall on the oracle's side."""
    B, gamma, V, top_p = 4, 6, 40000, 0.7
    X = _tied_logits(B, gamma + 1, V, 5, 11, dtype)
    Y = np.ascontiguousarray(X[:, :gamma])
    T = np.ones(B, np.float32)
    d = np.zeros((B, gamma), np.int32)
    kept = np.zeros((B, gamma), bool)
    for b in range(B):
        for i in range(gamma):
            p = oracle.filter_row(X[b, i], 1.0, 0, top_p)
            xf = synth.to_float(X[b, i])
            inside = np.nonzero(p > 0)[0]
            last = inside[np.argmin(xf[inside])]          # a token of the lowest kept level ...
            lvl = xf[last]
            group = np.nonzero(xf == lvl)[0]
            k_last = group[p[group] > 0].max()            # ... the last kept one of it
            dropped = group[p[group] == 0]
            # alternate: the last kept token, the first dropped one of the group
            d[b, i] = k_last if (i % 2 == 0 or dropped.size == 0) else dropped.min()
            kept[b, i] = p[d[b, i]] > 0
    assert kept.any() and not kept.all()
    Xd, Yd = _t(X), _t(Y)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok, ln, pq = dv.verify_audit(Xd, Yd, torch.from_numpy(d).to(DEV), torch.from_numpy(T).to(DEV), 0,
                                  top_p, 5, status=st)
    torch.cuda.synchronize()
    pq = pq.cpu().numpy()
    assert int(st.item()) == 0
    # a request stops at its first dropped draft (p = q = 0 rejects)
    ln = ln.cpu().numpy()
    for b in range(B):
        first_drop = np.nonzero(~kept[b])[0]
        want_len = (first_drop[0] if first_drop.size else gamma) + 1
        assert ln[b] == want_len
        for i in range(want_len - 1 if first_drop.size else gamma):
            assert pq[b, i, 0] > 0 and pq[b, i, 0] == pq[b, i, 1]
        if first_drop.size:
            assert pq[b, first_drop[0], 0] == 0 and pq[b, first_drop[0], 1] == 0


def test_fvtp_deterministic_drafts(dv):
    """dflash_verify_det with top-p over the full vocabulary: drafts from a
    greedy drafter mixed with uniform tokens (often outside the kept set)."""
    n_bad = total = 0
    for V, dtype in ((30011, "bf16"), (5003, "f32")):
        inp = synth.make_workload("b32_mixed_topp_v248320", data_seed=V, seed=4, B=12, V=V)
        if dtype == "f32":
            inp.target, inp.draft = synth.to_float(inp.target), synth.to_float(inp.draft)
        rng = np.random.default_rng(V)
        d = np.argmax(synth.to_float(inp.draft), axis=-1).astype(np.int32)
        d = np.where(rng.random(d.shape) < 0.25, rng.integers(0, V, d.shape), d).astype(np.int32)
        for top_p, seed in ((0.95, 1), (0.5, 2)):
            want_tok, want_len, (m_acc, m_cut, m_draw), want_st = oracle.verify_det(
                inp.target, d, inp.temperature, 0, top_p, seed, cut_margin=True)
            st = torch.zeros(1, dtype=torch.int32, device=DEV)
            tok, ln = dv.verify_det(_t(inp.target), torch.from_numpy(d).to(DEV),
                                    torch.from_numpy(inp.temperature).to(DEV), 0, top_p, seed, status=st)
            torch.cuda.synchronize()
            tok, ln = tok.cpu().numpy(), ln.cpu().numpy()
            assert int(st.item()) == want_st
            n_bad += compare_rows(tok, ln, want_tok, want_len,
                                  lambda b: excused_fvtp(V, top_p, m_acc[b], m_cut[b], m_draw[b]), "det")
            total += len(ln)
    assert n_bad <= ROW_BAR * total


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fvtp_sampler(dv, dtype):
    """dflash_sample with top-k off and top-p < 1: one token per row from the
    row's top-p set (T = 0 rows: the argmax). More than 2048 rows cross the
    launches the rows go in."""
    for R, V, top_p in ((2100, 300, 0.9), (24, 30011, 0.95), (40, 9000, 0.3)):
        X, _, _ = synth.make_logits(R, 0, V, dtype, data_seed=R + V)
        L = X.reshape(R, V)
        T = np.array([1.0, 0.0, 0.7, 1.3, -1.0], np.float32)[np.arange(R) % 5]
        for seed in (0, 31):
            want, margin, want_st = oracle.sample_rows(L, T, 0, top_p, seed)
            st = torch.zeros(1, dtype=torch.int32, device=DEV)
            got = dv.sample_rows(_t(L), torch.from_numpy(T).to(DEV), 0, top_p, seed, status=st)
            torch.cuda.synchronize()
            got = got.cpu().numpy()
            assert int(st.item()) == want_st == oracle.STATUS_BAD_TEMPERATURE
            greedy = T <= 0
            assert np.array_equal(got[greedy], want[greedy])
            diff = np.nonzero(got != want)[0]
            bound = max(FV_DRAW_ABS, fvtp_cut_rel(V, top_p))
            assert all(margin[r] < bound for r in diff), [(int(r), margin[r]) for r in diff[:5]]
            assert len(diff) <= ROW_BAR * R


def test_fvtp_full_size_headline_mix(dv):
    """B = 32, block 8, V = 248320, bf16, temperatures cycling greedy / 0.6 /
    1.0, top-k off, top-p 0.95: every request against the oracle, two seeds."""
    for data_seed in (0, 1):
        inp = synth.make_workload("b32_mixed_topp_v248320", data_seed=data_seed, seed=data_seed)
        d = _drafts(inp.draft, inp.temperature, inp.top_p, 100 + data_seed)
        n_bad, total = _check(dv, inp.target, inp.draft, d, inp.temperature, inp.top_p, inp.seed)
        assert n_bad <= ROW_BAR * total, n_bad


def test_fvtp_full_size_f32_block16(dv):
    """fp32 logits, block 16 (15 drafts), V = 248320, top-p 0.95, B = 128:
    every request against the oracle."""
    inp = synth.make_workload("b128_g15_topp_f32", data_seed=3, seed=3)
    d = _drafts(inp.draft, inp.temperature, inp.top_p, 7)
    n_bad, total = _check(dv, inp.target, inp.draft, d, inp.temperature, inp.top_p, 3)
    assert n_bad <= ROW_BAR * total, n_bad


def test_fvtp_audit_headline_mix(dv):
    """p(d), q(d) of every accept test against the oracle's fp64 top-p
    distributions: within 1e-5 absolute everywhere, and within fvtp_prob_rel
    relative on requests whose top-p cuts are clear of the cut bound (a cut
    inside the bound may keep one token more or less than the oracle)."""
    inp = synth.make_workload("b32_mixed_topp_v248320", data_seed=5, seed=5)
    B, gamma, V = inp.shape
    top_p = inp.top_p
    d = _drafts(inp.draft, inp.temperature, top_p, 9)
    X, Y = _t(inp.target), _t(inp.draft)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    _, _, pq = dv.verify_audit(X, Y, torch.from_numpy(d).to(DEV), torch.from_numpy(inp.temperature).to(DEV),
                               0, top_p, inp.seed, status=st)
    torch.cuda.synchronize()
    got = pq.cpu().numpy().astype(np.float64)
    _, _, (_, m_cut, _), _ = oracle.verify(inp.target, inp.draft, d, inp.temperature, 0, top_p, inp.seed,
                                           cut_margin=True)
    samp = inp.temperature > 0
    want = np.full_like(got, np.nan)
    for b in np.nonzero(samp)[0]:
        T = float(inp.temperature[b])
        for i in range(gamma):
            if np.isnan(got[b, i, 0]):
                continue  # the loop stopped before position i
            want[b, i, 0] = oracle.filter_row(inp.target[b, i], T, 0, top_p)[d[b, i]]
            want[b, i, 1] = oracle.filter_row(inp.draft[b, i], T, 0, top_p)[d[b, i]]
    seen = ~np.isnan(got)
    assert seen[samp].any() and not seen[~samp].any()
    assert np.max(np.abs(got[seen] - want[seen])) < 1e-5
    clear = samp & (m_cut >= fvtp_cut_rel(V, top_p))
    g, w = got[clear], want[clear]
    ok = ~np.isnan(g)
    rel = np.abs(g[ok] - w[ok]) / np.maximum(w[ok], 1e-300)
    assert np.all((w[ok] == 0) == (g[ok] == 0))
    assert np.max(rel[w[ok] > 0]) <= fvtp_prob_rel(V), np.max(rel[w[ok] > 0])


def test_fvtp_workspace_left_zero_across_modes(dv):
    """Top-p-over-the-vocabulary calls take turns with full-vocabulary, top-k
    and deterministic-draft calls on one workspace; each call agrees with the
    oracle and leaves the workspace at zero."""
    ws = dv.Workspace(64 << 20, DEV)
    B, gamma = 5, 4
    T = np.array([1.0, 0.0, 0.6, 1.0, 1.5], np.float32)
    for V, dtype, top_k, top_p in [(20000, "bf16", 0, 0.9), (20000, "bf16", 0, 1.0), (5003, "f32", 0, 0.5),
                                   (5003, "f32", 20, 0.95), (30011, "f32", 0, 0.95)]:
        X, Y, _ = synth.make_logits(B, gamma, V, dtype, data_seed=V + top_k)
        d, _, _ = oracle.sample_rows(Y.reshape(B * gamma, V), synth.draft_sampling_temperatures(T, gamma),
                                     top_k, top_p, 3)
        d = d.reshape(B, gamma)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        tok, ln = dv.verify(_t(X), _t(Y), torch.from_numpy(d).to(DEV), torch.from_numpy(T).to(DEV), top_k,
                            top_p, 4, status=st, workspace=ws)
        torch.cuda.synchronize()
        assert int(torch.count_nonzero(ws.buf).item()) == 0, f"workspace not left at zero after {V} {top_p}"
        want_tok, want_len, (m_acc, m_cut, m_draw), want_st = oracle.verify(X, Y, d, T, top_k, top_p, 4,
                                                                            cut_margin=True)
        assert int(st.item()) == want_st
        if top_k > 0:
            excused = lambda b: excused_topk(m_acc[b], m_cut[b], m_draw[b])
        elif top_p >= 1.0:
            excused = lambda b: excused_fullvocab(min(m_acc[b], m_cut[b]), m_draw[b])
        else:
            excused = lambda b: excused_fvtp(V, top_p, m_acc[b], m_cut[b], m_draw[b])
        assert compare_rows(tok.cpu().numpy(), ln.cpu().numpy(), want_tok, want_len, excused, "mixed") == 0
        # the same inputs as deterministic drafts
        tok2, ln2 = dv.verify_det(_t(X), torch.from_numpy(d).to(DEV), torch.from_numpy(T).to(DEV), top_k,
                                  top_p, 4, workspace=ws)
        torch.cuda.synchronize()
        assert int(torch.count_nonzero(ws.buf).item()) == 0, f"workspace not left at zero after det {V}"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_fvtp_rows_of_one_value(dv, dtype):
    """Every logit of a row equal: each row is one key group of V tokens, the
    kept set the first ceil(top_p V) or so by index. V = 2 x 65528 puts as
    many equal bf16 logits in one counting block as it may hold."""
    B, gamma, V = 2, 2, 2 * 65528
    X = np.full((B, gamma + 1, V), 0.75, np.float32)
    X[1] = -3.0
    Y = np.full((B, gamma, V), 0.25, np.float32)
    if dtype == "bf16":
        X, Y = synth.f32_to_bf16_bits(X), synth.f32_to_bf16_bits(Y)
    T = np.ones(B, np.float32)
    for top_p, seed in ((0.3, 1), (0.9, 2)):
        d = _drafts(Y, T, top_p, 3)
        n_bad, total = _check(dv, X, Y, d, T, top_p, seed)
        assert n_bad == 0
