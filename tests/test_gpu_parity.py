"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars: uniforms, greedy tokens and accept lengths, and status words are
bit-exact. Filtered probabilities agree within 1e-5 absolute (the sampling
bar) and, as the filter is float-float, within one fp32 rounding of the
oracle's fp64 value. Sampled tokens and accept lengths agree on every request
except ones whose oracle margin puts a decision within the GPU's rounding
(parity_bounds: 2^-21 relative for the accept tests and top-p cuts, 2^-21
absolute for the draw), and differing rows stay under 0.01% of the rows.
"""
import numpy as np
import pytest

import oracle
import synth
from parity_bounds import CUT_REL, DRAW_ABS, ROW_BAR, U, compare_rows, excused_fullvocab, excused_topk

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

PROB_TOL = 1e-5


@pytest.fixture(scope="module")
def dv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_83_gb300 as m

    m.build()
    m.load()
    return m


DEV = "cuda:0"


def _t(a):
    return synth.to_torch(a, DEV)


def _draft_tokens(inp, seed=77):
    B, gamma, V = inp.shape
    d, _, _ = oracle.sample_rows(inp.draft.reshape(B * gamma, V),
                                 synth.draft_sampling_temperatures(inp.temperature, gamma),
                                 inp.top_k, inp.top_p, seed)
    return d.reshape(B, gamma)


def _run_verify(dv, X, Y, d, T, top_k, top_p, seed):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok, ln = dv.verify(_t(X), _t(Y), torch.from_numpy(np.ascontiguousarray(d)).to(DEV),
                        torch.from_numpy(np.ascontiguousarray(T, np.float32)).to(DEV), top_k, top_p,
                        seed, status=st)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), ln.cpu().numpy(), int(st.item())


def _compare_sampling(tok, ln, want_tok, want_len, margins):
    """Rows must match unless the oracle's margins (accept, cut, draw) put a
    decision within the GPU's rounding."""
    m_acc, m_cut, m_draw = margins
    return compare_rows(tok, ln, want_tok, want_len,
                        lambda b: excused_topk(m_acc[b], m_cut[b], m_draw[b]))


# ---------------------------------------------------------------- uniforms
@pytest.mark.parametrize("seed", [0, 5, 2**40 + 17, 0xFFFFFFFFFFFFFFFF])
def test_uniforms_bit_exact(dv, seed):
    B, npos = 37, 17
    for stream_id in (0, 1):
        ua, ud = dv.uniforms(seed, B, npos, stream_id, device=DEV)
        ua, ud = ua.cpu().numpy(), ud.cpu().numpy()
        for b in range(B):
            for i in range(npos):
                wa, wd = oracle.uniforms(seed, b, i, stream_id)
                assert ua[b, i] == wa and ud[b, i] == wd


# ---------------------------------------------------------------- greedy
def _greedy_case(B, gamma, V, dtype, seed, ties):
    rng = np.random.default_rng(seed)
    if ties:
        X = rng.integers(-3, 4, size=(B, gamma + 1, V)).astype(np.float32)
    else:
        X = (rng.standard_normal((B, gamma + 1, V)) * 2).astype(np.float32)
    am = np.argmax(X, -1)
    d = np.where(rng.random((B, gamma)) < 0.7, am[:, :gamma], rng.integers(0, V, (B, gamma)))
    if dtype == "bf16":
        X = synth.f32_to_bf16_bits(X)
    return X, d.astype(np.int32)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [1, 5, 8, 9, 1000, 4097, 8192, 8200, 33001, 248320])
def test_greedy_bit_exact(dv, dtype, V):
    for B, gamma, ties in ((3, 7, False), (2, 4, True)):
        X, d = _greedy_case(B, gamma, V, dtype, V * 7 + B, ties)
        want_tok, want_len, want_st = oracle.verify_greedy(X, d)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        tok, ln = dv.verify_greedy(_t(X), torch.from_numpy(d).to(DEV), status=st)
        torch.cuda.synchronize()
        assert np.array_equal(tok.cpu().numpy(), want_tok)
        assert np.array_equal(ln.cpu().numpy(), want_len)
        assert int(st.item()) == want_st


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_greedy_misaligned_rows(dv, dtype):
    # rows start off a 16-byte boundary: heads and tails take the plain-load path
    B, gamma, V = 3, 5, 5003
    X, d = _greedy_case(B, gamma, V, dtype, 11, False)
    want_tok, want_len, _ = oracle.verify_greedy(X, d)
    flat = _t(np.concatenate([X.reshape(-1)[:1], X.reshape(-1)]))
    Xd = flat[1:].view(B, gamma + 1, V)
    assert Xd.data_ptr() % 16 != 0
    tok, ln = dv.verify_greedy(Xd, torch.from_numpy(d).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(tok.cpu().numpy(), want_tok)
    assert np.array_equal(ln.cpu().numpy(), want_len)


def test_greedy_all_equal_rows_take_lowest_index(dv):
    # every logit ties: the exact fallback selection runs; argmax is token 0
    B, gamma, V = 2, 3, 70000
    X = np.zeros((B, gamma + 1, V), np.float32)
    X[1, 2, 69999] = 1.0
    d = np.array([[0, 0, 5], [0, 0, 69999]], np.int32)
    want_tok, want_len, _ = oracle.verify_greedy(X, d)
    tok, ln = dv.verify_greedy(_t(X), torch.from_numpy(d).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(tok.cpu().numpy(), want_tok)
    assert np.array_equal(ln.cpu().numpy(), want_len)


# ---------------------------------------------------------------- filter
def _check_filter_rows(dv, L, T, top_k, top_p):
    R, V = L.shape
    idx, prob, cnt = dv.filter_rows(_t(L), torch.from_numpy(T).to(DEV), top_k, top_p)
    torch.cuda.synchronize()
    idx, prob, cnt = idx.cpu().numpy(), prob.cpu().numpy(), cnt.cpu().numpy()
    boundary = 0
    for r in range(R):
        w_idx, w_prob = oracle.filter_row_sparse(L[r], float(T[r]), top_k, top_p)
        n = cnt[r]
        if n != len(w_idx):
            # only a top-p cut within the GPU's rounding may differ, by one token
            full_idx, full_p = oracle.filter_row_sparse(L[r], float(T[r]), top_k, 1.0)
            m = min(n, len(w_idx))
            assert abs(n - len(w_idx)) == 1
            assert abs(full_p[:m].sum() - top_p) < CUT_REL * top_p
            boundary += 1
            continue
        assert np.array_equal(idx[r, :n], w_idx), f"row {r}"
        assert np.all(idx[r, n:] == -1)
        assert np.max(np.abs(prob[r, :n] - w_prob)) < PROB_TOL
        # one fp32 rounding of the exact value, plus the float-float exp's 1e-9
        assert np.all(np.abs(prob[r, :n] - w_prob) <= 1.05 * U * w_prob + 1e-30), f"row {r}"
        assert abs(prob[r, :n].sum() - 1.0) < 1e-5
    return boundary


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("top_k,top_p", [(1, 1.0), (5, 0.9), (20, 0.95), (20, 1.0), (32, 0.5)])
def test_filter_matches_oracle(dv, dtype, top_k, top_p):
    inp = synth.make_workload("b8_v248320", data_seed=3, B=2, V=50021, gamma=5)
    L = inp.draft.reshape(-1, inp.shape[2])
    if dtype == "f32":
        L = synth.to_float(L)
    R = L.shape[0]
    T = np.array([0.6, 1.0, 1.7, 0.3, 1.0] * 4, np.float32)[:R]
    assert _check_filter_rows(dv, L, T, top_k, top_p) == 0


def test_filter_full_vocab_rows(dv):
    inp = synth.make_workload("b32_mixed_v248320", data_seed=4, B=2, gamma=2)
    L = inp.target.reshape(-1, inp.shape[2])
    T = np.full(L.shape[0], 1.0, np.float32)
    assert _check_filter_rows(dv, L, T, 20, 0.95) == 0


# ---------------------------------------------------------------- sample
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_sample_matches_oracle(dv, dtype):
    inp = synth.make_workload("b8_v248320", data_seed=5, B=4, V=30011, gamma=7)
    L = inp.draft.reshape(-1, inp.shape[2])
    if dtype == "f32":
        L = synth.to_float(L)
    R = L.shape[0]
    T = np.array([1.0, 0.0, 0.6, 1.3], np.float32)[np.arange(R) % 4]
    for seed in (0, 9, 123):
        want, margin, want_st = oracle.sample_rows(L, T, 20, 0.95, seed)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        got = dv.sample_rows(_t(L), torch.from_numpy(T).to(DEV), 20, 0.95, seed, status=st)
        torch.cuda.synchronize()
        got = got.cpu().numpy()
        diff = np.nonzero(got != want)[0]
        # the sampler's margin is the smaller of its cut (relative) and draw
        # (absolute) margins; both are bounded by DRAW_ABS here
        assert all(margin[r] < DRAW_ABS for r in diff)
        assert int(st.item()) == want_st


# ---------------------------------------------------------------- verify
@pytest.mark.parametrize("V", [1024, 777, 20000])
def test_verify_small_many_seeds(dv, V):
    n_bad = total = 0
    for data_seed in range(6):
        inp = synth.make_workload("tiny_v1024", data_seed=data_seed, B=9, V=V)
        inp.temperature[:] = np.array([1.0, 0.0, 0.6, 1.0, 1.5, 0.0, 0.8, 1.0, 2.0], np.float32)
        d = _draft_tokens(inp, seed=data_seed)
        for seed in (data_seed, 1000 + data_seed):
            want_tok, want_len, margins, want_st = oracle.verify(
                inp.target, inp.draft, d, inp.temperature, inp.top_k, inp.top_p, seed, cut_margin=True)
            tok, ln, st = _run_verify(dv, inp.target, inp.draft, d, inp.temperature, inp.top_k,
                                      inp.top_p, seed)
            assert st == want_st
            n_bad += _compare_sampling(tok, ln, want_tok, want_len, margins)
            total += len(ln)
    assert n_bad <= ROW_BAR * total


@pytest.mark.parametrize("gamma", [1, 2, 15, 32])
def test_verify_gamma_range(dv, gamma):
    inp = synth.make_workload("b8_v248320", data_seed=gamma, B=3, V=4099, gamma=gamma)
    inp.temperature[:] = np.array([1.0, 0.0, 0.7], np.float32)
    d = _draft_tokens(inp)
    want_tok, want_len, margins, _ = oracle.verify(inp.target, inp.draft, d, inp.temperature,
                                                   inp.top_k, inp.top_p, 3, cut_margin=True)
    tok, ln, _ = _run_verify(dv, inp.target, inp.draft, d, inp.temperature, inp.top_k,
                             inp.top_p, 3)
    assert _compare_sampling(tok, ln, want_tok, want_len, margins) <= ROW_BAR * len(ln)


@pytest.mark.parametrize("name", ["b8_v248320", "b32_mixed_v248320", "b32_mixed_g3_v248320",
                                  "b32_mixed_g15_v248320"])
def test_verify_full_size_workloads(dv, name):
    """The full-size bf16 workloads, every request checked against the oracle."""
    inp = synth.make_workload(name, data_seed=0, seed=0)
    d = _draft_tokens(inp, seed=100)
    want_tok, want_len, margins, want_st = oracle.verify(
        inp.target, inp.draft, d, inp.temperature, inp.top_k, inp.top_p, inp.seed, cut_margin=True)
    tok, ln, st = _run_verify(dv, inp.target, inp.draft, d, inp.temperature, inp.top_k,
                              inp.top_p, inp.seed)
    assert st == want_st == 0
    n_bad = _compare_sampling(tok, ln, want_tok, want_len, margins)
    # greedy requests of the mix are bit-exact
    g = inp.temperature == 0
    assert np.array_equal(tok[g], want_tok[g]) and np.array_equal(ln[g], want_len[g])
    assert n_bad <= ROW_BAR * len(ln)


def test_verify_single_request_seeds_0_to_99(dv):
    """One request, block 8, V = 248320 bf16, T = 1, top-k 20, top-p 0.95:
    data and Philox seeds 0..99, each step checked against the oracle (the
    oracle calls run on the host threads side by side)."""
    from concurrent.futures import ThreadPoolExecutor

    n_bad = 0
    threads = oracle.default_threads()
    for s0 in range(0, 100, threads):
        cases = []
        for s in range(s0, min(100, s0 + threads)):
            inp = synth.make_workload("b1_v248320", data_seed=s, seed=s)
            cases.append((inp, _draft_tokens(inp, seed=100 + s)))
        with ThreadPoolExecutor(threads) as ex:
            wants = list(ex.map(lambda c: oracle.verify(c[0].target, c[0].draft, c[1], c[0].temperature,
                                                        c[0].top_k, c[0].top_p, c[0].seed, threads=1,
                                                        cut_margin=True), cases))
        for (inp, d), (want_tok, want_len, margins, want_st) in zip(cases, wants):
            tok, ln, st = _run_verify(dv, inp.target, inp.draft, d, inp.temperature, inp.top_k,
                                      inp.top_p, inp.seed)
            assert st == want_st == 0
            n_bad += _compare_sampling(tok, ln, want_tok, want_len, margins)
    assert n_bad <= ROW_BAR * 100


def test_verify_10k_sampled_rows(dv):
    """The sampling-mode bar on more than 10^4 sampled requests: 160 batches
    of 64 requests (temperatures cycling 0.6 / 1 / 1.3, top-k 20, top-p 0.95,
    draft noise sigma ~ U(0.3, 1.5)), V = 20011 bf16 (rows of several pieces
    spread over many CTAs, starts off 16-byte boundaries), every request
    checked against the oracle: a differing row must be excused by a margin
    within the GPU's rounding, and differing rows stay under 0.01%."""
    B, gamma, V = 64, 7, 20011
    n_bad = total = 0
    for s in range(160):
        inp = synth.make_workload("b32_mixed_v248320", data_seed=20_000 + s, seed=s, B=B, V=V)
        inp.temperature[:] = synth.cycle_temperatures(B, (0.6, 1.0, 1.3))
        d = _draft_tokens(inp, seed=500 + s)
        want_tok, want_len, margins, want_st = oracle.verify(
            inp.target, inp.draft, d, inp.temperature, inp.top_k, inp.top_p, inp.seed, cut_margin=True)
        tok, ln, st = _run_verify(dv, inp.target, inp.draft, d, inp.temperature, inp.top_k,
                                  inp.top_p, inp.seed)
        assert st == want_st == 0
        n_bad += _compare_sampling(tok, ln, want_tok, want_len, margins)
        total += B
    assert total >= 10_000
    assert n_bad <= ROW_BAR * total, f"{n_bad} of {total} rows differ"


def test_verify_b8_all_greedy_matches_greedy_entry(dv):
    inp = synth.make_workload("b8_v248320", data_seed=8)
    d = _draft_tokens(inp)
    T = np.zeros(inp.shape[0], np.float32)
    tok, ln, st = _run_verify(dv, inp.target, inp.draft, d, T, 20, 0.95, 0)
    g_tok, g_len = dv.verify_greedy(_t(inp.target), torch.from_numpy(d).to(DEV))
    want_tok, want_len, _ = oracle.verify_greedy(inp.target, d)
    assert np.array_equal(tok, want_tok) and np.array_equal(ln, want_len)
    assert np.array_equal(g_tok.cpu().numpy(), want_tok)
    assert np.array_equal(g_len.cpu().numpy(), want_len)


def test_status_bits_and_bad_inputs(dv):
    inp = synth.make_workload("tiny_v1024", data_seed=2, B=4, V=3001)
    inp.temperature[:] = np.array([1.0, 1.0, -1.0, np.nan], np.float32)
    d = _draft_tokens(synth.make_workload("tiny_v1024", data_seed=2, B=4, V=3001))
    d[0, 0] = 3001
    d[1, 3] = -5
    X = inp.target.copy()
    X[1, 6, 17] = np.nan
    want_tok, want_len, _, want_st = oracle.verify(X, inp.draft, d, inp.temperature,
                                                   inp.top_k, inp.top_p, 1)
    tok, ln, st = _run_verify(dv, X, inp.draft, d, inp.temperature, inp.top_k, inp.top_p, 1)
    assert st == want_st == (oracle.STATUS_BAD_TOKEN | oracle.STATUS_BAD_ROW
                             | oracle.STATUS_BAD_TEMPERATURE)
    assert np.all((tok >= -1) & (tok < 3001)) and np.all((ln >= 1) & (ln <= 8))
    # requests without a bad row agree with the oracle
    for b in (0, 2, 3):
        assert np.array_equal(tok[b], want_tok[b]) and ln[b] == want_len[b]


def test_workspace_reuse_and_repeatability(dv):
    inp = synth.make_workload("b8_v248320", data_seed=9, B=5, V=12345)
    d = _draft_tokens(inp)
    ws = dv.Workspace(dv.workspace_bytes(5, 7, 12345, dv.DFLASH_BF16, 20, 0.95), DEV)
    outs = []
    for _ in range(3):
        tok, ln = dv.verify(_t(inp.target), _t(inp.draft), torch.from_numpy(d).to(DEV),
                            torch.from_numpy(inp.temperature).to(DEV), 20, 0.95, 4, workspace=ws)
        outs.append((tok.cpu().numpy(), ln.cpu().numpy()))
    assert all(np.array_equal(o[0], outs[0][0]) and np.array_equal(o[1], outs[0][1]) for o in outs)
    want_tok, want_len, margins, _ = oracle.verify(inp.target, inp.draft, d, inp.temperature, 20,
                                                   0.95, 4, cut_margin=True)
    assert _compare_sampling(outs[0][0], outs[0][1], want_tok, want_len, margins) == 0


def test_verify_host_buffers(dv):
    inp = synth.make_workload("b32_mixed_v248320", data_seed=6, B=6, V=9000)
    B, gamma, V = inp.shape
    d = _draft_tokens(inp)

    def pin(a):
        return synth.to_torch(a, "cpu").pin_memory()

    out_tok = torch.empty((B, gamma + 1), dtype=torch.int32).pin_memory()
    out_len = torch.empty((B,), dtype=torch.int32).pin_memory()
    out_st = torch.zeros((1,), dtype=torch.int32).pin_memory()
    staging = torch.empty(dv.host_staging_bytes(B, gamma, V, 0), dtype=torch.uint8, device=DEV)
    ws = dv.Workspace(dv.workspace_bytes(B, gamma, V, 0, 20, 0.95), DEV)
    dv.verify_host(pin(inp.target), pin(inp.draft), pin(d), pin(inp.temperature), 20, 0.95, 8,
                   out_tok, out_len, out_st, staging, ws)
    want_tok, want_len, margins, want_st = oracle.verify(inp.target, inp.draft, d, inp.temperature,
                                                         20, 0.95, 8, cut_margin=True)
    assert _compare_sampling(out_tok.numpy(), out_len.numpy(), want_tok, want_len, margins) == 0
    assert int(out_st.item()) == want_st


def test_workspace_left_zero_across_shapes(dv):
    """Every call leaves its whole workspace at zero, whatever the shape.

    The workspace regions move with the shape: a larger call's tile keys can
    lie where a smaller call kept its filtered lists. Row finals treat
    non-zero tile keys as written, so the next call would see leftovers as
    finished keys. Calls of several shapes and modes run in turn on one
    workspace. Each is checked against the oracle, and the workspace must
    read back as zero after each call."""
    ws = dv.Workspace(48 << 20, DEV)
    cases = [(1024, "f32", 20, 0.95), (777, "f32", 20, 0.95), (20000, "f32", 20, 0.95),
             (5003, "bf16", 7, 0.9), (20000, "f32", 0, 1.0), (1024, "f32", 20, 0.95)]
    for V, dtype, top_k, top_p in cases:
        X, Y, _ = synth.make_logits(6, 5, V, dtype, data_seed=V)
        T = np.array([1.0, 0.0, 0.6, 1.0, 1.5, 0.0], np.float32)
        B, gamma = 6, 5
        d, _, _ = oracle.sample_rows(Y.reshape(B * gamma, V), synth.draft_sampling_temperatures(T, gamma),
                                     top_k, top_p, 3)
        d = d.reshape(B, gamma)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        tok, ln = dv.verify(_t(X), _t(Y), torch.from_numpy(d).to(DEV), torch.from_numpy(T).to(DEV), top_k,
                            top_p, 9, status=st, workspace=ws)
        torch.cuda.synchronize()
        want_tok, want_len, (m_acc, m_cut, m_draw), want_st = oracle.verify(X, Y, d, T, top_k, top_p, 9,
                                                                             cut_margin=True)
        assert int(st.item()) == want_st
        fv = top_k <= 0
        compare_rows(tok.cpu().numpy(), ln.cpu().numpy(), want_tok, want_len,
                     (lambda b: excused_fullvocab(m_acc[b], m_draw[b])) if fv
                     else (lambda b: excused_topk(m_acc[b], m_cut[b], m_draw[b])), f"V={V}")
        assert int(torch.count_nonzero(ws.buf).item()) == 0, f"workspace not left at zero after V={V}"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_verify_narrow_and_wide_top_tiles(dv, dtype):
    """Row finals find the k-th largest tile maximum by counting tile maxima in
    a window of buckets below the row's largest, or, when the k largest spread
    wider than that window, by a full histogram. Rows of both kinds, in one
    batch, against the oracle: a row is 'wide' when 20 spikes 100, 95, ..., 5
    sit in separate tiles above Gaussian logits."""
    B, gamma, V = 6, 3, 50000
    X, Y, _ = synth.make_logits(B, gamma, V, "f32", data_seed=123, sigma_d=0.3)
    X = X.copy()
    Y = Y.copy()
    rng = np.random.default_rng(5)
    for b in (1, 3, 4):
        for i in range(gamma + 1):
            pos = rng.choice(V // 300, size=20, replace=False) * 300 + 7
            X[b, i, pos] = np.arange(100, 0, -5, dtype=np.float32)
            if i < gamma:
                Y[b, i, pos] = X[b, i, pos] - 0.5
    if dtype == "bf16":
        X, Y = synth.f32_to_bf16_bits(X), synth.f32_to_bf16_bits(Y)
    T = np.array([1.0, 1.0, 0.7, 1.3, 0.0, 1.0], np.float32)
    d, _, _ = oracle.sample_rows(Y.reshape(B * gamma, V), synth.draft_sampling_temperatures(T, gamma),
                                 20, 0.95, 9)
    d = d.reshape(B, gamma)
    for seed in (1, 2, 3):
        want_tok, want_len, margins, want_st = oracle.verify(X, Y, d, T, 20, 0.95, seed, cut_margin=True)
        tok, ln, st = _run_verify(dv, X, Y, d, T, 20, 0.95, seed)
        assert st == want_st
        assert _compare_sampling(tok, ln, want_tok, want_len, margins) == 0
