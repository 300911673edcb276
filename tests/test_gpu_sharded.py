"""GPU parity of the vocabulary-sharded verification.

The shards of a rank group are played on one GPU: each shard's record comes
from dflash_shard_candidates on a contiguous copy of its vocabulary slice
(uneven slices, odd offsets, so rows start at every alignment), the records
are stacked as the all-gather would leave them, and dflash_verify_candidates
verifies from them. The outputs must equal dflash_verify's on the whole rows
bit for bit (tokens, accept lengths, status word), and agree with the oracle
within the bars of the unsharded parity tests.
"""
import numpy as np
import pytest

import oracle
import synth
from parity_bounds import ROW_BAR, compare_rows, excused_topk

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


def _bounds(V, n, seed):
    """n uneven shards, each at least V / (2n) wide, cut at odd offsets."""
    rng = np.random.default_rng(seed)
    step = V / n
    j = int(step // 4)
    cuts = [int(step * i + rng.integers(-j, j + 1)) | 1 for i in range(1, n)]
    return [0] + cuts + [V]


def _records(dv, X, Y, bounds, k, order=None):
    recs = []
    for s in range(len(bounds) - 1):
        lo, hi = bounds[s], bounds[s + 1]
        recs.append(dv.shard_candidates(_t(np.ascontiguousarray(X[:, :, lo:hi])),
                                        _t(np.ascontiguousarray(Y[:, :, lo:hi])), lo, k))
    if order is not None:
        recs = [recs[i] for i in order]
    return torch.stack(recs).contiguous()


def _sharded(dv, records, k, d, T, V, top_k, top_p, seed):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok, ln = dv.verify_candidates(records, k, torch.from_numpy(np.ascontiguousarray(d)).to(DEV),
                                   torch.from_numpy(np.ascontiguousarray(T, np.float32)).to(DEV), V, top_k,
                                   top_p, seed, status=st)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), ln.cpu().numpy(), int(st.item())


def _whole(dv, X, Y, d, T, top_k, top_p, seed):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok, ln = dv.verify(_t(X), _t(Y), torch.from_numpy(np.ascontiguousarray(d)).to(DEV),
                        torch.from_numpy(np.ascontiguousarray(T, np.float32)).to(DEV), top_k, top_p, seed,
                        status=st)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), ln.cpu().numpy(), int(st.item())


def _drafts(Y, T, top_k, top_p, seed):
    B, gamma, V = Y.shape
    d, _, _ = oracle.sample_rows(Y.reshape(B * gamma, V), synth.draft_sampling_temperatures(T, gamma), top_k,
                                 top_p, seed)
    return d.reshape(B, gamma)


@pytest.mark.parametrize("dtype,V", [("bf16", 20011), ("f32", 5003)])
@pytest.mark.parametrize("n_shards", [1, 2, 3, 8])
@pytest.mark.parametrize("top_k,top_p", [(20, 0.95), (5, 0.9), (1, 1.0), (32, 1.0)])
def test_sharded_equals_whole_rows(dv, dtype, V, n_shards, top_k, top_p):
    B, gamma = 9, 7
    X, Y, _ = synth.make_logits(B, gamma, V, dtype, data_seed=V + n_shards, sigma_d=0.5)
    T = np.array([1.0, 0.0, 0.6, 1.0, 1.5, 0.0, 0.8, 1.0, 2.0], np.float32)
    d = _drafts(Y, T, top_k, top_p, n_shards)
    recs = _records(dv, X, Y, _bounds(V, n_shards, seed=V * n_shards), top_k)
    for seed in (3, 4):
        tok, ln, st = _sharded(dv, recs, top_k, d, T, V, top_k, top_p, seed)
        w_tok, w_ln, w_st = _whole(dv, X, Y, d, T, top_k, top_p, seed)
        assert st == w_st == 0
        assert np.array_equal(tok, w_tok) and np.array_equal(ln, w_ln)
        o_tok, o_ln, (m_acc, m_cut, m_draw), o_st = oracle.verify(X, Y, d, T, top_k, top_p, seed,
                                                                  cut_margin=True)
        assert o_st == st
        n_bad = compare_rows(tok, ln, o_tok, o_ln, lambda b: excused_topk(m_acc[b], m_cut[b], m_draw[b]))
        assert n_bad <= ROW_BAR * B


def test_shard_order_and_wider_shard_lists(dv):
    """Records in any order, and shards that keep more candidates (k = 32)
    than the filter's top-k (20), give the same outputs."""
    B, gamma, V = 12, 7, 30011
    X, Y, _ = synth.make_logits(B, gamma, V, "bf16", data_seed=77, sigma_d=(0.3, 1.5))
    T = synth.cycle_temperatures(B)
    d = _drafts(Y, T, 20, 0.95, 5)
    bounds = _bounds(V, 5, seed=9)
    w_tok, w_ln, w_st = _whole(dv, X, Y, d, T, 20, 0.95, 11)
    for k, order in ((20, [4, 2, 0, 3, 1]), (32, None), (32, [1, 0, 4, 3, 2])):
        tok, ln, st = _sharded(dv, _records(dv, X, Y, bounds, k, order), k, d, T, V, 20, 0.95, 11)
        assert st == w_st
        assert np.array_equal(tok, w_tok) and np.array_equal(ln, w_ln)


def test_sharded_full_size_b32_mixed(dv):
    """The B=32 mixed bf16 workload (block 8, V=248320) in 4 shards of 62080."""
    inp = synth.make_workload("b32_mixed_v248320", data_seed=3, seed=3)
    B, gamma, V = inp.shape
    d = _drafts(inp.draft, inp.temperature, 20, 0.95, 8)
    recs = _records(dv, inp.target, inp.draft, [0, 62080, 124160, 186240, 248320], 20)
    tok, ln, st = _sharded(dv, recs, 20, d, inp.temperature, V, 20, 0.95, inp.seed)
    w_tok, w_ln, w_st = _whole(dv, inp.target, inp.draft, d, inp.temperature, 20, 0.95, inp.seed)
    assert st == w_st == 0
    assert np.array_equal(tok, w_tok) and np.array_equal(ln, w_ln)
    # and against the oracle on the whole rows
    o_tok, o_ln, (m_acc, m_cut, m_draw), o_st = oracle.verify(inp.target, inp.draft, d, inp.temperature, 20,
                                                              0.95, inp.seed, cut_margin=True)
    assert o_st == 0
    n_bad = compare_rows(tok, ln, o_tok, o_ln, lambda b: excused_topk(m_acc[b], m_cut[b], m_draw[b]))
    assert n_bad <= ROW_BAR * B


def test_sharded_greedy_only(dv):
    B, gamma, V = 8, 7, 12007
    X, Y, _ = synth.make_logits(B, gamma, V, "f32", data_seed=5)
    T = np.zeros(B, np.float32)
    am = np.argmax(X[:, :gamma], axis=-1)
    d = am.astype(np.int32).copy()
    d[::3, 2] = (d[::3, 2] + 1) % V
    recs = _records(dv, X, Y, _bounds(V, 3, seed=2), 20)
    tok, ln, st = _sharded(dv, recs, 20, d, T, V, 20, 0.95, 0)
    g_tok, g_ln, g_st = oracle.verify_greedy(X, d)
    assert st == g_st == 0
    assert np.array_equal(tok, g_tok) and np.array_equal(ln, g_ln)


def test_sharded_bad_rows_and_tokens(dv):
    """A NaN in one shard's part of a row, an infinite logit, and a shard whose
    part of a row is all -inf (the row as a whole is fine): the same status
    word as the whole rows, and the same outputs for the requests without a
    bad row."""
    B, gamma, V = 6, 7, 9001
    X, Y, _ = synth.make_logits(B, gamma, V, "f32", data_seed=13)
    X, Y = X.copy(), Y.copy()
    T = np.array([1.0, 1.0, 0.0, 1.0, -1.0, 0.7], np.float32)
    bounds = [0, 3000, 6001, 9001]
    X[1, 3, 4500] = np.nan            # shard 1 of request 1, target row 3
    Y[3, 2, 100] = np.inf             # shard 0 of request 3, draft row 2
    X[5, 1, 6001:9001] = -np.inf      # shard 2's part of request 5's target row 1
    X[2, 4, 7000] = np.nan            # a greedy request's row
    d = _drafts(np.nan_to_num(Y, nan=0.0, posinf=0.0), T, 20, 0.95, 3)
    d[0, 1] = V
    d[5, 0] = -3
    recs = _records(dv, X, Y, bounds, 20)
    tok, ln, st = _sharded(dv, recs, 20, d, T, V, 20, 0.95, 2)
    w_tok, w_ln, w_st = _whole(dv, X, Y, d, T, 20, 0.95, 2)
    assert st == w_st == (oracle.STATUS_BAD_TOKEN | oracle.STATUS_BAD_ROW | oracle.STATUS_BAD_TEMPERATURE)
    assert np.all((tok >= -1) & (tok < V)) and np.all((ln >= 1) & (ln <= gamma + 1))
    for b in (0, 4, 5):
        assert np.array_equal(tok[b], w_tok[b]) and ln[b] == w_ln[b]
