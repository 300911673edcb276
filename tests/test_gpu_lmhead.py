"""The LM head on the tensor cores (tcgen05 MMAs from TMA-loaded shared
memory, fp32 accumulators in tensor memory) and the verification fused into
its epilogue.

- dflash_lmhead_logits against the oracle's fp64 product of the same bf16
  values: each logit within the bound of fp32 accumulation (K 2^-23 times
  sum |h_k w_k|) plus one bf16 rounding (2^-8 relative), and nearly all
  exactly the bf16 rounding of the exact sum.
- dflash_lmhead_verify against dflash_lmhead_logits followed by
  dflash_verify: logits, tokens, accept lengths and status bit for bit, and
  the workspace left at zero.
"""
import numpy as np
import pytest

import oracle
import synth

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


def _bits(rng, shape, scale):
    return synth.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def _check_logits(got_bits, h_bits, w_bits):
    K = h_bits.shape[1]
    exact = oracle.lmhead_logits(h_bits, w_bits)
    scale = oracle.lmhead_abs(h_bits, w_bits)
    got = synth.bf16_bits_to_f32(got_bits).astype(np.float64)
    acc = K * 2.0 ** -23 * scale
    bound = acc + 2.0 ** -8 * (np.abs(exact) + acc)
    err = np.abs(got - exact)
    assert np.all(err <= bound), float(np.max(err / np.maximum(bound, 1e-300)))
    rounded = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(exact.astype(np.float32))).astype(np.float64)
    assert np.mean(got == rounded) > 0.99


@pytest.mark.parametrize("M,V,K", [(128, 128, 64), (1, 8, 64), (37, 1032, 128), (200, 1000, 256),
                                   (512, 4104, 512), (480, 2056, 1024), (256, 40000, 128),
                                   # the full vocabulary: about 13 tiles per SM pair, each accumulator
                                   # slot reused many times, with one token group and with two
                                   (200, 248320, 64), (480, 248320, 64)])
def test_lmhead_logits_match_the_oracle(dv, M, V, K):
    rng = np.random.default_rng(M * 7 + V + K)
    h = _bits(rng, (M, K), 1.0)
    w = _bits(rng, (V, K), 2.0 / np.sqrt(K))
    hd, wd = synth.to_torch(h, DEV), synth.to_torch(w, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = dv.lmhead_logits(hd, wd, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    _check_logits(got, h, w)


def _fused_vs_unfused(dv, B, gamma, V, K, T, top_k, top_p, seed, data_seed, edit_h=None):
    rng = np.random.default_rng(data_seed)
    M, Mt = B * (2 * gamma + 1), B * (gamma + 1)
    hb = _bits(rng, (M, K), 1.0)
    if edit_h is not None:
        edit_h(hb)
    h = synth.to_torch(hb, DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(data_seed)
    w = (torch.randn((V, K), generator=g, device=DEV) * (2.0 / K ** 0.5)).to(torch.bfloat16)
    d = torch.from_numpy(rng.integers(0, V, size=(B, gamma)).astype(np.int32)).to(DEV)
    Td = torch.from_numpy(np.asarray(T, np.float32)).to(DEV)
    ws = dv.Workspace(dv.workspace_bytes(B, gamma, V, dv.DFLASH_BF16, top_k, top_p), DEV)
    st_f = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok_f, len_f, logits_f = dv.lmhead_verify(h, w, B, gamma, d, Td, top_k, top_p, seed, status=st_f, workspace=ws)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(ws.buf).item()) == 0, "workspace not left at zero"
    st_u = torch.zeros(1, dtype=torch.int32, device=DEV)
    logits_u = dv.lmhead_logits(h, w)
    tok_u, len_u = dv.verify(logits_u[:Mt].view(B, gamma + 1, V), logits_u[Mt:].view(B, gamma, V), d, Td, top_k,
                             top_p, seed, status=st_u)
    torch.cuda.synchronize()
    assert torch.equal(logits_f.view(torch.int16), logits_u.view(torch.int16))
    assert torch.equal(tok_f, tok_u) and torch.equal(len_f, len_u)
    assert int(st_f.item()) == int(st_u.item())
    if edit_h is not None:
        assert int(st_f.item()) & dv.STATUS_BAD_ROW
    return tok_f.cpu().numpy(), len_f.cpu().numpy(), logits_u, d.cpu().numpy()


@pytest.mark.parametrize("B,gamma,V,K", [(4, 3, 20000, 256), (2, 7, 8192, 64), (6, 2, 33000, 128),
                                         (1, 1, 1032, 64), (34, 7, 4104, 128)])
def test_fused_equals_unfused_small(dv, B, gamma, V, K):
    T = np.resize(np.array([1.0, 0.0, 0.7, 1.3, 0.0, 2.0], np.float32), B)  # cycled over the requests
    for seed in (0, 5):
        tok, ln, logits, d = _fused_vs_unfused(dv, B, gamma, V, K, T, 20, 0.95, seed, B * 100 + V)
        # and the verification of those logits against the oracle
        Mt = B * (gamma + 1)
        L = logits.view(torch.int16).cpu().numpy().view(np.uint16)
        X, Y = L[:Mt].reshape(B, gamma + 1, V), L[Mt:].reshape(B, gamma, V)
        want_tok, want_len, (m_acc, m_cut, m_draw), _ = oracle.verify(X, Y, d, T, 20, 0.95, seed, cut_margin=True)
        from parity_bounds import compare_rows, excused_topk

        compare_rows(tok, ln, want_tok, want_len, lambda b: excused_topk(m_acc[b], m_cut[b], m_draw[b]), "lmhead")


def test_fused_equals_unfused_full_shape(dv):
    """B = 32 requests, block 8, hidden size 5120, V = 248320 (W of 2.54 GB,
    random init), temperatures cycling greedy / 0.6 / 1.0, top-k 20, top-p 0.95."""
    B, gamma, V, K = 32, 7, 248320, 5120
    T = np.array([(0.0, 0.6, 1.0)[b % 3] for b in range(B)], np.float32)
    _fused_vs_unfused(dv, B, gamma, V, K, T, 20, 0.95, 1, 7)


def test_fused_equals_unfused_zero_and_nan_rows(dv):
    """Hidden states that are zero (every logit of the row ties at 0: the
    argmax is column 0) or hold a NaN (the whole row is NaN: BAD_ROW, and the
    key order still decides the argmax), on target rows of greedy and of
    sampling requests."""
    B, gamma, V, K = 4, 3, 20000, 128
    T = np.array([0.0, 1.0, 0.0, 0.7], np.float32)
    g1 = gamma + 1

    def edit(hb):
        hb[0 * g1 + 1] = 0  # greedy request 0, position 1: zeros
        hb[2 * g1 + 0, 5] = 0x7FC0  # greedy request 2, position 0: a NaN
        hb[1 * g1 + 2, 0] = 0x7FC0  # sampling request 1, position 2: a NaN
        hb[3 * g1 + 0] = 0  # sampling request 3, position 0: zeros

    for seed in (0, 3):
        _fused_vs_unfused(dv, B, gamma, V, K, T, 20, 0.95, seed, 77, edit_h=edit)
