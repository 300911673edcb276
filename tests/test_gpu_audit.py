"""The probabilities each accept test used, audited against the oracle.

dflash_verify_audit returns, per sampling request and draft position, the
p(d) and q(d) that the test u < p(d)/q(d) compared. They are checked against
the oracle's fp64 filtered distributions of the same rows (filter_row, dense)
at the draft token:
  * the sampling-mode bar: within 1e-5 absolute;
  * top-k filter (float-float weights and sums): within one fp32 rounding
    (1.05 * 2^-24 relative);
  * full-vocabulary softmax (the stream's normalisers, exp on the
    special-function unit): within the derived bound FV_PROB_REL relative
    (parity_bounds).
The outputs of the audit call equal those of dflash_verify bit for bit.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
import synth
from parity_bounds import FV_PROB_REL, U

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


def _oracle_pq(inp, d, top_k, top_p):
    """p_i(d_i), q_i(d_i) of every sampling request from the oracle's dense filter."""
    B, gamma, V = inp.shape
    jobs = [(b, i) for b in range(B) if inp.temperature[b] > 0 for i in range(gamma)]
    out = np.full((B, gamma, 2), np.nan)

    def run(job):
        b, i = job
        T = float(inp.temperature[b])
        p = oracle.filter_row(inp.target[b, i], T, top_k, top_p)
        q = oracle.filter_row(inp.draft[b, i], T, top_k, top_p)
        out[b, i, 0] = p[d[b, i]]
        out[b, i, 1] = q[d[b, i]]

    with ThreadPoolExecutor(oracle.default_threads()) as ex:
        list(ex.map(run, jobs))
    return out


def _audit(dv, inp, d, top_k, top_p):
    X, Y = synth.to_torch(inp.target, DEV), synth.to_torch(inp.draft, DEV)
    dd = torch.from_numpy(d).to(DEV)
    T = torch.from_numpy(inp.temperature).to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok, ln, pq = dv.verify_audit(X, Y, dd, T, top_k, top_p, inp.seed, status=st)
    tok2, ln2 = dv.verify(X, Y, dd, T, top_k, top_p, inp.seed)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(tok, tok2) and torch.equal(ln, ln2)
    return pq.cpu().numpy().astype(np.float64)


def test_audit_topk_headline_workload(dv):
    inp = synth.make_workload("b32_mixed_v248320", data_seed=1, seed=1)
    B, gamma, V = inp.shape
    d, _, _ = oracle.sample_rows(inp.draft.reshape(B * gamma, V),
                                 synth.draft_sampling_temperatures(inp.temperature, gamma), 20, 0.95, 11)
    d = d.reshape(B, gamma)
    got = _audit(dv, inp, d, 20, 0.95)
    want = _oracle_pq(inp, d, 20, 0.95)
    samp = inp.temperature > 0
    g, w = got[samp], want[samp]
    assert np.all(np.isfinite(g))
    assert np.max(np.abs(g - w)) < 1e-5
    assert np.all(np.abs(g - w) <= 1.05 * U * w + 1e-30)
    # greedy requests are not audited
    assert np.all(np.isnan(got[~samp]))


def test_audit_fullvocab_workload(dv):
    inp = synth.make_workload("b128_g15_fullvocab_f32", data_seed=2, seed=2, B=32)
    B, gamma, V = inp.shape
    d, _, _ = oracle.sample_rows(inp.draft.reshape(B * gamma, V),
                                 synth.draft_sampling_temperatures(inp.temperature, gamma), 0, 1.0, 12)
    d = d.reshape(B, gamma)
    got = _audit(dv, inp, d, 0, 1.0)
    want = _oracle_pq(inp, d, 0, 1.0)
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - want)) < 1e-5
    # relative, for every probability a draw from q can plausibly meet (the
    # SFU's exp flushes weights below 2^-126 of the row's largest to zero)
    rel = np.abs(got - want) / np.maximum(want, 1e-300)
    assert np.max(rel[want > 1e-30]) <= FV_PROB_REL, np.max(rel[want > 1e-30])
