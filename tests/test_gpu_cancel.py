"""Cancellation and the abort exit path, without a GPU fault.

dflash_workspace_cancel sets the workspace's abort flag. A call launched on
a cancelled workspace reports DFLASH_STATUS_TIMEOUT and returns before it
issues a copy (its CTAs read the flag in their prologue); a call already
running gives up its bounded waits, lets its issued bulk copies land, and
returns with the same status. The context stays usable: after
dflash_workspace_init the same call gives the outputs of an uncancelled
call again. Every mode that runs the stream kernel is covered.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TIMEOUT = 4


@pytest.fixture(scope="module")
def dv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_83_gb300 as m

    m.build()
    m.load()
    return m


@pytest.mark.parametrize("mode", ["top_k", "full_vocab", "top_p_vocab", "det", "greedy", "sample_rows", "shard",
                                  "lmhead"])
def test_cancelled_call_reports_timeout_and_the_workspace_recovers(dv, mode):
    B, gamma, V = 6, 7, 20011 if mode != "lmhead" else 20008  # the LM head wants V % 8 == 0
    X, Y, _ = synth.make_logits(B, gamma, V, "bf16", data_seed=17, sigma_d=0.5)
    T = np.array([1.0, 0.0, 0.6, 1.0, 1.5, 0.0], np.float32)
    top_k, top_p = {"full_vocab": (0, 1.0), "top_p_vocab": (0, 0.9)}.get(mode, (20, 0.95))
    d, _, _ = oracle.sample_rows(Y.reshape(B * gamma, V), synth.draft_sampling_temperatures(T, gamma), top_k,
                                 top_p, 4)
    Xd, Yd = synth.to_torch(X, DEV), synth.to_torch(Y, DEV)
    dd, Td = torch.from_numpy(d.reshape(B, gamma)).to(DEV), torch.from_numpy(T).to(DEV)
    if mode == "sample_rows":
        ws = dv.Workspace(dv.rows_workspace_bytes(B * gamma, V, dv.DFLASH_BF16, 20, 0.95), DEV)
    elif mode == "shard":
        ws = dv.Workspace(dv.load().dflash_shard_workspace_bytes(B, gamma, V, dv.DFLASH_BF16, 20), DEV)
    else:
        ws = dv.Workspace(dv.workspace_bytes(B, gamma, V, dv.DFLASH_BF16, top_k, top_p), DEV)

    if mode == "lmhead":
        rng = np.random.default_rng(3)
        h = synth.to_torch(synth.f32_to_bf16_bits(rng.standard_normal((B * (2 * gamma + 1), 64)).astype(np.float32)),
                           DEV)
        w = synth.to_torch(synth.f32_to_bf16_bits((rng.standard_normal((V, 64)) * 0.25).astype(np.float32)), DEV)

    def call():
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        if mode in ("top_k", "full_vocab", "top_p_vocab"):
            out = dv.verify(Xd, Yd, dd, Td, top_k, top_p, 9, status=st, workspace=ws)
        elif mode == "det":
            out = dv.verify_det(Xd, dd, Td, top_k, top_p, 9, status=st, workspace=ws)
        elif mode == "greedy":
            out = dv.verify_greedy(Xd, dd, status=st, workspace=ws)
        elif mode == "sample_rows":
            out = (dv.sample_rows(Yd.view(B * gamma, V), Td.repeat_interleave(gamma), 20, 0.95, 3, status=st,
                                  workspace=ws),)
        elif mode == "shard":
            out = (dv.shard_candidates(Xd, Yd, 0, 20, status=st, workspace=ws),)
        else:  # the LM head runs whatever the flag; its finals-only verification reports the cancel
            out = dv.lmhead_verify(h, w, B, gamma, dd, Td, top_k, top_p, 9, status=st, workspace=ws)[:2]
        torch.cuda.synchronize()
        return [o.cpu().numpy() for o in out], int(st.item())

    want, st0 = call()
    assert st0 & TIMEOUT == 0
    ws.cancel()
    _, st = call()
    assert st & TIMEOUT, f"cancelled call reported status {st}"
    _, st = call()  # still cancelled until the workspace is prepared again
    assert st & TIMEOUT
    ws.reset()
    again, st2 = call()
    assert st2 == st0
    for a, b in zip(want, again):
        assert np.array_equal(a, b)
