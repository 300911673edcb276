"""dflash_verify_noalloc: the verification step for callers that cannot
allocate device memory (a framework's private memory pool, a plugin that does
not own the process's allocator, a path where cudaMalloc/cudaFree are not
allowed). It takes no workspace; its scratch is a fixed array the library keeps
on the GPU.

Called here through the C ABI and compared, on two calls in a row, with
dflash_verify given its own workspace: same inputs, same seed, so tokens,
accept lengths and status words must agree exactly (the deterministic kernel
meets any tolerance the other tests use). This file sorts last so that a run
stopping at the first failure has run every other test before it; it also
passes alone in a fresh process (the first call sets the scratch up).
"""
import ctypes

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


def _case(dtype, top_k, top_p):
    inp = synth.make_workload("b32_mixed_v248320", data_seed=21, seed=3, B=12, V=50021)
    if dtype == "f32":
        inp.target, inp.draft = synth.to_float(inp.target), synth.to_float(inp.draft)
    B, gamma, V = inp.shape
    d, _, _ = oracle.sample_rows(inp.draft.reshape(B * gamma, V),
                                 synth.draft_sampling_temperatures(inp.temperature, gamma),
                                 top_k, top_p, 5)
    return inp, d.reshape(B, gamma)


def _noalloc(lib, X, Y, d, T, B, gamma, V, dt, top_k, top_p, seed, out_tok, out_len, st):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.dflash_verify_noalloc(X.data_ptr(), Y.data_ptr(), d.data_ptr(), B, gamma, V,
                                     dt, T.data_ptr(), top_k, top_p, seed, out_tok.data_ptr(),
                                     out_len.data_ptr(), st.data_ptr(), stream)


# the top-k filter in bf16 and fp32, the full-vocabulary softmax (which also
# uses the draw's part of the scratch and a second pass of launches), and
# top-p over the full vocabulary (its cut's rounds and histograms too)
@pytest.mark.parametrize("dtype,top_k,top_p", [("bf16", 20, 0.95), ("f32", 20, 0.95), ("bf16", 0, 1.0),
                                               ("bf16", 0, 0.9)])
def test_noalloc_matches_workspace_entry_point_twice(dv, dtype, top_k, top_p):
    lib = dv.load()
    inp, d_np = _case(dtype, top_k, top_p)
    B, gamma, V = inp.shape
    dt = dv.DFLASH_BF16 if dtype == "bf16" else dv.DFLASH_F32
    X, Y = synth.to_torch(inp.target, DEV), synth.to_torch(inp.draft, DEV)
    d = torch.from_numpy(d_np).to(DEV)
    T = torch.from_numpy(inp.temperature).to(DEV)
    assert 0 < lib.dflash_workspace_bytes(B, gamma, V, dt, top_k, top_p) <= lib.dflash_noalloc_scratch_bytes()
    for seed in (3, 4):            # two calls in a row on the shared scratch
        want_st = torch.zeros(1, dtype=torch.int32, device=DEV)
        want_tok, want_len = dv.verify(X, Y, d, T, top_k, top_p, seed, status=want_st)
        tok = torch.full((B, gamma + 1), -7, dtype=torch.int32, device=DEV)
        ln = torch.full((B,), -7, dtype=torch.int32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        rc = _noalloc(lib, X, Y, d, T, B, gamma, V, dt, top_k, top_p, seed, tok, ln, st)
        assert rc == 0, lib.dflash_last_error()
        torch.cuda.synchronize()
        assert torch.equal(tok, want_tok) and torch.equal(ln, want_len)
        assert int(st.item()) == int(want_st.item()) == 0
        assert int(ln.min()) >= 1 and int(ln.max()) <= gamma + 1


def test_noalloc_rejects_shapes_beyond_its_scratch(dv):
    lib = dv.load()
    B, gamma, V = 32, 7, 2_000_000    # workspace far above the fixed scratch
    assert lib.dflash_workspace_bytes(B, gamma, V, 0, 20, 0.95) > lib.dflash_noalloc_scratch_bytes()
    p = ctypes.c_void_p(1 << 20)
    rc = lib.dflash_verify_noalloc(p, p, p, B, gamma, V, 0, p, 20, 0.95, 0, p, p, None, None)
    assert rc == dv.ERR_INVALID_ARG
    assert b"scratch" in lib.dflash_last_error()
