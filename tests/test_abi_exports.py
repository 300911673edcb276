"""The C-ABI library loads, exports every entry point include/dflash_verify.h
declares, and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_83_gb300 as dv

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "dflash_verify.h")


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    dv.build()
    return dv.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
        assert n in dv.EXPORTS, f"binding lacks {n}"
    assert lib.dflash_abi_version() == 1


def test_workspace_sizes(lib):
    n = lib.dflash_workspace_bytes(32, 7, 248320, dv.DFLASH_BF16, 20, 0.95)
    assert n > 0 and n % 256 == 0
    assert lib.dflash_workspace_bytes(0, 7, 248320, 0, 20, 0.95) == 0
    assert lib.dflash_workspace_bytes(32, 7, 248320, 7, 20, 0.95) == 0
    assert lib.dflash_workspace_bytes(32, 7, 248320, 0, 64, 0.95) == 0   # top_k > 32
    # top-p over the full vocabulary keeps per-row cuts and histograms on top
    # of the full-vocabulary regions
    fv = lib.dflash_workspace_bytes(32, 7, 248320, 0, 0, 1.0)
    tp = lib.dflash_workspace_bytes(32, 7, 248320, 0, 0, 0.9)
    assert 0 < fv < tp and tp % 256 == 0
    assert lib.dflash_workspace_bytes(32, 7, 248320, 0, -1, 0.5) == tp
    assert lib.dflash_rows_workspace_bytes(224, 248320, 0, 0, 0.9) > 0   # the sampler
    assert lib.dflash_rows_workspace_bytes(224, 248320, 0, 20, 0.95) > 0
    assert lib.dflash_host_staging_bytes(32, 7, 248320, 0) >= 32 * 15 * 248320 * 2


def _verify(lib, B=2, gamma=3, V=100, dtype=0, top_k=20, top_p=0.95, ptr=1 << 20):
    # non-null fake pointers: argument checks run before any CUDA call
    p = ctypes.c_void_p(ptr)
    return lib.dflash_verify(p, p, p, B, gamma, V, dtype, p, top_k, top_p, 0, p, p, p, 1 << 30,
                             None, None)


def test_argument_checks_happen_on_the_host(lib):
    assert _verify(lib, B=0) == dv.ERR_INVALID_ARG
    assert b"B=0" in lib.dflash_last_error()
    assert _verify(lib, gamma=0) == dv.ERR_INVALID_ARG
    assert _verify(lib, gamma=33) == dv.ERR_INVALID_ARG
    assert _verify(lib, V=0) == dv.ERR_INVALID_ARG
    assert _verify(lib, dtype=5) == dv.ERR_INVALID_ARG
    assert _verify(lib, top_p=0.0) == dv.ERR_INVALID_ARG
    assert _verify(lib, top_p=float("nan")) == dv.ERR_INVALID_ARG
    assert _verify(lib, top_k=33) == dv.ERR_UNSUPPORTED
    assert _verify(lib, top_k=40, top_p=0.9) == dv.ERR_UNSUPPORTED
    # top-p over the full vocabulary: up to 2^22 tokens (the fixed-point sums)
    assert _verify(lib, V=(1 << 22) + 1, top_k=0, top_p=0.9) == dv.ERR_UNSUPPORTED
    assert _verify(lib, dtype=1, ptr=(1 << 20) + 2) == dv.ERR_INVALID_ARG  # fp32 misaligned
    n = ctypes.c_void_p(0)
    assert lib.dflash_verify(n, n, n, 2, 3, 100, 0, n, 20, 0.95, 0, n, n, n, 0, None,
                             None) == dv.ERR_INVALID_ARG
    assert lib.dflash_uniforms(0, 0, 3, 0, None, None, None) == dv.ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        dv.load(str(tmp_path / "absent.so"))


def test_cancel_refuses_a_buffer_without_the_header(lib):
    assert lib.dflash_workspace_cancel(None, 1 << 20, None) == dv.ERR_INVALID_ARG
    assert lib.dflash_workspace_cancel(ctypes.c_void_p(256), 64, None) == dv.ERR_INVALID_ARG
    assert b"abort flag" in lib.dflash_last_error()


@pytest.mark.parametrize("top_k,top_p", [(33, 0.95), (64, 0.5), (40, 1.0)])
def test_noalloc_reports_unsupported_filters_like_verify(lib, top_k, top_p):
    """An unsupported filter gets DFLASH_ERR_UNSUPPORTED and the same message
    from the workspace-free entry point as from dflash_verify (no launch, no
    GPU needed: both reject the call on the host)."""
    p = ctypes.c_void_p(1 << 20)
    B, gamma, V = 4, 7, 50000
    rc = lib.dflash_verify(p, p, p, B, gamma, V, 0, p, top_k, top_p, 0, p, p, p, 1 << 30, None, None)
    want = lib.dflash_last_error()
    assert rc == dv.ERR_UNSUPPORTED
    rc2 = lib.dflash_verify_noalloc(p, p, p, B, gamma, V, 0, p, top_k, top_p, 0, p, p, None, None)
    assert rc2 == dv.ERR_UNSUPPORTED
    assert lib.dflash_last_error() == want


def test_audit_entry_point_checks_its_output(lib):
    p = ctypes.c_void_p(1 << 20)
    rc = lib.dflash_verify_audit(p, p, p, 4, 7, 5000, 0, p, 20, 0.95, 0, p, p, None, p, 1 << 30, None, None)
    assert rc == dv.ERR_INVALID_ARG and b"audit" in lib.dflash_last_error()


def test_lmhead_argument_checks_happen_on_the_host(lib):
    """The LM head's shape, alignment and filter checks return before any CUDA
    call (fake non-null pointers, no GPU needed)."""
    p, q = ctypes.c_void_p(1 << 20), ctypes.c_void_p((1 << 20) + 8)
    assert lib.dflash_lmhead_logits(p, p, 513, 4096, 64, p, None, None) == dv.ERR_INVALID_ARG   # M > 512
    assert lib.dflash_lmhead_logits(p, p, 16, 4100, 64, p, None, None) == dv.ERR_INVALID_ARG   # V % 8
    assert lib.dflash_lmhead_logits(p, p, 16, 4096, 96, p, None, None) == dv.ERR_INVALID_ARG   # K % 64
    assert lib.dflash_lmhead_logits(q, p, 16, 4096, 64, p, None, None) == dv.ERR_INVALID_ARG   # 16-byte alignment
    assert b"aligned" in lib.dflash_last_error()
    n = ctypes.c_void_p(0)
    assert lib.dflash_lmhead_logits(n, p, 16, 4096, 64, p, None, None) == dv.ERR_INVALID_ARG

    def fused(B, gamma, top_k, top_p, V=4096, K=64):
        return lib.dflash_lmhead_verify(p, p, B, gamma, V, K, p, p, top_k, top_p, 0, p, p, p, p, 1 << 30, None,
                                        None)

    assert fused(32, 8, 20, 0.95) == dv.ERR_INVALID_ARG      # 32 x 17 = 544 rows > 512
    assert b"rows" in lib.dflash_last_error()
    assert fused(4, 3, 0, 1.0) == dv.ERR_UNSUPPORTED         # the full-vocabulary filter
    assert fused(4, 3, 0, 0.9) == dv.ERR_UNSUPPORTED         # top-p over the full vocabulary
    assert fused(4, 3, 40, 0.9) == dv.ERR_UNSUPPORTED
    assert fused(4, 3, 20, 0.0) == dv.ERR_INVALID_ARG
