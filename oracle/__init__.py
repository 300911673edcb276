"""CPU oracle for the batched draft-verification step (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package. The GPU library never links or calls it, and
the two share no code: the oracle is plain C (``dflash_oracle.c``, fp64,
single-threaded per call) built here with gcc, and this module only marshals
numpy arrays into it. Request ranges may be spread over host threads (ctypes
releases the GIL during each call).

Logits are passed as numpy arrays: ``uint16`` holds raw bf16 bits, ``float32``
holds fp32 values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dflash_oracle.c")
_HDR = os.path.join(_HERE, "dflash_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libdflash_oracle.so")

BF16, F32 = 0, 1
STATUS_BAD_TOKEN, STATUS_BAD_ROW, STATUS_BAD_TEMPERATURE = 1, 2, 8

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest_src:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    P, I, U32, U64, F, D = (ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64,
                            ctypes.c_float, ctypes.c_double)
    lib.oracle_philox4x32_10.argtypes = [P, P, P]
    lib.oracle_philox4x32_10.restype = None
    lib.oracle_uniforms.argtypes = [U64, U32, U32, U32, P, P]
    lib.oracle_uniforms.restype = None
    lib.oracle_argmax_row.argtypes = [P, I, I, P]
    lib.oracle_argmax_row.restype = ctypes.c_int32
    lib.oracle_filter_row.argtypes = [P, I, I, D, I, F, P]
    lib.oracle_filter_row.restype = I
    lib.oracle_filter_row_sparse.argtypes = [P, I, I, D, I, F, P, P]
    lib.oracle_filter_row_sparse.restype = I
    lib.oracle_verify.argtypes = [P, P, P, I, I, I, I, P, I, F, U64, P, P, P, P, I, I]
    lib.oracle_verify.restype = I
    lib.oracle_verify_margins.argtypes = [P, P, P, I, I, I, I, P, I, F, U64, P, P, P, P, P, P, I, I]
    lib.oracle_verify_margins.restype = I
    lib.oracle_verify_det_margins.argtypes = [P, P, I, I, I, I, P, I, F, U64, P, P, P, P, P, P, I, I]
    lib.oracle_verify_det_margins.restype = I
    lib.oracle_verify_greedy.argtypes = [P, P, I, I, I, I, P, P, P, I, I]
    lib.oracle_verify_greedy.restype = I
    lib.oracle_sample_rows.argtypes = [P, I, I, I, P, I, F, U64, P, P, P, I, I]
    lib.oracle_sample_rows.restype = I
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    raise TypeError(f"logits must be uint16 (bf16 bits) or float32, got {a.dtype}")


def _contig(a, dtype=None):
    return np.ascontiguousarray(a if dtype is None else np.asarray(a, dtype=dtype))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def load_variant(path: str):
    """Bind a separately built copy of the oracle (used by the mutation tests,
    which compile deliberately broken copies and check that the pins fail)."""
    return _bind(ctypes.CDLL(os.path.abspath(path)))


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile oracle source text (same flags as ``build``) into ``out_path``."""
    src_path = out_path[:-3] + ".c"
    with open(src_path, "w") as f:
        f.write(source_text)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-I", _HERE, "-o", out_path, src_path, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def philox4x32_10(ctr, key, lib=None) -> np.ndarray:
    lib = lib or _load()
    c = _contig(ctr, np.uint32)
    k = _contig(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib.oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniforms(seed: int, request: int, position: int, stream: int = 0, lib=None):
    lib = lib or _load()
    ua, ud = ctypes.c_float(), ctypes.c_float()
    lib.oracle_uniforms(seed, request, position, stream, ctypes.byref(ua), ctypes.byref(ud))
    return ua.value, ud.value


def argmax_row(row: np.ndarray, lib=None):
    lib = lib or _load()
    row = _contig(row)
    st = np.zeros(1, np.uint32)
    j = lib.oracle_argmax_row(_ptr(row), row.shape[-1], _dtype_code(row), _ptr(st))
    return int(j), int(st[0])


def filter_row(row: np.ndarray, temperature: float, top_k: int, top_p: float, lib=None) -> np.ndarray | None:
    """Dense filtered distribution (fp64) of one row, or None for a bad row."""
    lib = lib or _load()
    row = _contig(row)
    V = row.shape[-1]
    prob = np.zeros(V, np.float64)
    n = lib.oracle_filter_row(_ptr(row), V, _dtype_code(row), float(temperature), int(top_k),
                              float(top_p), _ptr(prob))
    return None if n < 0 else prob


def filter_row_sparse(row: np.ndarray, temperature: float, top_k: int, top_p: float, lib=None):
    """Kept tokens in (logit desc, index asc) order and their probabilities."""
    lib = lib or _load()
    row = _contig(row)
    V = row.shape[-1]
    idx = np.zeros(V, np.int32)
    prob = np.zeros(V, np.float64)
    n = lib.oracle_filter_row_sparse(_ptr(row), V, _dtype_code(row), float(temperature),
                                     int(top_k), float(top_p), _ptr(idx), _ptr(prob))
    if n < 0:
        return None
    return idx[:n].copy(), prob[:n].copy()


def accept_rates(target, draft, temperature, top_k, top_p, threads=None, lib=None):
    """Per (request, draft position) probability that the draft token is
    accepted when it is a sample of q: alpha = sum_v min(p(v), q(v)) over the
    filtered target and draft distributions (standard speculative sampling;
    the accept rule of "DFlash2 用投机解码给 Qwen 提速", bml.asia, the
    draft/verify loop). Greedy requests (temperature 0) get NaN: their accept
    length is the argmax prefix match, not a random variable. Returns [B, gamma]."""
    lib = lib or _load()
    X = _contig(target)
    Y = _contig(draft)
    T = np.asarray(temperature, np.float32)
    B, g1, V = X.shape
    gamma = g1 - 1
    alpha = np.full((B, gamma), np.nan, np.float64)
    jobs = [(b, i) for b in range(B) if T[b] > 0 and np.isfinite(T[b]) for i in range(gamma)]

    def run(job):
        b, i = job
        p = filter_row(X[b, i], float(T[b]), top_k, top_p, lib=lib)
        q = filter_row(Y[b, i], float(T[b]), top_k, top_p, lib=lib)
        alpha[b, i] = np.nan if p is None or q is None else float(np.minimum(p, q).sum())

    nthreads = threads or default_threads()
    if nthreads <= 1:
        for j in jobs:
            run(j)
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(run, jobs))
    return alpha


def expected_accept_len(alpha) -> np.ndarray:
    """Closed-form mean accept length of each request from its accept rates:
    the step emits position i (i = 0..gamma) when every draft before it was
    accepted, so E[len] = sum_{i=0}^{gamma} prod_{j<i} alpha_j."""
    a = np.asarray(alpha, np.float64)
    surv = np.concatenate([np.ones((a.shape[0], 1)), np.cumprod(a, axis=1)], axis=1)
    return surv.sum(axis=1)


def _ranges(n: int, parts: int):
    parts = max(1, min(parts, n))
    step = (n + parts - 1) // parts
    return [(s, min(n, s + step)) for s in range(0, n, step)]


def verify(target, draft, draft_tokens, temperature, top_k, top_p, seed, threads=None,
           requests=None, lib=None, split_margins=False, cut_margin=False):
    """Sampling-mode verification (greedy for requests with temperature 0).

    Returns (tokens [B, gamma+1], accept_len [B], margin [B], status).
    ``requests`` (optional iterable of request indices) restricts the work to
    those requests; the other rows of the outputs stay -1 / 0.
    With ``split_margins`` the third item is the pair (accept margin [B],
    draw margin [B]): the accept tests and top-p cuts, and the final draw.
    With ``cut_margin`` it is the triple (accept [B], cut [B], draw [B]):
    the accept tests alone, the top-p cuts, and the final draw.
    """
    lib = lib or _load()
    X = _contig(target)
    Y = _contig(draft)
    d = _contig(draft_tokens, np.int32)
    T = _contig(temperature, np.float32)
    B, g1, V = X.shape
    gamma = g1 - 1
    assert Y.shape == (B, gamma, V) and d.shape == (B, gamma) and T.shape == (B,)
    assert X.dtype == Y.dtype
    dt = _dtype_code(X)
    tokens = np.full((B, gamma + 1), -1, np.int32)
    lens = np.zeros(B, np.int32)
    margin = np.full(B, np.inf, np.float64)
    margin_draw = np.full(B, np.inf, np.float64)
    margin_cut = np.full(B, np.inf, np.float64)
    nthreads = threads or default_threads()
    if requests is None:
        todo = _ranges(B, nthreads * 4)
    else:
        todo = [(b, b + 1) for b in sorted(set(int(b) for b in requests))]

    def run(rng):
        st = np.zeros(1, np.uint32)
        rc = lib.oracle_verify_margins(_ptr(X), _ptr(Y), _ptr(d), B, gamma, V, dt, _ptr(T),
                                       int(top_k), float(top_p), int(seed), _ptr(tokens),
                                       _ptr(lens), _ptr(margin), _ptr(margin_draw),
                                       _ptr(margin_cut) if cut_margin else None, _ptr(st),
                                       rng[0], rng[1])
        if rc != 0:
            raise RuntimeError(f"oracle_verify failed: {rc}")
        return int(st[0])

    if nthreads <= 1 or len(todo) <= 1:
        statuses = [run(r) for r in todo]
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            statuses = list(ex.map(run, todo))
    status = 0
    for s in statuses:
        status |= s
    if cut_margin:
        return tokens, lens, (margin, margin_cut, margin_draw), status
    if split_margins:
        return tokens, lens, (margin, margin_draw), status
    return tokens, lens, np.minimum(margin, margin_draw), status


def verify_det(target, draft_tokens, temperature, top_k, top_p, seed, threads=None, lib=None,
               split_margins=False, cut_margin=False):
    """Verification of deterministic drafts (q = the point mass at each draft
    token; no draft logits). Returns (tokens, accept_len, margin, status) as
    ``verify``, with the same ``split_margins`` and ``cut_margin`` options."""
    lib = lib or _load()
    X = _contig(target)
    d = _contig(draft_tokens, np.int32)
    T = _contig(temperature, np.float32)
    B, g1, V = X.shape
    gamma = g1 - 1
    assert d.shape == (B, gamma) and T.shape == (B,)
    dt = _dtype_code(X)
    tokens = np.full((B, gamma + 1), -1, np.int32)
    lens = np.zeros(B, np.int32)
    margin = np.full(B, np.inf, np.float64)
    margin_draw = np.full(B, np.inf, np.float64)
    margin_cut = np.full(B, np.inf, np.float64)
    nthreads = threads or default_threads()
    todo = _ranges(B, nthreads * 4)

    def run(rng):
        st = np.zeros(1, np.uint32)
        rc = lib.oracle_verify_det_margins(_ptr(X), _ptr(d), B, gamma, V, dt, _ptr(T), int(top_k),
                                           float(top_p), int(seed), _ptr(tokens), _ptr(lens),
                                           _ptr(margin), _ptr(margin_draw),
                                           _ptr(margin_cut) if cut_margin else None, _ptr(st), rng[0], rng[1])
        if rc != 0:
            raise RuntimeError(f"oracle_verify_det failed: {rc}")
        return int(st[0])

    if nthreads <= 1 or len(todo) <= 1:
        statuses = [run(r) for r in todo]
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            statuses = list(ex.map(run, todo))
    status = 0
    for st_ in statuses:
        status |= st_
    if cut_margin:
        return tokens, lens, (margin, margin_cut, margin_draw), status
    if split_margins:
        return tokens, lens, (margin, margin_draw), status
    return tokens, lens, np.minimum(margin, margin_draw), status


def verify_greedy(target, draft_tokens, threads=None, lib=None):
    lib = lib or _load()
    X = _contig(target)
    d = _contig(draft_tokens, np.int32)
    B, g1, V = X.shape
    gamma = g1 - 1
    assert d.shape == (B, gamma)
    dt = _dtype_code(X)
    tokens = np.full((B, gamma + 1), -1, np.int32)
    lens = np.zeros(B, np.int32)

    def run(rng):
        st = np.zeros(1, np.uint32)
        rc = lib.oracle_verify_greedy(_ptr(X), _ptr(d), B, gamma, V, dt, _ptr(tokens), _ptr(lens),
                                      _ptr(st), rng[0], rng[1])
        if rc != 0:
            raise RuntimeError(f"oracle_verify_greedy failed: {rc}")
        return int(st[0])

    nthreads = threads or default_threads()
    with ThreadPoolExecutor(nthreads) as ex:
        statuses = list(ex.map(run, _ranges(B, nthreads)))
    status = 0
    for s in statuses:
        status |= s
    return tokens, lens, status


def sample_rows(logits, temperature, top_k, top_p, seed, threads=None, lib=None):
    """One token per row of ``logits`` [R, V] from its filtered distribution.

    Returns (tokens [R], margin [R], status)."""
    lib = lib or _load()
    L = _contig(logits)
    R, V = L.shape
    T = _contig(temperature, np.float32)
    assert T.shape == (R,)
    dt = _dtype_code(L)
    out = np.zeros(R, np.int32)
    margin = np.full(R, np.inf, np.float64)

    def run(rng):
        st = np.zeros(1, np.uint32)
        rc = lib.oracle_sample_rows(_ptr(L), R, V, dt, _ptr(T), int(top_k), float(top_p),
                                    int(seed), _ptr(out), _ptr(margin), _ptr(st), rng[0], rng[1])
        if rc != 0:
            raise RuntimeError(f"oracle_sample_rows failed: {rc}")
        return int(st[0])

    nthreads = threads or default_threads()
    with ThreadPoolExecutor(nthreads) as ex:
        statuses = list(ex.map(run, _ranges(R, nthreads * 4)))
    status = 0
    for s in statuses:
        status |= s
    return out, margin, status


# ---- the LM head ---------------------------------------------------------------------------
def _bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def lmhead_logits(h_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """logits[m, n] = sum_k h[m, k] w[n, k] (the target's vocabulary projection
    of the positions' last hidden states, the logits the draft/verify loop of
    "DFlash2 用投机解码给 Qwen 提速" verifies from), from bf16 bit patterns
    (uint16 [M, K] and [V, K]). Every product of two bf16 values is exact in
    fp64, and the sum is accurate to about 2^-53 relative to sum |h_k w_k|
    (numpy's matmul as the summing step)."""
    return _bf16_to_f64(h_bits) @ _bf16_to_f64(w_bits).T


def lmhead_abs(h_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """sum_k |h[m, k] w[n, k]|: the scale of each logit's rounding error."""
    return np.abs(_bf16_to_f64(h_bits)) @ np.abs(_bf16_to_f64(w_bits)).T
