"""Python binding of the GB300 draft-verification library (libdflash_verify.so).

Argument marshalling only: every step of the verification runs in the CUDA
kernels behind the C ABI declared in ``include/dflash_verify.h``. PyTorch
provides device memory and streams. There is no CPU fallback: if the compiled
library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
_INCLUDE = os.path.join(_ROOT, "include")
_BUILD = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD, "libdflash_verify.so")
SOURCES = ["dflash_sweep.cu", "dflash_fullvocab.cu", "dflash_fvtp.cu", "dflash_candidates.cu", "dflash_lmhead.cu",
           "dflash_abi.cu",
           "dflash_noalloc.cu"]
HEADERS = ["dflash_device.cuh", "dflash_internal.h", "dflash_rule.cuh", "dflash_ff.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]

DFLASH_BF16, DFLASH_F32 = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA = 0, 1, 2, 3
STATUS_BAD_TOKEN, STATUS_BAD_ROW, STATUS_TIMEOUT, STATUS_BAD_TEMPERATURE = 1, 2, 4, 8
MAX_TOP_K = 32


class DFlashError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"dflash error {code}: {message}")
        self.code = code


def _nvcc() -> str:
    env = os.environ.get("NVCC")
    if env:
        return env
    if os.path.exists("/usr/local/cuda/bin/nvcc"):
        return "/usr/local/cuda/bin/nvcc"
    return "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(_CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(_INCLUDE, "dflash_verify.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA sources for sm_103a (in parallel) and link the library."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    nvcc = _nvcc()
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(_BUILD, src.replace(".cu", f".{os.getpid()}.o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-I", _INCLUDE, "-c", os.path.join(_CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    for cmd, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{out.decode(errors='replace')}")
        if verbose and out:
            print(out.decode(errors="replace"))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
            "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    res = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if res.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(link)}\n{res.stdout.decode(errors='replace')}")
    os.replace(tmp, LIB_PATH)
    for o in objs:
        os.remove(o)
    return LIB_PATH


_lock = threading.Lock()
_lib = None

EXPORTS = {
    # name: (restype, argtypes)
    "dflash_abi_version": ("i", ""),
    "dflash_last_error": ("s", ""),
    "dflash_workspace_bytes": ("z", "iiiiif"),
    "dflash_rows_workspace_bytes": ("z", "iiiif"),
    "dflash_workspace_init": ("i", "pzp"),
    "dflash_workspace_cancel": ("i", "pzp"),
    "dflash_verify": ("i", "pppiiiipifQppp" "zpp"),
    "dflash_verify_audit": ("i", "pppiiiipifQpppp" "zpp"),
    "dflash_verify_det": ("i", "ppiiiipifQpppzpp"),
    "dflash_verify_greedy": ("i", "ppiiiipppzpp"),
    "dflash_host_staging_bytes": ("z", "iiii"),
    "dflash_verify_host": ("i", "pppiiiipifQppppzpzp"),
    "dflash_filter": ("i", "piiipifpppp" "zpp"),
    "dflash_sample": ("i", "piiipifQp" "pzpp"),
    "dflash_uniforms": ("i", "Qiiippp"),
    "dflash_candidates_words": ("z", "iii"),
    "dflash_shard_workspace_bytes": ("z", "iiiii"),
    "dflash_shard_candidates": ("i", "ppiiiiiippzpp"),
    "dflash_verify_candidates": ("i", "piipiiipifQpppp"),
    "dflash_noalloc_scratch_bytes": ("z", ""),
    "dflash_verify_noalloc": ("i", "pppiiiipifQpppp"),
    "dflash_lmhead_logits": ("i", "ppiiippp"),
    "dflash_lmhead_verify": ("i", "ppiiiippifQppppzpp"),
}
_CT = {"i": ctypes.c_int, "p": ctypes.c_void_p, "z": ctypes.c_size_t, "f": ctypes.c_float,
       "Q": ctypes.c_uint64, "s": ctypes.c_char_p, "": None}


def load(path: str | None = None):
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libdflash_verify.so not found at {p}: run build() first "
                                   "(there is no CPU fallback)")
            lib = ctypes.CDLL(p)
            for name, (res, args) in EXPORTS.items():
                fn = getattr(lib, name)
                fn.restype = _CT[res]
                fn.argtypes = [_CT[c] for c in args]
            if lib.dflash_abi_version() != 1:
                raise RuntimeError("unexpected ABI version")
            if path is not None:
                return lib
            _lib = lib
    return _lib


def _check(rc: int):
    if rc != OK:
        raise DFlashError(rc, load().dflash_last_error().decode(errors="replace"))


# ---- torch marshalling -------------------------------------------------------------
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return DFLASH_BF16
    if t.dtype == torch.float32:
        return DFLASH_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _dev(t, name, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _shape(t, shape, name):
    """Every buffer the library reads or writes must have the shape the call's
    sizes imply: a short tensor would let a kernel run past its end."""
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _on(device, **tensors):
    for name, t in tensors.items():
        if t is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device}, the call's logits on {device}")


def _status_ok(status):
    if status is not None and status.numel() < 1:
        raise ValueError("status must hold one int32 word")


def _stream_ptr(stream, device):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def workspace_bytes(B, gamma, V, dtype_code, top_k, top_p) -> int:
    n = load().dflash_workspace_bytes(B, gamma, V, dtype_code, top_k, top_p)
    if n == 0:
        raise DFlashError(ERR_INVALID_ARG, "unsupported or invalid shape / filter for a workspace")
    return n


class Workspace:
    """Device scratch for the verification kernels: a caller-owned byte
    buffer (allocated through torch), zero-filled once before first use."""

    def __init__(self, nbytes: int, device="cuda", stream=None):
        torch = _torch()
        self.nbytes = int(nbytes)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.reset(stream)

    def reset(self, stream=None):
        _check(load().dflash_workspace_init(self.buf.data_ptr(), self.nbytes,
                                            _stream_ptr(stream, self.buf.device)))

    def cancel(self, stream=None):
        """dflash_workspace_cancel: calls on this workspace give up their waits
        and report DFLASH_STATUS_TIMEOUT; reset() before the next use."""
        _check(load().dflash_workspace_cancel(self.buf.data_ptr(), self.nbytes,
                                              _stream_ptr(stream, self.buf.device)))

    @property
    def ptr(self):
        return self.buf.data_ptr()


_ws_cache: dict = {}


def _workspace_for(nbytes, device, workspace):
    if workspace is not None:
        if workspace.nbytes < nbytes:
            raise ValueError(f"workspace of {workspace.nbytes} bytes < {nbytes} needed")
        return workspace
    key = (str(device), threading.get_ident())
    ws = _ws_cache.get(key)
    if ws is None or ws.nbytes < nbytes:
        ws = Workspace(nbytes, device)
        _ws_cache[key] = ws
    return ws


def verify(target, draft, draft_tokens, temperature, top_k: int, top_p: float, seed: int,
           out_tokens=None, out_accept_len=None, status=None, workspace=None, stream=None):
    """dflash_verify on torch CUDA tensors. Returns (out_tokens, out_accept_len)."""
    torch = _torch()
    B, g1, V = target.shape
    gamma = g1 - 1
    if tuple(draft.shape) != (B, gamma, V) or draft.dtype != target.dtype:
        raise ValueError("draft must be [B, gamma, V] with the target's dtype")
    dt = _dtype_code(target)
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    if out_accept_len is None:
        out_accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    _shape(draft_tokens, (B, gamma), "draft_tokens")
    _shape(temperature, (B,), "temperature")
    _shape(out_tokens, (B, gamma + 1), "out_tokens")
    _shape(out_accept_len, (B,), "out_accept_len")
    _status_ok(status)
    _on(dev, draft=draft, draft_tokens=draft_tokens, temperature=temperature, out_tokens=out_tokens,
        out_accept_len=out_accept_len, status=status)
    ws = _workspace_for(workspace_bytes(B, gamma, V, dt, top_k, top_p), dev, workspace)
    rc = load().dflash_verify(
        _dev(target, "target"), _dev(draft, "draft"), _dev(draft_tokens, "draft_tokens", torch.int32),
        B, gamma, V, dt, _dev(temperature, "temperature", torch.float32), int(top_k), float(top_p),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _dev(out_tokens, "out_tokens", torch.int32),
        _dev(out_accept_len, "out_accept_len", torch.int32), ws.ptr, ws.nbytes,
        None if status is None else _dev(status, "status", torch.int32), _stream_ptr(stream, dev))
    _check(rc)
    return out_tokens, out_accept_len


def verify_audit(target, draft, draft_tokens, temperature, top_k: int, top_p: float, seed: int,
                 status=None, workspace=None, stream=None):
    """dflash_verify_audit on torch CUDA tensors. Returns (out_tokens,
    out_accept_len, audit_pq): audit_pq [B, gamma, 2] holds p(d), q(d) of each
    accept test (NaN where the call wrote nothing: greedy requests)."""
    torch = _torch()
    B, g1, V = target.shape
    gamma = g1 - 1
    if tuple(draft.shape) != (B, gamma, V) or draft.dtype != target.dtype:
        raise ValueError("draft must be [B, gamma, V] with the target's dtype")
    dt = _dtype_code(target)
    dev = target.device
    out_tokens = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    out_accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    audit = torch.full((B, gamma, 2), float("nan"), dtype=torch.float32, device=dev)
    _shape(draft_tokens, (B, gamma), "draft_tokens")
    _shape(temperature, (B,), "temperature")
    _status_ok(status)
    _on(dev, draft=draft, draft_tokens=draft_tokens, temperature=temperature, status=status)
    ws = _workspace_for(workspace_bytes(B, gamma, V, dt, top_k, top_p), dev, workspace)
    rc = load().dflash_verify_audit(
        _dev(target, "target"), _dev(draft, "draft"), _dev(draft_tokens, "draft_tokens", torch.int32),
        B, gamma, V, dt, _dev(temperature, "temperature", torch.float32), int(top_k), float(top_p),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _dev(out_tokens, "out_tokens", torch.int32),
        _dev(out_accept_len, "out_accept_len", torch.int32), _dev(audit, "audit_pq", torch.float32),
        ws.ptr, ws.nbytes, None if status is None else _dev(status, "status", torch.int32),
        _stream_ptr(stream, dev))
    _check(rc)
    return out_tokens, out_accept_len, audit


def lmhead_logits(h, w, out=None, status=None, stream=None):
    """dflash_lmhead_logits: logits [M, V] = h [M, K] @ w [V, K]^T in bf16 on
    the tensor cores (fp32 accumulation). Returns the logits tensor."""
    torch = _torch()
    if h.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
        raise ValueError("h and w must be bfloat16")
    M, K = h.shape
    V, K2 = w.shape
    if K2 != K:
        raise ValueError("h and w must share the hidden size")
    dev = h.device
    if out is None:
        out = torch.empty((M, V), dtype=torch.bfloat16, device=dev)
    _shape(out, (M, V), "out")
    _status_ok(status)
    _on(dev, w=w, out=out, status=status)
    rc = load().dflash_lmhead_logits(_dev(h, "h"), _dev(w, "w"), M, V, K, _dev(out, "out"),
                                     None if status is None else _dev(status, "status", torch.int32),
                                     _stream_ptr(stream, dev))
    _check(rc)
    return out


def lmhead_verify(h, w, B: int, gamma: int, draft_tokens, temperature, top_k: int, top_p: float, seed: int,
                  logits=None, status=None, workspace=None, stream=None):
    """dflash_lmhead_verify: the LM head over h [B (gamma + 1) + B gamma, K]
    (target rows, then draft rows) with the verification's tile statistics in
    its epilogue, then the verification's finals. Returns (out_tokens,
    out_accept_len, logits)."""
    torch = _torch()
    M, K = h.shape
    V = w.shape[0]
    if M != B * (2 * gamma + 1):
        raise ValueError("h must hold B (gamma + 1) target rows and B gamma draft rows")
    dev = h.device
    if logits is None:
        logits = torch.empty((M, V), dtype=torch.bfloat16, device=dev)
    out_tokens = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    out_len = torch.empty((B,), dtype=torch.int32, device=dev)
    _shape(draft_tokens, (B, gamma), "draft_tokens")
    _shape(temperature, (B,), "temperature")
    _shape(logits, (M, V), "logits")
    _status_ok(status)
    _on(dev, w=w, draft_tokens=draft_tokens, temperature=temperature, logits=logits, status=status)
    ws = _workspace_for(workspace_bytes(B, gamma, V, DFLASH_BF16, top_k, top_p), dev, workspace)
    rc = load().dflash_lmhead_verify(
        _dev(h, "h"), _dev(w, "w"), B, gamma, V, K, _dev(draft_tokens, "draft_tokens", torch.int32),
        _dev(temperature, "temperature", torch.float32), int(top_k), float(top_p),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _dev(logits, "logits"), _dev(out_tokens, "out_tokens", torch.int32),
        _dev(out_len, "out_accept_len", torch.int32), ws.ptr, ws.nbytes,
        None if status is None else _dev(status, "status", torch.int32), _stream_ptr(stream, dev))
    _check(rc)
    return out_tokens, out_len, logits


def verify_det(target, draft_tokens, temperature, top_k: int, top_p: float, seed: int,
               out_tokens=None, out_accept_len=None, status=None, workspace=None, stream=None):
    """dflash_verify_det (deterministic drafts, no draft logits) on torch CUDA
    tensors. Returns (out_tokens, out_accept_len)."""
    torch = _torch()
    B, g1, V = target.shape
    gamma = g1 - 1
    dt = _dtype_code(target)
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    if out_accept_len is None:
        out_accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    _shape(draft_tokens, (B, gamma), "draft_tokens")
    _shape(temperature, (B,), "temperature")
    _shape(out_tokens, (B, gamma + 1), "out_tokens")
    _shape(out_accept_len, (B,), "out_accept_len")
    _status_ok(status)
    _on(dev, draft_tokens=draft_tokens, temperature=temperature, out_tokens=out_tokens,
        out_accept_len=out_accept_len, status=status)
    ws = _workspace_for(workspace_bytes(B, gamma, V, dt, top_k, top_p), dev, workspace)
    rc = load().dflash_verify_det(
        _dev(target, "target"), _dev(draft_tokens, "draft_tokens", torch.int32), B, gamma, V, dt,
        _dev(temperature, "temperature", torch.float32), int(top_k), float(top_p),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _dev(out_tokens, "out_tokens", torch.int32),
        _dev(out_accept_len, "out_accept_len", torch.int32), ws.ptr, ws.nbytes,
        None if status is None else _dev(status, "status", torch.int32), _stream_ptr(stream, dev))
    _check(rc)
    return out_tokens, out_accept_len


def verify_greedy(target, draft_tokens, out_tokens=None, out_accept_len=None, status=None,
                  workspace=None, stream=None):
    torch = _torch()
    B, g1, V = target.shape
    gamma = g1 - 1
    dt = _dtype_code(target)
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    if out_accept_len is None:
        out_accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    _shape(draft_tokens, (B, gamma), "draft_tokens")
    _shape(out_tokens, (B, gamma + 1), "out_tokens")
    _shape(out_accept_len, (B,), "out_accept_len")
    _status_ok(status)
    _on(dev, draft_tokens=draft_tokens, out_tokens=out_tokens, out_accept_len=out_accept_len, status=status)
    ws = _workspace_for(workspace_bytes(B, gamma, V, dt, 1, 1.0), dev, workspace)
    rc = load().dflash_verify_greedy(
        _dev(target, "target"), _dev(draft_tokens, "draft_tokens", torch.int32), B, gamma, V, dt,
        _dev(out_tokens, "out_tokens", torch.int32), _dev(out_accept_len, "out_accept_len", torch.int32),
        ws.ptr, ws.nbytes, None if status is None else _dev(status, "status", torch.int32),
        _stream_ptr(stream, dev))
    _check(rc)
    return out_tokens, out_accept_len


# ---- vocabulary-sharded verification -------------------------------------------------
def candidates_words(B: int, gamma: int, k: int) -> int:
    """32-bit words of one shard's candidate record (dflash_candidates_words)."""
    n = load().dflash_candidates_words(B, gamma, k)
    if n == 0:
        raise DFlashError(ERR_INVALID_ARG, f"invalid record shape B={B} gamma={gamma} k={k}")
    return n


def shard_candidates(target_shard, draft_shard, vocab_offset: int, k: int, record=None, status=None,
                     workspace=None, stream=None):
    """dflash_shard_candidates: this rank's record (int32 tensor of
    candidates_words(B, gamma, k) words) from its vocabulary shard of the
    target [B, gamma+1, V_shard] and draft [B, gamma, V_shard] logits."""
    torch = _torch()
    B, g1, Vs = target_shard.shape
    gamma = g1 - 1
    if tuple(draft_shard.shape) != (B, gamma, Vs) or draft_shard.dtype != target_shard.dtype:
        raise ValueError("draft_shard must be [B, gamma, V_shard] with the target's dtype")
    dt = _dtype_code(target_shard)
    dev = target_shard.device
    words = candidates_words(B, gamma, k)
    if record is None:
        record = torch.empty((words,), dtype=torch.int32, device=dev)
    if record.numel() < words:
        raise ValueError(f"record of {record.numel()} words < {words} needed")
    _status_ok(status)
    _on(dev, draft_shard=draft_shard, record=record, status=status)
    nbytes = load().dflash_shard_workspace_bytes(B, gamma, Vs, dt, k)
    if nbytes == 0:
        raise DFlashError(ERR_INVALID_ARG, f"k={k} must be in [1, 32] and below the shard's V={Vs}")
    ws = _workspace_for(nbytes, dev, workspace)
    rc = load().dflash_shard_candidates(
        _dev(target_shard, "target_shard"), _dev(draft_shard, "draft_shard"), B, gamma, Vs, dt, int(vocab_offset),
        int(k), _dev(record, "record", torch.int32), ws.ptr, ws.nbytes,
        None if status is None else _dev(status, "status", torch.int32), _stream_ptr(stream, dev))
    _check(rc)
    return record


def gather_records(record, group=None):
    """The step's one exchange: every rank's record, gathered into a
    [world, words] tensor in rank order (torch.distributed all-gather into
    the rows of one buffer; any backend)."""
    torch = _torch()
    import torch.distributed as dist

    world = dist.get_world_size(group)
    out = torch.empty((world, record.numel()), dtype=record.dtype, device=record.device)
    dist.all_gather(list(out.unbind(0)), record.contiguous(), group=group)
    return out


def verify_candidates(records, k: int, draft_tokens, temperature, V: int, top_k: int, top_p: float, seed: int,
                      out_tokens=None, out_accept_len=None, status=None, stream=None):
    """dflash_verify_candidates on gathered records [n_shards, words]."""
    torch = _torch()
    n_shards = records.shape[0]
    B, gamma = draft_tokens.shape
    dev = records.device
    if not records.is_contiguous() or records.shape[1] != candidates_words(B, gamma, k):
        raise ValueError("records must be a contiguous [n_shards, candidates_words(B, gamma, k)] tensor")
    if out_tokens is None:
        out_tokens = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    if out_accept_len is None:
        out_accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    _shape(temperature, (B,), "temperature")
    _shape(out_tokens, (B, gamma + 1), "out_tokens")
    _shape(out_accept_len, (B,), "out_accept_len")
    _status_ok(status)
    _on(dev, draft_tokens=draft_tokens, temperature=temperature, out_tokens=out_tokens,
        out_accept_len=out_accept_len, status=status)
    rc = load().dflash_verify_candidates(
        _dev(records, "records", torch.int32), n_shards, int(k),
        _dev(draft_tokens, "draft_tokens", torch.int32), B, gamma, int(V),
        _dev(temperature, "temperature", torch.float32), int(top_k), float(top_p),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _dev(out_tokens, "out_tokens", torch.int32),
        _dev(out_accept_len, "out_accept_len", torch.int32),
        None if status is None else _dev(status, "status", torch.int32), _stream_ptr(stream, dev))
    _check(rc)
    return out_tokens, out_accept_len


def verify_vocab_sharded(target_shard, draft_shard, vocab_offset: int, V: int, draft_tokens, temperature,
                         top_k: int, top_p: float, seed: int, group=None, status=None, workspace=None,
                         stream=None):
    """One verification step with the vocabulary split across the ranks of
    `group`: this rank's record, the all-gather, then the verification from
    every shard's candidates (identical on every rank)."""
    record = shard_candidates(target_shard, draft_shard, vocab_offset, top_k, status=status,
                              workspace=workspace, stream=stream)
    records = gather_records(record, group)
    return verify_candidates(records, top_k, draft_tokens, temperature, V, top_k, top_p, seed,
                             status=status, stream=stream)


def rows_workspace_bytes(R, V, dtype_code, top_k, top_p) -> int:
    n = load().dflash_rows_workspace_bytes(R, V, dtype_code, top_k, top_p)
    if n == 0:
        raise DFlashError(ERR_INVALID_ARG, "unsupported or invalid shape / filter for a workspace")
    return n


def filter_rows(logits, temperature, top_k: int, top_p: float, status=None, workspace=None,
                stream=None):
    """dflash_filter: per-row kept tokens, probabilities and counts."""
    torch = _torch()
    R, V = logits.shape
    dt = _dtype_code(logits)
    dev = logits.device
    _shape(temperature, (R,), "temperature")
    _status_ok(status)
    _on(dev, temperature=temperature, status=status)
    idx = torch.empty((R, top_k), dtype=torch.int32, device=dev)
    prob = torch.empty((R, top_k), dtype=torch.float32, device=dev)
    cnt = torch.empty((R,), dtype=torch.int32, device=dev)
    ws = _workspace_for(rows_workspace_bytes(R, V, dt, top_k, top_p), dev, workspace)
    rc = load().dflash_filter(
        _dev(logits, "logits"), R, V, dt, _dev(temperature, "temperature", torch.float32), int(top_k),
        float(top_p), idx.data_ptr(), prob.data_ptr(), cnt.data_ptr(), ws.ptr, ws.nbytes,
        None if status is None else _dev(status, "status", torch.int32), _stream_ptr(stream, dev))
    _check(rc)
    return idx, prob, cnt


def sample_rows(logits, temperature, top_k: int, top_p: float, seed: int, status=None,
                workspace=None, stream=None):
    """dflash_sample: one token per row from its filtered distribution."""
    torch = _torch()
    R, V = logits.shape
    dt = _dtype_code(logits)
    dev = logits.device
    _shape(temperature, (R,), "temperature")
    _status_ok(status)
    _on(dev, temperature=temperature, status=status)
    out = torch.empty((R,), dtype=torch.int32, device=dev)
    ws = _workspace_for(rows_workspace_bytes(R, V, dt, top_k, top_p), dev, workspace)
    rc = load().dflash_sample(
        _dev(logits, "logits"), R, V, dt, _dev(temperature, "temperature", torch.float32), int(top_k),
        float(top_p), int(seed) & 0xFFFFFFFFFFFFFFFF, out.data_ptr(), ws.ptr, ws.nbytes,
        None if status is None else _dev(status, "status", torch.int32), _stream_ptr(stream, dev))
    _check(rc)
    return out


def uniforms(seed: int, B: int, npos: int, stream_id: int = 0, device="cuda", stream=None):
    torch = _torch()
    ua = torch.empty((B, npos), dtype=torch.float32, device=device)
    ud = torch.empty((B, npos), dtype=torch.float32, device=device)
    _check(load().dflash_uniforms(int(seed) & 0xFFFFFFFFFFFFFFFF, B, npos, stream_id, ua.data_ptr(),
                                  ud.data_ptr(), _stream_ptr(stream, ua.device)))
    return ua, ud


def host_staging_bytes(B, gamma, V, dtype_code) -> int:
    return load().dflash_host_staging_bytes(B, gamma, V, dtype_code)


def verify_host(target, draft, draft_tokens, temperature, top_k, top_p, seed, out_tokens,
                out_accept_len, out_status, staging, workspace, stream=None):
    """dflash_verify_host: host (ideally pinned) torch CPU tensors in and out;
    ``staging`` and ``workspace`` are device buffers. Waits for the stream."""
    B, g1, V = target.shape
    gamma = g1 - 1
    dt = _dtype_code(target)
    torch = _torch()
    for t, n, shape, dtype in ((target, "target", (B, gamma + 1, V), target.dtype),
                               (draft, "draft", (B, gamma, V), target.dtype),
                               (draft_tokens, "draft_tokens", (B, gamma), torch.int32),
                               (temperature, "temperature", (B,), torch.float32),
                               (out_tokens, "out_tokens", (B, gamma + 1), torch.int32),
                               (out_accept_len, "out_accept_len", (B,), torch.int32),
                               (out_status, "out_status", (1,), torch.int32)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host tensor")
        _shape(t, shape, n)
        if t.dtype != dtype:
            raise TypeError(f"{n} must be {dtype}, got {t.dtype}")
    if not staging.is_cuda or staging.dtype != torch.uint8:
        raise ValueError("staging must be a uint8 CUDA tensor")
    rc = load().dflash_verify_host(
        target.data_ptr(), draft.data_ptr(), draft_tokens.data_ptr(), B, gamma, V, dt,
        temperature.data_ptr(), int(top_k), float(top_p), int(seed) & 0xFFFFFFFFFFFFFFFF,
        out_tokens.data_ptr(), out_accept_len.data_ptr(), out_status.data_ptr(),
        staging.data_ptr(), staging.numel(), workspace.ptr, workspace.nbytes,
        _stream_ptr(stream, staging.device))
    _check(rc)
    return out_tokens, out_accept_len


__all__ = [
    "build", "load", "verify", "verify_det", "verify_greedy", "shard_candidates", "gather_records",
    "verify_candidates", "verify_vocab_sharded", "candidates_words", "filter_rows", "sample_rows", "uniforms",
    "verify_host", "Workspace", "workspace_bytes", "rows_workspace_bytes", "host_staging_bytes",
    "DFlashError", "LIB_PATH", "EXPORTS",
]
