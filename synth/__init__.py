"""Seeded synthetic inputs for the draft-verification step.

This module is shared by the tests, the smoke check and the benchmark. It
holds none of the method's arithmetic (no temperature, filtering, softmax,
acceptance or sampling): it only draws logits with the structure the
workloads describe, rounds them to the storage type, and lays them out.
Draft tokens, which must be samples from the filtered draft distribution, are
drawn afterwards by each side's own sampler (the oracle's in the tests, the
library's in the benchmark).

Recipe (per request b, position i):
  target  x[b, i, :] ~ N(0, sigma=2) i.i.d., plus one spike of height
          U(4, 12) at a uniformly drawn token;            i in [0, gamma]
  draft   y[b, i, :] = x[b, i, :] + N(0, sigma_d[b])      i in [0, gamma)
  sigma_d is a constant (0.5) or drawn per request from U(lo, hi).
Values are drawn in fp32 and rounded to nearest-even bf16 when the storage
type is bf16; bf16 arrays are returned as uint16 bit patterns.

Draw order from ``numpy.random.Generator(PCG64(seed))``: target normals,
spike tokens, spike heights, per-request sigma_d (if a range), draft normals.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BF16 = "bf16"
F32 = "f32"


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even), as uint16 bits."""
    bits = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (bits + 0x7FFF + ((bits >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_float(a: np.ndarray) -> np.ndarray:
    """Logits as fp32 values whatever the storage type."""
    return bf16_bits_to_f32(a) if a.dtype == np.uint16 else np.asarray(a, np.float32)


@dataclass
class VerifyInputs:
    target: np.ndarray        # [B, gamma+1, V] uint16 (bf16 bits) or float32
    draft: np.ndarray         # [B, gamma, V]
    temperature: np.ndarray   # [B] float32, 0 = greedy
    sigma_d: np.ndarray       # [B] float32
    top_k: int
    top_p: float
    seed: int                 # Philox seed of the step
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        B, g1, V = self.target.shape
        return B, g1 - 1, V


def make_logits(B: int, gamma: int, V: int, dtype: str = BF16, data_seed: int = 0,
                sigma: float = 2.0, spike=(4.0, 12.0), sigma_d=0.5):
    """Target and draft logits following the recipe above.

    ``sigma_d`` is a float (same for every request) or a (lo, hi) tuple
    (drawn per request)."""
    rng = np.random.Generator(np.random.PCG64(data_seed))
    x = rng.standard_normal((B, gamma + 1, V), dtype=np.float32)
    x *= np.float32(sigma)
    tok = rng.integers(0, V, size=(B, gamma + 1))
    height = rng.uniform(spike[0], spike[1], size=(B, gamma + 1)).astype(np.float32)
    bi = np.arange(B)[:, None]
    ii = np.arange(gamma + 1)[None, :]
    x[bi, ii, tok] += height
    if isinstance(sigma_d, tuple):
        sd = rng.uniform(sigma_d[0], sigma_d[1], size=B).astype(np.float32)
    else:
        sd = np.full(B, sigma_d, np.float32)
    y = rng.standard_normal((B, gamma, V), dtype=np.float32)
    y *= sd[:, None, None]
    y += x[:, :gamma, :]
    if dtype == BF16:
        return f32_to_bf16_bits(x), f32_to_bf16_bits(y), sd
    if dtype == F32:
        return x, y, sd
    raise ValueError(dtype)


def cycle_temperatures(B: int, cycle=(0.0, 0.6, 1.0)) -> np.ndarray:
    return np.array([cycle[b % len(cycle)] for b in range(B)], np.float32)


# The workloads of the step (shapes, storage types, filters).
WORKLOADS = {
    # tiny CPU-checkable case: greedy and sampling on one request
    "tiny_v1024": dict(B=1, gamma=7, V=1024, dtype=F32, sigma_d=0.5, temperature=1.0,
                       top_k=20, top_p=0.95),
    # one request, full vocabulary, bf16
    "b1_v248320": dict(B=1, gamma=7, V=248320, dtype=BF16, sigma_d=0.5, temperature=1.0,
                       top_k=20, top_p=0.95),
    # concurrency 8, per-request draft noise spreading the accept lengths
    "b8_v248320": dict(B=8, gamma=7, V=248320, dtype=BF16, sigma_d=(0.3, 1.5),
                       temperature=1.0, top_k=20, top_p=0.95),
    # concurrency 32, temperatures cycling greedy / 0.6 / 1.0
    "b32_mixed_v248320": dict(B=32, gamma=7, V=248320, dtype=BF16, sigma_d=(0.3, 1.5),
                              temperature=(0.0, 0.6, 1.0), top_k=20, top_p=0.95),
    # the same concurrency-32 mix at blocks of 4 and 16 (3 and 15 verified drafts)
    "b32_mixed_g3_v248320": dict(B=32, gamma=3, V=248320, dtype=BF16, sigma_d=(0.3, 1.5),
                                 temperature=(0.0, 0.6, 1.0), top_k=20, top_p=0.95),
    "b32_mixed_g15_v248320": dict(B=32, gamma=15, V=248320, dtype=BF16, sigma_d=(0.3, 1.5),
                                  temperature=(0.0, 0.6, 1.0), top_k=20, top_p=0.95),
    # the concurrency-32 mix with top-k off: top-p 0.95 over the full vocabulary
    "b32_mixed_topp_v248320": dict(B=32, gamma=7, V=248320, dtype=BF16, sigma_d=(0.3, 1.5),
                                   temperature=(0.0, 0.6, 1.0), top_k=0, top_p=0.95),
    # block 16, fp32, top-k off and top-p 1: full-vocabulary softmax and residual
    "b128_g15_fullvocab_f32": dict(B=128, gamma=15, V=248320, dtype=F32, sigma_d=0.5,
                                   temperature=1.0, top_k=0, top_p=1.0),
    # the same with top-p 0.95 over the full vocabulary
    "b128_g15_topp_f32": dict(B=128, gamma=15, V=248320, dtype=F32, sigma_d=0.5,
                              temperature=1.0, top_k=0, top_p=0.95),
}


def make_workload(name: str, data_seed: int = 0, seed: int = 0, B: int | None = None,
                  V: int | None = None, gamma: int | None = None) -> VerifyInputs:
    """Logits, temperatures and filter settings of a named workload.

    B, V and gamma may be overridden (smaller cases of the same recipe)."""
    w = dict(WORKLOADS[name])
    B = B or w["B"]
    V = V or w["V"]
    gamma = gamma or w["gamma"]
    X, Y, sd = make_logits(B, gamma, V, w["dtype"], data_seed=data_seed, sigma_d=w["sigma_d"])
    t = w["temperature"]
    T = cycle_temperatures(B, t) if isinstance(t, tuple) else np.full(B, t, np.float32)
    return VerifyInputs(X, Y, T, sd, w["top_k"], w["top_p"], seed,
                        meta=dict(name=name, data_seed=data_seed, dtype=w["dtype"]))


def draft_sampling_temperatures(T: np.ndarray, gamma: int) -> np.ndarray:
    """Per-draft-row temperatures [B*gamma]: each request's temperature repeated."""
    return np.repeat(np.asarray(T, np.float32), gamma)


def to_torch(a: np.ndarray, device="cuda"):
    """A generated array as a torch tensor on ``device`` (uint16 bf16 bits
    become torch.bfloat16 with the same bits)."""
    import torch

    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)
