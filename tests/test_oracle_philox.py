"""Pins for the oracle's Philox4x32-10 and its uniforms.

The oracle writes Philox4x32-10 from Salmon et al., "Parallel Random Numbers:
As Easy as 1, 2, 3" (SC'11). It is pinned to an implementation that is not its
own: the curand library's block function, compiled for the host and called.
"""
import numpy as np
import pytest
from scipy import stats

import oracle


def test_philox_matches_curand(curand_pin):
    rng = np.random.default_rng(20261202)
    n = 4096
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2**32, size=(n, 2), dtype=np.uint64).astype(np.uint32)
    # structured counters too: the (position, request, stream, 0) layout the step uses
    ctr[:64] = np.stack([np.arange(64), np.arange(64) % 7, np.zeros(64), np.zeros(64)], 1)
    key[:64] = 0
    want = np.zeros((n, 4), np.uint32)
    curand_pin.pin_curand_philox4x32_10(ctr.ctypes.data, key.ctypes.data, want.ctypes.data, n)
    got = np.stack([oracle.philox4x32_10(ctr[i], key[i]) for i in range(n)])
    assert np.array_equal(got, want)


def test_uniform_layout_and_range():
    # u = (w >> 8) * 2^-24 of words 0 / 1 of philox((pos, req, stream, 0), seed words)
    for seed in (0, 1, 2**32 + 5, 0xDEADBEEFCAFEF00D):
        for req, pos, stream in ((0, 0, 0), (3, 7, 0), (31, 15, 1), (0, 4, 1)):
            w = oracle.philox4x32_10([pos, req, stream, 0], [seed & 0xFFFFFFFF, seed >> 32])
            ua, ud = oracle.uniforms(seed, req, pos, stream)
            assert ua == (int(w[0]) >> 8) / 2**24
            assert ud == (int(w[1]) >> 8) / 2**24
            assert 0.0 <= ua < 1.0 and 0.0 <= ud < 1.0


def test_uniforms_are_uniform_and_independent():
    us = np.array([oracle.uniforms(7, r, p) for r in range(200) for p in range(100)])
    for col in range(2):
        assert stats.kstest(us[:, col], "uniform").pvalue > 1e-3
    # accept and draw uniforms of one (request, position) are uncorrelated
    assert abs(np.corrcoef(us[:, 0], us[:, 1])[0, 1]) < 0.03
    # the stream word separates verification draws from sampling draws
    a = [oracle.uniforms(7, 0, p, 0)[0] for p in range(50)]
    b = [oracle.uniforms(7, 0, p, 1)[0] for p in range(50)]
    assert a != b


@pytest.mark.parametrize("seed", [0, 123456789])
def test_uniforms_depend_on_every_key_word(seed):
    base = oracle.uniforms(seed, 1, 2, 0)
    assert oracle.uniforms(seed ^ 1, 1, 2, 0) != base
    assert oracle.uniforms(seed ^ (1 << 40), 1, 2, 0) != base
    assert oracle.uniforms(seed, 2, 2, 0) != base
    assert oracle.uniforms(seed, 1, 3, 0) != base
