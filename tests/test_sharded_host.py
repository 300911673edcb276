"""Vocabulary-sharded verification: what can be checked without a GPU.

* The property the scheme rests on: the union of the shards' top k of a row
  holds the row's global top k, and ordering the union by (logit desc, token
  asc) gives the global top k in the global order. Checked by brute force on
  random rows with many ties and random uneven splits.
* The record size the library reports, and the host-side refusals of the two
  entry points (they return before any launch).
* The exchange over two gloo ranks: gather_records returns every rank's record
  in rank order, and verify_vocab_sharded hands the gathered records (and
  k = top_k) to the verification.
"""
import ctypes
import os
import socket

import numpy as np
import pytest

import speculative_decoding_verification_83_gb300 as dv

torch = pytest.importorskip("torch")
import torch.distributed as tdist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _topk(x, tokens, k):
    """(logit desc, token asc) order, first k."""
    order = np.lexsort((tokens, -x))
    return tokens[order[:k]], x[order[:k]]


@pytest.mark.parametrize("seed", range(6))
def test_union_of_shard_top_k_holds_the_global_top_k(seed):
    rng = np.random.default_rng(seed)
    for _ in range(50):
        V = int(rng.integers(40, 400))
        k = int(rng.integers(1, 33))
        # few distinct values: many ties, which the token order must break
        x = rng.integers(-4, 5, V).astype(np.float32) * 0.5
        tokens = np.arange(V)
        n_sh = int(rng.integers(1, 9))
        cuts = np.sort(rng.choice(np.arange(1, V), size=n_sh - 1, replace=False)) if n_sh > 1 else []
        bounds = np.concatenate([[0], cuts, [V]]).astype(int)
        ut, ux = [], []
        for s in range(n_sh):
            lo, hi = bounds[s], bounds[s + 1]
            t, v = _topk(x[lo:hi], tokens[lo:hi], k)
            ut.append(t)
            ux.append(v)
        ut, ux = np.concatenate(ut), np.concatenate(ux)
        gt, gx = _topk(x, tokens, k)
        mt, mx = _topk(ux, ut, k)
        assert np.array_equal(mt, gt) and np.array_equal(mx, gx)


@pytest.fixture(scope="module")
def lib():
    dv.build()
    return dv.load()


def test_record_words(lib):
    for B, g, k in ((1, 1, 1), (32, 7, 20), (2048, 32, 32), (3, 15, 7)):
        rows = B * (g + 1) + B * g
        assert lib.dflash_candidates_words(B, g, k) == rows * (2 * k + 1)
    assert lib.dflash_candidates_words(0, 7, 20) == 0
    assert lib.dflash_candidates_words(32, 33, 20) == 0
    assert lib.dflash_candidates_words(32, 7, 33) == 0
    assert lib.dflash_shard_workspace_bytes(32, 7, 62080, dv.DFLASH_BF16, 20) > 0
    assert lib.dflash_shard_workspace_bytes(32, 7, 20, dv.DFLASH_BF16, 20) == 0   # k >= V_shard


def test_host_refusals(lib):
    p = ctypes.c_void_p(256)   # never dereferenced: every case is refused on the host
    # verify from candidates: B, n_shards, k, top_k, top_p
    vc = lib.dflash_verify_candidates
    args = dict(n=4, k=20, B=8, g=7, V=1000, top_k=20, top_p=0.95)

    def call(**kw):
        a = dict(args, **kw)
        return vc(p, a["n"], a["k"], p, a["B"], a["g"], a["V"], p, a["top_k"], a["top_p"], 1, p, p, None, None)

    assert call(top_k=21) == dv.ERR_UNSUPPORTED                  # top_k above the shards' k
    assert call(top_k=0, top_p=1.0) == dv.ERR_UNSUPPORTED        # full vocabulary
    assert call(top_p=0.0) == dv.ERR_INVALID_ARG
    assert call(n=13) == dv.ERR_INVALID_ARG                      # 13 x 20 > 256 candidates per row
    assert b"n_shards=13" in lib.dflash_last_error()
    assert call(n=0) == dv.ERR_INVALID_ARG
    assert call(k=33) == dv.ERR_INVALID_ARG
    assert call(B=0) == dv.ERR_INVALID_ARG
    assert vc(None, 4, 20, p, 8, 7, 1000, p, 20, 0.95, 1, p, p, None, None) == dv.ERR_INVALID_ARG
    # shard candidates: k against the shard, the offset, the record's alignment
    sc = lib.dflash_shard_candidates
    big = ctypes.c_size_t(1 << 40)
    assert sc(p, p, 8, 7, 20, dv.DFLASH_BF16, 0, 20, p, p, big, None, None) == dv.ERR_INVALID_ARG
    assert sc(p, p, 8, 7, 5000, dv.DFLASH_BF16, -1, 20, p, p, big, None, None) == dv.ERR_INVALID_ARG
    assert sc(p, p, 8, 7, 5000, dv.DFLASH_BF16, 2**31 - 4000, 20, p, p, big, None, None) == dv.ERR_INVALID_ARG
    assert sc(p, p, 8, 7, 5000, dv.DFLASH_BF16, 0, 20, ctypes.c_void_p(258), p, big, None, None) == \
        dv.ERR_INVALID_ARG
    assert sc(p, p, 8, 7, 5000, dv.DFLASH_BF16, 0, 20, p, p, 16, None, None) == dv.ERR_INVALID_ARG  # workspace


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import speculative_decoding_verification_83_gb300 as m

        # the exchange itself
        rec = torch.arange(11, dtype=torch.int32) + 100 * rank
        got = m.gather_records(rec)
        results[("gather", rank)] = got.tolist()

        # the step's orchestration, with the two kernels stood in for
        seen = {}

        def fake_shard(target_shard, draft_shard, vocab_offset, k, **kw):
            seen["shard"] = (tuple(target_shard.shape), vocab_offset, k)
            return torch.full((7,), vocab_offset, dtype=torch.int32)

        def fake_verify(records, k, draft_tokens, temperature, V, top_k, top_p, seed, **kw):
            seen["verify"] = (records.tolist(), k, V, top_k, top_p, seed)
            return "tokens", "lens"

        m.shard_candidates, m.verify_candidates = fake_shard, fake_verify
        V_shard = 50
        X = torch.zeros((2, 4, V_shard))
        Y = torch.zeros((2, 3, V_shard))
        out = m.verify_vocab_sharded(X, Y, rank * V_shard, 2 * V_shard, torch.zeros((2, 3), dtype=torch.int32),
                                     torch.ones(2), 20, 0.95, 5)
        results[("step", rank)] = (out, seen["shard"], seen["verify"])
    finally:
        tdist.destroy_process_group()


def test_two_rank_exchange_and_orchestration():
    world = 2
    with mp.Manager() as manager:
        results = manager.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        res = dict(results)
    want = [list(range(100 * r, 100 * r + 11)) for r in range(world)]
    for rank in range(world):
        assert res[("gather", rank)] == want
        out, shard, verify = res[("step", rank)]
        assert out == ("tokens", "lens")
        assert shard == ((2, 4, 50), 50 * rank, 20)
        records, k, V, top_k, top_p, seed = verify
        assert records == [[0] * 7, [50] * 7]   # every rank's record, in rank order
        assert (k, V, top_k, seed) == (20, 100, 20, 5) and top_p == pytest.approx(0.95)
