"""The Python binding refuses buffers whose shape, dtype or device does not
match the call's sizes, before any pointer reaches the library: a short
temperature or output tensor would otherwise let a kernel read or write past
its end. These checks run on the host (CPU tensors, no GPU needed)."""
import pytest

import speculative_decoding_verification_83_gb300 as dv

torch = pytest.importorskip("torch")

B, G, V = 4, 3, 64


def _logits(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def _i32(*shape):
    return torch.zeros(shape, dtype=torch.int32)


def test_verify_shapes():
    X, Y = _logits(B, G + 1, V), _logits(B, G, V)
    with pytest.raises(ValueError, match="temperature must have shape"):
        dv.verify(X, Y, _i32(B, G), torch.ones(B - 1), 20, 0.95, 1)
    with pytest.raises(ValueError, match="draft_tokens must have shape"):
        dv.verify(X, Y, _i32(B, G + 1), torch.ones(B), 20, 0.95, 1)
    with pytest.raises(ValueError, match="out_tokens must have shape"):
        dv.verify(X, Y, _i32(B, G), torch.ones(B), 20, 0.95, 1, out_tokens=_i32(B, G))
    with pytest.raises(ValueError, match="out_accept_len must have shape"):
        dv.verify(X, Y, _i32(B, G), torch.ones(B), 20, 0.95, 1, out_accept_len=_i32(B - 1))
    with pytest.raises(ValueError, match="status"):
        dv.verify(X, Y, _i32(B, G), torch.ones(B), 20, 0.95, 1, status=_i32(0))
    with pytest.raises(ValueError, match="draft must be"):
        dv.verify(X, _logits(B, G, V + 1), _i32(B, G), torch.ones(B), 20, 0.95, 1)


def test_verify_det_and_greedy_shapes():
    X = _logits(B, G + 1, V)
    with pytest.raises(ValueError, match="draft_tokens must have shape"):
        dv.verify_det(X, _i32(B + 1, G), torch.ones(B), 20, 0.95, 1)
    with pytest.raises(ValueError, match="temperature must have shape"):
        dv.verify_det(X, _i32(B, G), torch.ones(2 * B), 20, 0.95, 1)
    with pytest.raises(ValueError, match="out_tokens must have shape"):
        dv.verify_greedy(X, _i32(B, G), out_tokens=_i32(B, G + 2))


def test_rows_and_candidates_shapes():
    with pytest.raises(ValueError, match="temperature must have shape"):
        dv.filter_rows(_logits(5, V), torch.ones(4), 20, 0.95)
    with pytest.raises(ValueError, match="temperature must have shape"):
        dv.sample_rows(_logits(5, V), torch.ones(6), 20, 0.95, 1)
    words = dv.candidates_words(B, G, 20)
    recs = _i32(2, words)
    with pytest.raises(ValueError, match="temperature must have shape"):
        dv.verify_candidates(recs, 20, _i32(B, G), torch.ones(B + 1), V, 20, 0.95, 1)
    with pytest.raises(ValueError, match="contiguous"):
        dv.verify_candidates(_i32(2, words + 1), 20, _i32(B, G), torch.ones(B), V, 20, 0.95, 1)


def test_host_entry_types_and_shapes():
    X, Y = _logits(B, G + 1, V), _logits(B, G, V)
    outs = (_i32(B, G + 1), _i32(B), _i32(1))
    with pytest.raises(TypeError, match="draft_tokens must be"):
        dv.verify_host(X, Y, torch.zeros((B, G), dtype=torch.int64), torch.ones(B), 20, 0.95, 1, *outs, None, None)
    with pytest.raises(ValueError, match="temperature must have shape"):
        dv.verify_host(X, Y, _i32(B, G), torch.ones(B - 1), 20, 0.95, 1, *outs, None, None)
    with pytest.raises(ValueError, match="out_status must have shape"):
        dv.verify_host(X, Y, _i32(B, G), torch.ones(B), 20, 0.95, 1, outs[0], outs[1], _i32(2), None, None)
