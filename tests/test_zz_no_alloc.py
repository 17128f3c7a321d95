"""The indexer chain for callers that cannot allocate device memory.

Some callers of this library have no way to call cudaMalloc: a plugin inside
a serving framework that has reserved the device memory for its own pool,
or code on a latency-critical or captured path where an allocation would
synchronize the device or is refused.  topk_ragged_indexer_static serves
them: the chain's intermediate scores go to a fixed array that the library
holds, and the caller passes only inputs and outputs.

These tests call it through the C ABI and compare it with
topk_ragged_indexer, whose scores go to a caller buffer, bit for bit (the
tolerance of every selection test here: the same scores give the same
selection).  Two calls run in a row on different shapes, so the second
reads an array that still holds the first call's scores.  A size beyond the
array is refused before anything is launched.

The file sits last in the collection order, so a run that stops at the
first failure has run every other test before this one; it also passes
alone in a fresh process (the module fixture builds and prepares the
library).
"""
import ctypes

import pytest
import torch

import sparse_attention_deterministic_gb300 as pkg
import workloads as W

pytestmark = pytest.mark.gpu

STATIC_SCORES = 1 << 23          # TOPK_RAGGED_STATIC_SCORES
SCRATCH_TOO_SMALL = 5            # TOPK_ERR_SCRATCH_TOO_SMALL


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkg.build()
    pkg.init()


def _static_call(iw, n_scores, out_idx, out_val, flags=0):
    """One call of the C entry point, on the current stream."""
    so = pkg.lib()
    return so.topk_ragged_indexer_static(
        iw.q.data_ptr(), iw.w.data_ptr(), iw.bias.data_ptr(), iw.keys.data_ptr(), iw.keys.shape[0],
        iw.key_starts.data_ptr(), iw.lengths.data_ptr(), iw.score_starts.data_ptr(), iw.B,
        ctypes.c_float(iw.scale), n_scores, iw.k, flags, out_idx.data_ptr(),
        out_val.data_ptr() if out_val is not None else None, torch.cuda.current_stream().cuda_stream)


def _shapes():
    # The first call fills about 3 M entries of the array; the second, on
    # fewer and shorter rows, reads windows that still hold the first
    # call's scores around them.
    return [W.decode_indexer(device="cuda", B=16, lmin=4096, lmax=400000, k=2048),
            W.decode_indexer(device="cuda", B=5, lmin=100, lmax=9000, k=512)]


def test_static_scores_match_caller_scratch():
    for flags in (0, pkg.TOPK_EXCLUDE_NEG_INF):
        for iw in _shapes():
            assert iw.n_scores <= STATIC_SCORES
            ref_idx, ref_val, _ = pkg.topk_ragged_indexer(
                iw.q, iw.w, iw.keys, iw.key_starts, iw.lengths, iw.score_starts, k=iw.k, flags=flags,
                bias=iw.bias, scale=iw.scale, n_scores=iw.n_scores, with_values=True)
            out_idx = torch.full((iw.B, iw.k), 7, dtype=torch.int32, device="cuda")
            out_val = torch.zeros((iw.B, iw.k), dtype=torch.float32, device="cuda")
            assert _static_call(iw, iw.n_scores, out_idx, out_val, flags) == 0
            torch.cuda.synchronize()
            assert torch.equal(out_idx, ref_idx)
            assert torch.equal(out_val.view(torch.int32), ref_val.view(torch.int32))
    assert pkg.device_status() == 0


def test_binding_and_refusal_beyond_the_array():
    iw = _shapes()[1]
    ref_idx, _, _ = pkg.topk_ragged_indexer(iw.q, iw.w, iw.keys, iw.key_starts, iw.lengths, iw.score_starts,
                                            k=iw.k, bias=iw.bias, scale=iw.scale, n_scores=iw.n_scores)
    got, _ = pkg.topk_ragged_indexer_static(iw.q, iw.w, iw.keys, iw.key_starts, iw.lengths,
                                            iw.score_starts, iw.n_scores, k=iw.k, bias=iw.bias,
                                            scale=iw.scale)
    torch.cuda.synchronize()
    assert torch.equal(got, ref_idx)
    # One score past the array: refused on the host, nothing launched.
    out_idx = torch.full((iw.B, iw.k), 7, dtype=torch.int32, device="cuda")
    assert _static_call(iw, STATIC_SCORES + 1, out_idx, None) == SCRATCH_TOO_SMALL
    torch.cuda.synchronize()
    assert bool((out_idx == 7).all())
    assert "fixed score array" in pkg.strerror(SCRATCH_TOO_SMALL)
