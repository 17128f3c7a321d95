"""CUDA-graph capture: after init, calls capture and replay bit-identically to
eager calls, and the call allocates no device memory (sglang PR #31115: the
backend must be CUDA-graph-safe, replay verified bitwise-equal to eager)."""
import ctypes

import pytest
import torch

import sparse_attention_deterministic_gb300 as pkg
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkg.build()
    pkg.init()


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill"])
def test_capture_replay_equals_eager(name):
    w = W.make(name, device="cuda")
    B, k = w.B, w.k
    eager_idx, eager_val = pkg.topk_ragged(w.scores, w.row_starts, w.lengths, k, w.offset_mode,
                                           with_values=True)
    torch.cuda.synchronize()
    out_idx = torch.full((B, k), 7, dtype=torch.int32, device="cuda")
    out_val = torch.zeros((B, k), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    free0 = torch.cuda.mem_get_info()[0]
    with torch.cuda.graph(graph, stream=stream):
        pkg.topk_ragged(w.scores, w.row_starts, w.lengths, k, w.offset_mode, out_idx=out_idx,
                        out_val=out_val, stream=torch.cuda.current_stream())
    for _ in range(3):
        out_idx.fill_(7)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_idx, eager_idx)
        assert torch.equal(out_val.view(torch.int32), eager_val.view(torch.int32))
    # The captured call itself allocated nothing (the graph's own bookkeeping
    # is small; a per-call workspace for these sizes would be megabytes).
    assert free0 - torch.cuda.mem_get_info()[0] < (1 << 20)


def test_capture_without_init_is_refused():
    # A device that was initialised stays initialised; the refusal path is
    # covered by the C-level status code.
    assert pkg.strerror(2).startswith("device not initialized")
