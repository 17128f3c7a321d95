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


CAPTURE_BEFORE_INIT = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import sparse_attention_deterministic_gb300 as pkg
so = pkg.lib()                        # loaded; no entry point has run on the device yet
dev = torch.device("cuda", 0)
scores = torch.rand(3 * 5000, device=dev)
starts = torch.tensor([0, 5000, 10000], dtype=torch.int32, device=dev)
lengths = torch.full((3,), 5000, dtype=torch.int32, device=dev)
out = torch.full((3, 64), 7, dtype=torch.int32, device=dev)
marker = torch.zeros(1, device=dev)
torch.cuda.synchronize()
side = torch.cuda.Stream()
graph = torch.cuda.CUDAGraph()
with torch.cuda.graph(graph, stream=side):
    marker.add_(1.0)                  # one captured node of torch's own
    rc = so.topk_ragged(scores.data_ptr(), scores.numel(), starts.data_ptr(), lengths.data_ptr(), 3, 64, 0,
                        out.data_ptr(), None, side.cuda_stream)
    rc_stats = so.topk_ragged_stats(scores.data_ptr(), scores.numel(), starts.data_ptr(), lengths.data_ptr(),
                                    3, 64, out.data_ptr(), side.cuda_stream)
graph.replay()                        # the captured graph holds no launch of the library
torch.cuda.synchronize()
untouched = bool((out == 7).all().item()) and float(marker.item()) == 1.0
pkg.init(dev)                         # outside capture: the device becomes ready
rc_eager = so.topk_ragged(scores.data_ptr(), scores.numel(), starts.data_ptr(), lengths.data_ptr(), 3, 64, 0,
                          out.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
torch.cuda.synchronize()
graph2 = torch.cuda.CUDAGraph()
with torch.cuda.graph(graph2, stream=side):
    rc_cap = so.topk_ragged(scores.data_ptr(), scores.numel(), starts.data_ptr(), lengths.data_ptr(), 3, 64, 0,
                            out.data_ptr(), None, side.cuda_stream)
print(rc, rc_stats, int(untouched), rc_eager, rc_cap)
"""


def test_capture_without_init_is_refused():
    """A call under stream capture on a device that no entry point has
    prepared yet returns TOPK_ERR_NOT_INITIALIZED and launches nothing (the
    replayed graph leaves the output as it was); after topk_ragged_init the
    same call runs eagerly and captures (the sglang page's hardening commit:
    graph-safe after one eager warm-up).  Run in a fresh process, since a
    device stays prepared for the life of the process."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", CAPTURE_BEFORE_INIT, root], capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-3000:]
    rc, rc_stats, untouched, rc_eager, rc_cap = (int(x) for x in out.stdout.split()[-5:])
    assert (rc, rc_stats) == (2, 2)
    assert untouched == 1
    assert (rc_eager, rc_cap) == (0, 0)
    assert pkg.strerror(2).startswith("device not initialized")
