"""The tie / plateau statistics op (topk_ragged_stats) on the GPU, field for
field against the oracle's row_stats: the five named workloads at full size,
the tie-study families, lengths around k, unaligned and overlapping windows,
rejected rows, repeated calls and CUDA-graph replay."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_deterministic_gb300 as pkg
import workloads as W
from helpers import ragged

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkg.build()
    pkg.init()


def _gpu(w, k=None):
    d = w.to("cuda")
    out = pkg.topk_ragged_stats(d.scores, d.row_starts, d.lengths, w.k if k is None else k)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint32)


def assert_stats(w, k=None):
    k = w.k if k is None else k
    got = _gpu(w, k)
    s, st, ln = w.numpy()
    want, flags = oracle.row_stats(s, st, ln, k)
    bad = np.flatnonzero((got != want).any(axis=1))
    assert bad.size == 0, (f"{w.name} k={k}: {bad.size} rows differ; first row {bad[0]}: "
                           f"got {got[bad[0]].tolist()} want {want[bad[0]].tolist()}")
    expected = int(np.bitwise_or.reduce(flags)) if flags.size else 0
    assert pkg.device_status() == expected
    return got


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "adversarial", "long"])
def test_named_workload_full_size(name):
    w = W.make(name, device="cuda").to("cpu")
    got = assert_stats(w)
    if name == "adversarial":
        # the families that straddle: all 0.0, all -inf and the 3000-entry tie block
        assert (got[:, 5] & pkg.TOPK_STAT_STRADDLE).any()


@pytest.mark.parametrize("B,L", [(4, 32768), (640, 8192)])
@pytest.mark.parametrize("k", [1, 2048, 4096])
def test_families(B, L, k):
    for w in (W.plateau(B, L, 1024, k), W.tie_block(B, L, k, 512), W.relu_shifted(B, L, k),
              W.narrow(B, L, k)):
        assert_stats(w)


@pytest.mark.parametrize("alphabet", [None, [0, 0x80000000, 0x3F800000, 0x7FC00001, 0xFFC00001,
                                             0xFF800000, 0x7F800000, 0x00000001]])
def test_random_bit_patterns(alphabet):
    for k in (1, 7, 1024):
        assert_stats(W.random_bits(300, 5003, k, alphabet=alphabet))


@pytest.mark.parametrize("k", [1, 2, 100, 2047, 2048, 4096])
def test_lengths_around_k_and_unaligned(k):
    g = torch.Generator().manual_seed(k)
    choices = [0, 1, 2, 3, 4, 5, k - 1, k, k + 1, 2 * k + 3, 40000]
    rows = []
    for i in range(60):
        L = max(0, choices[i] if i < len(choices) else int(torch.randint(0, 3 * k + 10, (1,), generator=g)))
        r = torch.randn(L, generator=g)
        r[torch.rand(L, generator=g) < 0.4] = 0.0
        rows.append(r)
    for lead in (0, 1, 2, 3):
        assert_stats(ragged(f"around_k{k}", rows, k, gap=lead % 3, lead=lead))


def test_overlapping_windows_and_long_rows():
    g = torch.Generator().manual_seed(5)
    buf = torch.relu(torch.randn(100000, generator=g))
    starts = torch.tensor([0, 1, 2, 3, 50000, 50001, 12345, 0], dtype=torch.int32)
    lengths = torch.tensor([100000, 99999, 5000, 3, 50000, 49999, 77777, 2048], dtype=torch.int32)
    for k in (1, 2048, 4096):
        assert_stats(W.Workload("overlap", buf, starts, lengths, k, 0, {}))
    rows = [torch.relu(torch.randn(L, generator=g) - 2.5) for L in (3_000_000, 800_001)]
    assert_stats(ragged("huge", rows, 4096, lead=1))


def test_rejected_rows_set_status():
    buf = torch.ones(64)
    starts = torch.tensor([0, -1, 60, 0, 10], dtype=torch.int32)
    lengths = torch.tensor([8, 4, 8, 1 << 24, -3], dtype=torch.int32)
    got = assert_stats(W.Workload("bad", buf, starts, lengths, 4, 0, {}))
    assert got[1:4].tolist() == [[0] * 6] * 3


def test_repeatable_and_graph_replay():
    w = W.make("decode", device="cuda")
    a = pkg.topk_ragged_stats(w.scores, w.row_starts, w.lengths, w.k)
    out = torch.empty_like(a)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkg.topk_ragged_stats(w.scores, w.row_starts, w.lengths, w.k, out=out)   # warm
    torch.cuda.synchronize()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkg.topk_ragged_stats(w.scores, w.row_starts, w.lengths, w.k, out=out)
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, a)
    for _ in range(3):
        assert torch.equal(pkg.topk_ragged_stats(w.scores, w.row_starts, w.lengths, w.k), a)


def test_rejected_and_empty_rows_in_clusters():
    # Few long rows: the library splits each over a cluster of CTAs.
    g = torch.Generator().manual_seed(21)
    buf = torch.relu(torch.randn(3_000_000, generator=g) - 0.5)
    starts = torch.tensor([0, -5, 2_000_000, 100, 2_999_000, 7], dtype=torch.int32)
    lengths = torch.tensor([900_000, 10, 999_999, 0, 5_000, 1 << 24], dtype=torch.int32)
    for k in (1, 2048, 4096):
        got = assert_stats(W.Workload("bad_cluster", buf, starts, lengths, k, 0, {}))
        assert got[[1, 4, 5]].tolist() == [[0] * 6] * 3
        assert got[3].tolist() == [0, 0, 0, 0, 0, 0]
