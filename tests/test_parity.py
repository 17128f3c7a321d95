"""Bit-exact parity of the CUDA path with the CPU oracle (out_idx and the bit
patterns of out_val), on the five named workloads at full size and on the
tie-study families, edge lengths, unaligned and overlapping windows and every
launch shape the host planner picks."""
import numpy as np
import pytest
import torch

import workloads as W
from helpers import assert_parity, ragged

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import sparse_attention_deterministic_gb300 as pkg
    pkg.build()
    pkg.init()


# --- the five named workloads, full size (the launch shapes bench.py times) --
@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "adversarial", "long"])
def test_named_workload_full_size(name):
    w = W.make(name, device="cuda").to("cpu")
    assert_parity(w)


# --- tie-study families of the pages ----------------------------------------
@pytest.mark.parametrize("B,L", [(64, 32768), (4, 32768), (8, 131072)])
@pytest.mark.parametrize("m", [0, 256, 1024, 4095, 8192])
def test_plateau_family(B, L, m):
    assert_parity(W.plateau(B, L, m, 2048))


@pytest.mark.parametrize("B,L", [(64, 32768), (4, 32768), (8, 131072)])
@pytest.mark.parametrize("T", [64, 512, 4096, 16384])
def test_tie_family(B, L, T):
    assert_parity(W.tie_block(B, L, 2048, T))


@pytest.mark.parametrize("B,L", [(64, 16384), (256, 16384), (64, 32768)])
def test_relu_shifted_family(B, L):
    assert_parity(W.relu_shifted(B, L, 2048))


@pytest.mark.parametrize("B,L", [(64, 32768), (8, 131072)])
def test_narrow_family(B, L):
    assert_parity(W.narrow(B, L, 2048))


@pytest.mark.parametrize("alphabet", [None, [0, 0x80000000, 0x3F800000, 0x7FC00001, 0xFFC00001,
                                             0xFF800000, 0x7F800000, 0x00000001]])
@pytest.mark.parametrize("B", [3, 50, 700])
def test_random_bit_patterns(alphabet, B):
    assert_parity(W.random_bits(B, 5003, 1024, alphabet=alphabet))


# --- every k, every planner class, ragged lengths around k --------------------
@pytest.mark.parametrize("k", [1, 2, 7, 100, 512, 1024, 2047, 2048, 3000, 4096])
@pytest.mark.parametrize("B", [1, 5, 40, 160, 300, 400, 700])
def test_lengths_around_k(k, B):
    g = torch.Generator().manual_seed(1000 * k + B)
    choices = [0, 1, 2, 3, 4, 5, k - 1, k, k + 1, 2 * k + 3, 4 * k + 1, 40000]
    rows = []
    for i in range(B):
        L = max(0, choices[i % len(choices)] if i < len(choices) else
                int(torch.randint(0, 3 * k + 10, (1,), generator=g)))
        r = torch.randn(L, generator=g)
        r[torch.rand(L, generator=g) < 0.4] = 0.0
        rows.append(r)
    assert_parity(ragged(f"around_k{k}_B{B}", rows, k, offset_mode=B % 2, gap=1, lead=3))


@pytest.mark.parametrize("lead", [0, 1, 2, 3, 5])
@pytest.mark.parametrize("B", [2, 64, 1000])
def test_unaligned_row_starts(lead, B):
    g = torch.Generator().manual_seed(lead * 7 + B)
    rows = [torch.relu(torch.randn(int(torch.randint(1, 9000, (1,), generator=g)), generator=g))
            for _ in range(B)]
    assert_parity(ragged(f"unaligned{lead}", rows, 512, gap=lead % 3 + 1, lead=lead))


def test_overlapping_windows():
    g = torch.Generator().manual_seed(5)
    buf = torch.relu(torch.randn(100000, generator=g))
    starts = torch.tensor([0, 1, 2, 3, 50000, 50001, 12345, 0], dtype=torch.int32)
    lengths = torch.tensor([100000, 99999, 5000, 3, 50000, 49999, 77777, 2048], dtype=torch.int32)
    for k in (1, 2048, 4096):
        for mode in (0, 1):
            assert_parity(W.Workload("overlap", buf, starts, lengths, k, mode, {}))


def test_long_rows_beyond_shared_memory():
    # Rows longer than a cluster's staging capacity exercise the L2 re-read path.
    g = torch.Generator().manual_seed(9)
    rows = [torch.relu(torch.randn(L, generator=g) - 2.5) for L in (3_000_000, 800_001)]
    assert_parity(ragged("huge", rows, 4096, lead=1))
    rows = [torch.randn(1_500_000, generator=g) for _ in range(3)]
    assert_parity(ragged("huge2", rows, 2048))


def test_values_optional_gives_same_indices():
    w = W.decode(B=16, lmin=1000, lmax=70000, k=2048)
    a = assert_parity(w, with_values=True)
    b = assert_parity(w, with_values=False)
    assert np.array_equal(a, b)
