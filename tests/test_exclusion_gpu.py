"""The -inf exclusion flag (offset_mode bit 2) on the GPU, bit for bit
against the oracle, in both kernels and on every path that writes entries:
the short and general one-CTA-per-row paths, cluster rows settled by a key
range, and exact thresholds whose tie set is -inf itself."""
import numpy as np
import pytest
import torch

import workloads as W
from helpers import assert_parity, ragged

pytestmark = pytest.mark.gpu

NEG_INF, NEG_NAN = float("-inf"), np.array([0xFFC00000], np.uint32).view(np.float32)[0]


def _row(g, L, p_neg_inf, p_neg_nan, p_zero=0.3):
    x = torch.randn(L, generator=g)
    u = torch.rand(L, generator=g)
    x[u < p_zero] = 0.0
    x[(u >= p_zero) & (u < p_zero + p_neg_inf)] = NEG_INF
    x[(u >= p_zero + p_neg_inf) & (u < p_zero + p_neg_inf + p_neg_nan)] = float(NEG_NAN)
    return x


@pytest.mark.parametrize("mode", [2, 3])
@pytest.mark.parametrize("B,L,k", [(64, 3000, 2048), (5, 20000, 2048), (700, 2500, 2048), (3, 9000, 64)])
def test_exclusion_mixed_rows(mode, B, L, k):
    g = torch.Generator().manual_seed(B * 1000 + L + mode)
    rows = [_row(g, int(torch.randint(1, L + 1, (1,), generator=g)), 0.4, 0.05) for _ in range(B)]
    assert_parity(ragged(f"excl{mode}_{B}_{L}", rows, k, offset_mode=mode, lead=3))


@pytest.mark.parametrize("mode", [2, 3])
def test_exclusion_tie_set_is_neg_inf(mode):
    # Fewer finite entries than k: the boundary lies in the -inf block, whose
    # members are ties of an exact threshold; long rows take the clusters.
    g = torch.Generator().manual_seed(5 + mode)
    rows = [_row(g, 70000, 0.97, 0.0, p_zero=0.0) for _ in range(6)]
    rows.append(torch.full((50000,), NEG_INF))
    assert_parity(ragged(f"excl_ties{mode}", rows, 4096, offset_mode=mode))


def test_exclusion_off_ranks_neg_inf():
    g = torch.Generator().manual_seed(9)
    rows = [_row(g, 3000, 0.5, 0.05) for _ in range(40)]
    assert_parity(ragged("excl_off", rows, 2048, offset_mode=0))


def test_exclusion_named_workloads():
    for name in ("adversarial", "tiny"):
        w = W.make(name)
        w = W.Workload(w.name + "_excl", w.scores, w.row_starts, w.lengths, w.k,
                       w.offset_mode | 2, w.info)
        assert_parity(w)
