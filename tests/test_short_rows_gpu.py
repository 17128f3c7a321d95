"""The row kernel's register-resident short path, branch by branch.

Batches of 700 rows (more than four per SM, so every row goes to the
one-CTA-per-row kernel) whose rows steer the short path into each of its
cases, checked against the oracle bit for bit:

- lengths around 4 x 256 quads (4090 .. 4100) at every alignment of the row
  start, so rows fall on both sides of the register limit (the longest ones
  take the general path);
- both signs around +0.0 (the bucket grid is shifted to put a bucket edge on
  +0.0's key), only negatives with +0.0 entries, only +0.0, only one sign;
- a block of equal non-zero scores of 40 .. 200 entries inside the output
  (more than 48 members in one bucket sends the row to the general path);
- NaNs of both signs and -inf, with and without the exclusion flag;
- k from 1 to 4096 (the ranked count and the buffer of composites).
"""
import pytest
import torch

from helpers import assert_parity, ragged

pytestmark = pytest.mark.gpu

B = 700


def _row(kind: int, L: int, g: torch.Generator) -> torch.Tensor:
    x = torch.randn(L, generator=g)
    if kind == 0:            # both signs, a third +0.0
        x[torch.rand(L, generator=g) < 0.33] = 0.0
    elif kind == 1:          # negatives and +0.0 only
        x = -x.abs()
        x[torch.rand(L, generator=g) < 0.5] = 0.0
    elif kind == 2:          # all +0.0
        x = torch.zeros(L)
    elif kind == 3:          # positives only (relu of a shifted normal, the indexer's shape)
        x = torch.relu(x - 0.3)
    elif kind == 4:          # a block of equal scores near the top
        n = int(torch.randint(40, 201, (1,), generator=g))
        pos = torch.randperm(L, generator=g)[:min(n, L)]
        x[pos] = 1.25
    elif kind == 5:          # NaNs of both signs and -inf
        u = torch.rand(L, generator=g)
        x[u < 0.02] = float("nan")
        x[(u >= 0.02) & (u < 0.04)] = -float("nan")
        x[(u >= 0.04) & (u < 0.06)] = -float("inf")
    return x


@pytest.mark.parametrize("k", [1, 64, 2048, 4096])
@pytest.mark.parametrize("mode", [0, 1, 2, 3])   # row-local / row-start offsets, with and without exclusion
def test_short_path_cases(k, mode):
    g = torch.Generator().manual_seed(17 * k + mode)
    rows = []
    for i in range(B):
        if i < 72:
            L = 4090 + i % 11          # around the 1024-quad limit, starts at every alignment below
        else:
            L = int(torch.randint(1, 4100, (1,), generator=g))
        rows.append(_row(i % 6, L, g))
    assert_parity(ragged(f"short_k{k}_m{mode}", rows, k, offset_mode=mode, gap=1 + mode, lead=mode))
