"""Property tests of the oracle over arbitrary fp32 bit patterns.

The fixed alphabets of the exhaustive pins cover the order's special values;
here hypothesis draws any 32-bit patterns (every NaN payload, denormals, both
zeros, the extremes), any k and any placement of the row in its buffer, and
checks the selection and the tie/plateau statistics against sort-free brute
force written from the order's definition (fp32 comparison, NaN placed by
sign and payload, -0.0 below +0.0), which shares nothing with the oracle's key.
"""
import numpy as np
import pytest

import oracle
from test_oracle import brute_force_topk, order_tuple

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies

SPECIAL = [0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000, 0x00000001,
           0x80000001, 0x7F7FFFFF, 0xFF7FFFFF, 0x3F800000, 0xBF800000, 0x7FFFFFFF, 0xFFFFFFFF]
# Half arbitrary patterns, half drawn from a few specials, so ties occur.
bits32 = st.one_of(st.integers(0, 0xFFFFFFFF), st.sampled_from(SPECIAL))
rows = st.lists(bits32, min_size=0, max_size=40)


def _place(row, pad):
    flat = np.zeros(pad + len(row) + 3, dtype=np.uint32)
    flat[pad:pad + len(row)] = row
    return flat.view(np.float32), np.array([pad], dtype=np.int32), np.array([len(row)], dtype=np.int32)


@hypothesis.settings(max_examples=400, deadline=None)
@hypothesis.given(row=rows, k=st.integers(1, 48), pad=st.integers(0, 5), row_start=st.booleans())
def test_selection_equals_rank_count(row, k, pad, row_start):
    s, starts, lengths = _place(row, pad)
    mode = oracle.OFFSET_ROW_START if row_start else 0
    idx, val, flags = oracle.topk_ragged(s, starts, lengths, k, mode)
    want = brute_force_topk(row, k)
    off = pad if row_start else 0
    assert idx[0].tolist() == [j + off if j >= 0 else -1 for j in want]
    assert val[0].view(np.uint32).tolist() == [row[j] if j >= 0 else 0xFF800000 for j in want]
    assert int(flags[0]) == 0


def brute_force_stats(row, k):
    """The tie/plateau statistics from the order tuple alone."""
    t = [order_tuple(b) for b in row]
    L = len(row)
    n_zero = sum(1 for b in row if b & 0x7FFFFFFF == 0)
    if L <= k:
        return (L, n_zero, 0, 0, L, 0)
    order = sorted(range(L), key=lambda j: (t[j], -j), reverse=True)
    b = row[order[k - 1]]
    tb = t[order[k - 1]]
    tie = sum(1 for x in t if x == tb)
    above = sum(1 for x in t if x > tb)
    flags = oracle.STAT_HAS_BOUNDARY
    if tie > 1 and above + tie > k:
        flags |= oracle.STAT_STRADDLE
    if b & 0x7FFFFFFF == 0:
        flags |= oracle.STAT_ZERO_BOUND
    return (L, n_zero, b, tie, above, flags)


@hypothesis.settings(max_examples=400, deadline=None)
@hypothesis.given(row=rows, k=st.integers(1, 48), pad=st.integers(0, 5))
def test_row_stats_equal_brute_force(row, k, pad):
    s, starts, lengths = _place(row, pad)
    stats, flags = oracle.row_stats(s, starts, lengths, k)
    assert tuple(int(v) for v in stats[0]) == brute_force_stats(row, k)
    assert int(flags[0]) == 0


@hypothesis.settings(max_examples=200, deadline=None)
@hypothesis.given(row=rows, k=st.integers(1, 48))
def test_exclusion_keeps_the_selection_of_the_rest(row, k):
    """Excluding -inf and negative NaN equals selecting over the other
    entries alone (their original indices kept), then -1."""
    s, starts, lengths = _place(row, 0)
    idx, _, _ = oracle.topk_ragged(s, starts, lengths, k, oracle.EXCLUDE_NEG_INF)
    kept = [j for j, b in enumerate(row) if order_tuple(b) > order_tuple(0xFF800000)]
    sub = brute_force_topk([row[j] for j in kept], k)
    assert idx[0].tolist() == [kept[j] if j >= 0 else -1 for j in sub]
