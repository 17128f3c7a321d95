"""Pins for the oracle's tie/plateau statistics (oracle.row_stats).

The statistics are those of the sglang page's score-statistics script
(row_stats): plateau fraction, the k-th score, its tie-set size, the count
strictly above it, straddle and zero_bound.  They are pinned three ways, none
of which uses the oracle's own order key or sort:
  * hand-worked rows (ties across position k, signed zeros, NaN payloads,
    rows no longer than k, rejected windows);
  * the page's float definition restated with torch's sort, on rows without
    NaN or -0.0 (where the bitwise order and the float order agree);
  * invariants that tie the statistics to the selection itself: the k-th
    selected value is the boundary and exactly k - above selected entries
    equal it.
Planted slips in a copy of row_stats (a flipped comparison, an off-by-one at
the boundary, the wrong zero test) each fail at least one of these.
"""
import inspect
import textwrap

import numpy as np
import pytest
import torch

import oracle
import workloads as W

HAS, STR, ZB = oracle.STAT_HAS_BOUNDARY, oracle.STAT_STRADDLE, oracle.STAT_ZERO_BOUND


def _bits(*vals):
    return np.array(vals, dtype=np.uint32)


def _one(fn, bits, k):
    x = np.asarray(bits, dtype=np.uint32).view(np.float32)
    st, fl = fn(x, [0], [x.size], k)
    return tuple(int(v) for v in st[0]), int(fl[0])


# --------------------------------------------------------------------------- #
# The three pins, as functions of the statistics routine under test.
# --------------------------------------------------------------------------- #

def pin_hand_cases(fn):
    one, two, three = 0x3F800000, 0x40000000, 0x40400000
    row = _bits(three, two, two, two, one)               # 3, 2, 2, 2, 1
    assert _one(fn, row, 1) == ((5, 0, three, 1, 0, HAS), 0)
    assert _one(fn, row, 2) == ((5, 0, two, 3, 1, HAS | STR), 0)   # 1 above, 3 tied, k = 2
    assert _one(fn, row, 4) == ((5, 0, two, 3, 1, HAS), 0)         # the tie set ends at k
    assert _one(fn, row, 5) == ((5, 0, 0, 0, 5, 0), 0)             # L <= k: no boundary
    # +0.0 ranks above -0.0 (not bitwise equal); both count as 0.0.
    z = _bits(0x00000000, 0x80000000, 0x80000000, 0x3F000000)
    assert _one(fn, z, 1) == ((4, 3, 0x3F000000, 1, 0, HAS), 0)
    assert _one(fn, z, 2) == ((4, 3, 0x00000000, 1, 1, HAS | ZB), 0)
    assert _one(fn, z, 3) == ((4, 3, 0x80000000, 2, 2, HAS | STR | ZB), 0)
    # Two copies of one +NaN pattern sit above +inf; another payload is apart.
    nan = _bits(0x7FC00001, 0x7F800000, 0x7FC00001, 0x7FC00002, 0xFFC00000)
    assert _one(fn, nan, 1) == ((5, 0, 0x7FC00002, 1, 0, HAS), 0)
    assert _one(fn, nan, 2) == ((5, 0, 0x7FC00001, 2, 1, HAS | STR), 0)
    assert _one(fn, nan, 4) == ((5, 0, 0x7F800000, 1, 3, HAS), 0)
    # An all-equal row longer than k straddles; an all-zero one is zero-bound.
    assert _one(fn, _bits(*[0] * 10), 4) == ((10, 10, 0, 10, 0, HAS | STR | ZB), 0)
    # Empty rows, rejected windows and lengths.
    x = np.ones(8, dtype=np.float32)
    st, fl = fn(x, [0, 3, -1, 6, 0], [0, -5, 2, 4, 1 << 24], 2)
    assert st[:2].tolist() == [[0, 0, 0, 0, 0, 0]] * 2 and fl[:2].tolist() == [0, 0]
    assert st[2:].tolist() == [[0] * 6] * 3
    assert fl[2:].tolist() == [oracle.FLAG_BAD_WINDOW, oracle.FLAG_BAD_WINDOW, oracle.FLAG_LEN_ENVELOPE]


def torch_float_stats(row: torch.Tensor, k: int):
    """The page's definition with float comparisons and torch's sort."""
    n = row.numel()
    n_zero = int((row == 0.0).sum())
    if n <= k:
        return (n, n_zero, 0, 0, n, 0)
    v = torch.sort(row, descending=True).values[k - 1]
    tie = int((row == v).sum())
    above = int((row > v).sum())
    flags = HAS | (STR if tie > 1 and above + tie > k else 0) | (ZB if float(v) == 0.0 else 0)
    return (n, n_zero, int(v.view(torch.int32)) & 0xFFFFFFFF, tie, above, flags)


def pin_float_definition(fn):
    g = torch.Generator().manual_seed(5)
    rows = []
    for t in range(40):
        L = int(torch.randint(1, 3000, (1,), generator=g))
        x = torch.randn(L, generator=g)
        if t % 3 == 0:
            x = torch.round(x * 4) / 4            # ties everywhere
        if t % 4 == 1:
            x = torch.relu(x - 0.3)               # a +0.0 plateau
        if t % 5 == 2:
            x = -torch.relu(x)                    # negative side, -0.0 replaced below
        x = torch.where(x == 0, torch.zeros_like(x), x)   # every zero is +0.0
        rows.append(x)
    flat = torch.cat(rows).numpy()
    lengths = np.array([r.numel() for r in rows])
    starts = np.concatenate([[0], np.cumsum(lengths)[:-1]])
    for k in (1, 7, 512, 2048):
        st, fl = fn(flat, starts, lengths, k)
        assert not fl.any()
        for i, r in enumerate(rows):
            assert tuple(int(v) for v in st[i]) == torch_float_stats(r, k), (k, i)


def pin_selection_invariants(fn):
    alphabet = [0, 0x80000000, 0x3F800000, 0x7FC00001, 0xFFC00001, 0xFF800000, 0x7F800000, 1]
    for w in (W.random_bits(30, 3001, 1000, alphabet=alphabet), W.random_bits(20, 5003, 7),
              W.tie_block(4, 8192, 2048, 512), W.plateau(4, 8192, 1024, 2048)):
        s, st0, ln = w.numpy()
        st, fl = fn(s, st0, ln, w.k)
        _, val, _ = oracle.topk_ragged(s, st0, ln, w.k, 0)
        val = val.view(np.uint32)
        for i in range(w.B):
            L, n_zero, bb, tie, above, flags = (int(v) for v in st[i])
            row = s[st0[i]:st0[i] + ln[i]].view(np.uint32)
            assert n_zero == int(np.count_nonzero((row & 0x7FFFFFFF) == 0))
            if L <= w.k:
                continue
            assert above < w.k <= above + tie
            assert int(val[i, w.k - 1]) == bb
            assert int(np.count_nonzero(val[i] == bb)) == w.k - above
            assert bool(flags & STR) == (tie > 1 and above + tie > w.k)


PINS = (pin_hand_cases, pin_float_definition, pin_selection_invariants)


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_row_stats_pins(pin):
    pin(oracle.row_stats)


# --------------------------------------------------------------------------- #
# Planted slips in a copy of row_stats; each must fail one of the pins.
# --------------------------------------------------------------------------- #
MUTATIONS = {
    "tie_ge": ("tie = int(np.count_nonzero(key == T))", "tie = int(np.count_nonzero(key >= T))"),
    "above_ge": ("above = int(np.count_nonzero(key > T))", "above = int(np.count_nonzero(key >= T))"),
    "boundary_off_by_one": ("[::-1][k - 1]", "[::-1][k]"),
    "ascending": ("np.sort(key)[::-1][k - 1]", "np.sort(key)[k - 1]"),
    "straddle_ge": ("above + tie > k:", "above + tie >= k:"),
    "zero_plus_only": ("(b & 0x7FFFFFFF) == 0))", "b == 0))"),
    "short_rows_lt": ("if L <= k:", "if L < k:"),
    "zero_bound_plus_only": ("if bb & 0x7FFFFFFF == 0:", "if bb == 0:"),
}


def _mutant(name):
    before, after = MUTATIONS[name]
    src = textwrap.dedent(inspect.getsource(oracle.row_stats))
    assert src.count(before) == 1, name
    ns = dict(vars(oracle))
    exec(compile(src.replace(before, after), f"<row_stats {name}>", "exec"), ns)
    return ns["row_stats"]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_slip_is_caught(name):
    fn = _mutant(name)
    failed = []
    for pin in PINS:
        try:
            pin(fn)
        except (AssertionError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught {name}"


# --------------------------------------------------------------------------- #
# Closed forms of the sglang page's tie-safety families: a plateau row of m
# distinct positives and L - m exact zeros has, for m < k, its boundary on
# the zero plateau with a tie set of L - m; a tie block of T copies of 1.0
# with `above` distinct larger values, where the block straddles the k-th
# place (above < k < above + T), has the boundary 1.0 with tie T.
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("m", [0, 1, 256, 1024, 2047])
def test_plateau_family_closed_form(m):
    L, k = 8192, 2048
    w = W.plateau(3, L, m, k)
    s, st, ln = w.numpy()
    stats, fl = oracle.row_stats(s, st, ln, k)
    assert not fl.any()
    for row in stats.tolist():
        assert row == [L, L - m, 0, L - m, m, HAS | STR | ZB]


@pytest.mark.parametrize("T", [2, 64, 512, 4096])
def test_tie_block_family_closed_form(T):
    L, k = 16384, 2048
    w = W.tie_block(3, L, k, T)
    s, st, ln = w.numpy()
    stats, _ = oracle.row_stats(s, st, ln, k)
    above = w.info["above"]
    assert max(0, k - T + 1) <= above < k
    for row in stats.tolist():
        assert row == [L, 0, 0x3F800000, T, above, HAS | STR]
