"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test pins the oracle to an independent statement of what the pages fix:
a brute-force rank count written from the order's definition, hand-derived
golden rows, a library stable sort, the torch.topk + two-stable-sorts recipe
of the blog post, closed forms and invariants.  A plausible slip in the oracle
(a flipped comparator, the key's negative branch wrong, a dropped tie rule,
an off-by-one in the padding or the offset) fails at least one of them.
"""
import glob
import itertools
import os
import struct

import numpy as np
import pytest
import torch

import oracle
import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def f32_from_bits(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


# --------------------------------------------------------------------------- #
# An order stated without the oracle's key: fp32 comparison plus the two rules
# the pages add (NaN placed by sign and payload, not maximal; -0.0 below +0.0
# because they are not bitwise-equal).
# --------------------------------------------------------------------------- #

def order_tuple(bits: int):
    sign = bits >> 31
    exp = (bits >> 23) & 0xFF
    mant = bits & 0x7FFFFF
    if exp == 0xFF and mant != 0:                     # NaN
        return (2, float(mant), 0) if sign == 0 else (-2, -float(mant), 0)
    value = struct.unpack("<f", struct.pack("<I", bits))[0]
    zero_rank = 1 if (value == 0.0 and sign == 0) else 0
    return (0, value, zero_rank)


def brute_force_topk(row_bits, k):
    """rank(j) = #{i : t_i > t_j or (t_i == t_j and i < j)}; slot rank(j) = j."""
    t = [order_tuple(b) for b in row_bits]
    out = [-1] * k
    for j in range(len(t)):
        rank = sum(1 for i in range(len(t)) if t[i] > t[j] or (t[i] == t[j] and i < j))
        if rank < k:
            out[rank] = j
    return out


ALPHABET = [
    0x7FC00000, 0x7F800001,            # +NaN, two payloads
    0xFFC00000, 0xFF800001,            # -NaN, two payloads
    0xFF800000, 0xBF800000,            # -inf, -1.0
    0x80000000, 0x00000000,            # -0.0, +0.0
    0x3F800000, 0x7F800000,            # 1.0, +inf
]


def _levels(alphabet):
    ranked = sorted(set(order_tuple(b) for b in alphabet))
    return np.array([ranked.index(order_tuple(b)) for b in alphabet], dtype=np.int64)


def _run_oracle_rows(rows_bits, k, offset_mode=0, pad_before=0):
    lengths = np.array([len(r) for r in rows_bits], dtype=np.int32)
    starts = (np.cumsum(lengths) - lengths + pad_before).astype(np.int32)
    flat = np.zeros(pad_before + int(lengths.sum()), dtype=np.uint32)
    for s, r in zip(starts, rows_bits):
        flat[s:s + len(r)] = r
    idx, val, flags = oracle.topk_ragged(flat.view(np.float32), starts, lengths, k,
                                         offset_mode)
    return idx, val, flags, starts


@pytest.mark.parametrize("length", [0, 1, 2, 3, 4, 5])
def test_brute_force_exhaustive(length):
    """Every row of length <= 5 over a 10-pattern alphabet, every k in 1..7:
    the oracle equals the sort-free rank count (vectorised per length)."""
    levels = _levels(ALPHABET)
    combos = list(itertools.product(range(len(ALPHABET)), repeat=length))
    sym = np.array(combos, dtype=np.int64).reshape(len(combos), length)
    bits = np.array(ALPHABET, dtype=np.uint32)[sym]
    lv = levels[sym]                                            # [R, n]
    pos = np.arange(length)
    # rank[r, j] = #{i: lv[i] > lv[j]} + #{i < j: lv[i] == lv[j]}
    gt = (lv[:, :, None] > lv[:, None, :]).sum(1)
    eq_before = ((lv[:, :, None] == lv[:, None, :]) & (pos[:, None] < pos[None, :])).sum(1)
    rank = gt + eq_before
    for k in range(1, 8):
        expect = np.full((sym.shape[0], k), -1, dtype=np.int32)
        rr, jj = np.nonzero(rank < k)
        expect[rr, rank[rr, jj]] = jj
        idx, val, _, _ = _run_oracle_rows(list(bits), k)
        np.testing.assert_array_equal(idx, expect)
        # values: the selected patterns, pad = -inf bits
        if length:
            picked = bits[np.arange(sym.shape[0])[:, None], np.maximum(expect, 0)]
        else:
            picked = np.zeros(expect.shape, dtype=np.uint32)
        sel = np.where(expect >= 0, picked, 0xFF800000).astype(np.uint32)
        np.testing.assert_array_equal(val.view(np.uint32), sel)


def test_brute_force_scalar_cross_check():
    """The vectorised brute force above and the scalar one agree with the oracle
    on random longer rows drawn from a wider alphabet (denormals, max, ties)."""
    wide = ALPHABET + [0x00000001, 0x80000001, 0x7F7FFFFF, 0xFF7FFFFF, 0x3FC00000,
                       0xBFC00000]
    rng = np.random.default_rng(1234)
    rows = [rng.choice(np.array(wide, dtype=np.uint32), size=int(rng.integers(0, 24)))
            for _ in range(300)]
    for k in (1, 3, 8, 16, 30):
        idx, _, _, _ = _run_oracle_rows(rows, k)
        for r, row in enumerate(rows):
            assert list(idx[r]) == brute_force_topk([int(b) for b in row], k)


# --------------------------------------------------------------------------- #
# Golden rows worked out by hand (tests/golden/*.txt).
# --------------------------------------------------------------------------- #

def _parse_golden(path):
    fields = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            fields[key.strip()] = val.strip()
    return fields


GOLDEN = sorted(glob.glob(os.path.join(HERE, "golden", "*.txt")))


def test_golden_files_exist_and_cite():
    assert len(GOLDEN) >= 8
    for p in GOLDEN:
        assert "cite" in _parse_golden(p), p


@pytest.mark.parametrize("path", GOLDEN, ids=[os.path.basename(p) for p in GOLDEN])
def test_golden(path):
    g = _parse_golden(path)
    k = int(g["k"])
    mode = int(g["offset_mode"])
    start = int(g["row_start"])
    row = [int(x, 16) for x in g["scores"].split()]
    flat = np.zeros(start + len(row) + 3, dtype=np.uint32)
    flat[start:start + len(row)] = row
    idx, val, flags = oracle.topk_ragged(flat.view(np.float32), np.array([start]),
                                         np.array([len(row)]), k, mode)
    assert list(idx[0]) == [int(x) for x in g["expected_idx"].split()]
    assert list(val[0].view(np.uint32)) == [int(x, 16) for x in g["expected_val"].split()]
    assert flags[0] == 0


# --------------------------------------------------------------------------- #
# The order key: bijective, float-order preserving, NaN groups at the ends.
# --------------------------------------------------------------------------- #

def _structured_patterns():
    mants = np.array([0, 1, 2, 3, 0x1FFFFF, 0x3FFFFF, 0x400000, 0x400001, 0x7FFFFE, 0x7FFFFF],
                     dtype=np.uint32)
    se = np.arange(512, dtype=np.uint32) << 23
    grid = (se[:, None] | mants[None, :]).reshape(-1)
    rnd = np.random.default_rng(5).integers(0, 1 << 32, size=1 << 21, dtype=np.uint64)
    return np.unique(np.concatenate([grid, rnd.astype(np.uint32)]))


def test_order_key_bijective_and_monotone():
    bits = _structured_patterns()
    keys = oracle.order_key(bits)
    assert np.unique(keys).size == bits.size                      # injective
    vals = bits.view(np.float32)
    nan = np.isnan(vals)
    # Sorting by key must put non-NaN floats in non-decreasing order ...
    order = np.argsort(keys[~nan], kind="stable")
    v = vals[~nan][order]
    b = bits[~nan][order]
    assert np.all(v[1:] >= v[:-1])
    # ... and the only equal floats (the two zeros) in -0.0, +0.0 order.
    zero_pos = np.nonzero(v == 0)[0]
    assert list(b[zero_pos]) == [0x80000000, 0x00000000]
    # NaN groups: +NaN above +inf, -NaN below -inf, payload order inside.
    k_pinf = oracle.order_key(np.array([0x7F800000], dtype=np.uint32))[0]
    k_ninf = oracle.order_key(np.array([0xFF800000], dtype=np.uint32))[0]
    pos_nan = nan & (bits >> 31 == 0)
    neg_nan = nan & (bits >> 31 == 1)
    assert np.all(keys[pos_nan] > k_pinf)
    assert np.all(keys[neg_nan] < k_ninf)
    pay = bits & 0x7FFFFF
    o = np.argsort(keys[pos_nan])
    assert np.all(np.diff(pay[pos_nan][o].astype(np.int64)) > 0)
    o = np.argsort(keys[neg_nan])
    assert np.all(np.diff(pay[neg_nan][o].astype(np.int64)) < 0)


# --------------------------------------------------------------------------- #
# Library and recipe pins (rows without NaN and without -0.0, where the
# bitwise total order coincides with fp32 comparison).
# --------------------------------------------------------------------------- #

def _float_rows(seed, B, L, quantise):
    g = torch.Generator().manual_seed(seed)
    rows = torch.randn(B, L, generator=g)
    if quantise:
        rows = torch.round(rows * quantise) / quantise         # many exact ties
    rows = torch.where(rows == 0, torch.zeros_like(rows), rows)  # no -0.0
    rows[:, ::7] = torch.relu(rows[:, ::7])                    # a 0.0 plateau
    return rows.contiguous()


@pytest.mark.parametrize("quantise", [0, 4, 64])
@pytest.mark.parametrize("k", [1, 17, 256, 1000])
def test_library_stable_sort_pin(quantise, k):
    """torch.sort(descending, stable) keeps ascending index among equal values:
    its first k indices are the canonical top-k."""
    B, L = 6, 999
    rows = _float_rows(100 + k + quantise, B, L, quantise)
    starts = np.arange(B, dtype=np.int32) * L
    lengths = np.full(B, L, dtype=np.int32)
    idx, val, _ = oracle.topk_ragged(rows.numpy().reshape(-1), starts, lengths, k)
    ref = torch.sort(rows, dim=1, descending=True, stable=True).indices[:, :k]
    np.testing.assert_array_equal(idx[:, :min(k, L)], ref.numpy())
    np.testing.assert_array_equal(val[:, :min(k, L)], rows.gather(1, ref).numpy())


@pytest.mark.parametrize("k", [8, 300, 2048])
def test_blog_recipe_pin(k):
    """The blog post's exact-selection recipe (torch.topk unsorted, a stable
    sort by index ascending, a stable sort by value descending, -1 pad when the
    row is shorter than k) equals the oracle on rows whose k-th boundary is not
    tied (where torch.topk's unsorted set is unique)."""
    g = torch.Generator().manual_seed(k)
    for L in (k // 2, k, k + 1, 3 * k + 5):
        rows = torch.randn(5, L, generator=g)
        vals, ind = torch.topk(rows, min(k, L), dim=1, sorted=False)
        o = torch.sort(ind, dim=1, stable=True).indices
        ind, vals = ind.gather(1, o), vals.gather(1, o)
        o = torch.sort(vals, dim=1, descending=True, stable=True).indices
        ind = ind.gather(1, o)
        expect = torch.full((5, k), -1, dtype=torch.int64)
        expect[:, :ind.shape[1]] = ind
        starts = np.arange(5, dtype=np.int32) * L
        idx, _, _ = oracle.topk_ragged(rows.numpy().reshape(-1), starts,
                                       np.full(5, L, dtype=np.int32), k)
        np.testing.assert_array_equal(idx, expect.numpy())


# --------------------------------------------------------------------------- #
# Closed forms.
# --------------------------------------------------------------------------- #

def test_all_zero_and_all_neg_inf():
    for pattern in (0x00000000, 0xFF800000, 0x80000000):
        L, k = 5000, 2048
        flat = np.full(L, pattern, dtype=np.uint32).view(np.float32)
        idx, val, _ = oracle.topk_ragged(flat, np.array([0]), np.array([L]), k)
        assert list(idx[0]) == list(range(k))
        assert np.all(val.view(np.uint32) == pattern)


def test_empty_and_negative_lengths():
    flat = np.ones(10, dtype=np.float32)
    idx, val, flags = oracle.topk_ragged(flat, np.array([0, 3]), np.array([0, -5]), 4)
    assert np.all(idx == -1)
    assert np.all(val.view(np.uint32) == oracle.PAD_VALUE_BITS)
    assert list(flags) == [0, 0]


def test_envelope_and_window_flags():
    flat = np.ones(100, dtype=np.float32)
    starts = np.array([0, 90, -1, 10])
    lengths = np.array([1 << 24, 20, 5, 10])
    idx, _, flags = oracle.topk_ragged(flat, starts, lengths, 3)
    assert list(flags) == [oracle.FLAG_LEN_ENVELOPE, oracle.FLAG_BAD_WINDOW,
                           oracle.FLAG_BAD_WINDOW, 0]
    assert np.all(idx[:3] == -1)
    assert list(idx[3]) == [0, 1, 2]


def test_empty_batch_and_bad_args():
    flat = np.ones(4, dtype=np.float32)
    idx, _, _ = oracle.topk_ragged(flat, np.zeros(0), np.zeros(0), 5)
    assert idx.shape == (0, 5)
    for k in (0, 4097):
        with pytest.raises(ValueError):
            oracle.topk_ragged(flat, np.array([0]), np.array([4]), k)
    with pytest.raises(ValueError):
        oracle.topk_ragged(flat, np.array([0]), np.array([4]), 2, offset_mode=4)


@pytest.mark.parametrize("T", [64, 512, 4096])
def test_tie_block_closed_form(T):
    """T equal values straddling the boundary: the `above` larger values in
    value order, then the smallest (k - above) indices of the tie set."""
    k, L = 2048, 16384
    w = W.tie_block(2, L, k, T)
    s, st, ln = w.numpy()
    idx, _, _ = oracle.topk_ragged(s, st, ln, k)
    above = w.info["above"]
    for b in range(2):
        row = s[st[b]:st[b] + L]
        big = np.nonzero(row > 1.0)[0]
        big = big[np.argsort(-row[big], kind="stable")]
        ties = np.nonzero(row == 1.0)[0][:k - above]
        assert list(idx[b]) == list(big) + list(ties)


@pytest.mark.parametrize("m", [0, 256, 2047, 4095])
def test_plateau_closed_form(m):
    """m distinct positives, rest 0.0: positives in value order, then zeros in
    ascending index order, exactly k entries."""
    k, L = 2048, 8192
    w = W.plateau(2, L, m, k)
    s, st, ln = w.numpy()
    idx, _, _ = oracle.topk_ragged(s, st, ln, k)
    for b in range(2):
        row = s[st[b]:st[b] + L]
        pos = np.nonzero(row > 0)[0]
        pos = pos[np.argsort(-row[pos], kind="stable")]
        zeros = np.nonzero(row == 0)[0]
        assert list(idx[b]) == (list(pos) + list(zeros))[:k]


def test_offset_mode_shift():
    w = W.decode(B=3, lmin=3000, lmax=5000, k=512)
    s, st, ln = w.numpy()
    local, v0, _ = oracle.topk_ragged(s, st, ln, 512, 0)
    glob_, v1, _ = oracle.topk_ragged(s, st, ln, 512, 1)
    np.testing.assert_array_equal(glob_, np.where(local >= 0, local + st[:, None], -1))
    np.testing.assert_array_equal(v0.view(np.uint32), v1.view(np.uint32))


# --------------------------------------------------------------------------- #
# The -inf exclusion flag (offset_mode bit 2): -inf and every negative NaN
# are left out of the selection (the sglang page's torch-compatible backend,
# Modifications, leaves -inf scores out; the negative NaNs rank below -inf
# and go with them).
# --------------------------------------------------------------------------- #

def _bits(values):
    return np.array(values, dtype=np.uint32).view(np.float32)


def test_exclusion_closed_form():
    # [3, -inf, 1, -NaN, 2, -inf]: the three finite scores in value order,
    # then -1; values -inf in the padding.
    row = _bits([0x40400000, 0xFF800000, 0x3F800000, 0xFFC00000, 0x40000000, 0xFF800000])
    idx, val, _ = oracle.topk_ragged(row, np.array([0], np.int32), np.array([6], np.int32), 6,
                                     oracle.EXCLUDE_NEG_INF)
    assert list(idx[0]) == [0, 4, 2, -1, -1, -1]
    assert list(val[0].view(np.uint32)) == [0x40400000, 0x40000000, 0x3F800000] + [0xFF800000] * 3
    # Without the flag -inf ranks by its key above the negative NaN.
    idx, _, _ = oracle.topk_ragged(row, np.array([0], np.int32), np.array([6], np.int32), 6, 0)
    assert list(idx[0]) == [0, 4, 2, 1, 5, 3]


def test_exclusion_all_neg_inf_row():
    row = np.full(100, -np.inf, dtype=np.float32)
    idx, val, _ = oracle.topk_ragged(row, np.array([0], np.int32), np.array([100], np.int32), 64,
                                     oracle.EXCLUDE_NEG_INF | oracle.OFFSET_ROW_START)
    assert (idx == -1).all()
    assert (val.view(np.uint32) == 0xFF800000).all()


@pytest.mark.parametrize("mode", [oracle.EXCLUDE_NEG_INF, oracle.EXCLUDE_NEG_INF | oracle.OFFSET_ROW_START])
def test_exclusion_equals_selection_of_the_kept_entries(mode):
    """Flag on == the plain selection of the row with the excluded entries
    removed, indices mapped back: a second route to the same result."""
    rng = np.random.default_rng(29)
    alphabet = np.array([0xFF800000, 0xFFC00000, 0xFFC00123, 0x7FC00000, 0x80000000, 0,
                         0x3F800000, 0xBF800000, 0x7F800000, 0x40000000], dtype=np.uint32)
    for _ in range(300):
        L = int(rng.integers(0, 40))
        k = int(rng.integers(1, 48))
        start = int(rng.integers(0, 5))
        bits = rng.choice(alphabet, size=L)
        flat = np.concatenate([np.zeros(start, np.uint32), bits]).view(np.float32)
        got, _, _ = oracle.topk_ragged(flat, np.array([start], np.int32), np.array([L], np.int32), k, mode)
        keys = oracle.order_key(bits).astype(np.int64)
        neg_inf_key = int(oracle.order_key(np.array([0xFF800000], np.uint32))[0])
        keep = np.nonzero(keys > neg_inf_key)[0]
        sub = bits[keep].view(np.float32)
        ref, _, _ = oracle.topk_ragged(sub, np.array([0], np.int32), np.array([keep.size], np.int32), k, 0)
        ref = np.where(ref[0] >= 0, keep[np.maximum(ref[0], 0)], -1) if keep.size else ref[0]
        if mode & oracle.OFFSET_ROW_START:
            ref = np.where(ref >= 0, ref + start, -1)
        assert list(got[0]) == list(ref)


# --------------------------------------------------------------------------- #
# The page-table transform (the KV-cache slot of each selected index).
# --------------------------------------------------------------------------- #

def test_paged_slots_hand_case():
    # Selected [5, 0, 3, -1], pages of 2 entries, row pages [7, 2, 9]:
    # 5 -> page 9 offset 1 = 19; 0 -> page 7 offset 0 = 14; 3 -> page 2
    # offset 1 = 5.
    got = oracle.paged_slots(np.array([[5, 0, 3, -1]]), np.array([[7, 2, 9]]), 2)
    assert got.tolist() == [[19, 14, 5, -1]]


def test_paged_slots_identity_and_shared_table():
    rng = np.random.default_rng(3)
    idx = np.where(rng.random((4, 50)) < 0.2, -1, rng.integers(0, 64, (4, 50)))
    # One entry per page and pages 0, 1, 2, ...: slots are the indices.
    assert (oracle.paged_slots(idx, np.arange(64), 1) == idx).all()
    # 16 entries per page, identity pages: still the indices.
    assert (oracle.paged_slots(idx, np.tile(np.arange(4), (4, 1)), 16) == idx).all()


# --------------------------------------------------------------------------- #
# Invariants on arbitrary bit patterns, and thread-count independence.
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("alphabet", [None, [0, 0x80000000, 0x3F800000, 0x7FC00001,
                                             0xFFC00001, 0xFF800000]])
def test_invariants_random_bits(alphabet):
    k = 300
    w = W.random_bits(8, 2000, k, alphabet=alphabet)
    s, st, ln = w.numpy()
    idx, val, _ = oracle.topk_ragged(s, st, ln, k)
    bits = s.view(np.uint32)
    for b in range(8):
        row_bits = bits[st[b]:st[b] + ln[b]]
        sel = idx[b]
        assert np.all((sel >= 0) & (sel < ln[b]))
        assert np.unique(sel).size == k
        np.testing.assert_array_equal(val[b].view(np.uint32), row_bits[sel])
        # order tuples: selected multiset == the k best of the row, and in order
        t = [order_tuple(int(x)) for x in row_bits]
        best = sorted(t, reverse=True)[:k]
        got = [t[j] for j in sel]
        assert got == best
        # boundary ties are the smallest indices of the tie set
        boundary = got[-1]
        tie_idx = [j for j in range(len(t)) if t[j] == boundary]
        n_taken = sum(1 for x in got if x == boundary)
        assert [j for j in sel if t[j] == boundary] == tie_idx[:n_taken]


def test_thread_count_independent():
    w = W.decode(B=9, lmin=1000, lmax=20000, k=700)
    s, st, ln = w.numpy()
    a = oracle.topk_ragged(s, st, ln, 700, n_threads=1)
    b = oracle.topk_ragged(s, st, ln, 700, n_threads=4)
    for x, y in zip(a, b):
        assert x.tobytes() == y.tobytes()


def test_page_shape_set_equals_torch_topk():
    """The pages' standalone probe shape, [4, 4096] fp32 with k = 2048: on rows
    of distinct values the selected set equals torch.topk's set."""
    g = torch.Generator().manual_seed(4096)
    rows = (torch.randperm(4 * 4096, generator=g).float() - 8192.0).reshape(4, 4096) / 512
    assert torch.unique(rows).numel() == rows.numel()
    idx, _, _ = oracle.topk_ragged(rows.numpy().reshape(-1), np.arange(4) * 4096,
                                   np.full(4, 4096), 2048)
    ref = torch.topk(rows, 2048, dim=1).indices
    for b in range(4):
        assert set(idx[b].tolist()) == set(ref[b].tolist())
