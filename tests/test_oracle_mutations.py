"""The oracle's pins catch plausible mistakes.

Each case compiles a copy of the oracle with one deliberate slip planted in it
(on the CPU, in a temporary directory) and checks that the pin suite's
independent checks reject it.  The shipped oracle itself passes the same
checks in test_oracle.py.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTATIONS = {
    "tie_index_descending": ("return a->idx < b->idx ? -1 : 1;", "return a->idx > b->idx ? -1 : 1;"),
    "key_ascending": ("return a->key > b->key ? -1 : 1;", "return a->key < b->key ? -1 : 1;"),
    "negative_branch_sign_flip": ("return ~bits;", "return bits ^ 0x80000000u;"),
    "positive_branch_no_or": ("return bits | 0x80000000u;", "return bits;"),
    "pad_value_zero": ("neg_inf_bits = 0xFF800000u", "neg_inf_bits = 0x00000000u"),
    "offset_ignored": ("(job->offset_mode & ORACLE_OFFSET_ROW_START) ? (int32_t)(start + j) : j", "j"),
    "exclusion_ignored": ("if (exclude && key <= neg_inf_key)", "if (0)"),
    "one_short": ("int32_t n = m < job->k ? (int32_t)m : job->k;",
                  "int32_t n = m < job->k ? (int32_t)m : job->k - 1;"),
    "length_envelope_off": ("if (len >= ORACLE_MAX_LEN)", "if (len > ORACLE_MAX_LEN)"),
}


def _build_mutant(tmp_path, name):
    before, after = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(before, after))
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-pthread", str(path),
                    "-o", str(lib)], check=True)
    so = ctypes.CDLL(str(lib))
    so.oracle_topk_ragged.argtypes = [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int]
    return so


def _call(so, flat_bits, starts, lengths, k, mode):
    flat = np.ascontiguousarray(flat_bits, dtype=np.uint32)
    starts = np.ascontiguousarray(starts, dtype=np.int32)
    lengths = np.ascontiguousarray(lengths, dtype=np.int32)
    B = starts.size
    idx = np.empty((B, k), dtype=np.int32)
    val = np.empty((B, k), dtype=np.uint32)
    flags = np.empty(B, dtype=np.uint32)
    so.oracle_topk_ragged(flat.ctypes.data, flat.size, starts.ctypes.data, lengths.ctypes.data,
                          B, k, mode, idx.ctypes.data, val.ctypes.data, flags.ctypes.data, 1)
    return idx, val, flags


def _pins_pass(so):
    """A compact run of independent pins; False as soon as one rejects."""
    from test_oracle import GOLDEN, _parse_golden, brute_force_topk
    for path in GOLDEN:
        g = _parse_golden(path)
        k, mode, start = int(g["k"]), int(g["offset_mode"]), int(g["row_start"])
        row = [int(x, 16) for x in g["scores"].split()]
        flat = np.zeros(start + len(row) + 3, dtype=np.uint32)
        flat[start:start + len(row)] = row
        idx, val, _ = _call(so, flat, [start], [len(row)], k, mode)
        if list(idx[0]) != [int(x) for x in g["expected_idx"].split()]:
            return False
        if list(val[0]) != [int(x, 16) for x in g["expected_val"].split()]:
            return False
    rng = np.random.default_rng(3)
    alphabet = np.array([0x7FC00000, 0xFFC00000, 0xFF800000, 0xBF800000, 0x80000000, 0,
                         0x3F800000, 0x40000000, 0xC0000000, 0x7F800000], dtype=np.uint32)
    rows = [rng.choice(alphabet, size=int(rng.integers(0, 12))) for _ in range(200)]
    lengths = np.array([len(r) for r in rows])
    starts = np.cumsum(lengths) - lengths
    flat = np.concatenate(rows).astype(np.uint32)
    for k in (1, 4, 9):
        idx, _, _ = _call(so, flat, starts, lengths, k, 0)
        for r, row in enumerate(rows):
            if list(idx[r]) != brute_force_topk([int(b) for b in row], k):
                return False
    # Exclusion of -inf and negative NaN (offset_mode bit 2), with and
    # without the row-start offset: [3, -inf, 1, -NaN, 2, -inf], k = 6.
    row = np.array([0x40400000, 0xFF800000, 0x3F800000, 0xFFC00000, 0x40000000, 0xFF800000],
                   dtype=np.uint32)
    flat = np.concatenate([np.zeros(5, np.uint32), row])
    for mode, want in ((2, [0, 4, 2, -1, -1, -1]), (3, [5, 9, 7, -1, -1, -1]),
                       (0, [0, 4, 2, 1, 5, 3])):
        idx, _, _ = _call(so, flat, [5], [6], 6, mode)
        if list(idx[0]) != want:
            return False
    ones = np.ones(64, dtype=np.float32).view(np.uint32)
    _, _, flags = _call(so, ones, [0, 0], [1 << 24, 4], 2, 0)
    if list(flags) != [oracle.FLAG_LEN_ENVELOPE, 0]:
        return False
    return True


def test_shipped_oracle_passes_compact_pins(tmp_path):
    src = open(SRC).read()
    path = tmp_path / "same.c"
    path.write_text(src)
    lib = tmp_path / "libsame.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-pthread", str(path),
                    "-o", str(lib)], check=True)
    so = ctypes.CDLL(str(lib))
    so.oracle_topk_ragged.argtypes = [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int]
    assert _pins_pass(so)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    assert not _pins_pass(_build_mutant(tmp_path, name))
