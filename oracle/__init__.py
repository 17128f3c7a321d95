"""CPU oracle for deterministic exact ragged top-k (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference arm may import this package.  The product path (the CUDA library and
its Python binding) never touches it, and the oracle shares no code with that
path: ``oracle.c`` is compiled on its own with the host C compiler.

Every function pins to the definition in sglang PR #31115 "Add opt-in
deterministic CuTe-DSL DSA top-k backend" (PR summary, hardening commit,
Modifications): canonical order score desc / index asc on bitwise-equal
scores under the bitwise total order of fp32 patterns, front-packed output,
-1 padding.  The pinning tests live in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

FLAG_LEN_ENVELOPE = 1
FLAG_BAD_WINDOW = 2
# offset_mode bits
OFFSET_ROW_START = 1
EXCLUDE_NEG_INF = 2   # leave out -inf and every negative NaN
PAD_VALUE_BITS = 0xFF800000


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library beside it (host C compiler)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-shared", "-fPIC",
           "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_order_key.argtypes = [ctypes.c_uint32]
            lib.oracle_order_key.restype = ctypes.c_uint32
            lib.oracle_order_key_batch.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_int64]
            lib.oracle_order_key_batch.restype = None
            lib.oracle_topk_ragged.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_topk_ragged.restype = ctypes.c_int
            _lib = lib
    return _lib


def order_key(bits: np.ndarray) -> np.ndarray:
    """Order keys of fp32 bit patterns (uint32 in, uint32 out)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint32)
    out = np.empty_like(bits)
    _load().oracle_order_key_batch(bits.ctypes.data, out.ctypes.data, bits.size)
    return out


def topk_ragged(scores: np.ndarray, row_starts: np.ndarray, lengths: np.ndarray,
                k: int, offset_mode: int = 0, n_threads: int = 1,
                with_values: bool = True):
    """Oracle top-k over a flat ragged fp32 buffer.

    Returns ``(out_idx int32[B, k], out_val float32[B, k] or None,
    row_flags uint32[B])``.  Bit patterns of ``out_val`` are the input's.
    """
    scores = np.ascontiguousarray(scores, dtype=np.float32).reshape(-1)
    row_starts = np.ascontiguousarray(row_starts, dtype=np.int32).reshape(-1)
    lengths = np.ascontiguousarray(lengths, dtype=np.int32).reshape(-1)
    B = row_starts.size
    if lengths.size != B:
        raise ValueError("row_starts and lengths differ in size")
    out_idx = np.empty((B, k), dtype=np.int32)
    out_val = np.empty((B, k), dtype=np.float32) if with_values else None
    flags = np.empty(B, dtype=np.uint32)
    rc = _load().oracle_topk_ragged(
        scores.ctypes.data if scores.size else None, scores.size,
        row_starts.ctypes.data, lengths.ctypes.data, B, k, offset_mode,
        out_idx.ctypes.data, out_val.ctypes.data if with_values else None,
        flags.ctypes.data, int(n_threads))
    if rc == -1:
        raise ValueError(f"oracle: invalid argument (k={k}, offset_mode={offset_mode})")
    if rc != 0:
        raise MemoryError("oracle: worker allocation failed")
    return out_idx, out_val, flags


def paged_slots(out_idx: np.ndarray, page_table: np.ndarray, page_size: int) -> np.ndarray:
    """The page-table transform written out: row i's selected in-row index j
    becomes page_table[i, j // page_size] * page_size + j % page_size, and -1
    stays -1.  page_table is [B, P], or [P] shared by every row."""
    out_idx = np.asarray(out_idx, dtype=np.int64)
    pt = np.asarray(page_table, dtype=np.int64)
    if pt.ndim == 1:
        pt = np.broadcast_to(pt, (out_idx.shape[0], pt.size))
    j = np.maximum(out_idx, 0)
    rows = np.arange(out_idx.shape[0])[:, None]
    slots = pt[rows, j // page_size] * page_size + j % page_size
    return np.where(out_idx >= 0, slots, -1).astype(np.int32)


# --- tie / plateau statistics at the k-th boundary ----------------------------
# Fields of one row of row_stats(), in order.
ROW_STATS_FIELDS = ("len", "n_zero", "boundary_bits", "tie", "above", "flags")
STAT_HAS_BOUNDARY = 1   # L > k: the row has a k-th entry
STAT_STRADDLE = 2       # the tie set of the boundary crosses position k
STAT_ZERO_BOUND = 4     # the boundary score is 0.0 (either sign)
MAX_LEN = 1 << 24


def row_stats(scores: np.ndarray, row_starts: np.ndarray, lengths: np.ndarray, k: int):
    """Per-row statistics of the k-th boundary, as the sglang page's score
    statistics script defines them (its row_stats: plateau fraction, the k-th
    largest score, the size of its tie set, the count strictly above it, and
    whether the tie set straddles position k or the boundary sits on 0.0),
    written out on the same bitwise order as the selection (C1, C2): the
    boundary is the k-th entry in canonical order, "tie" counts the entries
    bitwise equal to it and "above" those with a larger order key.  n_zero
    counts the entries whose value is 0.0 (+0.0 or -0.0).

    A row with L <= k has no boundary: (L, n_zero, 0, 0, L, 0).  Window and
    length checks are topk_ragged's; a rejected row is all zero and its flag
    is set in the returned row_flags.

    Returns ``(stats uint32[B, 6] in ROW_STATS_FIELDS order, row_flags uint32[B])``.
    """
    if not 1 <= k <= 4096:
        raise ValueError(f"k={k} outside [1, 4096]")
    bits = np.ascontiguousarray(scores, dtype=np.float32).reshape(-1).view(np.uint32)
    row_starts = np.asarray(row_starts, dtype=np.int64).reshape(-1)
    lengths = np.asarray(lengths, dtype=np.int64).reshape(-1)
    B = row_starts.size
    out = np.zeros((B, 6), dtype=np.uint32)
    row_flags = np.zeros(B, dtype=np.uint32)
    for i in range(B):
        L = max(int(lengths[i]), 0)
        s0 = int(row_starts[i])
        if L >= MAX_LEN:
            row_flags[i] = FLAG_LEN_ENVELOPE
            continue
        if s0 < 0 or s0 + L > bits.size:
            row_flags[i] = FLAG_BAD_WINDOW
            continue
        b = bits[s0:s0 + L]
        n_zero = int(np.count_nonzero((b & 0x7FFFFFFF) == 0))
        if L <= k:
            out[i] = (L, n_zero, 0, 0, L, 0)
            continue
        key = order_key(b)
        T = np.sort(key)[::-1][k - 1]          # the k-th key in canonical order
        tie = int(np.count_nonzero(key == T))
        above = int(np.count_nonzero(key > T))
        bb = int(b[np.flatnonzero(key == T)[0]])   # the key is a bijection: one pattern
        flags = STAT_HAS_BOUNDARY
        if tie > 1 and above + tie > k:
            flags |= STAT_STRADDLE
        if bb & 0x7FFFFFFF == 0:
            flags |= STAT_ZERO_BOUND
        out[i] = (L, n_zero, bb, tie, above, flags)
    return out, row_flags


# --- the lightning-indexer scores that feed the selection ----------------------
INDEXER_HEADS = 64
INDEXER_DIM = 128


def indexer_scores(q: np.ndarray, w: np.ndarray, bias, keys: np.ndarray, key_starts: np.ndarray,
                   lengths: np.ndarray, score_starts: np.ndarray, n_scores: int, scale: float):
    """The indexer scores of the DSA lightning indexer as the pages state
    them (the decode batch of the vLLM / sglang pages' workloads: each
    key t of row i scores s_t = sum over heads h of w[i, h] *
    relu(scale * q[i, h] . k_t + b_i), with 64 heads of dimension 128; b_i is
    an optional per-row logit shift, 0 for the plain indexer), in float64
    from the given (bf16-valued) inputs.

    Row i reads keys[key_starts[i] : key_starts[i] + L_i] and its scores go
    to [score_starts[i], score_starts[i] + L_i) of an n_scores buffer.
    Returns (scores float64[n_scores], written bool[n_scores]).  A row whose
    windows leave [0, len(keys)) or [0, n_scores), or whose length is at
    least 2^24, writes nothing.
    """
    q = np.asarray(q, dtype=np.float64).reshape(-1, INDEXER_HEADS, INDEXER_DIM)
    w = np.asarray(w, dtype=np.float64).reshape(-1, INDEXER_HEADS)
    keys = np.asarray(keys, dtype=np.float64).reshape(-1, INDEXER_DIM)
    B = q.shape[0]
    b = np.zeros(B) if bias is None else np.asarray(bias, dtype=np.float64).reshape(-1)
    out = np.zeros(n_scores, dtype=np.float64)
    written = np.zeros(n_scores, dtype=bool)
    for i in range(B):
        L = max(int(lengths[i]), 0)
        ks, ss = int(key_starts[i]), int(score_starts[i])
        if L == 0 or L >= MAX_LEN or ks < 0 or ks + L > keys.shape[0] or ss < 0 or ss + L > n_scores:
            continue
        logits = scale * (keys[ks:ks + L] @ q[i].T) + b[i]          # [L, H]
        out[ss:ss + L] = np.maximum(logits, 0.0) @ w[i]
        written[ss:ss + L] = True
    return out, written
