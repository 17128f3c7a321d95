"""Python binding of the C ABI in ``include/topk_ragged.h``.

Argument marshalling only: tensors are checked (dtype, device, layout) and
their device pointers, sizes and the current CUDA stream are passed to the
library.  Every step of the selection runs in the library's kernels; output
tensors are allocated here with torch only when the caller does not pass them
(the library call itself allocates nothing).
"""
from __future__ import annotations

import ctypes

import torch

from ._native import LaunchInfo, TopkError, lib

TOPK_OFFSET_ROW_LOCAL = 0
TOPK_OFFSET_ROW_START = 1
TOPK_EXCLUDE_NEG_INF = 2   # or-ed into offset_mode: leave out -inf and negative NaN
TOPK_DEV_LEN_ENVELOPE = 1
TOPK_DEV_BAD_WINDOW = 2
TOPK_DEV_INTERNAL = 4
# topk_row_stats: six 32-bit fields per row, and its flag bits
ROW_STATS_FIELDS = ("len", "n_zero", "boundary_bits", "tie", "above", "flags")
TOPK_STAT_HAS_BOUNDARY = 1
TOPK_STAT_STRADDLE = 2
TOPK_STAT_ZERO_BOUND = 4
MAX_K = 4096
MAX_LEN = 1 << 24
PAD_VALUE_BITS = 0xFF800000
_STATUS_INVALID_ARG = 1   # TOPK_ERR_INVALID_ARG


def _device(device) -> torch.device:
    """The CUDA device named by `device` (an index, a string or a torch.device);
    None or a bare "cuda" is the current one."""
    d = torch.device("cuda", device) if isinstance(device, int) else torch.device(device or "cuda")
    if d.type != "cuda":
        raise ValueError(f"expected a CUDA device, got {d}")
    return d if d.index is not None else torch.device("cuda", torch.cuda.current_device())


def _check_k(k: int, B: int, what: str) -> None:
    """The library's own k and B * k limits, checked before an output of B * k
    entries is allocated for a call that would be refused."""
    if not 1 <= int(k) <= MAX_K or B * int(k) >= 1 << 31:
        raise TopkError(_STATUS_INVALID_ARG, f"{what} (k = {k}, B = {B})")


def _stream_handle(device: torch.device, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(t: torch.Tensor, name: str, dtype, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor, got {t.device}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _outputs(out_idx, out_val, with_values: bool, B: int, k: int, dev, what: str):
    """The selection's outputs: the caller's, checked to hold B * k entries,
    or new ones."""
    _check_k(k, B, what)
    if out_idx is None:
        out_idx = torch.empty((B, k), dtype=torch.int32, device=dev)
    else:
        _check(out_idx, "out_idx", torch.int32, dev)
        if out_idx.numel() != B * k:
            raise ValueError("out_idx must hold B * k entries")
    if out_val is None and with_values:
        out_val = torch.empty((B, k), dtype=torch.float32, device=dev)
    elif out_val is not None:
        _check(out_val, "out_val", torch.float32, dev)
        if out_val.numel() != B * k:
            raise ValueError("out_val must hold B * k entries")
    return out_idx, out_val


def init(device=None) -> None:
    """Prepare a device (outside stream capture); see topk_ragged_init."""
    dev = _device(device)
    with torch.cuda.device(dev):
        rc = lib().topk_ragged_init(dev.index)
    if rc != 0:
        raise TopkError(rc, "topk_ragged_init")


def topk_ragged(scores: torch.Tensor, row_starts: torch.Tensor, lengths: torch.Tensor,
                k: int = 2048, offset_mode: int = TOPK_OFFSET_ROW_LOCAL,
                out_idx: torch.Tensor | None = None, out_val: torch.Tensor | None = None,
                with_values: bool = False, stream=None, page_table: torch.Tensor | None = None,
                page_size: int = 1):
    """Deterministic exact top-k of each ragged row of a flat fp32 buffer.

    scores      float32 CUDA tensor (any shape, contiguous; used as flat).
    row_starts  int32 CUDA tensor [B]; lengths int32 CUDA tensor [B].
    page_table  optional int32 CUDA tensor [B, P] (or [P], shared by every
                row): the selected indices are written as KV-cache slots
                page_table[i, j // page_size] * page_size + j % page_size
                (topk_ragged_paged); offset_mode may then only carry
                TOPK_EXCLUDE_NEG_INF.
    Returns (out_idx int32 [B, k], out_val float32 [B, k] or None).
    """
    _check(scores, "scores", torch.float32)
    dev = scores.device
    _check(row_starts, "row_starts", torch.int32, dev)
    _check(lengths, "lengths", torch.int32, dev)
    B = row_starts.numel()
    if lengths.numel() != B:
        raise ValueError(f"row_starts has {B} entries, lengths has {lengths.numel()}")
    if page_table is not None:
        _check(page_table, "page_table", torch.int32, dev)
        if page_table.dim() > 2 or (page_table.dim() == 2 and page_table.shape[0] != B):
            raise ValueError("page_table must be [B, pages] (one row per query row) or [pages] (shared)")
    out_idx, out_val = _outputs(out_idx, out_val, with_values, B, k, dev,
                                "topk_ragged" if page_table is None else "topk_ragged_paged")
    common = (scores.data_ptr() if scores.numel() else None, scores.numel(),
              row_starts.data_ptr() if B else None, lengths.data_ptr() if B else None,
              B, int(k), int(offset_mode))
    tail = (out_idx.data_ptr() if B else None, out_val.data_ptr() if (out_val is not None and B) else None,
            _stream_handle(dev, stream))
    with torch.cuda.device(dev):
        if page_table is None:
            rc = lib().topk_ragged(*common, *tail)
            name = "topk_ragged"
        else:
            stride = page_table.shape[-1] if page_table.dim() == 2 else 0
            rc = lib().topk_ragged_paged(*common, page_table.data_ptr() if page_table.numel() else None,
                                         stride, int(page_size), *tail)
            name = "topk_ragged_paged"
    if rc != 0:
        raise TopkError(rc, name)
    return out_idx, out_val


def topk_ragged_stats(scores: torch.Tensor, row_starts: torch.Tensor, lengths: torch.Tensor,
                      k: int = 2048, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Tie / plateau statistics of each row at its k-th boundary.

    Returns an int32 CUDA tensor [B, 6] holding topk_row_stats per row, in
    ROW_STATS_FIELDS order; every field is an unsigned 32-bit value (read
    boundary_bits as the fp32 pattern of the k-th score).
    """
    _check(scores, "scores", torch.float32)
    dev = scores.device
    _check(row_starts, "row_starts", torch.int32, dev)
    _check(lengths, "lengths", torch.int32, dev)
    B = row_starts.numel()
    if lengths.numel() != B:
        raise ValueError(f"row_starts has {B} entries, lengths has {lengths.numel()}")
    if out is None:
        out = torch.empty((B, len(ROW_STATS_FIELDS)), dtype=torch.int32, device=dev)
    else:
        _check(out, "out", torch.int32, dev)
        if out.numel() != B * len(ROW_STATS_FIELDS):
            raise ValueError("out must hold B * 6 entries")
    with torch.cuda.device(dev):
        rc = lib().topk_ragged_stats(scores.data_ptr() if scores.numel() else None, scores.numel(),
                                     row_starts.data_ptr() if B else None, lengths.data_ptr() if B else None,
                                     B, int(k), out.data_ptr() if B else None, _stream_handle(dev, stream))
    if rc != 0:
        raise TopkError(rc, "topk_ragged_stats")
    return out


INDEXER_HEADS = 64
INDEXER_DIM = 128


def _indexer_args(q, w, keys, key_starts, lengths, score_starts, bias, scale):
    _check(q, "q", torch.bfloat16)
    dev = q.device
    _check(w, "w", torch.float32, dev)
    _check(keys, "keys", torch.bfloat16, dev)
    for t, name in ((key_starts, "key_starts"), (lengths, "lengths"), (score_starts, "score_starts")):
        _check(t, name, torch.int32, dev)
    B = key_starts.numel()
    if q.numel() != B * INDEXER_HEADS * INDEXER_DIM or w.numel() != B * INDEXER_HEADS:
        raise ValueError(f"q must be [B, {INDEXER_HEADS}, {INDEXER_DIM}] and w [B, {INDEXER_HEADS}]")
    if lengths.numel() != B or score_starts.numel() != B:
        raise ValueError("key_starts, lengths and score_starts differ in size")
    if keys.numel() % INDEXER_DIM:
        raise ValueError(f"keys must be [n_keys, {INDEXER_DIM}]")
    for t, name in ((q, "q"), (keys, "keys"), (w, "w")):
        if t.numel() and t.data_ptr() % 16:
            raise ValueError(f"{name} must start on a 16-byte boundary (the TMA and vector loads need it)")
    if bias is not None:
        _check(bias, "bias", torch.float32, dev)
        if bias.numel() != B:
            raise ValueError("bias must hold B entries")
    scale = 1.0 / INDEXER_DIM ** 0.5 if scale is None else float(scale)
    return dev, B, scale


def indexer_scores(q: torch.Tensor, w: torch.Tensor, keys: torch.Tensor, key_starts: torch.Tensor,
                   lengths: torch.Tensor, score_starts: torch.Tensor, n_scores: int | None = None,
                   scale: float | None = None, bias: torch.Tensor | None = None,
                   out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Lightning-indexer scores on the tensor cores (topk_ragged_indexer_scores).

    q bf16 [B, 64, 128], w fp32 [B, 64], keys bf16 [n_keys, 128], bias fp32
    [B] or None, key_starts / lengths / score_starts int32 [B]; scale defaults
    to 1/sqrt(128).  Writes row i's scores to out[score_starts[i] + j] and
    returns out (fp32 [n_scores], allocated with zeros when not given).
    """
    dev, B, scale = _indexer_args(q, w, keys, key_starts, lengths, score_starts, bias, scale)
    if out is None:
        if n_scores is None:
            raise ValueError("give n_scores or out")
        out = torch.zeros(int(n_scores), dtype=torch.float32, device=dev)
    else:
        _check(out, "out", torch.float32, dev)
    with torch.cuda.device(dev):
        rc = lib().topk_ragged_indexer_scores(
            q.data_ptr() if B else None, w.data_ptr() if B else None,
            bias.data_ptr() if (bias is not None and B) else None, keys.data_ptr() if keys.numel() else None,
            keys.numel() // INDEXER_DIM, key_starts.data_ptr() if B else None, lengths.data_ptr() if B else None,
            score_starts.data_ptr() if B else None, B, scale, out.data_ptr() if out.numel() else None,
            out.numel(), _stream_handle(dev, stream))
    if rc != 0:
        raise TopkError(rc, "topk_ragged_indexer_scores")
    return out


def topk_ragged_indexer(q: torch.Tensor, w: torch.Tensor, keys: torch.Tensor, key_starts: torch.Tensor,
                        lengths: torch.Tensor, score_starts: torch.Tensor, k: int = 2048, flags: int = 0,
                        scale: float | None = None, bias: torch.Tensor | None = None,
                        scores: torch.Tensor | None = None, n_scores: int | None = None,
                        out_idx: torch.Tensor | None = None, out_val: torch.Tensor | None = None,
                        with_values: bool = False, stream=None):
    """Indexer scores, then the deterministic top-k over them
    (topk_ragged_indexer).  `scores` is the caller's scratch (allocated when
    not given).  Returns (out_idx, out_val or None, scores)."""
    dev, B, scale = _indexer_args(q, w, keys, key_starts, lengths, score_starts, bias, scale)
    if scores is None:
        if n_scores is None:
            raise ValueError("give n_scores or scores")
        scores = torch.zeros(int(n_scores), dtype=torch.float32, device=dev)
    else:
        _check(scores, "scores", torch.float32, dev)
    out_idx, out_val = _outputs(out_idx, out_val, with_values, B, k, dev, "topk_ragged_indexer")
    with torch.cuda.device(dev):
        rc = lib().topk_ragged_indexer(
            q.data_ptr() if B else None, w.data_ptr() if B else None,
            bias.data_ptr() if (bias is not None and B) else None, keys.data_ptr() if keys.numel() else None,
            keys.numel() // INDEXER_DIM, key_starts.data_ptr() if B else None, lengths.data_ptr() if B else None,
            score_starts.data_ptr() if B else None, B, scale, scores.data_ptr() if scores.numel() else None,
            scores.numel(), int(k), int(flags), out_idx.data_ptr() if B else None,
            out_val.data_ptr() if (out_val is not None and B) else None, _stream_handle(dev, stream))
    if rc != 0:
        raise TopkError(rc, "topk_ragged_indexer")
    return out_idx, out_val, scores


STATIC_SCORES = 1 << 23   # TOPK_RAGGED_STATIC_SCORES: scores the library's own array holds


def topk_ragged_indexer_static(q: torch.Tensor, w: torch.Tensor, keys: torch.Tensor, key_starts: torch.Tensor,
                               lengths: torch.Tensor, score_starts: torch.Tensor, n_scores: int, k: int = 2048,
                               flags: int = 0, scale: float | None = None, bias: torch.Tensor | None = None,
                               out_idx: torch.Tensor | None = None, out_val: torch.Tensor | None = None,
                               with_values: bool = False, stream=None):
    """The indexer chain with its scores in the library's own fixed array
    (topk_ragged_indexer_static), for callers that cannot allocate device
    memory: such a caller passes out_idx (and out_val) and nothing is
    allocated; n_scores (at most STATIC_SCORES) bounds the score windows that
    score_starts lays out in the array.  Returns (out_idx, out_val or None)."""
    dev, B, scale = _indexer_args(q, w, keys, key_starts, lengths, score_starts, bias, scale)
    out_idx, out_val = _outputs(out_idx, out_val, with_values, B, k, dev, "topk_ragged_indexer_static")
    with torch.cuda.device(dev):
        rc = lib().topk_ragged_indexer_static(
            q.data_ptr() if B else None, w.data_ptr() if B else None,
            bias.data_ptr() if (bias is not None and B) else None, keys.data_ptr() if keys.numel() else None,
            keys.numel() // INDEXER_DIM, key_starts.data_ptr() if B else None, lengths.data_ptr() if B else None,
            score_starts.data_ptr() if B else None, B, scale, int(n_scores), int(k), int(flags),
            out_idx.data_ptr() if B else None, out_val.data_ptr() if (out_val is not None and B) else None,
            _stream_handle(dev, stream))
    if rc != 0:
        raise TopkError(rc, "topk_ragged_indexer_static")
    return out_idx, out_val


def device_status(device=None, stream=None) -> int:
    """Read and clear the device status word (synchronises the stream)."""
    dev = _device(device)
    v = ctypes.c_uint32(0)
    with torch.cuda.device(dev):
        rc = lib().topk_ragged_device_status(ctypes.byref(v), _stream_handle(dev, stream))
    if rc != 0:
        raise TopkError(rc, "topk_ragged_device_status")
    return int(v.value)


def wait_probe(polls: int = 4096, device=None, stream=None) -> None:
    """Launch the bounded-wait diagnostic: one CTA waits, with the kernels'
    own bounded wait (``polls`` polls per bound), on an mbarrier that nothing
    completes, so that the next device_status() reads TOPK_DEV_INTERNAL."""
    dev = _device(device)
    with torch.cuda.device(dev):
        rc = lib().topk_ragged_wait_probe(int(polls), _stream_handle(dev, stream))
    if rc != 0:
        raise TopkError(rc, "topk_ragged_wait_probe")


def launch_info(n_scores: int, B: int, k: int, device=None) -> dict:
    """How a call with (n_scores, B, k) is launched on the device: threads,
    cluster, grid, ..."""
    dev = _device(device)
    info = LaunchInfo()
    with torch.cuda.device(dev):
        rc = lib().topk_ragged_launch_info(int(n_scores), int(B), int(k), ctypes.byref(info))
    if rc != 0:
        raise TopkError(rc, "topk_ragged_launch_info")
    return {name: int(getattr(info, name)) for name, _ in LaunchInfo._fields_}
