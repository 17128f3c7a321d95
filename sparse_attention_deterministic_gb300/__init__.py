"""Deterministic exact ragged top-k for GB300 (sm_103a).

The selection step of a sparse-attention lightning indexer: per ragged row of
fp32 scores, the k best positions in canonical order (score descending under
the bitwise fp32 total order, index ascending on bitwise-equal scores),
-1 padded.  The work runs in the CUDA library built from ``csrc/`` and exposed
through the C ABI in ``include/topk_ragged.h``; this package only builds,
loads and calls it.
"""
from ._native import EXPORTS, LIB_PATH, TopkError, build, lib, strerror
from .binding import (MAX_K, MAX_LEN, PAD_VALUE_BITS, ROW_STATS_FIELDS, TOPK_DEV_BAD_WINDOW,
                      TOPK_DEV_INTERNAL, TOPK_DEV_LEN_ENVELOPE, TOPK_OFFSET_ROW_LOCAL,
                      TOPK_EXCLUDE_NEG_INF, TOPK_OFFSET_ROW_START, TOPK_STAT_HAS_BOUNDARY,
                      TOPK_STAT_STRADDLE, TOPK_STAT_ZERO_BOUND, INDEXER_DIM, INDEXER_HEADS, device_status,
                      indexer_scores, init, launch_info, topk_ragged, topk_ragged_indexer, topk_ragged_stats,
                      STATIC_SCORES, topk_ragged_indexer_static, wait_probe)

__all__ = [
    "EXPORTS", "LIB_PATH", "TopkError", "build", "lib", "strerror", "MAX_K", "MAX_LEN",
    "PAD_VALUE_BITS", "TOPK_DEV_BAD_WINDOW", "TOPK_DEV_INTERNAL", "TOPK_DEV_LEN_ENVELOPE",
    "TOPK_OFFSET_ROW_LOCAL", "TOPK_OFFSET_ROW_START", "TOPK_EXCLUDE_NEG_INF", "device_status", "init",
    "launch_info", "ROW_STATS_FIELDS", "TOPK_STAT_HAS_BOUNDARY", "TOPK_STAT_STRADDLE",
    "TOPK_STAT_ZERO_BOUND", "topk_ragged", "topk_ragged_stats", "INDEXER_HEADS", "INDEXER_DIM",
    "indexer_scores", "topk_ragged_indexer", "STATIC_SCORES", "topk_ragged_indexer_static", "wait_probe",
]
