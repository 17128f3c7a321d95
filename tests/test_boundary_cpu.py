"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol the header declares, and rejects out-of-contract arguments before
touching the device."""
import ctypes
import os
import re

import pytest

import sparse_attention_deterministic_gb300 as pkg
from sparse_attention_deterministic_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def so():
    pkg.build()
    return pkg.lib()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(topk_ragged\w*)\s*\(", text)
    return sorted(set(names))


def test_exports_every_declared_symbol(so):
    declared = _declared_functions()
    assert declared, "no declarations found"
    assert set(declared) == set(_native.EXPORTS)
    for name in declared:
        assert hasattr(so, name), name


def test_abi_version_and_strerror(so):
    assert so.topk_ragged_abi_version() == 4
    for st in range(5):
        assert pkg.strerror(st)
    assert pkg.strerror(99) == "unknown status"


def _call(so, scores=0x1000, n=16, rs=0x2000, ln=0x3000, B=1, k=4, mode=0, oi=0x4000):
    return so.topk_ragged(scores, n, rs, ln, B, k, mode, oi, None, None)


@pytest.mark.parametrize("kw", [
    dict(k=0), dict(k=4097), dict(k=-1), dict(B=-1), dict(mode=4), dict(mode=-1),
    dict(rs=None), dict(ln=None), dict(oi=None), dict(scores=None),
    dict(scores=0x1002), dict(n=-1), dict(n=1 << 31), dict(B=1 << 20, k=4096),
])
def test_invalid_arguments_rejected_on_host(so, kw):
    # Pointers here are never dereferenced: validation fails first.
    assert _call(so, **kw) == 1


@pytest.mark.parametrize("args", [
    (0x1000, 16, 0x2000, 0x3000, 1, 0, 0x4000), (0x1000, 16, 0x2000, 0x3000, 1, 4097, 0x4000),
    (0x1000, 16, 0x2000, 0x3000, -1, 4, 0x4000), (0x1000, 16, None, 0x3000, 1, 4, 0x4000),
    (0x1000, 16, 0x2000, None, 1, 4, 0x4000), (0x1000, 16, 0x2000, 0x3000, 1, 4, None),
    (None, 16, 0x2000, 0x3000, 1, 4, 0x4000), (0x1002, 16, 0x2000, 0x3000, 1, 4, 0x4000),
    (0x1000, -1, 0x2000, 0x3000, 1, 4, 0x4000), (0x1000, 1 << 31, 0x2000, 0x3000, 1, 4, 0x4000),
])
def test_stats_invalid_arguments_rejected_on_host(so, args):
    assert so.topk_ragged_stats(*args, None) == 1


def test_stats_empty_batch_and_header_flags(so):
    assert so.topk_ragged_stats(None, 0, None, None, 0, 2048, None, None) == 0
    text = open(os.path.join(ROOT, "include", "topk_ragged.h")).read()
    assert re.search(r"TOPK_STAT_HAS_BOUNDARY = 1u", text) and pkg.TOPK_STAT_HAS_BOUNDARY == 1
    assert re.search(r"TOPK_STAT_STRADDLE = 2u", text) and pkg.TOPK_STAT_STRADDLE == 2
    assert re.search(r"TOPK_STAT_ZERO_BOUND = 4u", text) and pkg.TOPK_STAT_ZERO_BOUND == 4
    fields = re.search(r"typedef struct \{(.*?)\} topk_row_stats;", text, re.S).group(1)
    assert re.findall(r"uint32_t (\w+);", fields) == list(pkg.ROW_STATS_FIELDS)


def test_empty_batch_is_ok_without_device(so):
    assert _call(so, B=0, rs=None, ln=None, oi=None, scores=None, n=0) == 0


def test_device_status_null(so):
    assert so.topk_ragged_device_status(None, None) == 1


def test_launch_info_null(so):
    assert so.topk_ragged_launch_info(16384, 4, 2048, None) == 1


def test_header_defines_match_binding():
    text = open(os.path.join(ROOT, "include", "topk_ragged.h")).read()
    assert "#define TOPK_RAGGED_MAX_K 4096" in text
    assert pkg.MAX_K == 4096 and pkg.MAX_LEN == 1 << 24
    assert re.search(r"TOPK_DEV_LEN_ENVELOPE = 1u", text)
    assert re.search(r"TOPK_DEV_BAD_WINDOW = 2u", text)
    assert re.search(r"TOPK_DEV_INTERNAL = 4u", text)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_native, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_native, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _native.lib()


def _ix_args(**kw):
    a = dict(q=0x10000, w=0x20000, bias=None, keys=0x30000, n_keys=100, ks=0x40000, ln=0x50000, ss=0x60000,
             B=2, scale=0.088, scores=0x70000, n_scores=1000)
    a.update(kw)
    return (a["q"], a["w"], a["bias"], a["keys"], a["n_keys"], a["ks"], a["ln"], a["ss"], a["B"], a["scale"],
            a["scores"], a["n_scores"])


@pytest.mark.parametrize("kw", [
    dict(B=-1), dict(n_keys=0), dict(n_keys=1 << 31), dict(n_keys=(1 << 31) - 127), dict(n_scores=-1), dict(n_scores=1 << 31),
    dict(B=1 << 25), dict(scale=float("nan")), dict(scale=float("inf")), dict(q=None), dict(w=None),
    dict(keys=None), dict(ks=None), dict(ln=None), dict(ss=None), dict(scores=None), dict(q=0x10008),
    dict(keys=0x30004), dict(w=0x20004), dict(bias=0x2), dict(scores=0x70002),
])
def test_indexer_invalid_arguments_rejected_on_host(so, kw):
    # Pointers here are never dereferenced: validation fails first.
    assert so.topk_ragged_indexer_scores(*_ix_args(**kw), None) == 1
    assert so.topk_ragged_indexer(*_ix_args(**kw), 2048, 0, 0x80000, None, None) == 1


@pytest.mark.parametrize("k,flags,oi", [(0, 0, 0x80000), (4097, 0, 0x80000), (16, 1, 0x80000), (16, 4, 0x80000),
                                        (16, 0, None)])
def test_indexer_chain_selection_arguments_rejected(so, k, flags, oi):
    assert so.topk_ragged_indexer(*_ix_args(), k, flags, oi, None, None) == 1


def test_indexer_empty_batch_is_ok_without_device(so):
    assert so.topk_ragged_indexer_scores(*_ix_args(B=0, q=None, w=None, ks=None, ln=None, ss=None), None) == 0
