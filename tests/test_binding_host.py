"""The Python binding's marshalling on the CPU, against a fake library.

Every binding function checks its tensors and passes pointers, sizes and a
stream to the C entry point of the same name.  Here the library is replaced
by a recorder and the CUDA-device test of `_check` by a CPU one (dtype,
size and contiguity checks stay), so the argument order, the page-table
stride rule, the size checks that guard the library's writes and the
status-to-exception path run without a GPU.
"""
import contextlib

import pytest
import torch

from sparse_attention_deterministic_gb300 import binding as bd
from sparse_attention_deterministic_gb300._native import TopkError


class FakeLib:
    def __init__(self, status=0):
        self.calls = []
        self.status = status

    def __getattr__(self, name):
        def call(*args):
            self.calls.append((name, args))
            return self.status
        return call


@pytest.fixture
def fake(monkeypatch):
    lib = FakeLib()
    real_check = bd._check

    def cpu_check(t, name, dtype, device=None):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")

    monkeypatch.setattr(bd, "_check", cpu_check)
    monkeypatch.setattr(bd, "lib", lambda: lib)
    monkeypatch.setattr(bd, "_stream_handle", lambda dev, stream: 77)
    monkeypatch.setattr(bd.torch.cuda, "device", lambda dev: contextlib.nullcontext())
    lib.real_check = real_check
    return lib


def _rows(B=3, n=100):
    scores = torch.zeros(n)
    starts = torch.arange(B, dtype=torch.int32) * 10
    lengths = torch.full((B,), 10, dtype=torch.int32)
    return scores, starts, lengths


def test_real_check_rejects_host_tensors(fake):
    with pytest.raises(ValueError, match="CUDA tensor"):
        fake.real_check(torch.zeros(4), "scores", torch.float32)


def test_selection_arguments_in_header_order(fake):
    s, st, ln = _rows()
    idx, val = bd.topk_ragged(s, st, ln, k=8, offset_mode=bd.TOPK_OFFSET_ROW_START, with_values=True)
    assert idx.shape == (3, 8) and idx.dtype == torch.int32 and val.shape == (3, 8)
    (name, a), = fake.calls
    assert name == "topk_ragged"
    assert a == (s.data_ptr(), 100, st.data_ptr(), ln.data_ptr(), 3, 8, 1, idx.data_ptr(), val.data_ptr(), 77)


def test_empty_batch_passes_null_pointers(fake):
    s = torch.zeros(0)
    e = torch.zeros(0, dtype=torch.int32)
    idx, val = bd.topk_ragged(s, e, e, k=8)
    assert idx.shape == (0, 8) and val is None
    (_, a), = fake.calls
    assert a == (None, 0, None, None, 0, 8, 0, None, None, 77)


def test_page_table_stride_per_row_or_shared(fake):
    s, st, ln = _rows()
    pt = torch.zeros((3, 5), dtype=torch.int32)
    bd.topk_ragged(s, st, ln, k=8, page_table=pt, page_size=4)
    shared = torch.zeros(5, dtype=torch.int32)
    bd.topk_ragged(s, st, ln, k=8, page_table=shared, page_size=4)
    (n0, a0), (n1, a1) = fake.calls
    assert n0 == n1 == "topk_ragged_paged"
    assert a0[7:10] == (pt.data_ptr(), 5, 4) and a1[7:10] == (shared.data_ptr(), 0, 4)


@pytest.mark.parametrize("shape", [(2, 5), (3, 5, 1)])
def test_page_table_of_wrong_shape_is_refused(fake, shape):
    s, st, ln = _rows()
    with pytest.raises(ValueError, match="page_table"):
        bd.topk_ragged(s, st, ln, k=8, page_table=torch.zeros(shape, dtype=torch.int32), page_size=4)
    assert not fake.calls


@pytest.mark.parametrize("k,B", [(0, 3), (4097, 3), (4096, 1 << 19)])
def test_k_outside_the_library_limits_is_refused_before_allocating(fake, k, B):
    st = torch.zeros(B, dtype=torch.int32)
    with pytest.raises(TopkError) as e:
        bd.topk_ragged(torch.zeros(4), st, st, k=k)
    assert e.value.status == bd._STATUS_INVALID_ARG
    assert not fake.calls


def test_caller_outputs_must_hold_b_times_k(fake):
    s, st, ln = _rows()
    with pytest.raises(ValueError, match="out_idx"):
        bd.topk_ragged(s, st, ln, k=8, out_idx=torch.empty((3, 7), dtype=torch.int32))
    with pytest.raises(ValueError, match="out_val"):
        bd.topk_ragged(s, st, ln, k=8, out_val=torch.empty((3, 7)))
    assert not fake.calls


def test_library_status_becomes_topk_error(fake):
    fake.status = 4
    s, st, ln = _rows()
    with pytest.raises(TopkError) as e:
        bd.topk_ragged(s, st, ln, k=8)
    assert e.value.status == 4 and "topk_ragged" in str(e.value)


def test_stats_arguments(fake):
    s, st, ln = _rows()
    out = bd.topk_ragged_stats(s, st, ln, k=16)
    assert out.shape == (3, len(bd.ROW_STATS_FIELDS)) and out.dtype == torch.int32
    (name, a), = fake.calls
    assert name == "topk_ragged_stats"
    assert a == (s.data_ptr(), 100, st.data_ptr(), ln.data_ptr(), 3, 16, out.data_ptr(), 77)


def _indexer_inputs(B=2, n_keys=300):
    g = torch.Generator().manual_seed(0)
    q = torch.randn((B, bd.INDEXER_HEADS, bd.INDEXER_DIM), generator=g).to(torch.bfloat16)
    w = torch.rand((B, bd.INDEXER_HEADS), generator=g)
    keys = torch.randn((n_keys, bd.INDEXER_DIM), generator=g).to(torch.bfloat16)
    ks = torch.tensor([0, 100], dtype=torch.int32)
    ln = torch.tensor([100, 200], dtype=torch.int32)
    ss = torch.tensor([0, 100], dtype=torch.int32)
    return q, w, keys, ks, ln, ss


def test_indexer_scores_arguments(fake):
    q, w, keys, ks, ln, ss = _indexer_inputs()
    out = bd.indexer_scores(q, w, keys, ks, ln, ss, n_scores=300)
    assert out.shape == (300,) and float(out.abs().sum()) == 0.0
    (name, a), = fake.calls
    assert name == "topk_ragged_indexer_scores"
    assert a[:4] == (q.data_ptr(), w.data_ptr(), None, keys.data_ptr())
    assert a[4:9] == (300, ks.data_ptr(), ln.data_ptr(), ss.data_ptr(), 2)
    assert a[9] == pytest.approx(128 ** -0.5) and a[10:] == (out.data_ptr(), 300, 77)


def test_indexer_chain_checks_its_outputs(fake):
    q, w, keys, ks, ln, ss = _indexer_inputs()
    with pytest.raises(ValueError, match="out_val"):
        bd.topk_ragged_indexer(q, w, keys, ks, ln, ss, k=16, n_scores=300, out_val=torch.empty(2 * 16 - 1))
    with pytest.raises(TopkError):
        bd.topk_ragged_indexer(q, w, keys, ks, ln, ss, k=4097, n_scores=300)
    assert not fake.calls
    idx, val, scores = bd.topk_ragged_indexer(q, w, keys, ks, ln, ss, k=16, n_scores=300, with_values=True,
                                              bias=torch.zeros(2), scale=0.5)
    (name, a), = fake.calls
    assert name == "topk_ragged_indexer"
    assert a[10:] == (scores.data_ptr(), 300, 16, 0, idx.data_ptr(), val.data_ptr(), 77)
    assert a[9] == 0.5 and a[2] is not None


def test_indexer_shapes_are_checked(fake):
    q, w, keys, ks, ln, ss = _indexer_inputs()
    with pytest.raises(ValueError, match="q must be"):
        bd.indexer_scores(q[:, :32].contiguous(), w, keys, ks, ln, ss, n_scores=300)
    with pytest.raises(ValueError, match="keys must be"):
        bd.indexer_scores(q, w, keys.view(-1)[:1000], ks, ln, ss, n_scores=300)
    with pytest.raises(ValueError, match="n_scores"):
        bd.indexer_scores(q, w, keys, ks, ln, ss)
    assert not fake.calls


def test_device_names():
    assert bd._device(3) == torch.device("cuda", 3)
    assert bd._device("cuda:2") == torch.device("cuda", 2)
    assert bd._device(torch.device("cuda", 1)) == torch.device("cuda", 1)
    with pytest.raises(ValueError, match="CUDA device"):
        bd._device("cpu")
