"""Edge cases of the contract on the GPU: empty rows and batch, envelope and
window violations (reported through the device status word, rows written as
-1), degenerate rows (all equal, all -inf, NaN only), k extremes."""
import numpy as np
import pytest
import torch

import sparse_attention_deterministic_gb300 as pkg
import workloads as W
from helpers import assert_parity, ragged

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkg.build()
    pkg.init()
    pkg.device_status()   # start from a clear status word


def test_empty_batch():
    s = torch.zeros(4, device="cuda")
    e = torch.zeros(0, dtype=torch.int32, device="cuda")
    idx, val = pkg.topk_ragged(s, e, e, 16, with_values=True)
    assert idx.shape == (0, 16)


def test_zero_and_negative_lengths():
    buf = torch.ones(64)
    w = W.Workload("neg", buf, torch.tensor([0, 5, 9], dtype=torch.int32),
                   torch.tensor([0, -3, 7], dtype=torch.int32), 8, 0, {})
    idx = assert_parity(w)
    assert (idx[:2] == -1).all()


def test_length_envelope_flag():
    buf = torch.ones(64)
    w = W.Workload("env", buf, torch.tensor([0, 0, 3], dtype=torch.int32),
                   torch.tensor([1 << 24, (1 << 24) + 5, 10], dtype=torch.int32), 4, 0, {})
    idx = assert_parity(w)      # asserts the status bits equal the oracle's flags
    assert (idx[:2] == -1).all() and list(idx[2]) == [0, 1, 2, 3]


def test_bad_window_flag():
    buf = torch.ones(100)
    w = W.Workload("win", buf, torch.tensor([-1, 95, 90, 0], dtype=torch.int32),
                   torch.tensor([5, 6, 10, 100], dtype=torch.int32), 4, 1, {})
    idx = assert_parity(w)
    assert (idx[:2] == -1).all()


def test_status_word_clears():
    buf = torch.ones(8)
    w = W.Workload("env", buf, torch.tensor([0], dtype=torch.int32),
                   torch.tensor([1 << 24], dtype=torch.int32), 4, 0, {})
    assert_parity(w)
    assert pkg.device_status() == 0


@pytest.mark.parametrize("pattern", [0x00000000, 0x80000000, 0xFF800000, 0x7F800000,
                                     0x7FC00000, 0xFFC00000, 0x3F800000])
@pytest.mark.parametrize("L", [1, 3, 2048, 2049, 65536, 300000])
def test_constant_rows(pattern, L):
    bits = torch.full((L,), pattern, dtype=torch.int64)
    bits = (bits - ((bits >> 31) << 32)).to(torch.int32)
    rows = [bits.view(torch.float32)] * 3
    assert_parity(ragged(f"const{pattern:x}", rows, 2048, gap=2, lead=1))


def test_signed_zero_and_nan_mix():
    g = torch.Generator().manual_seed(77)
    alphabet = [0x00000000, 0x80000000, 0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF800001,
                0xFF800000, 0x7F800000]
    assert_parity(W.random_bits(40, 12000, 4096, alphabet=alphabet))
    assert_parity(W.random_bits(2000, 700, 512, alphabet=alphabet))


def test_k_equals_one_and_max():
    for k in (1, 4096):
        w = W.decode(B=12, lmin=100, lmax=200000, k=k)
        assert_parity(w)
