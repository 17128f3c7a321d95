"""The fused page-table transform (topk_ragged_paged) on the GPU, bit for
bit against the oracle's selection mapped through the page table, in both
kernels, with per-row and shared tables and with the -inf exclusion."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_deterministic_gb300 as pkg
import workloads as W
from helpers import ragged

pytestmark = pytest.mark.gpu


def _pages(g, B, L_max, page_size, shared):
    n = -(-L_max // page_size)
    if shared:
        return torch.randperm(4 * n, generator=g)[:n].to(torch.int32)
    return torch.stack([torch.randperm(4 * n, generator=g)[:n] for _ in range(B)]).to(torch.int32)


def _check(w, page_size, shared, flags=0):
    g = torch.Generator().manual_seed(w.B * 7 + page_size + flags)
    L_max = int(w.lengths.max()) if w.B else 1
    pt = _pages(g, w.B, max(L_max, 1), page_size, shared)
    d = w.to("cuda")
    idx, val = pkg.topk_ragged(d.scores, d.row_starts, d.lengths, w.k, flags, with_values=True,
                               page_table=pt.cuda(), page_size=page_size)
    torch.cuda.synchronize()
    s, st, ln = w.numpy()
    ref_idx, ref_val, ref_flags = oracle.topk_ragged(s, st, ln, w.k, flags, n_threads=8)
    want = oracle.paged_slots(ref_idx, pt.numpy(), page_size)
    got = idx.cpu().numpy()
    assert (got == want).all(), f"{w.name}: {int((got != want).any(1).sum())} rows differ"
    assert (val.cpu().numpy().view(np.uint32) == ref_val.view(np.uint32)).all()
    assert pkg.device_status() == int(np.bitwise_or.reduce(ref_flags)) if ref_flags.size else True


@pytest.mark.parametrize("page_size", [1, 16, 64])
@pytest.mark.parametrize("shared", [False, True])
def test_paged_decode_rows(page_size, shared):
    _check(W.decode(B=20, lmin=4096, lmax=40000), page_size, shared)


@pytest.mark.parametrize("page_size", [1, 64])
def test_paged_short_rows(page_size):
    g = torch.Generator().manual_seed(11)
    rows = [torch.relu(torch.randn(int(torch.randint(1, 4000, (1,), generator=g)), generator=g) - 0.2)
            for _ in range(700)]
    _check(ragged("paged_short", rows, 2048, lead=5), page_size, False)


def test_paged_with_exclusion():
    g = torch.Generator().manual_seed(13)
    rows = []
    for _ in range(30):
        x = torch.randn(int(torch.randint(100, 9000, (1,), generator=g)), generator=g)
        x[torch.rand(x.numel(), generator=g) < 0.5] = float("-inf")
        rows.append(x)
    _check(ragged("paged_excl", rows, 2048), 16, False, flags=pkg.TOPK_EXCLUDE_NEG_INF)


def test_paged_rejects_row_start_offset():
    d = W.tiny().to("cuda")
    pt = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(pkg.TopkError):
        pkg.topk_ragged(d.scores, d.row_starts, d.lengths, d.k, pkg.TOPK_OFFSET_ROW_START,
                        page_table=pt, page_size=64)


# Every exit of both kernels: the +0.0 plateau and the exact tie block
# (cluster kernel at B=4, row kernel's general path at B=640), a narrow
# value band (two refinement levels) and the bit-pattern alphabet.
@pytest.mark.parametrize("B,L", [(4, 32768), (640, 8192)])
def test_paged_plateau_and_ties(B, L):
    _check(W.plateau(B, L, 1024, 2048), 32, False)
    _check(W.tie_block(B, L, 2048, 512), 32, False)


def test_paged_narrow_and_bit_patterns():
    _check(W.narrow(8, 131072, 2048), 128, False)
    _check(W.random_bits(50, 5003, 1024, alphabet=[0, 0x80000000, 0x3F800000, 0x7FC00001, 0xFFC00001,
                                                  0xFF800000, 0x7F800000, 0x00000001]),
           7, True, flags=pkg.TOPK_EXCLUDE_NEG_INF)


@pytest.mark.parametrize("k", [1, 7, 1001, 4096])
def test_paged_k_not_multiple_of_four_and_max(k):
    # k % 4 != 0 leaves output rows unaligned: the scalar mapping path.
    _check(W.random_bits(40, 5003, k), 16, False)
    _check(W.decode(B=6, lmin=k, lmax=60000, k=k) if k >= 2 else W.random_bits(6, 60000, k), 8, True)
