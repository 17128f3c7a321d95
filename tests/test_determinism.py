"""Run-to-run and batch-composition determinism of the CUDA path.

Repeats under scheduling noise (a busy sibling stream, the method of the tie
study in sglang PR #31115) must be byte-identical, and a row's output must not
depend on which rows share its batch: the batch size changes the launch shape
(one CTA per row, grouped clusters, one cluster per row) and the grouped
clusters deal CTAs to rows by length, so each row is split differently in
each of these runs."""
import numpy as np
import pytest
import torch

import sparse_attention_deterministic_gb300 as pkg
import workloads as W
from helpers import oracle_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkg.build()
    pkg.init()


def _run(scores, starts, lengths, k, mode, stream=None):
    idx, val = pkg.topk_ragged(scores, starts, lengths, k, mode, with_values=True, stream=stream)
    return idx, val


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "adversarial", "long"])
def test_repeats_identical_under_noise(name):
    """100 repeats on one stream while a sibling stream keeps the GPU busy
    with matmuls: every repeat's indices and value bits equal the first
    repeat's, compared as raw 32-bit words on the device.  Prefill runs the
    one-CTA-per-row kernel's register path, long the 16-CTA clusters whose
    slices are partly re-read from L2, decode and adversarial the 4- and
    2-CTA clusters."""
    w = W.make(name, device="cuda")
    noise = torch.randn(2048, 2048, device="cuda")
    side = torch.cuda.Stream()
    main = torch.cuda.Stream()
    first = None
    differ = 0
    for rep in range(100):
        with torch.cuda.stream(side):
            for _ in range(2):
                noise = noise @ noise
                noise = noise / noise.norm()
        with torch.cuda.stream(main):
            idx, val = _run(w.scores, w.row_starts, w.lengths, w.k, w.offset_mode, stream=main)
            if first is None:
                first = (idx.clone(), val.view(torch.int32).clone())
            elif not (torch.equal(idx, first[0]) and torch.equal(val.view(torch.int32), first[1])):
                differ += 1
        main.synchronize()
    torch.cuda.synchronize()
    assert differ == 0, f"{differ} of 99 repeats differ from the first"
    # The repeated output is also the right one.
    ref_idx, ref_val, _ = oracle_run(w.to("cpu"))
    assert np.array_equal(first[0].cpu().numpy(), ref_idx)
    assert np.array_equal(first[1].cpu().numpy().view(np.uint32), ref_val)


def _row_bytes(idx, val):
    return [bytes(idx[i].cpu().numpy().tobytes()) + bytes(val[i].cpu().numpy().tobytes())
            for i in range(idx.shape[0])]


def test_batch_composition_invariance():
    w = W.decode(B=64, k=2048).to("cuda")
    base_idx, base_val = _run(w.scores, w.row_starts, w.lengths, w.k, 0)
    base = _row_bytes(base_idx, base_val)
    g = torch.Generator().manual_seed(3)
    perm = torch.randperm(64, generator=g).cuda()
    subsets = [perm, torch.arange(0, 64, 3).cuda(), torch.arange(1).cuda(), torch.tensor([63]).cuda(),
               torch.arange(0, 8).cuda(), torch.arange(0, 20).cuda()]
    for sel in subsets:
        idx, val = _run(w.scores, w.row_starts[sel].contiguous(), w.lengths[sel].contiguous(), w.k, 0)
        got = _row_bytes(idx, val)
        for j, i in enumerate(sel.tolist()):
            assert got[j] == base[i], (sel.numel(), i)
    # Embed the rows in a batch large enough for the one-CTA-per-row shape.
    rep = torch.arange(64, device="cuda").repeat(12)
    idx, val = _run(w.scores, w.row_starts[rep].contiguous(), w.lengths[rep].contiguous(), w.k, 0)
    got = _row_bytes(idx, val)
    for j, i in enumerate(rep.tolist()):
        assert got[j] == base[i]


def _same_rows(sel, idx, val, base_idx, base_val):
    assert torch.equal(idx, base_idx[sel]), sel[:8].tolist()
    assert torch.equal(val.view(torch.int32), base_val.view(torch.int32)[sel]), sel[:8].tolist()


def test_prefill_rows_batch_composition():
    """Prefill rows, shorter and longer than k, keep their bytes in any batch:
    the whole chunk runs one CTA per row; 64 permuted rows over the same
    33.5 M-score buffer run in clusters (the planner sizes by the buffer);
    2000 rows and the rows around L = k run one CTA per row again."""
    w = W.prefill(device="cuda")
    base_idx, base_val = _run(w.scores, w.row_starts, w.lengths, w.k, w.offset_mode)
    n = int(w.scores.numel())
    assert pkg.launch_info(n, w.B, w.k)["cluster"] == 1
    assert pkg.launch_info(n, 64, w.k)["cluster"] > 1
    g = torch.Generator().manual_seed(5)
    picks = [torch.randperm(w.B, generator=g)[:64], torch.randperm(w.B, generator=g)[:2000],
             torch.arange(8180, 8200), torch.tensor([16383, 0, 8190, 8191, 8194])]
    for sel in picks:
        sel = sel.cuda()
        idx, val = _run(w.scores, w.row_starts[sel].contiguous(), w.lengths[sel].contiguous(), w.k,
                        w.offset_mode)
        _same_rows(sel, idx, val, base_idx, base_val)


def test_long_rows_batch_composition():
    """Rows of 2^20 scores keep their bytes whether a 16-CTA cluster takes one
    of them alone, the eight share the grid, or 640 copies run one CTA per
    row (most of each row then streams from L2 in every pass)."""
    w = W.long_context(device="cuda")
    base_idx, base_val = _run(w.scores, w.row_starts, w.lengths, w.k, w.offset_mode)
    n = int(w.scores.numel())
    assert pkg.launch_info(n, 640, w.k)["cluster"] == 1
    g = torch.Generator().manual_seed(6)
    for sel in (torch.tensor([3]), torch.tensor([6, 1]), torch.randperm(8, generator=g),
                torch.arange(8).repeat(80)):
        sel = sel.cuda()
        idx, val = _run(w.scores, w.row_starts[sel].contiguous(), w.lengths[sel].contiguous(), w.k,
                        w.offset_mode)
        _same_rows(sel, idx, val, base_idx, base_val)


def test_launch_shapes_cover_all_variants():
    # Rows of 64k scores on average: clusters below four rows per SM.
    shapes = {B: pkg.launch_info(B << 16, B, 2048) for B in (1, 4, 64, 300, 400, 4096)}
    kinds = {(info["threads"], info["cluster"] > 1) for info in shapes.values()}
    # 1024-thread clusters, 512-thread clusters (two CTAs per SM) and one
    # 256-thread CTA per row are all reached by some batch size.
    assert {(1024, True), (512, True), (256, False)} <= kinds, shapes
    assert shapes[4]["cluster"] == 16
    # Batches of short rows (at most 4096 scores per row on average) take the
    # one-CTA-per-row kernel whatever their size.
    for B in (1, 4, 64):
        info = pkg.launch_info(B * 4096, B, 2048)
        assert info["cluster"] == 1 and info["grid"] == B
    assert shapes[4096]["cluster"] == 1 and shapes[4096]["grid"] == 4096
    for info in shapes.values():
        assert info["launches"] == 1


@pytest.mark.parametrize("B", [300, 400])
def test_batches_between_shapes(B):
    g = torch.Generator().manual_seed(B)
    lengths = torch.randint(0, 30000, (B,), generator=g).to(torch.int32)
    starts = (torch.cumsum(lengths.to(torch.int64), 0) - lengths.to(torch.int64)).to(torch.int32)
    scores = torch.relu(torch.randn(int(lengths.sum()), generator=g) - 0.3)
    w = W.Workload(f"mid{B}", scores, starts, lengths, 2048, 1, {})
    g_ = w.to("cuda")
    idx, val = _run(g_.scores, g_.row_starts, g_.lengths, w.k, 1)
    ref_idx, ref_val, _ = oracle_run(w)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert np.array_equal(val.cpu().numpy().view(np.uint32), ref_val)
