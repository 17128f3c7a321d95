"""Stream order with programmatic dependent launch: every library kernel may be
staged before the grid ahead of it finishes, so each must wait for it before
touching memory.  These tests chain calls with no synchronisation between
them, each reading what the kernel just before it wrote (a torch kernel that
rewrites the scores, the previous call's output, a scratch buffer reused by
the next call), and check every result against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_deterministic_gb300 as pkg
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkg.build()
    pkg.init()


def test_inputs_rewritten_just_before_each_call():
    w = W.decode(B=16, lmin=4096, lmax=60000)
    d = w.to("cuda")
    scores = d.scores.clone()
    gens = [torch.Generator(device="cuda").manual_seed(s) for s in range(6)]
    outs, stats, inputs = [], [], []
    for g in gens:
        # a torch kernel rewrites the whole score buffer; the library reads it next
        scores.copy_(torch.relu(torch.randn(scores.shape, generator=g, device="cuda") - 0.3))
        idx, _ = pkg.topk_ragged(scores, d.row_starts, d.lengths, w.k)
        st = pkg.topk_ragged_stats(scores, d.row_starts, d.lengths, w.k)
        outs.append(idx)
        stats.append(st)
        inputs.append(scores.clone())   # a copy kernel after the library's
    torch.cuda.synchronize()
    st0, ln0 = w.row_starts.numpy(), w.lengths.numpy()
    for s, idx, st in zip(inputs, outs, stats):
        s_np = s.cpu().numpy()
        ref, _, _ = oracle.topk_ragged(s_np, st0, ln0, w.k, 0, n_threads=8, with_values=False)
        assert np.array_equal(idx.cpu().numpy(), ref)
        want, _ = oracle.row_stats(s_np, st0, ln0, w.k)
        assert np.array_equal(st.cpu().numpy().view(np.uint32), want)


def test_outputs_reused_as_inputs_and_scratch_reused():
    # The indexer chain writes `scores`; the next chain rewrites the same
    # scratch while a torch kernel reads the previous selection.
    iw = W.decode_indexer(device="cuda", B=8, lmin=2000, lmax=40000, k=512)
    scores = torch.zeros(iw.n_scores, device="cuda")
    idx = torch.empty((iw.B, iw.k), dtype=torch.int32, device="cuda")
    snapshots, selections = [], []
    for t in range(4):
        w_t = iw.w * (1.0 + 0.25 * t)                      # new head weights each round
        pkg.topk_ragged_indexer(iw.q, w_t, iw.keys, iw.key_starts, iw.lengths, iw.score_starts, k=iw.k,
                                bias=iw.bias, scale=iw.scale, scores=scores, out_idx=idx)
        selections.append(idx.clone())                     # reads the selection just written
        snapshots.append(scores.clone())
    torch.cuda.synchronize()
    st_np, ln_np = iw.score_starts.cpu().numpy(), iw.lengths.cpu().numpy()
    for s, sel in zip(snapshots, selections):
        ref, _, _ = oracle.topk_ragged(s.cpu().numpy(), st_np, ln_np, iw.k, 0, with_values=False)
        assert np.array_equal(sel.cpu().numpy(), ref)
    # the rounds differ (the weights changed), so a stale read would show
    assert not torch.equal(snapshots[0], snapshots[-1])


def test_paged_after_plain_on_one_output_buffer():
    w = W.decode(B=12, lmin=4096, lmax=50000)
    d = w.to("cuda")
    n_pages = -(-int(w.lengths.max()) // 16)
    g = torch.Generator().manual_seed(3)
    pt = torch.stack([torch.randperm(4 * n_pages, generator=g)[:n_pages] for _ in range(w.B)]).to(torch.int32)
    out = torch.empty((w.B, w.k), dtype=torch.int32, device="cuda")
    pkg.topk_ragged(d.scores, d.row_starts, d.lengths, w.k, out_idx=out)
    plain = out.clone()
    pkg.topk_ragged(d.scores, d.row_starts, d.lengths, w.k, out_idx=out, page_table=pt.cuda(), page_size=16)
    paged = out.clone()
    torch.cuda.synchronize()
    s, st, ln = w.numpy()
    ref, _, _ = oracle.topk_ragged(s, st, ln, w.k, 0, n_threads=8, with_values=False)
    assert np.array_equal(plain.cpu().numpy(), ref)
    assert np.array_equal(paged.cpu().numpy(), oracle.paged_slots(ref, pt.numpy(), 16))
