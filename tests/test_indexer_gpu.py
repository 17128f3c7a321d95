"""The lightning-indexer scores on the tensor cores (topk_ragged_indexer_scores)
against the oracle's float64 scores, and the indexer + top-k chain
(topk_ragged_indexer) against the oracle's selection over the GPU's own scores.

Tolerance.  The inputs are bf16, so every product q_hd * k_td is exact in
fp32; the tensor cores sum 128 of them per head in fp32, and the epilogue
applies scale and bias (one fused multiply-add), the relu and a 64-term
fused multiply-add chain over heads.  With u = 2^-24 per rounding, the error
is at most about 128 * 2u * scale * sum_h w_h sum_d |q_hd k_td| (allowing the
tensor-core adds one extra bit) plus about 66 u * sum_h w_h |x_h| for the
epilogue, x_h the head logit.  2^-16 times the sum of those two magnitudes
bounds both with room to spare; it is the bar below, per element.

The selection is decided in fp32 on both sides: the oracle's top-k runs over
the GPU's scores, so the indices must agree bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_deterministic_gb300 as pkg

pytestmark = pytest.mark.gpu
H, D = 64, 128
SENTINEL = -7.25


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkg.build()
    pkg.init()


def make_case(lengths, shared_keys=False, seed=0, bias=True, rho=0.99, gap=0, score_gap=3, extra_keys=0):
    """Correlated-head queries (as the workloads' indexer), U(0,1) head
    weights, N(0,1) bf16 keys; decode layout (own keys per row) or a causal
    prefill layout (every row reads the first L_i keys).  Score windows are
    score_gap apart.  The library groups rows that share key tiles when the
    score buffer holds at least twice as many entries as the key buffer has
    rows, so score_gap also picks which of its two kernels runs."""
    g = torch.Generator().manual_seed(seed)
    B = len(lengths)
    lengths = torch.tensor(lengths, dtype=torch.int32)
    qbar = torch.randn(B, 1, D, generator=g)
    q = (rho ** 0.5 * qbar + (1 - rho) ** 0.5 * torch.randn(B, H, D, generator=g)).to(torch.bfloat16)
    w = torch.rand(B, H, generator=g)
    b = (-0.6 * torch.rand(B, generator=g)) if bias else None
    if shared_keys:
        n_keys = max(1, int(lengths.max()))
        key_starts = torch.zeros(B, dtype=torch.int32)
    else:
        key_starts = torch.zeros(B, dtype=torch.int32)
        key_starts[1:] = torch.cumsum(lengths + gap, 0)[:-1].to(torch.int32)
        n_keys = max(1, int((lengths + gap).sum()))
    n_keys += extra_keys
    keys = torch.randn(n_keys, D, generator=g).to(torch.bfloat16)
    score_starts = torch.zeros(B, dtype=torch.int32)
    score_starts[1:] = torch.cumsum(lengths + score_gap, 0)[:-1].to(torch.int32)
    n_scores = int((lengths + score_gap).sum())
    return dict(q=q, w=w, bias=b, keys=keys, key_starts=key_starts, lengths=lengths,
                score_starts=score_starts, n_scores=n_scores)


def gpu_scores(c, scale=None):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in c.items()}
    out = torch.full((c["n_scores"],), SENTINEL, dtype=torch.float32, device="cuda")
    pkg.indexer_scores(d["q"], d["w"], d["keys"], d["key_starts"], d["lengths"], d["score_starts"],
                       scale=scale, bias=d["bias"], out=out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def oracle_scores(c, scale):
    q = c["q"].float().numpy()
    keys = c["keys"].float().numpy()
    s, written = oracle.indexer_scores(q, c["w"].numpy(), None if c["bias"] is None else c["bias"].numpy(),
                                       keys, c["key_starts"].numpy(), c["lengths"].numpy(),
                                       c["score_starts"].numpy(), c["n_scores"], scale)
    # the error bound's magnitudes, per written score
    mag = np.zeros(c["n_scores"])
    qa, w = np.abs(q.astype(np.float64)), c["w"].numpy().astype(np.float64)
    b = np.zeros(len(c["lengths"])) if c["bias"] is None else c["bias"].numpy().astype(np.float64)
    for i in range(len(c["lengths"])):
        L, ks, ss = int(c["lengths"][i]), int(c["key_starts"][i]), int(c["score_starts"][i])
        if L <= 0 or not written[ss:ss + L].all():
            continue
        k64 = keys[ks:ks + L].astype(np.float64)
        x = scale * (k64 @ q[i].astype(np.float64).T) + b[i]
        mag[ss:ss + L] = scale * ((np.abs(k64) @ qa[i].T) @ w[i]) + np.abs(x) @ w[i]
    return s, written, mag


def assert_scores(c, scale=None):
    scale = 1.0 / D ** 0.5 if scale is None else scale
    got = gpu_scores(c, scale)
    want, written, mag = oracle_scores(c, scale)
    assert (got[~written] == SENTINEL).all(), "a score outside the rows' windows was written"
    err = np.abs(got[written].astype(np.float64) - want[written])
    tol = 2.0 ** -16 * mag[written] + 1e-30
    bad = np.flatnonzero(err > tol)
    assert bad.size == 0, (f"{bad.size} scores out of tolerance; worst ratio "
                           f"{(err / tol).max():.3g}, first at {np.flatnonzero(written)[bad[0]]}")
    return got


def test_single_tile_single_row():
    assert_scores(make_case([128], bias=False))


@pytest.mark.parametrize("L", [1, 2, 127, 129, 255, 256, 1000])
def test_partial_tiles(L):
    assert_scores(make_case([L], seed=L))


def test_rows_mixed_lengths_and_empty():
    assert_scores(make_case([0, 5, 300, 0, 128, 4097, 1, 700], seed=3, gap=7))


def test_shared_keys_causal_prefill_layout():
    lengths = [max(1, (i + 1) // 4) for i in range(600)]
    assert_scores(make_case(lengths, shared_keys=True, seed=4))


def test_decode_layout_many_rows():
    g = torch.Generator().manual_seed(5)
    lengths = torch.randint(1, 20000, (64,), generator=g).tolist()
    assert_scores(make_case(lengths, seed=5))


@pytest.mark.parametrize("scale", [1.0, 0.01])
def test_other_scales(scale):
    assert_scores(make_case([3000, 17], seed=6), scale=scale)


def test_repeatable_and_rejected_rows():
    c = make_case([200, 300, 50], seed=7)
    pkg.device_status()   # clear what earlier calls left
    a = gpu_scores(c)
    assert np.array_equal(a, gpu_scores(c))
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in c.items()}
    bad_starts = d["key_starts"].clone()
    bad_starts[1] = int(d["keys"].shape[0]) - 10          # key window leaves the buffer
    out = torch.full((c["n_scores"],), SENTINEL, device="cuda")
    pkg.indexer_scores(d["q"], d["w"], d["keys"], bad_starts, d["lengths"], d["score_starts"],
                       bias=d["bias"], out=out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert pkg.device_status() == pkg.TOPK_DEV_BAD_WINDOW
    ss = c["score_starts"].numpy()
    assert (got[ss[1]:ss[1] + 300] == SENTINEL).all()
    assert np.array_equal(got[ss[0]:ss[0] + 200], a[ss[0]:ss[0] + 200])


@pytest.mark.parametrize("k", [1, 2048, 4096])
def test_indexer_then_topk_equals_oracle_selection(k):
    g = torch.Generator().manual_seed(8)
    c = make_case(torch.randint(1, 30000, (40,), generator=g).tolist(), seed=8)
    d = {kk: (v.cuda() if isinstance(v, torch.Tensor) else v) for kk, v in c.items()}
    idx, val, scores = pkg.topk_ragged_indexer(d["q"], d["w"], d["keys"], d["key_starts"], d["lengths"],
                                               d["score_starts"], k=k, bias=d["bias"], n_scores=c["n_scores"],
                                               with_values=True)
    torch.cuda.synchronize()
    s = scores.cpu().numpy()
    ref_idx, ref_val, _ = oracle.topk_ragged(s, c["score_starts"].numpy(), c["lengths"].numpy(), k, 0)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert np.array_equal(val.cpu().numpy().view(np.uint32), ref_val.view(np.uint32))
    # the chain's scores are the standalone op's
    alone = gpu_scores(c)
    for i in range(len(c["lengths"])):
        a, L = int(c["score_starts"][i]), int(c["lengths"][i])
        assert np.array_equal(s[a:a + L], alone[a:a + L])


def test_graph_capture_of_the_chain():
    c = make_case([5000, 70000, 1234], seed=9)
    d = {kk: (v.cuda() if isinstance(v, torch.Tensor) else v) for kk, v in c.items()}
    scores = torch.zeros(c["n_scores"], device="cuda")
    idx = torch.empty((3, 2048), dtype=torch.int32, device="cuda")
    args = (d["q"], d["w"], d["keys"], d["key_starts"], d["lengths"], d["score_starts"])
    ref, _, _ = pkg.topk_ragged_indexer(*args, bias=d["bias"], scores=scores.clone())
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        pkg.topk_ragged_indexer(*args, bias=d["bias"], scores=scores, out_idx=idx)
    torch.cuda.synchronize()
    idx.zero_()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=st):
        pkg.topk_ragged_indexer(*args, bias=d["bias"], scores=scores, out_idx=idx)
    gr.replay()
    torch.cuda.synchronize()
    assert torch.equal(idx, ref)


def test_row_groups_and_their_edges():
    # Aligned blocks of four rows that read the same key window share key
    # tiles; blocks that break the rule (another key start, a rejected row,
    # a batch that is not a multiple of four) fall back to single rows.
    c = make_case([300, 299, 0, 1000, 7, 7, 7, 7, 50, 4000, 129, 128, 5, 6, 70], shared_keys=True, seed=10,
                  score_gap=1000)
    assert 2 * c["keys"].shape[0] <= c["n_scores"]                               # the grouping kernel
    c["key_starts"][4:8] = torch.tensor([0, 0, 1, 0], dtype=torch.int32)      # block 1: one start differs
    assert_scores(c)
    d = make_case([500, 400, 300, 200, 100, 90, 80, 70], shared_keys=True, seed=11)
    assert 2 * d["keys"].shape[0] <= d["n_scores"]
    d["score_starts"][6] = d["n_scores"] - 10                                    # block 1: row 6 rejected
    pkg.device_status()
    got = gpu_scores(d)
    want, written, mag = oracle_scores(d, 1.0 / D ** 0.5)
    ok = written & (got != SENTINEL)
    assert written[:d["score_starts"][6]].sum() > 0 and pkg.device_status() == pkg.TOPK_DEV_BAD_WINDOW
    assert np.all(np.abs(got[ok] - want[ok]) <= 2.0 ** -16 * mag[ok] + 1e-30)
    assert (got[written] != SENTINEL).all()


@pytest.mark.parametrize("shared,score_gap,extra_keys,grouping", [
    (False, 0, 0, False),          # own keys per row, the single-row kernel
    (False, 12000, 0, True),       # own keys per row through the grouping kernel (no group forms)
    (True, 0, 40000, False),       # shared keys through the single-row kernel
    (True, 0, 0, True),            # shared keys, grouped
])
def test_both_kernels_on_the_same_rows(shared, score_gap, extra_keys, grouping):
    lengths = [max(1, (i + 1) // 3) * 37 % 3000 + 1 for i in range(64)]
    c = make_case(lengths, shared_keys=shared, seed=12, score_gap=score_gap, extra_keys=extra_keys)
    assert (2 * c["keys"].shape[0] <= c["n_scores"]) == grouping
    assert_scores(c)


def test_scores_do_not_depend_on_the_kernel_instance():
    # The same shared-key rows, once grouped (four rows per MMA, N = 256) and
    # once one row per MMA (N = 64, forced by a larger key buffer): the fp32
    # scores must agree bit for bit, so a row's scores do not depend on the
    # rest of its batch.
    lengths = [max(1, (i + 1) // 3) * 37 % 3000 + 1 for i in range(64)]
    grouped = make_case(lengths, shared_keys=True, seed=13)
    single = dict(grouped)
    single["keys"] = torch.cat([grouped["keys"], torch.zeros(40000, D, dtype=torch.bfloat16)])
    assert 2 * grouped["keys"].shape[0] <= grouped["n_scores"] < 2 * single["keys"].shape[0]
    a, b = gpu_scores(grouped), gpu_scores(single)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_misaligned_inputs_are_refused_with_a_message():
    c = make_case([100, 50], seed=14)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in c.items()}
    w_off = torch.empty(2 * H + 1, device="cuda")[1:].view(2, H)          # 4 bytes off a 16-byte boundary
    w_off.copy_(d["w"])
    with pytest.raises(ValueError, match="16-byte"):
        pkg.indexer_scores(d["q"], w_off, d["keys"], d["key_starts"], d["lengths"], d["score_starts"],
                           n_scores=c["n_scores"])
