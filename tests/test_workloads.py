"""The synthetic inputs have the shapes the pages' workloads describe (no
selection arithmetic here, only the generator's documented properties):
decode rows hold roughly 40-70 % exact 0.0 scores, the long-context rows
alternate between a boundary inside the 0.0 plateau (fewer than k nonzero
scores) and one among the positives, the prefill lengths follow
L_i = max(1, (i+1)//4), and every generator is reproducible from its seed.
Sizes are reduced where the full ones would be slow on the CPU."""
import numpy as np
import torch

import workloads as W


def test_decode_zero_fraction_band():
    w = W.decode(B=8, lmin=4096, lmax=20000)
    s, st, ln = w.numpy()
    for i in range(w.B):
        row = s[st[i]:st[i] + ln[i]]
        frac = float(np.mean(row == 0.0))
        assert 0.35 <= frac <= 0.75, (i, frac)
        assert (row >= 0).all()            # a sum of non-negative weights times relu


def test_long_rows_alternate_plateau_boundary():
    w = W.long_context(B=4, L=1 << 18, k=4096)
    nz = w.info["nonzero_per_row"]
    assert [i for i in range(4) if nz[i] < w.k] == [0, 2]
    assert all(nz[i] > 4 * w.k for i in (1, 3))


def test_prefill_lengths_and_layout():
    w = W.prefill(rows=64, nkeys=64, chunk_rows=16)
    ln = w.lengths.numpy()
    assert ln.tolist() == [max(1, (i + 1) // 4) for i in range(64)]
    st = w.row_starts.numpy()
    assert st[0] == 0 and (st[1:] == np.cumsum(ln)[:-1]).all()
    assert w.offset_mode == 1


def test_generators_are_seeded():
    a, b = W.decode(B=3, lmin=100, lmax=300), W.decode(B=3, lmin=100, lmax=300)
    assert torch.equal(a.scores, b.scores) and torch.equal(a.lengths, b.lengths)
    x, y = W.decode_indexer(B=2, lmin=50, lmax=90), W.decode_indexer(B=2, lmin=50, lmax=90)
    assert torch.equal(x.keys, y.keys) and torch.equal(x.q, y.q) and torch.equal(x.lengths, y.lengths)
