"""Shared helpers for the GPU tests: run the CUDA path and the oracle on the
same seeded inputs and compare them bit for bit."""
import numpy as np
import torch

import oracle
import sparse_attention_deterministic_gb300 as pkg
import workloads as W


def gpu_run(w: W.Workload, with_values=True, stream=None):
    g = w.to("cuda")
    idx, val = pkg.topk_ragged(g.scores, g.row_starts, g.lengths, w.k, w.offset_mode,
                               with_values=with_values, stream=stream)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), (val.cpu().numpy().view(np.uint32) if val is not None else None)


def oracle_run(w: W.Workload, n_threads=8):
    s, st, ln = w.numpy()
    idx, val, flags = oracle.topk_ragged(s, st, ln, w.k, w.offset_mode, n_threads=n_threads)
    return idx, val.view(np.uint32), flags


def assert_parity(w: W.Workload, with_values=True):
    got_idx, got_val = gpu_run(w, with_values)
    ref_idx, ref_val, flags = oracle_run(w)
    bad = np.nonzero((got_idx != ref_idx).any(1))[0]
    if bad.size:
        r = int(bad[0])
        cols = np.nonzero(got_idx[r] != ref_idx[r])[0]
        raise AssertionError(
            f"{w.name}: {bad.size} rows differ in out_idx; row {r} (len "
            f"{int(w.lengths[r])}) first cols {cols[:6].tolist()}: got "
            f"{got_idx[r, cols[:6]].tolist()} want {ref_idx[r, cols[:6]].tolist()}")
    if with_values:
        badv = np.nonzero((got_val != ref_val).any(1))[0]
        assert badv.size == 0, f"{w.name}: out_val bits differ in rows {badv[:8].tolist()}"
    status = pkg.device_status()
    expected = 0
    for f in flags:
        expected |= int(f)
    assert status == expected, f"{w.name}: device status {status:#x}, expected {expected:#x}"
    return got_idx


def ragged(name, rows, k, offset_mode=0, gap=0, lead=0):
    """Pack a list of 1-D float32 tensors into one flat buffer with `gap`
    entries between rows and `lead` entries before the first (both filled
    with +inf so that a window overrun would be visible in the output)."""
    lengths = torch.tensor([r.numel() for r in rows], dtype=torch.int32)
    total = lead + int(lengths.sum()) + gap * len(rows)
    buf = torch.full((max(total, 1),), float("inf"), dtype=torch.float32)
    starts = []
    pos = lead
    for r in rows:
        starts.append(pos)
        buf[pos:pos + r.numel()] = r
        pos += r.numel() + gap
    return W.Workload(name, buf[:total] if total else buf[:0], torch.tensor(starts, dtype=torch.int32),
                      lengths, k, offset_mode, {})
