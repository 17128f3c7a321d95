"""Seeded synthetic inputs for deterministic exact ragged top-k.

This module only builds inputs: it holds none of the selection's arithmetic
and is shared by the tests, the benchmark and the smoke check, so that the CPU
oracle and the CUDA library read the very same buffers.  Every buffer is flat
(ragged rows addressed by ``row_starts``/``lengths``), fp32 scores, int32
metadata.

Score models, read from the pages:

* Lightning-indexer scores ``s_t = sum_h w_h * relu(q_h . k_t / sqrt(128) + mu)``
  with 64 heads of dim 128, q and k ~ N(0,1) rounded to bf16, the products in
  fp32, w_h ~ U(0,1) (sglang PR #31115, discussion: the score is a sum of
  ReLU-ed per-head dot products, so every row holds an exact-0.0 plateau).
  Heads are equicorrelated, ``q_h = sqrt(rho) qbar + sqrt(1-rho) eps_h``,
  following the correlated-Gaussian model of the same page's
  ``dsa_topk_score_stats.py`` ("synthetic_rows"): with independent heads no
  entry is ever exactly 0.0, so the 40-70 % plateau needs rho near 1.  The
  reading used here is rho = 0.99 and a per-row mean logit mu ~ U(-0.6, 0).
* Tie-study families of the same page's ``topk_v2_tie_safety.py``: plateau
  (m distinct positives, rest 0.0), a tie block straddling the boundary,
  the ReLU-of-shifted-Gaussian fixture and the narrow range near 1.0.

Seeds come from ``zlib.crc32`` of the workload name, the stable-seed practice
of the same page's hardening commit.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
import zlib

import numpy as np
import torch

HEADS = 64
HEAD_DIM = 128
RHO = 0.99
MAX_LEN = 1 << 24


@dataclasses.dataclass
class Workload:
    name: str
    scores: torch.Tensor        # float32, 1-D flat buffer
    row_starts: torch.Tensor    # int32 [B]
    lengths: torch.Tensor       # int32 [B]
    k: int
    offset_mode: int
    info: dict

    @property
    def B(self) -> int:
        return int(self.row_starts.numel())

    def total_len(self) -> int:
        return int(self.lengths.clamp(min=0).to(torch.int64).sum().item())

    def to(self, device) -> "Workload":
        return dataclasses.replace(
            self, scores=self.scores.to(device), row_starts=self.row_starts.to(device),
            lengths=self.lengths.to(device))

    def numpy(self):
        return (self.scores.cpu().numpy(), self.row_starts.cpu().numpy(),
                self.lengths.cpu().numpy())


def seed_of(name: str) -> int:
    return zlib.crc32(name.encode()) & 0x7FFFFFFF


def digest(t: torch.Tensor) -> str:
    return hashlib.sha256(t.detach().cpu().contiguous().numpy().tobytes()).hexdigest()[:16]


def _gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=device).manual_seed(seed)


def _contiguous_starts(lengths: torch.Tensor) -> torch.Tensor:
    ends = torch.cumsum(lengths.to(torch.int64), 0)
    return (ends - lengths.to(torch.int64)).to(torch.int32)


def _bf16_normal(shape, g, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device).to(torch.bfloat16).to(torch.float32)


def indexer_scores(q: torch.Tensor, keys: torch.Tensor, w: torch.Tensor, mu: float,
                   chunk: int = 1 << 16) -> torch.Tensor:
    """Scores of one query against a key block.

    q [H, D] (bf16-valued fp32), keys [L, D] (bf16-valued fp32), w [H].
    Returns fp32 [L]; heads are summed in one fixed order per call.
    """
    out = torch.empty(keys.shape[0], dtype=torch.float32, device=keys.device)
    scale = 1.0 / math.sqrt(q.shape[1])
    for s in range(0, keys.shape[0], chunk):
        x = (q @ keys[s:s + chunk].T) * scale + mu          # [H, chunk]
        out[s:s + chunk] = (w[:, None] * torch.relu(x)).sum(0)
    return out


def _indexer_query(g, device, rho: float = RHO):
    qbar = torch.randn(HEAD_DIM, generator=g, device=device)
    eps = torch.randn(HEADS, HEAD_DIM, generator=g, device=device)
    q = math.sqrt(rho) * qbar[None, :] + math.sqrt(1.0 - rho) * eps
    q = q.to(torch.bfloat16).to(torch.float32)
    w = torch.rand(HEADS, generator=g, device=device)
    return q, w


def _matmul_precision_guard():
    # fp32 products must not silently drop to TF32 on the GPU.
    torch.backends.cuda.matmul.allow_tf32 = False


# --------------------------------------------------------------------------- #
# The five named workloads.
# --------------------------------------------------------------------------- #

def tiny(device="cpu") -> Workload:
    """B=4 rows of L=4096, row_starts = i*4096, k=2048; each entry 0.0 with
    probability 1/2, else |N(0,1)| (a ReLU plateau)."""
    B, L, k = 4, 4096, 2048
    g = _gen(seed_of("tiny"), device)
    mag = torch.randn(B * L, generator=g, device=device).abs()
    keep = torch.rand(B * L, generator=g, device=device) < 0.5
    scores = torch.where(keep, mag, torch.zeros_like(mag)).to(torch.float32)
    lengths = torch.full((B,), L, dtype=torch.int32, device=device)
    starts = torch.arange(B, dtype=torch.int32, device=device) * L
    return Workload("tiny", scores, starts, lengths, k, 0, {"L": L})


def decode(device="cpu", B: int = 64, lmin: int = 4096, lmax: int = 131072,
           k: int = 2048) -> Workload:
    """B query rows, lengths ~ U{lmin..lmax}, contiguous ragged layout, one
    indexer query and its own key block per row, mu ~ U(-0.6, 0) per row."""
    _matmul_precision_guard()
    g = _gen(seed_of("decode"), device)
    lengths = torch.randint(lmin, lmax + 1, (B,), generator=g, device=device).to(torch.int32)
    starts = _contiguous_starts(lengths)
    total = int(lengths.to(torch.int64).sum().item())
    scores = torch.empty(total, dtype=torch.float32, device=device)
    zero_frac = []
    for i in range(B):
        q, w = _indexer_query(g, device)
        mu = -0.6 * float(torch.rand(1, generator=g, device=device).item())
        L = int(lengths[i].item())
        keys = _bf16_normal((L, HEAD_DIM), g, device)
        s = indexer_scores(q, keys, w, mu)
        st = int(starts[i].item())
        scores[st:st + L] = s
        zero_frac.append(float((s == 0).float().mean().item()))
    return Workload("decode", scores, starts, lengths, k, 0,
                    {"total_len": total, "zero_frac_min": min(zero_frac),
                     "zero_frac_max": max(zero_frac)})


def prefill(device="cpu", rows: int = 16384, nkeys: int = 4096, k: int = 2048,
            chunk_rows: int = 256) -> Workload:
    """``rows`` query rows over one causal sequence of ``nkeys`` compressed
    keys: row i sees the first L_i = max(1, (i+1)//4) keys.  One query per row,
    mu ~ U(-0.6, 0) per row, contiguous ragged layout, offset_mode 1."""
    _matmul_precision_guard()
    g = _gen(seed_of("prefill"), device)
    keys = _bf16_normal((nkeys, HEAD_DIM), g, device)
    idx = torch.arange(rows, device=device, dtype=torch.int64)
    lengths64 = torch.clamp((idx + 1) // 4, min=1, max=nkeys)
    lengths = lengths64.to(torch.int32)
    starts = _contiguous_starts(lengths)
    total = int(lengths64.sum().item())
    scores = torch.empty(total, dtype=torch.float32, device=device)
    scale = 1.0 / math.sqrt(HEAD_DIM)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        R = r1 - r0
        Lmax = int(lengths64[r1 - 1].item())
        qbar = torch.randn(R, 1, HEAD_DIM, generator=g, device=device)
        eps = torch.randn(R, HEADS, HEAD_DIM, generator=g, device=device)
        q = (math.sqrt(RHO) * qbar + math.sqrt(1 - RHO) * eps).to(torch.bfloat16).to(torch.float32)
        w = torch.rand(R, HEADS, 1, generator=g, device=device)
        mu = -0.6 * torch.rand(R, 1, 1, generator=g, device=device)
        x = torch.matmul(q, keys[:Lmax].T) * scale + mu          # [R, H, Lmax]
        s = (w * torch.relu(x)).sum(1)                           # [R, Lmax]
        Lr = lengths64[r0:r1]
        mask = torch.arange(Lmax, device=device)[None, :] < Lr[:, None]
        st = int(starts[r0].item())
        scores[st:st + int(Lr.sum().item())] = s[mask]
    return Workload("prefill", scores, starts, lengths, k, 1, {"total_len": total})


def adversarial(device="cpu", B: int = 128, L: int = 65536, k: int = 4096) -> Workload:
    """Five tie/NaN families dealt round-robin by row id (family = i mod 5):
    (a) uniform over the 2^13 fp32 patterns of [1.0, 1.0 + 2^-10);
    (b) all 0.0; (c) all -inf;
    (d) N(0,1) with 3000 entries set to one value v chosen so that k - 1500
        other entries exceed it (the boundary lands inside the tie set);
    (e) N(0,1) with ~1 % NaN of random sign and random nonzero payload."""
    g = _gen(seed_of("adversarial"), "cpu")
    rows = []
    fam_names = "abcde"
    for i in range(B):
        fam = fam_names[i % 5]
        if fam == "a":
            bits = 0x3F800000 + torch.randint(0, 1 << 13, (L,), generator=g, dtype=torch.int64)
            row = bits.to(torch.int32).view(torch.float32)
        elif fam == "b":
            row = torch.zeros(L, dtype=torch.float32)
        elif fam == "c":
            row = torch.full((L,), float("-inf"), dtype=torch.float32)
        elif fam == "d":
            row = torch.randn(L, generator=g)
            perm = torch.randperm(L, generator=g)
            tie_pos, other = perm[:3000], perm[3000:]
            ranked = torch.sort(row[other], descending=True).values
            v = ranked[k - 1500]
            row[tie_pos] = v
            above = int((row > v).sum().item())
            ties = int((row == v).sum().item())
            assert above < k <= above + ties, (above, ties)
        else:
            row = torch.randn(L, generator=g)
            nan_pos = torch.rand(L, generator=g) < 0.01
            n = int(nan_pos.sum().item())
            sign = torch.randint(0, 2, (n,), generator=g, dtype=torch.int64) << 31
            payload = torch.randint(1, 1 << 23, (n,), generator=g, dtype=torch.int64)
            bits64 = sign | 0x7F800000 | payload
            nan_bits = (bits64 - ((bits64 >> 31) << 32)).to(torch.int32)
            row = row.clone()
            row.view(torch.int32)[nan_pos] = nan_bits
        rows.append(row)
    scores = torch.cat(rows).to(device)
    lengths = torch.full((B,), L, dtype=torch.int32, device=device)
    starts = torch.arange(B, dtype=torch.int32, device=device) * L
    return Workload("adversarial", scores, starts, lengths, k, 0,
                    {"families": "row i -> family 'abcde'[i % 5]"})


def long_context(device="cpu", B: int = 8, L: int = 1 << 20, k: int = 4096,
                 low_mu: float = -3.0) -> Workload:
    """B rows of L indexer scores.  Even rows use mu = low_mu, so fewer than k
    entries are nonzero and the k-th boundary falls inside the 0.0 plateau;
    odd rows use mu ~ U(-0.6, 0)."""
    _matmul_precision_guard()
    g = _gen(seed_of("long"), device)
    lengths = torch.full((B,), L, dtype=torch.int32, device=device)
    starts = torch.arange(B, dtype=torch.int32, device=device) * L
    scores = torch.empty(B * L, dtype=torch.float32, device=device)
    nonzero = []
    for i in range(B):
        q, w = _indexer_query(g, device)
        u = float(torch.rand(1, generator=g, device=device).item())
        mu = low_mu if i % 2 == 0 else -0.6 * u
        chunk = 1 << 16
        for s in range(0, L, chunk):
            keys = _bf16_normal((min(chunk, L - s), HEAD_DIM), g, device)
            scores[i * L + s:i * L + s + keys.shape[0]] = indexer_scores(q, keys, w, mu)
        nz = int((scores[i * L:(i + 1) * L] != 0).sum().item())
        nonzero.append(nz)
    return Workload("long", scores, starts, lengths, k, 0,
                    {"nonzero_per_row": nonzero,
                     "plateau_rows": [i for i in range(B) if nonzero[i] < k]})


NAMED = {
    "tiny": tiny,
    "decode": decode,
    "prefill": prefill,
    "adversarial": adversarial,
    "long": long_context,
}


def make(name: str, device="cpu", **kw) -> Workload:
    return NAMED[name](device=device, **kw)


# --------------------------------------------------------------------------- #
# Tie-study families (uniform-length rows, row_starts = i * L).
# --------------------------------------------------------------------------- #

def _uniform(name, rows: torch.Tensor, k: int, offset_mode: int = 0, info=None) -> Workload:
    B, L = rows.shape
    return Workload(name, rows.reshape(-1).contiguous().to(torch.float32),
                    torch.arange(B, dtype=torch.int32) * L,
                    torch.full((B,), L, dtype=torch.int32), k, offset_mode, info or {})


def plateau(B: int, L: int, m: int, k: int, seed: int = 7) -> Workload:
    """The plateau family: every row holds m distinct positive scores and
    L - m exact zeros.  Positions come from one random ordering of the row
    (argsort of uniform draws), and the positives are a random arrangement of
    the integers 1..m, so they are distinct and exact in fp32."""
    assert 0 <= m <= L < (1 << 24)
    g = _gen(seed, "cpu")
    rows = torch.zeros(B, L)
    if m:
        where = torch.rand(B, L, generator=g).argsort(dim=1)[:, :m]
        vals = torch.rand(B, m, generator=g).argsort(dim=1).to(torch.float32) + 1.0
        rows.scatter_(1, where, vals)
    return _uniform(f"plateau_m{m}", rows, k, info={"m": m})


def tie_block(B: int, L: int, k: int, T: int, seed: int = 11) -> Workload:
    """The tie-block family: T copies of 1.0 that straddle the k-th boundary.
    Per row, the number of larger scores `above` is drawn so that the
    boundary falls strictly inside the block (max(0, k - T + 1) <= above
    <= k - 1, so the selection takes part of the tie set); the larger scores
    are distinct values in (1, 2] and the rest distinct values in (0, 1).
    Every row of a call uses the same `above` (in ``info``)."""
    assert 2 <= T and k <= 4096
    g = _gen(seed, "cpu")
    lo = max(0, k - T + 1)
    above = int(torch.randint(lo, k, (1,), generator=g).item())
    below = L - above - T
    assert below >= 0 and below < (1 << 18)
    order = torch.rand(B, L, generator=g).argsort(dim=1)
    # Ranks 0..L-1 of a random ordering: the first `above` places get the
    # larger values, the next T the tie value, the rest the smaller ones.
    vals = torch.empty(L)
    vals[:above] = 1.0 + (torch.randperm(above, generator=g).to(torch.float32) + 1.0) * 2.0 ** -12
    vals[above:above + T] = 1.0
    vals[above + T:] = (torch.randperm(below, generator=g).to(torch.float32) + 1.0) * 2.0 ** -18
    rows = torch.empty(B, L)
    rows.scatter_(1, order, vals.expand(B, L).contiguous())
    return _uniform(f"tie_T{T}", rows, k, info={"T": T, "above": above})


def relu_shifted(B: int, L: int, k: int, seed: int = 13) -> Workload:
    """relu(N(0,1) - 1.28) * 11.3: about 10 % nonzero."""
    g = _gen(seed, "cpu")
    rows = torch.relu(torch.randn(B, L, generator=g) - 1.28) * 11.3
    return _uniform(f"relu_L{L}", rows, k)


def narrow(B: int, L: int, k: int, seed: int = 17) -> Workload:
    """1 + N(0,1)*1e-7: a handful of distinct fp32 patterns near 1.0."""
    g = _gen(seed, "cpu")
    rows = 1.0 + torch.randn(B, L, generator=g) * 1e-7
    return _uniform(f"narrow_L{L}", rows, k)


def random_bits(B: int, L: int, k: int, seed: int = 19, alphabet=None) -> Workload:
    """Arbitrary fp32 bit patterns (every NaN payload, both zeros, denormals),
    or draws from a small ``alphabet`` of patterns to force ties."""
    g = _gen(seed, "cpu")
    if alphabet is None:
        bits = torch.randint(-(1 << 31), 1 << 31, (B, L), generator=g, dtype=torch.int64)
    else:
        a = torch.tensor(alphabet, dtype=torch.int64)
        bits = a[torch.randint(0, len(alphabet), (B, L), generator=g)]
    bits = (bits - ((bits >> 31) << 32)).to(torch.int32)
    return _uniform("random_bits", bits.view(torch.float32), k)


# --------------------------------------------------------------------------- #
# Indexer inputs: the queries, head weights and keys the decode and prefill
# scores are made from, for the indexer + top-k chain.
# --------------------------------------------------------------------------- #

@dataclasses.dataclass
class IndexerWorkload:
    name: str
    q: torch.Tensor             # bf16 [B, 64, 128]
    w: torch.Tensor             # fp32 [B, 64]
    bias: torch.Tensor          # fp32 [B]: the per-row logit shift mu
    keys: torch.Tensor          # bf16 [n_keys, 128]
    key_starts: torch.Tensor    # int32 [B]
    lengths: torch.Tensor       # int32 [B]
    score_starts: torch.Tensor  # int32 [B]
    n_scores: int
    k: int
    scale: float = 1.0 / math.sqrt(HEAD_DIM)

    @property
    def B(self) -> int:
        return int(self.lengths.numel())

    def unique_key_rows(self) -> int:
        return int(self.keys.shape[0])


def decode_indexer(device="cpu", B: int = 64, lmin: int = 4096, lmax: int = 131072,
                   k: int = 2048) -> IndexerWorkload:
    """The decode batch's shape as indexer inputs: B rows, lengths ~
    U{lmin..lmax} (the decode workload's lengths), each row its own block of
    N(0,1) bf16 keys, correlated-head bf16 queries, w ~ U(0,1), mu ~
    U(-0.6, 0); keys and scores laid out contiguously."""
    g = _gen(seed_of("decode"), device)
    lengths = torch.randint(lmin, lmax + 1, (B,), generator=g, device=device).to(torch.int32)
    starts = _contiguous_starts(lengths)
    total = int(lengths.to(torch.int64).sum().item())
    gi = _gen(seed_of("decode_indexer"), device)
    qbar = torch.randn(B, 1, HEAD_DIM, generator=gi, device=device)
    eps = torch.randn(B, HEADS, HEAD_DIM, generator=gi, device=device)
    q = (math.sqrt(RHO) * qbar + math.sqrt(1.0 - RHO) * eps).to(torch.bfloat16)
    w = torch.rand(B, HEADS, generator=gi, device=device)
    bias = -0.6 * torch.rand(B, generator=gi, device=device)
    keys = torch.randn(total, HEAD_DIM, generator=gi, device=device).to(torch.bfloat16)
    return IndexerWorkload("decode_indexer", q, w, bias, keys, starts, lengths, starts.clone(), total, k)


def prefill_indexer(device="cpu", rows: int = 16384, nkeys: int = 4096, k: int = 2048) -> IndexerWorkload:
    """The prefill chunk's shape as indexer inputs: ``rows`` queries over one
    causal sequence of ``nkeys`` shared keys (row i reads the first
    L_i = max(1, (i+1)//4)), scores laid out contiguously."""
    gi = _gen(seed_of("prefill_indexer"), device)
    keys = torch.randn(nkeys, HEAD_DIM, generator=gi, device=device).to(torch.bfloat16)
    idx = torch.arange(rows, device=device, dtype=torch.int64)
    lengths = torch.clamp((idx + 1) // 4, min=1, max=nkeys).to(torch.int32)
    starts = _contiguous_starts(lengths)
    total = int(lengths.to(torch.int64).sum().item())
    qbar = torch.randn(rows, 1, HEAD_DIM, generator=gi, device=device)
    eps = torch.randn(rows, HEADS, HEAD_DIM, generator=gi, device=device)
    q = (math.sqrt(RHO) * qbar + math.sqrt(1.0 - RHO) * eps).to(torch.bfloat16)
    w = torch.rand(rows, HEADS, generator=gi, device=device)
    bias = -0.6 * torch.rand(rows, generator=gi, device=device)
    return IndexerWorkload("prefill_indexer", q, w, bias, keys, torch.zeros(rows, dtype=torch.int32, device=device),
                           lengths, starts, total, k)


INDEXER = {"decode": decode_indexer, "prefill": prefill_indexer}
