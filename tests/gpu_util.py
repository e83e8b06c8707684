"""Helpers for the GPU parity tests: run the CUDA path through the binding, run the oracle
on the same input bytes, and compare with the stated tolerances.

Tolerances (fixed by the method's stated acceptance criteria):
  * Qp and A_g: bf16 results within 1 unit in the last place of the oracle's (the GPU
    accumulates in fp32, the oracle in fp64; both round once to bf16, so only sums lying
    within an fp32 rounding error of a bf16 rounding boundary can differ, by one step);
  * scores: |gpu - oracle| <= 2e-3 * sum_j |Qp_j A_j| + 1e-6 (the largest such sum over the
    block's candidates);
  * victims: exact, except for blocks whose oracle score lies within that tolerance of the
    oracle's k-th smallest score.
"""
from __future__ import annotations

import numpy as np
import torch

import kv_cache_block_lowrank_gb300 as hss
import oracle


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def ordered(b: np.ndarray) -> np.ndarray:
    """bf16 bits -> integers in value order (+0 and -0 both map to 0)."""
    b = b.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp(b: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at the magnitude of each bf16 pattern (subnormal floor 2^-133)."""
    v = np.abs((np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32))
    e = np.floor(np.log2(np.maximum(v.astype(np.float64), 2.0 ** -126)))
    return 2.0 ** (np.maximum(e, -126) - 7)


def abs_sum_scale(X_bits: np.ndarray, P_bits: np.ndarray) -> np.ndarray:
    """sum_d |X_d| |P_dj| for every output of X . P (the size of the summed terms), in fp64."""
    f = lambda b: (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    return np.abs(f(X_bits).astype(np.float64)) @ np.abs(f(P_bits).astype(np.float64))


def assert_bf16_within_ulp(gpu_bits, orc_bits, max_ulp: int = 1, what: str = "",
                           scale=None, n_terms: int = 0, max_cancel_frac: float = 1e-3):
    """bf16 results within max_ulp of the oracle's.

    Where `scale` (sum of |terms| of each output) is given, an output may instead lie within
    1 ulp plus the fp32 accumulation bound 2 * n_terms * 2^-24 * scale: when the exact sum
    nearly cancels, one bf16 step of the small result is finer than any fp32 accumulation
    can resolve, for the GPU and for any other fp32 implementation alike.  `scale` is an
    array shaped like the outputs, or a function from flat output indices to their scales
    (evaluated only where an output is more than max_ulp off).  The outputs that need this
    allowance are counted, and their number is bounded by max(4, max_cancel_frac * size),
    so that a systematic error cannot hide inside it.
    """
    g = np.asarray(gpu_bits).reshape(-1)
    o = np.asarray(orc_bits).reshape(-1)
    d = np.abs(ordered(g) - ordered(o))
    bad = d > max_ulp
    n_off = int((d > 0).sum())
    n_cancel = 0
    if scale is not None and bad.any():
        idx = np.flatnonzero(bad)
        sc = scale(idx) if callable(scale) else np.asarray(scale).reshape(-1)[idx]
        f = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        allow = bf16_ulp(o[idx]) + 2.0 * n_terms * 2.0 ** -24 * np.asarray(sc)
        cancel = np.abs(f(g[idx]) - f(o[idx])) <= allow
        n_cancel = int(cancel.sum())
        bad[idx[cancel]] = False
    worst = int(d.max()) if d.size else 0
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {d.size} beyond tolerance "
                           f"({n_off} differ at all, worst {worst} ulp)")
    assert n_cancel <= max(4, max_cancel_frac * d.size), (
        f"{what}: {n_cancel} of {d.size} outputs needed the cancellation allowance")
    return n_off, n_cancel


def assert_scores_close(gpu: np.ndarray, orc: np.ndarray, tsum: np.ndarray, what: str = ""):
    gpu = np.asarray(gpu, dtype=np.float64)
    tol = oracle.score_tolerance(tsum)
    inf_g, inf_o = np.isinf(gpu), np.isinf(orc)
    assert np.array_equal(inf_g, inf_o), f"{what}: +inf entries differ"
    fin = ~inf_o
    err = np.abs(gpu[fin] - orc[fin])
    bad = np.nonzero(err > tol[fin])[0]
    assert bad.size == 0, (f"{what}: {bad.size} scores out of tolerance, worst "
                           f"{(err / tol[fin]).max():.3g} x tol")
    return float((err / np.maximum(tsum[fin], 1e-30)).max()) if err.size else 0.0


def assert_victims_match(gpu_vic: np.ndarray, orc_scores: np.ndarray, tsum: np.ndarray,
                         seq_offsets: np.ndarray, k: int, gpu_scores: np.ndarray | None = None):
    """Victim sets agree outside the tolerance band around the oracle's k-th score.

    Also checks, where the GPU's own scores are given, that the GPU list is exactly the
    ascending (score, index) order of those scores (a property check done here in numpy).
    """
    tol = oracle.score_tolerance(tsum)
    S = len(seq_offsets) - 1
    amb_total = 0
    for s in range(S):
        a, b = int(seq_offsets[s]), int(seq_offsets[s + 1])
        n = b - a
        take = min(k, n)
        row = gpu_vic[s]
        assert (row[take:] == -1).all() and (row[:take] >= 0).all() and (row[:take] < n).all()
        assert len(set(row[:take].tolist())) == take
        if take == 0:
            continue
        so = orc_scores[a:b]
        order = np.lexsort((np.arange(n), so))
        c = so[order[take - 1]]
        amb = np.abs(so - c) <= tol[a:b]
        amb_total += int(amb.sum())
        want = set(order[:take].tolist())
        got = set(row[:take].tolist())
        diff = (want ^ got)
        assert all(amb[i] for i in diff), f"seq {s}: victims differ outside the tolerance band"
        if gpu_scores is not None:
            sg = gpu_scores[a:b].astype(np.float32).astype(np.float64)
            sg = np.where(np.isnan(sg), np.inf, sg)
            exp = np.lexsort((np.arange(n), sg))[:take]
            assert np.array_equal(row[:take], exp), f"seq {s}: not the order of the GPU's scores"
    return amb_total


SENTINEL = 0x7FC1  # a bf16 NaN pattern no projection produces: marks slots never written


class GpuRun:
    """The four library calls on one case, on the current device and stream."""

    def __init__(self, case, device="cuda"):
        self.case = case
        self.device = device
        d = case.dims
        self.dims = d
        self.P = case.P.to(device)
        self.A = torch.empty(d.a_g_shape, dtype=torch.bfloat16, device=device)
        self.ids = case.block_ids.to(device)
        self.table = case.table.to(device)
        self.offs = case.seq_offsets.to(device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def fill_sentinel(self):
        self.A.view(torch.int16).fill_(SENTINEL)

    def ingest(self, li: int, layer: int, K=None, ids=None):
        K = self.case.K[li] if K is None else K
        ids = self.ids if ids is None else ids
        hss.hss_project_kv_blocks(self.dims, self.P, K.to(self.device), layer, ids,
                                  ids.numel(), self.A, self.status)

    def project_q(self, q_layer: int = 0):
        c = self.case
        Q = c.Q[q_layer].to(self.device)
        Qp = torch.empty(c.num_seqs, c.rows_per_seq, self.dims.num_q_heads, self.dims.r,
                         dtype=torch.bfloat16, device=self.device)
        hss.hss_project_q(self.dims, self.P, Q, c.num_seqs * c.rows_per_seq, Qp)
        return Qp

    def score(self, Qp, layer: int, path: int = hss.HSS_PATH_AUTO):
        c = self.case
        scores = torch.empty(c.total_blocks, dtype=torch.float32, device=self.device)
        hss.hss_score_blocks(self.dims, Qp, c.rows_per_seq, self.A, layer, self.table, self.offs,
                             c.num_seqs, c.total_blocks, scores, path, self.status)
        return scores

    def rank(self, scores, k=None):
        c = self.case
        k = c.k_victims if k is None else k
        vic = torch.empty(c.num_seqs, k, dtype=torch.int32, device=self.device)
        hss.hss_rank_victims(scores, self.offs, c.num_seqs, c.total_blocks, k, vic)
        return vic


def oracle_slots(case, li: int, block_positions, nthreads: int | None = None):
    """Oracle A_g slots [len(positions), nkv, bs, r] for the K blocks at the given positions."""
    d = case.dims
    pos = np.asarray(block_positions)
    K = bits(case.K[li][torch.as_tensor(pos)])
    A = np.zeros((1, len(pos), d.num_kv_heads, d.block_size, d.r), dtype=np.uint16)
    st = oracle.project_kv_blocks(bits(case.P), K, 0, np.arange(len(pos), dtype=np.int32), A,
                                  nthreads=nthreads or oracle.default_threads())
    assert st == 0
    return A[0]


def slot_scale(case, li: int, block_positions) -> np.ndarray:
    """sum_d |K_d| |P_dj| for the A_g slots of the given K blocks, slot layout [n, nkv, bs, r]."""
    K = bits(case.K[li][torch.as_tensor(np.asarray(block_positions))])
    return abs_sum_scale(K, bits(case.P)).transpose(0, 2, 1, 3)


def q_scale(case, q_layer: int = 0) -> np.ndarray:
    return abs_sum_scale(bits(case.Q[q_layer]), bits(case.P))


def _bf16_f64(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def slot_scale_fn(K: torch.Tensor, P: torch.Tensor):
    """Lazy sum_d |K_d| |P_dj| for A_g slots made from the key blocks K [n, bs, nkv, hd]
    (any device): a function from flat indices into [n, nkv, bs, r] to their scales."""
    n, bs, nkv, hd = K.shape
    Pa = np.abs(_bf16_f64(bits(P)))
    r = Pa.shape[1]

    def f(idx):
        blk, h, t, j = np.unravel_index(np.asarray(idx), (n, nkv, bs, r))
        dev = K.device
        rows = K[torch.as_tensor(blk, device=dev), torch.as_tensor(t, device=dev),
                 torch.as_tensor(h, device=dev)]
        return (np.abs(_bf16_f64(bits(rows))) * Pa[:, j].T).sum(axis=1)
    return f
