"""Masked block scores (valid-length and causal masks) on both scoring kernels, against the
oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import kv_cache_block_lowrank_gb300 as hss
import oracle
import workloads as W
from gpu_util import assert_scores_close, bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_block_lowrank_gb300 import _build

    _build.build()
    hss.load()


def case(nq, nkv, r, bs, rows, lengths, seed):
    g = torch.Generator().manual_seed(seed)
    total = sum(lengths)
    d = W.Dims(1, nq, nkv, 128, r, bs, max(total, 8) + 3)
    A = W.bf16_normal(g, d.a_g_shape)
    Qp = W.bf16_normal(g, (len(lengths), rows, nq, r))
    table = torch.randperm(d.max_blocks, generator=g)[:total].to(torch.int32)
    offs = W.identity_offsets(lengths)
    # Context lengths: inside the last block, several blocks short, zero, and the full table.
    ctx = []
    for i, n in enumerate(lengths):
        choice = i % 4
        full = n * bs
        ctx.append([max(full - int(torch.randint(1, bs, (1,), generator=g)), 0),
                    max(full - 3 * bs - 5, 0), 0, full][choice])
    pos0 = [int(torch.randint(-rows, max(n * bs, 1), (1,), generator=g)) for n in lengths]
    return d, A, Qp, table, offs, torch.tensor(ctx, dtype=torch.int32), \
        torch.tensor(pos0, dtype=torch.int32)


def run(d, A, Qp, table, offs, rows, ctx, pos0, path):
    sc = torch.full((table.numel(),), 123.0, dtype=torch.float32, device=DEV)
    hss.hss_score_blocks_masked(d, Qp.to(DEV), rows, A.to(DEV), 0, table.to(DEV), offs.to(DEV),
                                offs.numel() - 1, table.numel(),
                                None if ctx is None else ctx.to(DEV),
                                None if pos0 is None else pos0.to(DEV), sc, path)
    torch.cuda.synchronize()
    return sc.cpu().numpy()


SHAPES = [
    (32, 8, 32, 16, 1, [300, 41, 7, 120], hss.HSS_PATH_DECODE),
    (8, 2, 32, 16, 4, [33, 0, 50, 9, 64], hss.HSS_PATH_DECODE),
    (8, 8, 64, 32, 2, [21, 13], hss.HSS_PATH_DECODE),
    (64, 8, 64, 16, 40, [37, 80, 5], hss.HSS_PATH_TCGEN05),
    (16, 4, 32, 32, 100, [20, 9, 31, 4], hss.HSS_PATH_TCGEN05),
    (32, 8, 32, 16, 1, [300, 41], hss.HSS_PATH_TCGEN05),
]


@pytest.mark.parametrize("nq,nkv,r,bs,rows,lengths,path", SHAPES)
@pytest.mark.parametrize("masks", ["length", "causal", "both"])
def test_masked_scores(nq, nkv, r, bs, rows, lengths, path, masks):
    d, A, Qp, table, offs, ctx, pos0 = case(nq, nkv, r, bs, rows, lengths,
                                            seed=nq + r + bs + rows + len(lengths))
    ctx_m = ctx if masks in ("length", "both") else None
    pos_m = pos0 if masks in ("causal", "both") else None
    got = run(d, A, Qp, table, offs, rows, ctx_m, pos_m, path)
    ref, tsum, _ = oracle.score_blocks_masked(
        bits(Qp), bits(A), 0, table.numpy(), offs.numpy().astype(np.int64),
        ctx_len=None if ctx_m is None else ctx_m.numpy(),
        row_pos0=None if pos_m is None else pos_m.numpy(), nthreads=8)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), "hidden blocks differ"
    fin = np.isfinite(ref)
    assert fin.any() or masks != "length"
    assert_scores_close(got[fin], ref[fin], tsum[fin], f"{masks} scores")


@pytest.mark.parametrize("path", [hss.HSS_PATH_DECODE, hss.HSS_PATH_TCGEN05])
def test_no_masks_is_the_plain_score(path):
    d, A, Qp, table, offs, ctx, pos0 = case(32, 8, 32, 16, 2, [100, 30], seed=5)
    got = run(d, A, Qp, table, offs, 2, None, None, path)
    sc = torch.empty(table.numel(), dtype=torch.float32, device=DEV)
    hss.hss_score_blocks(d, Qp.to(DEV), 2, A.to(DEV), 0, table.to(DEV), offs.to(DEV), 2,
                         table.numel(), sc, path)
    torch.cuda.synchronize()
    assert np.array_equal(got, sc.cpu().numpy())


def test_full_length_mask_changes_nothing():
    d, A, Qp, table, offs, ctx, pos0 = case(32, 8, 32, 16, 1, [64, 17], seed=9)
    full = torch.tensor([64 * 16, 17 * 16], dtype=torch.int32)
    got = run(d, A, Qp, table, offs, 1, full, None, hss.HSS_PATH_DECODE)
    plain = run(d, A, Qp, table, offs, 1, None, None, hss.HSS_PATH_DECODE)
    assert np.array_equal(got, plain)
