"""Per-row block scores (hss_score_rows) and per-row top-k selection (hss_select_rows)
against the oracle."""
import math

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


def case(nq, nkv, hd, r, bs, B, R, n, seed, layers=2, layer=1):
    g = torch.Generator().manual_seed(seed)
    d = W.Dims(layers, nq, nkv, hd, r, bs, B)
    A = W.bf16_normal(g, d.a_g_shape)  # projected-looking slots, written directly
    Qp = W.bf16_normal(g, (R, nq, r))
    table = torch.randperm(B, generator=g)[:n].to(torch.int32)
    return d, A, Qp, table, layer


def gpu_rows(d, A, Qp, table, layer):
    R, n = Qp.shape[0], table.numel()
    sc = torch.empty(R, n, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_score_rows(d, Qp.to(DEV), R, A.to(DEV), layer, table.to(DEV), n, sc, st)
    torch.cuda.synchronize()
    return sc, int(st.item())


@pytest.mark.parametrize("nq,nkv,hd,r,bs,B,R,n", [
    (64, 8, 128, 64, 16, 600, 40, 300),    # g 8 (the prefill chunk's GQA), 320 vectors
    (32, 8, 128, 32, 16, 400, 70, 257),    # g 4, ragged tail of blocks
    (16, 16, 64, 16, 16, 300, 300, 130),   # g 1: 300 vectors per kv head (two chunks)
    (32, 16, 64, 64, 32, 200, 129, 99),    # g 2, block size 32
    (64, 4, 128, 128, 16, 300, 33, 150),   # g 16, r 128
])
def test_score_rows_against_oracle(nq, nkv, hd, r, bs, B, R, n):
    d, A, Qp, table, layer = case(nq, nkv, hd, r, bs, B, R, n, seed=nq + nkv + R + n)
    sc, st = gpu_rows(d, A, Qp, table, layer)
    assert st == 0
    s_o, t_o, bad = oracle.score_rows(bits(Qp), bits(A), layer, table.numpy(), nthreads=8)
    assert bad == 0
    assert_scores_close(sc.cpu().numpy().reshape(-1), s_o.reshape(-1), t_o.reshape(-1),
                        what="per-row scores")
    # The max over rows is the block score, bit for bit (the same accumulators).
    blk = torch.empty(n, dtype=torch.float32, device=DEV)
    offs = torch.tensor([0, n], dtype=torch.int32, device=DEV)
    hss.hss_score_blocks(d, Qp.to(DEV)[None], R, A.to(DEV), layer, table.to(DEV), offs, 1, n,
                         blk, 2)
    torch.cuda.synchronize()
    assert torch.equal(sc.max(dim=0).values, blk)


def test_score_rows_bad_id():
    d, A, Qp, table, layer = case(64, 8, 128, 64, 16, 300, 24, 40, seed=3)
    table[5] = 300
    sc, st = gpu_rows(d, A, Qp, table, layer)
    assert st == hss.HSS_ERR_OUT_OF_RANGE
    assert hss.hss_read_device_error() == hss.HSS_ERR_OUT_OF_RANGE
    s = sc.cpu().numpy()
    assert np.all(np.isneginf(s[:, 5]))
    assert np.all(np.isfinite(np.delete(s, 5, axis=1)))


def gpu_select(sc, n, first_pos, bs, topk):
    R = sc.shape[0]
    lists = torch.full((R, topk), 777, dtype=torch.int32, device=DEV)
    hss.hss_select_rows(sc, R, n, first_pos, bs, topk, lists)
    torch.cuda.synchronize()
    return lists.cpu().numpy()


@pytest.mark.parametrize("R,n,first_pos,bs,topk", [
    (40, 300, 4700, 16, 64),     # every row sees every block
    (70, 257, 0, 16, 8),         # the first rows see no whole block yet
    (33, 150, 1000, 32, 200),    # topk above what a row has seen: -1 tail
    (9, 5000, 70000, 16, 1024),  # long rows (1024-thread path), topk 1024
])
def test_select_rows_exact(R, n, first_pos, bs, topk):
    g = torch.Generator().manual_seed(R + n)
    sc = torch.randint(-40, 40, (R, n), generator=g).float() / 8  # many ties
    sc[0, :7] = float("nan")
    sc[1, 3] = -0.0
    sc[1, 4] = 0.0
    got = gpu_select(sc.to(DEV), n, first_pos, bs, topk)
    exp = oracle.select_rows(sc.numpy(), n, first_pos, bs, topk)
    assert np.array_equal(got, exp)


def assert_lists_match(gpu_lists, s_o, t_o, rows, n, first_pos, bs, topk):
    """Per-row top-k lists against the oracle's per-row scores: for each row, the set of its
    first min(topk, seen) entries equals the oracle's, except for blocks whose oracle score
    lies within the score tolerance of the oracle's topk-th largest; the -1 tail matches."""
    tol = oracle.score_tolerance(t_o)
    for i, row in enumerate(rows):
        seen = min(n, (first_pos + int(row) + 1) // bs)
        take = min(topk, seen)
        got = gpu_lists[i]
        assert (got[take:] == -1).all() and (got[:take] >= 0).all() and (got[:take] < seen).all()
        assert len(set(got[:take].tolist())) == take
        if take == 0:
            continue
        so = s_o[i, :seen]
        order = np.lexsort((np.arange(seen), -so))
        c = so[order[take - 1]]
        amb = np.abs(so - c) <= tol[i, :seen]
        diff = set(order[:take].tolist()) ^ set(got[:take].tolist())
        assert all(amb[j] for j in diff), f"row {row}: lists differ outside the tolerance band"


def test_rows_end_to_end_prefill_chunk_full_size():
    # The prefill chunk at full size: 512 rows x 64 q heads against 8192 blocks (r 64, g 8).
    # The max over rows equals the block scores exactly; 64 rows spread over the chunk (every
    # 1024-vector query slice of every kv group) are compared with the oracle on all 8192
    # blocks (every tile and CTA of the persistent scheduler), and their top-128 lists with
    # the oracle's inside the tolerance band; the selection of every row is exact for the
    # GPU's own scores.
    d, A, Qp, table, layer = case(64, 8, 128, 64, 16, 8192, 512, 8192, seed=21, layers=1,
                                  layer=0)
    sc, st = gpu_rows(d, A, Qp, table, layer)
    assert st == 0
    blk = torch.empty(8192, dtype=torch.float32, device=DEV)
    offs = torch.tensor([0, 8192], dtype=torch.int32, device=DEV)
    hss.hss_score_blocks(d, Qp.to(DEV)[None], 512, A.to(DEV), layer, table.to(DEV), offs, 1,
                         8192, blk, 2)
    torch.cuda.synchronize()
    assert torch.equal(sc.max(dim=0).values, blk)
    first_pos = 131072 - 512
    rows = np.arange(3, 512, 8)
    s_o, t_o, bad = oracle.score_rows(bits(Qp[torch.as_tensor(rows)]), bits(A), layer,
                                      table.numpy(), nthreads=oracle.default_threads())
    assert bad == 0
    got = sc[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    assert_scores_close(got.reshape(-1), s_o.reshape(-1), t_o.reshape(-1),
                        what="64 rows x 8192 blocks")
    lists = gpu_select(sc, 8192, first_pos, 16, 128)
    exp = oracle.select_rows(sc.cpu().numpy(), 8192, first_pos, 16, 128)
    assert np.array_equal(lists, exp)
    assert_lists_match(lists[rows], s_o, t_o, rows, 8192, first_pos, 16, 128)
