"""Each CUDA kernel against the oracle on the same seeded inputs (small and ragged sizes).

All calls go through the C ABI (the ctypes binding of libhss.so)."""
import math

import numpy as np
import pytest
import torch

import kv_cache_block_lowrank_gb300 as hss
import oracle
import workloads as W
from gpu_util import (SENTINEL, GpuRun, abs_sum_scale, assert_bf16_within_ulp,
                      assert_scores_close, bits)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_block_lowrank_gb300 import _build

    _build.build()
    hss.load()
    assert torch.cuda.is_available()


def gen(seed):
    return torch.Generator().manual_seed(seed)


def dims(L=1, nq=8, nkv=2, hd=128, r=32, bs=16, B=64):
    return W.Dims(L, nq, nkv, hd, r, bs, B)


# ----------------------------------------------------------------------------- projections

@pytest.mark.parametrize("hd,r", [(64, 16), (128, 32), (128, 64), (256, 128), (64, 128),
                                  (192, 32)])
def test_project_q(hd, r):
    g = gen(hd * 1000 + r)
    d = dims(nq=8, nkv=2, hd=hd, r=r)
    rows = 37                                   # 296 GEMM rows: 2 full 128-row tiles + 40
    P = W.projection(g, hd, r)
    Q = W.bf16_normal(g, (rows, d.num_q_heads, hd))
    Qp = torch.full((rows, d.num_q_heads, r), float("nan"), dtype=torch.bfloat16, device=DEV)
    hss.hss_project_q(d, P.to(DEV), Q.to(DEV), rows, Qp)
    torch.cuda.synchronize()
    ref = oracle.project_q(bits(Q), bits(P), nthreads=4)
    assert_bf16_within_ulp(bits(Qp), ref, what="Qp", scale=abs_sum_scale(bits(Q), bits(P)),
                           n_terms=hd)


def test_project_q_single_row_decode_shape():
    g = gen(5)
    d = W.DECODE
    P = W.projection(g, 128, 32)
    Q = W.bf16_normal(g, (1, 32, 128))
    Qp = torch.empty((1, 32, 32), dtype=torch.bfloat16, device=DEV)
    hss.hss_project_q(d, P.to(DEV), Q.to(DEV), 1, Qp)
    torch.cuda.synchronize()
    assert_bf16_within_ulp(bits(Qp), oracle.project_q(bits(Q), bits(P)), what="Qp",
                           scale=abs_sum_scale(bits(Q), bits(P)), n_terms=128)


@pytest.mark.parametrize("nkv,bs,r,n", [(2, 16, 32, 13), (8, 16, 32, 9), (8, 32, 64, 5),
                                        (1, 16, 16, 3), (4, 48, 32, 7)])
def test_project_kv_blocks(nkv, bs, r, n):
    g = gen(nkv * 100 + bs + r)
    L, B, layer, hd = 3, 40, 2, 128
    d = dims(L=L, nq=nkv * 2, nkv=nkv, hd=hd, r=r, bs=bs, B=B)
    P = W.projection(g, hd, r)
    K = W.bf16_normal(g, (n, bs, nkv, hd))
    ids = torch.randperm(B, generator=g)[:n].to(torch.int32)
    A = torch.empty(d.a_g_shape, dtype=torch.bfloat16, device=DEV)
    A.view(torch.int16).fill_(SENTINEL)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_project_kv_blocks(d, P.to(DEV), K.to(DEV), layer, ids.to(DEV), n, A, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = np.zeros((1, B, nkv, bs, r), dtype=np.uint16)
    oracle.project_kv_blocks(bits(P), bits(K), 0, ids.numpy(), ref, nthreads=4)
    got = bits(A)
    scale = abs_sum_scale(bits(K), bits(P)).transpose(0, 2, 1, 3)  # [n, nkv, bs, r]
    assert_bf16_within_ulp(got[layer][ids.numpy()], ref[0][ids.numpy()], what="A_g slots",
                           scale=scale, n_terms=hd)
    untouched = np.ones(B, dtype=bool)
    untouched[ids.numpy()] = False
    assert (got[layer][untouched] == SENTINEL).all(), "wrote a slot that was not addressed"
    assert (got[:layer] == SENTINEL).all(), "wrote another layer"


@pytest.mark.parametrize("per_cta", [2, 3, 5])
def test_project_kv_blocks_stage_rings(per_cta):
    # The projection's ring has as many stages as a CTA has tiles (at least two): 152 * (k - 1)
    # + 1 one-tile blocks give some CTAs k tiles, so rings of 2, 3 and 5 stages wrap.
    g = gen(300 + per_cta)
    n = 152 * (per_cta - 1) + 1
    B, hd, r = n + 50, 128, 32
    d = dims(L=1, nq=32, nkv=8, hd=hd, r=r, bs=16, B=B)
    P = W.projection(g, hd, r)
    K = W.bf16_normal(g, (n, 16, 8, hd))
    ids = torch.randperm(B, generator=g)[:n].to(torch.int32)
    A = torch.empty(d.a_g_shape, dtype=torch.bfloat16, device=DEV)
    A.view(torch.int16).fill_(SENTINEL)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_project_kv_blocks(d, P.to(DEV), K.to(DEV), 0, ids.to(DEV), n, A, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = np.zeros((1, B, 8, 16, r), dtype=np.uint16)
    oracle.project_kv_blocks(bits(P), bits(K), 0, ids.numpy(), ref, nthreads=8)
    got = bits(A)
    scale = abs_sum_scale(bits(K), bits(P)).transpose(0, 2, 1, 3)
    assert_bf16_within_ulp(got[0][ids.numpy()], ref[0][ids.numpy()], what="A_g slots",
                           scale=scale, n_terms=hd)
    untouched = np.ones(B, dtype=bool)
    untouched[ids.numpy()] = False
    assert (got[0][untouched] == SENTINEL).all()


def test_project_kv_out_of_range_ids_are_skipped_and_reported():
    g = gen(77)
    d = dims(L=2, nq=8, nkv=8, hd=128, r=32, bs=16, B=16)
    P = W.projection(g, 128, 32)
    K = W.bf16_normal(g, (4, 16, 8, 128))
    ids = torch.tensor([3, -1, 16, 7], dtype=torch.int32)
    A = torch.empty(d.a_g_shape, dtype=torch.bfloat16, device=DEV)
    A.view(torch.int16).fill_(SENTINEL)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_project_kv_blocks(d, P.to(DEV), K.to(DEV), 1, ids.to(DEV), 4, A, st)
    torch.cuda.synchronize()
    assert int(st.item()) == hss.HSS_ERR_OUT_OF_RANGE
    assert hss.hss_read_device_error() == hss.HSS_ERR_OUT_OF_RANGE
    assert hss.hss_read_device_error() == hss.HSS_OK  # read clears it
    got = bits(A)[1]
    ref = np.zeros((1, 16, 8, 16, 32), dtype=np.uint16)
    oracle.project_kv_blocks(bits(P), bits(K[[0, 3]]), 0, np.array([3, 7]), ref)
    scale = abs_sum_scale(bits(K[[0, 3]]), bits(P)).transpose(0, 2, 1, 3)
    assert_bf16_within_ulp(got[[3, 7]], ref[0][[3, 7]], scale=scale, n_terms=128)
    keep = np.ones(16, dtype=bool)
    keep[[3, 7]] = False
    assert (got[keep] == SENTINEL).all()


def test_project_kv_identity_P_is_exact():
    """P = I (r = head_dim = 64): A_g holds K transposed to head-major, bit for bit."""
    g = gen(3)
    d = dims(L=1, nq=4, nkv=2, hd=64, r=64, bs=16, B=12)
    P = torch.eye(64, dtype=torch.bfloat16)
    K = W.bf16_normal(g, (12, 16, 2, 64))
    A = torch.empty(d.a_g_shape, dtype=torch.bfloat16, device=DEV)
    hss.hss_project_kv_blocks(d, P.to(DEV), K.to(DEV), 0, torch.arange(12, dtype=torch.int32,
                                                                       device=DEV), 12, A)
    Qp = torch.empty((3, 4, 64), dtype=torch.bfloat16, device=DEV)
    Q = W.bf16_normal(g, (3, 4, 64))
    hss.hss_project_q(d, P.to(DEV), Q.to(DEV), 3, Qp)
    torch.cuda.synchronize()
    assert np.array_equal(bits(A)[0], bits(K).transpose(0, 2, 1, 3))
    assert np.array_equal(bits(Qp), bits(Q))


# ----------------------------------------------------------------------------- scores

def synthetic_store(g, d, pool):
    """A_g filled directly with N(0,1) bf16 values (exercises the scorer alone)."""
    return W.bf16_normal(g, d.a_g_shape)


@pytest.mark.parametrize("nq,nkv,r,bs,rows,lengths", [
    (32, 8, 32, 16, 1, [2048]),                  # the decode layer shape
    (4, 2, 16, 16, 1, [64]),                     # tiny
    (8, 2, 32, 16, 2, [0, 5, 130, 1, 77]),       # several sequences, an empty one, 2 rows
    (16, 4, 64, 16, 4, [33, 200]),               # 16 query vectors per kv head (two n-tiles)
    (8, 8, 128, 32, 3, [17, 9]),                 # g = 1, r = 128, two token tiles per head
    (6, 3, 32, 16, 5, [40]),                     # g = 2, 10 vectors: a ragged second n-tile
])
def test_score_decode(nq, nkv, r, bs, rows, lengths):
    g = gen(nq + 7 * nkv + r + bs + rows)
    total = sum(lengths)
    L, layer = 2, 1
    B = max(total, 8) + 3
    d = dims(L=L, nq=nq, nkv=nkv, hd=128, r=r, bs=bs, B=B)
    A = synthetic_store(g, d, B)
    S = len(lengths)
    Qp = W.bf16_normal(g, (S, rows, nq, r))
    table = torch.randperm(B, generator=g)[:total].to(torch.int32)
    offs = W.identity_offsets(lengths)
    scores = torch.empty(total, dtype=torch.float32, device=DEV)
    hss.hss_score_blocks(d, Qp.to(DEV), rows, A.to(DEV), layer, table.to(DEV), offs.to(DEV), S,
                         total, scores, hss.HSS_PATH_DECODE)
    torch.cuda.synchronize()
    ref, tsum, bad = oracle.score_blocks(bits(Qp), bits(A), layer, table.numpy(),
                                         offs.numpy().astype(np.int64), nthreads=4)
    assert bad == 0
    worst = assert_scores_close(scores.cpu().numpy(), ref, tsum, "decode scores")
    assert worst < 1e-5  # fp32 accumulation of r bf16 products: far inside the tolerance


def test_score_identity_table_is_the_contiguous_layout():
    """An identity table scores the first n slots, like the page's contiguous k_lr_seq."""
    g = gen(12)
    d = dims(L=1, nq=32, nkv=8, hd=128, r=32, bs=16, B=300)
    A = synthetic_store(g, d, 300)
    Qp = W.bf16_normal(g, (1, 1, 32, 32))
    n = 257
    table = torch.arange(n, dtype=torch.int32)
    offs = torch.tensor([0, n], dtype=torch.int32)
    scores = torch.empty(n, dtype=torch.float32, device=DEV)
    hss.hss_score_blocks(d, Qp.to(DEV), 1, A.to(DEV), 0, table.to(DEV), offs.to(DEV), 1, n,
                         scores)
    ref, tsum, _ = oracle.score_blocks(bits(Qp), bits(A), 0, table.numpy(), np.array([0, n]))
    assert_scores_close(scores.cpu().numpy(), ref, tsum)


def test_score_out_of_range_ids():
    g = gen(13)
    d = dims(L=1, nq=8, nkv=2, hd=128, r=32, bs=16, B=10)
    A = synthetic_store(g, d, 10)
    Qp = W.bf16_normal(g, (1, 1, 8, 32))
    table = torch.tensor([0, 10, -5, 9, 3], dtype=torch.int32)
    offs = torch.tensor([0, 5], dtype=torch.int32)
    scores = torch.empty(5, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_score_blocks(d, Qp.to(DEV), 1, A.to(DEV), 0, table.to(DEV), offs.to(DEV), 1, 5,
                         scores, hss.HSS_PATH_AUTO, st)
    torch.cuda.synchronize()
    assert int(st.item()) == hss.HSS_ERR_OUT_OF_RANGE
    hss.hss_read_device_error()
    s = scores.cpu().numpy()
    assert math.isinf(s[1]) and s[1] > 0 and math.isinf(s[2]) and s[2] > 0
    ref, tsum, bad = oracle.score_blocks(bits(Qp), bits(A), 0, table.numpy(), np.array([0, 5]))
    assert bad == 2
    assert_scores_close(s, ref, tsum)


# ----------------------------------------------------------------------------- victims

@pytest.mark.parametrize("lengths,k", [
    ([64], 8), ([2048], 256), ([0, 1, 5, 300], 4), ([3, 3000, 17], 64),
    ([20000], 4096),            # beyond the shared-memory key cache: keys re-read per pass
    ([8192], 1024), ([65536], 4096), ([100, 7000], 8192), ([5000], 1),
])
def test_rank_victims_exact(lengths, k):
    s, offs = W.random_scores(sum(lengths) + k, lengths, ties=0.2)
    vic = torch.empty(len(lengths), k, dtype=torch.int32, device=DEV)
    hss.hss_rank_victims(s.to(DEV), offs.to(DEV), len(lengths), int(offs[-1]), k, vic)
    torch.cuda.synchronize()
    ref = oracle.rank_victims(s.numpy(), offs.numpy().astype(np.int64), k)
    assert np.array_equal(vic.cpu().numpy(), ref)


def test_rank_victims_special_values():
    s = torch.tensor([3.0, 1.0, 1.0, -2.0, 0.0, -0.0, 5.0, float("nan"), float("inf"),
                      -float("inf"), 2.0, 0.5, 0.5, 0.5], dtype=torch.float32)
    offs = torch.tensor([0, 7, 11, 11, 14], dtype=torch.int32)
    vic = torch.empty(4, 5, dtype=torch.int32, device=DEV)
    hss.hss_rank_victims(s.to(DEV), offs.to(DEV), 4, 14, 5, vic)
    torch.cuda.synchronize()
    exp = [[3, 4, 5, 1, 2], [2, 3, 0, 1, -1], [-1] * 5, [0, 1, 2, -1, -1]]
    assert vic.cpu().tolist() == exp
    ref = oracle.rank_victims(s.numpy(), offs.numpy().astype(np.int64), 5)
    assert ref.tolist() == exp


def test_rank_victims_all_equal():
    n, k = 5000, 700
    s = torch.full((n,), 1.25, dtype=torch.float32)
    offs = torch.tensor([0, n], dtype=torch.int32)
    vic = torch.empty(1, k, dtype=torch.int32, device=DEV)
    hss.hss_rank_victims(s.to(DEV), offs.to(DEV), 1, n, k, vic)
    assert vic.cpu().numpy()[0].tolist() == list(range(k))


# ----------------------------------------------------------------------------- tcgen05 scorer

@pytest.mark.parametrize("nq,nkv,r,bs,rows,lengths", [
    (64, 8, 64, 16, 40, [37]),           # 320 vectors per kv head: one full and one ragged chunk
    (16, 4, 32, 16, 100, [0, 20, 9]),    # several sequences, one empty, ragged tiles
    (8, 8, 128, 32, 600, [15]),          # g = 1, r = 128 (two K chunks), 2 slices of 512
    (32, 2, 16, 16, 70, [11]),           # g = 16, r = 16 (32-byte swizzle), 1120 vectors
    (32, 8, 32, 16, 1, [300]),           # the decode shape forced onto the tensor-core path
    (64, 8, 64, 16, 512, [24]),          # the prefill chunk shape, few blocks
    (16, 4, 32, 16, 3, [5, 0, 0, 40, 0, 17, 0]),   # empty sequences between and after
    (32, 8, 64, 16, 2, [1] * 30 + [0] * 3 + [100]),  # a CTA's units span many sequences
])
def test_score_tcgen05(nq, nkv, r, bs, rows, lengths):
    g = gen(nq * 3 + nkv + r + bs + rows)
    total = sum(lengths)
    L, layer = 2, 1
    B = max(total, 8) + 5
    d = dims(L=L, nq=nq, nkv=nkv, hd=128, r=r, bs=bs, B=B)
    A = synthetic_store(g, d, B)
    S = len(lengths)
    Qp = W.bf16_normal(g, (S, rows, nq, r))
    table = torch.randperm(B, generator=g)[:total].to(torch.int32)
    offs = W.identity_offsets(lengths)
    scores = torch.full((total,), 7.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_score_blocks(d, Qp.to(DEV), rows, A.to(DEV), layer, table.to(DEV), offs.to(DEV), S,
                         total, scores, hss.HSS_PATH_TCGEN05, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and hss.hss_read_device_error() == 0
    ref, tsum, bad = oracle.score_blocks(bits(Qp), bits(A), layer, table.numpy(),
                                         offs.numpy().astype(np.int64), nthreads=8)
    assert bad == 0
    worst = assert_scores_close(scores.cpu().numpy(), ref, tsum, "tcgen05 scores")
    assert worst < 1e-5


def test_score_tcgen05_out_of_range_ids():
    g = gen(31)
    d = dims(L=1, nq=64, nkv=8, hd=128, r=64, bs=16, B=20)
    A = synthetic_store(g, d, 20)
    Qp = W.bf16_normal(g, (1, 64, 64, 64))
    table = torch.tensor([0, 20, 5, -3, 19, 7, 8, 9, 10, 11], dtype=torch.int32)
    offs = torch.tensor([0, 10], dtype=torch.int32)
    scores = torch.empty(10, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_score_blocks(d, Qp.to(DEV), 64, A.to(DEV), 0, table.to(DEV), offs.to(DEV), 1, 10,
                         scores, hss.HSS_PATH_TCGEN05, st)
    torch.cuda.synchronize()
    assert int(st.item()) == hss.HSS_ERR_OUT_OF_RANGE
    hss.hss_read_device_error()
    ref, tsum, bad = oracle.score_blocks(bits(Qp), bits(A), 0, table.numpy(), np.array([0, 10]))
    assert bad == 2
    assert_scores_close(scores.cpu().numpy(), ref, tsum)


def test_decode_and_tcgen05_paths_agree():
    """Both kernels on the same decode-shaped inputs (each also checked against the oracle)."""
    g = gen(41)
    d = dims(L=1, nq=32, nkv=8, hd=128, r=32, bs=16, B=700)
    A = synthetic_store(g, d, 700).to(DEV)
    Qp = W.bf16_normal(g, (2, 2, 32, 32)).to(DEV)
    table = torch.randperm(700, generator=g)[:650].to(torch.int32).to(DEV)
    offs = torch.tensor([0, 300, 650], dtype=torch.int32, device=DEV)
    out = []
    for path in (hss.HSS_PATH_DECODE, hss.HSS_PATH_TCGEN05):
        sc = torch.empty(650, dtype=torch.float32, device=DEV)
        hss.hss_score_blocks(d, Qp, 2, A, 0, table, offs, 2, 650, sc, path)
        out.append(sc)
    torch.cuda.synchronize()
    ref, tsum, _ = oracle.score_blocks(bits(Qp), bits(A), 0, table.cpu().numpy(),
                                       offs.cpu().numpy().astype(np.int64), nthreads=8)
    for sc in out:
        assert_scores_close(sc.cpu().numpy(), ref, tsum)


def test_binding_uses_the_current_stream():
    # The binding reads the current stream's raw handle; it must be torch's current stream,
    # on the default stream and inside a stream context.
    assert hss._stream(None) == torch.cuda.current_stream().cuda_stream
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert hss._stream(None) == s.cuda_stream
