"""hss_write_kv_tokens (the paged cache write with the A_g projection, one token at a time)
against the oracle and against hss_project_kv_blocks."""
import numpy as np
import pytest
import torch

import kv_cache_block_lowrank_gb300 as hss
import oracle
import workloads as W
from gpu_util import SENTINEL, abs_sum_scale, assert_bf16_within_ulp, bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_block_lowrank_gb300 import _build

    _build.build()
    hss.load()


def run_tokens(d, P, K_tok, slots, layer, with_cache=True):
    """Call the GPU path on sentinel-filled A_g and cache; return (A_g bits, cache bits,
    status)."""
    A = torch.empty(d.a_g_shape, dtype=torch.bfloat16, device=DEV)
    A.view(torch.int16).fill_(SENTINEL)
    C = None
    if with_cache:
        C = torch.empty(d.max_blocks, d.block_size, d.num_kv_heads, d.head_dim,
                        dtype=torch.bfloat16, device=DEV)
        C.view(torch.int16).fill_(SENTINEL)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_write_kv_tokens(d, P.to(DEV), K_tok.to(DEV), slots.to(DEV), slots.numel(), C, A,
                            layer, st)
    torch.cuda.synchronize()
    return bits(A), (bits(C) if with_cache else None), int(st.item())


def oracle_tokens(d, P, K_tok, slots, layer):
    A = np.full(d.a_g_shape, SENTINEL, dtype=np.uint16)
    C = np.full((d.max_blocks, d.block_size, d.num_kv_heads, d.head_dim), SENTINEL,
                dtype=np.uint16)
    st = oracle.write_kv_tokens(bits(P), bits(K_tok), slots.numpy(), layer, A, K_cache=C,
                                nthreads=4)
    return A, C, st


@pytest.mark.parametrize("nkv,hd,r,bs,B,n", [
    (8, 128, 32, 16, 64, 700),     # the decode layer's dims, several hundred tokens
    (1, 64, 16, 16, 8, 100),       # one kv head, small r
    (4, 192, 64, 32, 20, 333),     # head_dim 192, block 32
    (2, 256, 128, 16, 12, 150),    # head_dim 256, r 128
    (8, 128, 32, 16, 4, 3),        # fewer rows than one tile
])
def test_tokens_against_oracle(nkv, hd, r, bs, B, n):
    g = torch.Generator().manual_seed(nkv * 1000 + hd + r + n)
    d = W.Dims(2, nkv * 2, nkv, hd, r, bs, B)
    P = W.projection(g, hd, r)
    K_tok = W.bf16_normal(g, (n, nkv, hd))
    perm = torch.randperm(B * bs, generator=g)[:n].to(torch.int64)
    perm[::17] = -1  # padding tokens
    A, C, st = run_tokens(d, P, K_tok, perm, layer=1)
    A_o, C_o, st_o = oracle_tokens(d, P, K_tok, perm, layer=1)
    assert st == 0 and st_o == 0
    assert np.array_equal(C, C_o), "cache rows differ (they are copies)"
    written = (A_o[1] != SENTINEL).any(axis=-1)  # [B, nkv, bs]
    assert np.array_equal((A[1] != SENTINEL).any(axis=-1), written)
    scale_tok = abs_sum_scale(bits(K_tok), bits(P))  # [n, nkv, r]
    scale = np.zeros(A_o.shape[1:])
    for i, s in enumerate(perm.tolist()):
        if s >= 0:
            scale[s // bs, :, s % bs] = scale_tok[i]
    assert_bf16_within_ulp(A[1][written], A_o[1][written], what="A_g rows",
                           scale=scale[written], n_terms=hd)
    assert (A[0] == SENTINEL).all(), "wrote another layer"


def test_tokens_equal_block_projection():
    # Whole blocks written one token at a time (shuffled) give exactly the slots that
    # hss_project_kv_blocks writes for those blocks: the same kernel computes every row.
    g = torch.Generator().manual_seed(5)
    d = W.Dims(1, 32, 8, 128, 32, 16, 40)
    P = W.projection(g, 128, 32)
    n_blk = 24
    ids = torch.randperm(40, generator=g)[:n_blk].to(torch.int32)
    K = W.bf16_normal(g, (n_blk, 16, 8, 128))
    A_blk = torch.empty(d.a_g_shape, dtype=torch.bfloat16, device=DEV)
    A_blk.view(torch.int16).fill_(SENTINEL)
    hss.hss_project_kv_blocks(d, P.to(DEV), K.to(DEV), 0, ids.to(DEV), n_blk, A_blk)
    order = torch.randperm(n_blk * 16, generator=g)
    blk_of = order // 16
    slots = (ids[blk_of].to(torch.int64) * 16 + order % 16)
    K_tok = K.reshape(n_blk * 16, 8, 128)[order]
    A, C, st = run_tokens(d, P, K_tok, slots, layer=0)
    assert st == 0
    assert np.array_equal(A, bits(A_blk))
    assert np.array_equal(C[ids.numpy()], bits(K))


def test_tokens_out_of_range_and_no_cache():
    g = torch.Generator().manual_seed(9)
    d = W.Dims(1, 16, 8, 128, 32, 16, 10)
    P = W.projection(g, 128, 32)
    K_tok = W.bf16_normal(g, (4, 8, 128))
    slots = torch.tensor([3, 10 * 16, -5, 159], dtype=torch.int64)
    A, C, st = run_tokens(d, P, K_tok, slots, layer=0, with_cache=False)
    assert C is None
    assert st == hss.HSS_ERR_OUT_OF_RANGE
    assert hss.hss_read_device_error() == hss.HSS_ERR_OUT_OF_RANGE
    A_o, _, st_o = oracle_tokens(d, P, K_tok, slots, layer=0)
    assert st_o == 2
    rows = (A_o[0] != SENTINEL).any(axis=-1)
    assert rows.sum() == 2 * 8  # the two valid tokens, every kv head
    assert np.array_equal((A[0] != SENTINEL).any(axis=-1), rows)
    scale = abs_sum_scale(bits(K_tok), bits(P))
    sc = np.zeros(A_o.shape[1:])
    sc[0, :, 3] = scale[0]
    sc[9, :, 15] = scale[3]
    assert_bf16_within_ulp(A[0][rows], A_o[0][rows], scale=sc[rows], n_terms=128)


def test_tokens_decode_step_full_size():
    # One decode step of a 4096-sequence batch: one new token per sequence into a
    # 65536-block pool (the ingest workload's dims); sampled rows against the oracle.
    g = torch.Generator().manual_seed(11)
    d = W.Dims(32, 32, 8, 128, 32, 16, 65536)
    P = W.projection(g, 128, 32)
    n = 4096
    K_tok = W.bf16_normal(g, (n, 8, 128))
    slots = torch.randperm(65536 * 16, generator=g)[:n].to(torch.int64)
    A = torch.empty(d.a_g_shape, dtype=torch.bfloat16, device=DEV)
    C = torch.empty(65536, 16, 8, 128, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_write_kv_tokens(d, P.to(DEV), K_tok.to(DEV), slots.to(DEV), n, C, A, 17, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    pick = torch.randperm(n, generator=g)[:64]
    sl = slots[pick]
    blk, t = (sl // 16).to(DEV), (sl % 16).to(DEV)
    got_A = bits(A[17][blk, :, t])          # [64, nkv, r]
    got_C = bits(C[blk, t])                 # [64, nkv, hd]
    assert np.array_equal(got_C, bits(K_tok[pick]))
    ref = oracle.project_q(bits(K_tok[pick]), bits(P))  # same row math: bf16(row . P)
    assert_bf16_within_ulp(got_A, ref, scale=abs_sum_scale(bits(K_tok[pick]), bits(P)),
                           n_terms=128, what="A_g rows")
