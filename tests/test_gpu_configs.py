"""End to end on the five workloads: project K into A_g, project Q, score, rank victims --
all through the C ABI -- against the oracle on the same seeded inputs.

Every workload is compared in full, at its full size: the scored layer's whole A_g, Qp,
every block score (within 2e-3 * sum|terms| + 1e-6) and every sequence's victim set (exact
outside the tolerance band around the oracle's k-th score).  The GPU victim list is also
checked to be the exact ascending (score, index) order of the GPU's own scores.  Layers
that are written but not scored are checked on sampled slots."""
import json
import os

import numpy as np
import pytest
import torch

import kv_cache_block_lowrank_gb300 as hss
import oracle
import workloads as W
from gpu_util import (SENTINEL, GpuRun, assert_bf16_within_ulp, assert_scores_close,
                      assert_victims_match, bits, oracle_slots, q_scale, slot_scale,
                      slot_scale_fn)

pytestmark = pytest.mark.gpu
DEV = "cuda"
NT = oracle.default_threads()
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_block_lowrank_gb300 import _build

    _build.build()
    hss.load()


def offsets64(case):
    return case.seq_offsets.numpy().astype(np.int64)


def test_tiny_end_to_end():
    case = W.tiny(seed=0)
    d = case.dims
    run = GpuRun(case)
    run.fill_sentinel()
    run.ingest(0, 0)
    Qp = run.project_q(0)
    scores = run.score(Qp, 0)
    vic = run.rank(scores)
    torch.cuda.synchronize()
    assert int(run.status.item()) == 0

    P = bits(case.P)
    A_o = np.zeros(d.a_g_shape, dtype=np.uint16)
    assert oracle.project_kv_blocks(P, bits(case.K[0]), 0, case.block_ids.numpy(), A_o) == 0
    Qp_o = oracle.project_q(bits(case.Q[0]), P)
    s_o, t_o, bad = oracle.score_blocks(Qp_o, A_o, 0, case.table.numpy(), offsets64(case))
    assert bad == 0
    hd = d.head_dim
    assert_bf16_within_ulp(bits(run.A)[0], A_o[0], what="A_g",
                           scale=slot_scale(case, 0, np.arange(d.max_blocks)), n_terms=hd)
    assert_bf16_within_ulp(bits(Qp), Qp_o, what="Qp", scale=q_scale(case), n_terms=hd)
    s_g = scores.cpu().numpy()
    assert_scores_close(s_g, s_o, t_o, "scores")
    assert_victims_match(vic.cpu().numpy(), s_o, t_o, offsets64(case), case.k_victims,
                         gpu_scores=s_g)


def test_hand_example_on_gpu():
    """The hand-worked three-block example, zero-padded to a supported shape.

    head_dim 2 -> 64 and r 2 -> 16 with zeros (adds nothing to any dot product); block_size
    2 -> 16 by repeating the block's two tokens (a max over repeated candidates is unchanged).
    """
    g = json.load(open(os.path.join(GOLDEN, "hand_three_block.json")))
    hd, r, bs, nb = 64, 16, 16, 3
    d = W.Dims(1, 2, 1, hd, r, bs, nb)
    P = torch.zeros(hd, r)
    P[:2, :2] = torch.tensor(g["P"], dtype=torch.float32)
    Q = torch.zeros(1, 2, hd)
    Q[0, :, :2] = torch.tensor(g["Q"], dtype=torch.float32)
    K = torch.zeros(nb, bs, 1, hd)
    k2 = torch.tensor(g["K"], dtype=torch.float32)          # [3 blocks, 2 tokens, 1 head, 2]
    for t in range(bs):
        K[:, t, :, :2] = k2[:, t % 2]
    P, Q, K = (x.to(torch.bfloat16).to(DEV) for x in (P, Q, K))
    A = torch.zeros(d.a_g_shape, dtype=torch.bfloat16, device=DEV)
    hss.hss_project_kv_blocks(d, P, K, 0, torch.arange(nb, dtype=torch.int32, device=DEV), nb, A)
    Qp = torch.empty(1, 2, r, dtype=torch.bfloat16, device=DEV)
    hss.hss_project_q(d, P, Q, 1, Qp)
    torch.cuda.synchronize()
    assert Qp[0, :, :2].float().cpu().tolist() == g["expected_Qp"]
    assert (Qp[0, :, 2:] == 0).all()
    assert A[0, :, :, :2, :2].float().cpu().tolist() == g["expected_A_g_slots"]
    for c in g["cases"]:
        table = torch.tensor(c["table"], dtype=torch.int32, device=DEV)
        offs = torch.tensor(c["seq_offsets"], dtype=torch.int32, device=DEV)
        S = len(c["seq_offsets"]) - 1
        QpS = Qp.reshape(1, 1, 2, r).repeat(S, 1, 1, 1).contiguous()
        sc = torch.empty(len(c["table"]), dtype=torch.float32, device=DEV)
        hss.hss_score_blocks(d, QpS, 1, A, 0, table, offs, S, len(c["table"]), sc)
        vic = torch.empty(S, c["k"], dtype=torch.int32, device=DEV)
        hss.hss_rank_victims(sc, offs, S, len(c["table"]), c["k"], vic)
        torch.cuda.synchronize()
        assert sc.cpu().tolist() == [float(x) for x in c["expected_scores"]]
        assert vic.cpu().tolist() == c["expected_victims"]


def oracle_layer(case, parts):
    """The oracle's A_g for one layer: parts = [(K blocks [n, bs, nkv, hd], ids [n])]."""
    d = case.dims
    A_o = np.zeros((1,) + d.a_g_shape[1:], dtype=np.uint16)
    for K, ids in parts:
        st = oracle.project_kv_blocks(bits(case.P), bits(K), 0, np.asarray(ids, dtype=np.int32),
                                      A_o, nthreads=NT)
        assert st == 0
    return A_o


def test_decode_layer_full_size():
    """2048 blocks x 32 layers (Llama-3-8B-like decode layer), bottom-256, seed 0."""
    case = W.decode(seed=0, device=DEV)
    d = case.dims
    run = GpuRun(case)
    for layer in range(d.num_layers):
        run.ingest(layer, layer)
    torch.cuda.synchronize()
    assert int(run.status.item()) == 0
    rng = np.random.default_rng(0)
    A_g = run.A
    for layer in (0, 13, 31):
        pos = rng.choice(d.max_blocks, 24, replace=False)
        ids = case.block_ids.numpy()[pos]
        assert_bf16_within_ulp(bits(A_g[layer][torch.as_tensor(ids)]),
                               oracle_slots(case, layer, pos), what=f"A_g layer {layer}",
                               scale=slot_scale(case, layer, pos), n_terms=d.head_dim)
    layer = 17
    Qp = run.project_q(layer)
    scores = run.score(Qp, layer)
    vic = run.rank(scores)
    torch.cuda.synchronize()
    # Oracle: every slot of the layer (compared in full), Qp, all 2048 scores, the victims.
    ids = case.block_ids.numpy()
    A_o = oracle_layer(case, [(case.K[layer], ids)])
    assert_bf16_within_ulp(bits(A_g[layer][case.block_ids.long().to(DEV)]), A_o[0][ids],
                           what="A_g layer 17 (every slot)",
                           scale=slot_scale_fn(case.K[layer], case.P), n_terms=d.head_dim)
    Qp_o = oracle.project_q(bits(case.Q[layer]), bits(case.P))
    assert_bf16_within_ulp(bits(Qp), Qp_o, what="Qp", scale=q_scale(case, layer),
                           n_terms=d.head_dim)
    s_o, t_o, _ = oracle.score_blocks(Qp_o, A_o, 0, case.table.numpy(), offsets64(case),
                                      nthreads=NT)
    s_g = scores.cpu().numpy()
    assert_scores_close(s_g, s_o, t_o, "scores")
    assert_victims_match(vic.cpu().numpy(), s_o, t_o, offsets64(case), case.k_victims,
                         gpu_scores=s_g)


def test_batched_decode_full_size():
    """64 sequences from a 40000-block pool, bottom-64 each: every slot of the pool, every
    score and all 64 victim sets against the oracle."""
    case = W.batched(seed=0, device=DEV)
    d = case.dims
    run = GpuRun(case)
    run.ingest(0, 0)
    Qp = run.project_q(0)
    scores = run.score(Qp, 0)
    vic = run.rank(scores)
    torch.cuda.synchronize()
    assert int(run.status.item()) == 0
    ids = case.block_ids.numpy()                    # the whole pool, id == position
    A_o = oracle_layer(case, [(case.K[0], ids)])
    assert_bf16_within_ulp(bits(run.A[0][case.block_ids.long().to(DEV)]), A_o[0][ids],
                           what="A_g (every pool slot)", scale=slot_scale_fn(case.K[0], case.P),
                           n_terms=d.head_dim)
    Qp_o = oracle.project_q(bits(case.Q[0]), bits(case.P))
    assert_bf16_within_ulp(bits(Qp), Qp_o, what="Qp", scale=q_scale(case), n_terms=d.head_dim)
    s_o, t_o, bad = oracle.score_blocks(Qp_o, A_o, 0, case.table.numpy(), offsets64(case),
                                        nthreads=NT)
    assert bad == 0
    s_g = scores.cpu().numpy()
    assert_scores_close(s_g, s_o, t_o, "scores (all 64 sequences)")
    assert_victims_match(vic.cpu().numpy(), s_o, t_o, offsets64(case), case.k_victims,
                         gpu_scores=s_g)


def test_ingest_and_score_full_size():
    """4096 new blocks into each of 32 layers (skewed keys), then 65536 blocks scored: the
    scored layer's every slot, every score and the bottom-4096 set against the oracle."""
    case = W.ingest(seed=0, device=DEV)
    d = case.dims
    run = GpuRun(case)
    for li, layer in enumerate(case.ingest_layers):
        run.ingest(li, layer)
    L = case.score_layer
    fill_ids = case.fill_ids.to(DEV)
    hss.hss_project_kv_blocks(d, run.P, case.K_fill, L, fill_ids, fill_ids.numel(), run.A,
                              run.status)
    Qp = run.project_q(0)
    scores = run.score(Qp, L)
    vic = run.rank(scores)
    torch.cuda.synchronize()
    assert int(run.status.item()) == 0
    rng = np.random.default_rng(1)
    new_ids = case.block_ids.numpy()
    for layer in (0, 31):
        pos = rng.choice(len(new_ids), 16, replace=False)
        assert_bf16_within_ulp(bits(run.A[layer][torch.as_tensor(new_ids[pos])]),
                               oracle_slots(case, layer, pos), what=f"A_g layer {layer}",
                               scale=slot_scale(case, layer, pos), n_terms=d.head_dim)
    li = case.ingest_layers.index(L)
    A_o = oracle_layer(case, [(case.K[li], new_ids), (case.K_fill, case.fill_ids.numpy())])
    for K, ids, what in ((case.K[li], case.block_ids, "new"), (case.K_fill, case.fill_ids,
                                                               "filled")):
        assert_bf16_within_ulp(bits(run.A[L][ids.long().to(DEV)]), A_o[0][ids.numpy()],
                               what=f"A_g layer {L}, {what} slots",
                               scale=slot_scale_fn(K, case.P), n_terms=d.head_dim)
    Qp_o = oracle.project_q(bits(case.Q[0]), bits(case.P))
    assert_bf16_within_ulp(bits(Qp), Qp_o, what="Qp", scale=q_scale(case), n_terms=d.head_dim)
    s_o, t_o, bad = oracle.score_blocks(Qp_o, A_o, 0, case.table.numpy(), offsets64(case),
                                        nthreads=NT)
    assert bad == 0
    s_g = scores.cpu().numpy()
    assert_scores_close(s_g, s_o, t_o, "scores (all 65536)")
    assert_victims_match(vic.cpu().numpy(), s_o, t_o, offsets64(case), case.k_victims,
                         gpu_scores=s_g)


def test_prefill_chunk_full_size():
    """512 query rows x 64 heads against 8192 blocks (tensor-core path), bottom-1024: every
    slot, every score (the oracle's ~2.7e11 fp64 multiply-adds) and the victim set."""
    case = W.prefill(seed=0, device=DEV)
    d = case.dims
    run = GpuRun(case)
    run.ingest(0, 0)
    Qp = run.project_q(0)
    scores = run.score(Qp, 0)            # auto: 4096 query vectors per kv head -> tcgen05
    vic = run.rank(scores)
    torch.cuda.synchronize()
    assert int(run.status.item()) == 0 and hss.hss_read_device_error() == 0
    ids = case.block_ids.numpy()
    A_o = oracle_layer(case, [(case.K[0], ids)])
    assert_bf16_within_ulp(bits(run.A[0][case.block_ids.long().to(DEV)]), A_o[0][ids],
                           what="A_g (every slot)", scale=slot_scale_fn(case.K[0], case.P),
                           n_terms=d.head_dim)
    Qp_o = oracle.project_q(bits(case.Q[0]), bits(case.P), nthreads=NT)
    assert_bf16_within_ulp(bits(Qp), Qp_o, what="Qp", scale=q_scale(case), n_terms=d.head_dim)
    s_o, t_o, bad = oracle.score_blocks(Qp_o, A_o, 0, case.table.numpy(), offsets64(case),
                                        nthreads=NT)
    assert bad == 0
    s_g = scores.cpu().numpy()
    assert_scores_close(s_g, s_o, t_o, "scores (all 8192)")
    assert_victims_match(vic.cpu().numpy(), s_o, t_o, offsets64(case), case.k_victims,
                         gpu_scores=s_g)
