"""End to end on the five workloads: project K into A_g, project Q, score, rank victims --
all through the C ABI -- against the oracle on the same seeded inputs.

Small cases are compared in full.  At full size the oracle recomputes sampled outputs one
by one (A_g slots, block scores), and properties that hold at any size are checked on the
rest (the GPU victim list is the ascending order of the GPU's own scores)."""
import json
import os

import numpy as np
import pytest
import torch

import kv_cache_block_lowrank_gb300 as hss
import oracle
import workloads as W
from gpu_util import (SENTINEL, GpuRun, assert_bf16_within_ulp, assert_scores_close,
                      assert_victims_match, bits, oracle_slots, q_scale, slot_scale)

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
    # Oracle: every slot of the layer, Qp, all 2048 scores, the victims.
    A_o = np.zeros((1,) + d.a_g_shape[1:], dtype=np.uint16)
    oracle.project_kv_blocks(bits(case.P), bits(case.K[layer]), 0, case.block_ids.numpy(), A_o,
                             nthreads=NT)
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
    """64 sequences from a 40000-block pool, bottom-64 each."""
    case = W.batched(seed=0, device=DEV)
    d = case.dims
    run = GpuRun(case)
    run.ingest(0, 0)
    Qp = run.project_q(0)
    scores = run.score(Qp, 0)
    vic = run.rank(scores)
    torch.cuda.synchronize()
    assert int(run.status.item()) == 0
    offs = offsets64(case)
    table = case.table.numpy()
    s_g = scores.cpu().numpy()
    v_g = vic.cpu().numpy()
    Qp_o = oracle.project_q(bits(case.Q[0]), bits(case.P))
    assert_bf16_within_ulp(bits(Qp), Qp_o, what="Qp", scale=q_scale(case), n_terms=d.head_dim)
    # Two whole sequences: every score and the victim set.
    for s in (0, 37):
        a, b = int(offs[s]), int(offs[s + 1])
        ids = table[a:b]
        A_o = np.zeros((1, d.max_blocks, d.num_kv_heads, d.block_size, d.r), dtype=np.uint16)
        A_o[0, ids] = oracle_slots(case, 0, ids)  # pool position == block id here
        sub_offs = np.array([0, b - a])
        s_o, t_o, _ = oracle.score_blocks(Qp_o[s:s + 1], A_o, 0, ids, sub_offs, nthreads=NT)
        assert_scores_close(s_g[a:b], s_o, t_o, f"seq {s}")
        assert_victims_match(v_g[s:s + 1], s_o, t_o, sub_offs, case.k_victims,
                             gpu_scores=s_g[a:b])
    # Every other sequence: its victim list is the order of its GPU scores.
    for s in range(case.num_seqs):
        a, b = int(offs[s]), int(offs[s + 1])
        n = b - a
        exp = np.lexsort((np.arange(n), s_g[a:b]))[:case.k_victims]
        assert np.array_equal(v_g[s][:len(exp)], exp)


def test_ingest_and_score_full_size():
    """4096 new blocks into each of 32 layers (skewed keys), then 65536 blocks scored."""
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
    for layer in (0, L, 31):
        pos = rng.choice(len(new_ids), 16, replace=False)
        assert_bf16_within_ulp(bits(run.A[layer][torch.as_tensor(new_ids[pos])]),
                               oracle_slots(case, layer, pos), what=f"A_g layer {layer}",
                               scale=slot_scale(case, layer, pos), n_terms=d.head_dim)
    Qp_o = oracle.project_q(bits(case.Q[0]), bits(case.P))
    assert_bf16_within_ulp(bits(Qp), Qp_o, what="Qp", scale=q_scale(case), n_terms=d.head_dim)
    # Sampled scores: the oracle projects each sampled block from its own K.
    table = case.table.numpy()
    where_new = {int(b): i for i, b in enumerate(new_ids)}
    where_fill = {int(b): i for i, b in enumerate(case.fill_ids.numpy())}
    ent = rng.choice(d.max_blocks, 384, replace=False)
    A_o = np.zeros((1, d.max_blocks, d.num_kv_heads, d.block_size, d.r), dtype=np.uint16)
    for e in ent:
        bid = int(table[e])
        if bid in where_new:
            A_o[0, bid] = oracle_slots(case, L, [where_new[bid]], nthreads=1)[0]
        else:
            Kb = bits(case.K_fill[where_fill[bid]:where_fill[bid] + 1])
            tmp = np.zeros((1, 1, d.num_kv_heads, d.block_size, d.r), dtype=np.uint16)
            oracle.project_kv_blocks(bits(case.P), Kb, 0, np.array([0]), tmp)
            A_o[0, bid] = tmp[0, 0]
    s_o, t_o, _ = oracle.score_entries(Qp_o, A_o, 0, table, offsets64(case), ent)
    s_g = scores.cpu().numpy()
    assert_scores_close(s_g[ent], s_o, t_o, "sampled scores")
    v_g = vic.cpu().numpy()[0]
    exp = np.lexsort((np.arange(d.max_blocks), s_g))[:case.k_victims]
    assert np.array_equal(v_g, exp)


def test_prefill_chunk_full_size():
    """512 query rows x 64 heads against 8192 blocks (tensor-core path), bottom-1024."""
    case = W.prefill(seed=0, device=DEV)
    d = case.dims
    run = GpuRun(case)
    run.ingest(0, 0)
    Qp = run.project_q(0)
    scores = run.score(Qp, 0)            # auto: 4096 query vectors per kv head -> tcgen05
    vic = run.rank(scores)
    torch.cuda.synchronize()
    assert int(run.status.item()) == 0 and hss.hss_read_device_error() == 0
    Qp_o = oracle.project_q(bits(case.Q[0]), bits(case.P), nthreads=NT)
    assert_bf16_within_ulp(bits(Qp), Qp_o, what="Qp", scale=q_scale(case), n_terms=d.head_dim)
    rng = np.random.default_rng(4)
    ent = rng.choice(d.max_blocks, 24, replace=False)
    table = case.table.numpy()
    A_o = np.zeros((1, d.max_blocks, d.num_kv_heads, d.block_size, d.r), dtype=np.uint16)
    ids = table[ent]
    A_o[0, ids] = oracle_slots(case, 0, ids)
    s_o, t_o, _ = oracle.score_entries(Qp_o, A_o, 0, table, offsets64(case), ent)
    s_g = scores.cpu().numpy()
    assert_scores_close(s_g[ent], s_o, t_o, "sampled prefill scores")
    exp = np.lexsort((np.arange(d.max_blocks), s_g))[:case.k_victims]
    assert np.array_equal(vic.cpu().numpy()[0], exp)
