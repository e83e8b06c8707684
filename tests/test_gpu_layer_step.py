"""hss_layer_step (one fused layer call) against the four separate calls and the oracle."""
import numpy as np
import pytest
import torch

import kv_cache_block_lowrank_gb300 as hss
import oracle
import workloads as W
from gpu_util import assert_scores_close, assert_victims_match, bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_block_lowrank_gb300 import _build

    _build.build()
    hss.load()


def make(dims, lengths, rows, n_new, seed, pool_extra=7):
    g = torch.Generator().manual_seed(seed)
    total = sum(lengths)
    B = dims.max_blocks
    P = W.projection(g, dims.head_dim, dims.r).to(DEV)
    A = W.bf16_normal(g, dims.a_g_shape).to(DEV)
    table = torch.randperm(B, generator=g)[:total].to(torch.int32)
    new_ids = table[torch.randperm(total, generator=g)[:n_new]].contiguous() if n_new else \
        torch.zeros(0, dtype=torch.int32)
    K_new = W.bf16_normal(g, (max(n_new, 1), dims.block_size, dims.num_kv_heads, dims.head_dim))
    S = len(lengths)
    Q = W.bf16_normal(g, (S, rows, dims.num_q_heads, dims.head_dim))
    offs = W.identity_offsets(lengths)
    return dict(P=P, A=A, table=table.to(DEV), new_ids=new_ids.to(DEV), K_new=K_new.to(DEV),
                Q=Q.to(DEV), offs=offs.to(DEV), S=S, rows=rows, total=total, n_new=n_new)


def separate(d, x, layer, k):
    A = x["A"].clone()
    if x["n_new"]:
        hss.hss_project_kv_blocks(d, x["P"], x["K_new"], layer, x["new_ids"], x["n_new"], A)
    Qp = torch.empty(x["S"], x["rows"], d.num_q_heads, d.r, dtype=torch.bfloat16, device=DEV)
    hss.hss_project_q(d, x["P"], x["Q"], x["S"] * x["rows"], Qp)
    sc = torch.empty(x["total"], dtype=torch.float32, device=DEV)
    hss.hss_score_blocks(d, Qp, x["rows"], A, layer, x["table"], x["offs"], x["S"], x["total"], sc)
    vic = torch.empty(x["S"], k, dtype=torch.int32, device=DEV)
    hss.hss_rank_victims(sc, x["offs"], x["S"], x["total"], k, vic)
    torch.cuda.synchronize()
    return A, Qp, sc, vic


def fused(d, x, layer, k, ws=None, A=None):
    A = x["A"].clone() if A is None else A
    Qp = torch.empty(x["S"], x["rows"], d.num_q_heads, d.r, dtype=torch.bfloat16, device=DEV)
    sc = torch.empty(x["total"], dtype=torch.float32, device=DEV)
    vic = torch.full((x["S"], k), 12345, dtype=torch.int32, device=DEV)
    nb = hss.hss_layer_step_workspace_bytes(x["S"])
    if ws is None:
        ws = torch.zeros(max(nb, 4) // 4, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_layer_step(d, x["P"], x["K_new"], x["new_ids"], x["n_new"], x["Q"], x["rows"], Qp, A,
                       layer, x["table"], x["offs"], x["S"], x["total"], sc, k, vic, ws, nb, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return A, Qp, sc, vic, ws


@pytest.mark.parametrize("shape,lengths,rows,n_new,k", [
    ((2, 32, 8, 128, 32, 16, 2100), [2048], 1, 1, 256),           # the decode layer
    ((1, 8, 2, 128, 32, 16, 900), [0, 5, 300, 1, 0, 77, 400], 2, 3, 8),   # many sequences
    ((1, 16, 4, 128, 64, 16, 700), [600], 4, 2, 600),            # k == n
    ((1, 32, 8, 128, 32, 16, 40000), [20000, 15000], 1, 4, 64),  # beyond the fused cache
    ((1, 64, 8, 128, 64, 16, 600), [300, 200], 24, 2, 100),      # tcgen05 scorer
])
def test_layer_step_equals_separate_calls(shape, lengths, rows, n_new, k):
    d = W.Dims(*shape)
    x = make(d, lengths, rows, n_new, seed=sum(shape) + rows)
    layer = d.num_layers - 1
    A1, Qp1, sc1, vic1 = separate(d, x, layer, k)
    A2, Qp2, sc2, vic2, ws = fused(d, x, layer, k)
    assert torch.equal(A1.view(torch.int16), A2.view(torch.int16))
    assert torch.equal(Qp1.view(torch.int16), Qp2.view(torch.int16))
    assert torch.equal(sc1, sc2)
    assert torch.equal(vic1, vic2)
    assert int(ws.abs().sum()) == 0, "the workspace must be left zeroed"
    # A second call on the same workspace gives the same answer.
    _, _, sc3, vic3, _ = fused(d, x, layer, k, ws=ws)
    assert torch.equal(sc2, sc3) and torch.equal(vic2, vic3)


def test_layer_step_against_oracle():
    case = W.tiny(seed=3)
    d = case.dims
    P = case.P.to(DEV)
    A = torch.zeros(d.a_g_shape, dtype=torch.bfloat16, device=DEV)
    ids = case.block_ids.to(DEV)
    hss.hss_project_kv_blocks(d, P, case.K[0][:60].to(DEV), 0, ids[:60], 60, A)  # context
    new_ids = ids[60:].contiguous()                                           # this step's blocks
    Qp = torch.empty(1, 1, d.num_q_heads, d.r, dtype=torch.bfloat16, device=DEV)
    sc = torch.empty(64, dtype=torch.float32, device=DEV)
    vic = torch.empty(1, 8, dtype=torch.int32, device=DEV)
    ws = torch.zeros(64, dtype=torch.int32, device=DEV)
    table, offs = case.table.to(DEV), case.seq_offsets.to(DEV)
    hss.hss_layer_step(d, P, case.K[0][60:].to(DEV), new_ids, 4, case.Q[0].to(DEV), 1, Qp, A, 0,
                       table, offs, 1, 64, sc, 8, vic, ws, 256)
    torch.cuda.synchronize()
    A_o = np.zeros(d.a_g_shape, dtype=np.uint16)
    oracle.project_kv_blocks(bits(case.P), bits(case.K[0]), 0, case.block_ids.numpy(), A_o)
    Qp_o = oracle.project_q(bits(case.Q[0]), bits(case.P))
    s_o, t_o, _ = oracle.score_blocks(Qp_o, A_o, 0, case.table.numpy(),
                                      case.seq_offsets.numpy().astype(np.int64))
    s_g = sc.cpu().numpy()
    assert_scores_close(s_g, s_o, t_o)
    assert_victims_match(vic.cpu().numpy(), s_o, t_o, case.seq_offsets.numpy(), 8, gpu_scores=s_g)


def inline_vs_oracle(d, x, layer, k):
    """hss_layer_step with Qp = NULL (queries projected inside the scorer) against the
    oracle; the new slots must equal the projection kernel's, bit for bit."""
    A = x["A"].clone()
    sc = torch.empty(x["total"], dtype=torch.float32, device=DEV)
    vic = torch.full((x["S"], k), 12345, dtype=torch.int32, device=DEV)
    nb = hss.hss_layer_step_workspace_bytes(x["S"])
    ws = torch.zeros(max(nb, 4) // 4, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_layer_step(d, x["P"], x["K_new"], x["new_ids"], x["n_new"], x["Q"], x["rows"], None,
                       A, layer, x["table"], x["offs"], x["S"], x["total"], sc, k, vic, ws, nb, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert int(ws.abs().sum()) == 0, "the workspace must be left zeroed"
    A_ref, _, _, _ = separate(d, x, layer, k)
    assert torch.equal(A.view(torch.int16), A_ref.view(torch.int16))
    Qp_o = oracle.project_q(bits(x["Q"].cpu()).reshape(-1, d.num_q_heads, d.head_dim),
                            bits(x["P"].cpu()))
    Qp_o = Qp_o.reshape(x["S"], x["rows"], d.num_q_heads, d.r)
    offs = x["offs"].cpu().numpy().astype(np.int64)
    s_o, t_o, _ = oracle.score_blocks(Qp_o, bits(A_ref.cpu()), layer, x["table"].cpu().numpy(),
                                      offs)
    s_g = sc.cpu().numpy()
    assert_scores_close(s_g, s_o, t_o)
    assert_victims_match(vic.cpu().numpy(), s_o, t_o, offs, k, gpu_scores=s_g)


@pytest.mark.parametrize("shape,lengths,rows,n_new,k", [
    ((2, 32, 8, 128, 32, 16, 2100), [2048], 1, 1, 256),             # the decode layer
    ((2, 32, 8, 128, 32, 16, 2100), [2048], 1, 0, 256),             # no new block: full wait
    ((1, 32, 8, 128, 32, 16, 3000), [1500, 0, 700, 9], 1, 40, 64),  # > 32 new blocks, 4 seqs
    ((1, 8, 2, 64, 16, 16, 900), [0, 5, 300, 1, 0, 77, 400, 2], 2, 3, 8),  # 8 seqs, r 16
    ((1, 16, 4, 192, 64, 32, 700), [333], 4, 2, 50),                # nvec 16, r 64, bs 32
    ((1, 64, 8, 256, 32, 16, 500), [450], 2, 5, 33),                # hd 256, nvec 16 (NT 2)
    ((1, 40, 8, 128, 128, 16, 300), [257], 1, 1, 16),               # r 128, g 5
])
def test_layer_step_inline_query_projection(shape, lengths, rows, n_new, k):
    d = W.Dims(*shape)
    x = make(d, lengths, rows, n_new, seed=7 * sum(shape) + rows)
    inline_vs_oracle(d, x, d.num_layers - 1, k)


def test_layer_step_inline_new_block_outside_the_table():
    # A new block that no table entry names is still written; the scorer waits for the
    # projection only where it reads a new block.
    d = W.Dims(1, 32, 8, 128, 32, 16, 600)
    x = make(d, [500], 1, 2, seed=99)
    in_table = set(x["table"].tolist())
    outside = next(b for b in range(d.max_blocks) if b not in in_table)
    x["new_ids"] = torch.tensor([int(x["table"][7]), outside], dtype=torch.int32, device=DEV)
    inline_vs_oracle(d, x, 0, 32)
