"""hss_layer_step (one fused layer call) against the four separate calls and the oracle."""
import numpy as np
import pytest
import torch

import kv_cache_block_lowrank_gb300 as hss
import oracle
import workloads as W
from gpu_util import (assert_bf16_within_ulp, assert_scores_close, assert_victims_match, bits,
                      slot_scale_fn)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_block_lowrank_gb300 import _build

    _build.build()
    hss.load()


SPREAD_REGION_WORDS = 33024 // 4  # the one-sequence ranking's call number and tagged keys


def counters_zero(ws, num_seqs):
    """The per-sequence completion counters (4 * num_seqs bytes, rounded up to 256, after the
    one-sequence ranking's region) are back at zero; that region carries over to the next
    call."""
    words = (4 * num_seqs + 255) // 256 * 64
    return int(ws[SPREAD_REGION_WORDS:SPREAD_REGION_WORDS + words].abs().sum()) == 0


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
    assert counters_zero(ws, x["S"]), "the counters must be left zeroed"
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
    nb = hss.hss_layer_step_workspace_bytes(1)
    ws = torch.zeros(nb // 4, dtype=torch.int32, device=DEV)
    table, offs = case.table.to(DEV), case.seq_offsets.to(DEV)
    hss.hss_layer_step(d, P, case.K[0][60:].to(DEV), new_ids, 4, case.Q[0].to(DEV), 1, Qp, A, 0,
                       table, offs, 1, 64, sc, 8, vic, ws, nb)
    torch.cuda.synchronize()
    A_o = np.zeros(d.a_g_shape, dtype=np.uint16)
    oracle.project_kv_blocks(bits(case.P), bits(case.K[0]), 0, case.block_ids.numpy(), A_o)
    Qp_o = oracle.project_q(bits(case.Q[0]), bits(case.P))
    s_o, t_o, _ = oracle.score_blocks(Qp_o, A_o, 0, case.table.numpy(),
                                      case.seq_offsets.numpy().astype(np.int64))
    s_g = sc.cpu().numpy()
    assert_scores_close(s_g, s_o, t_o)
    assert_victims_match(vic.cpu().numpy(), s_o, t_o, case.seq_offsets.numpy(), 8, gpu_scores=s_g)


def oracle_new_slots(d, x, layer):
    """The caller's A_g with the oracle's projection of this call's new blocks written in."""
    A_o = bits(x["A"].cpu()).copy()
    if x["n_new"]:
        st = oracle.project_kv_blocks(bits(x["P"].cpu()), bits(x["K_new"][:x["n_new"]].cpu()),
                                      layer, x["new_ids"].cpu().numpy(), A_o, nthreads=8)
        assert st == 0 or x.get("bad_new", False)
    return A_o


def inline_vs_oracle(d, x, layer, k, status=0):
    """hss_layer_step with Qp = NULL (queries projected inside the scorer) against the oracle:
    the new slots within 1 bf16 ulp of the oracle's, every other slot untouched, scores within
    tolerance, victims exact outside the tolerance band and exactly the ranking kernel's order
    of the call's own scores."""
    A = x["A"].clone()
    sc = torch.empty(x["total"], dtype=torch.float32, device=DEV)
    vic = torch.full((x["S"], k), 12345, dtype=torch.int32, device=DEV)
    nb = hss.hss_layer_step_workspace_bytes(x["S"])
    ws = torch.zeros(max(nb, 4) // 4, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_layer_step(d, x["P"], x["K_new"], x["new_ids"], x["n_new"], x["Q"], x["rows"], None,
                       A, layer, x["table"], x["offs"], x["S"], x["total"], sc, k, vic, ws, nb, st)
    torch.cuda.synchronize()
    assert int(st.item()) == status
    assert counters_zero(ws, x["S"]), "the counters must be left zeroed"
    A_o = oracle_new_slots(d, x, layer)
    A_g = bits(A.cpu())
    new = x["new_ids"].cpu().numpy()[:x["n_new"]]
    new = new[(new >= 0) & (new < d.max_blocks)]
    keep = np.ones(d.max_blocks, dtype=bool)
    keep[new] = False
    assert np.array_equal(A_g[layer][keep], A_o[layer][keep]), "wrote a slot that is not new"
    assert np.array_equal(np.delete(A_g, layer, axis=0), np.delete(A_o, layer, axis=0))
    if new.size:
        pos = [int(np.nonzero(x["new_ids"].cpu().numpy() == b)[0][0]) for b in new]
        scale = slot_scale_fn(x["K_new"][torch.as_tensor(pos)], x["P"])
        assert_bf16_within_ulp(A_g[layer][new], A_o[layer][new], what="new slots", scale=scale,
                               n_terms=d.head_dim)
    Qp_o = oracle.project_q(bits(x["Q"].cpu()).reshape(-1, d.num_q_heads, d.head_dim),
                            bits(x["P"].cpu()))
    Qp_o = Qp_o.reshape(x["S"], x["rows"], d.num_q_heads, d.r)
    offs = x["offs"].cpu().numpy().astype(np.int64)
    s_o, t_o, _ = oracle.score_blocks(Qp_o, A_o, layer, x["table"].cpu().numpy(), offs)
    s_g = sc.cpu().numpy()
    assert_scores_close(s_g, s_o, t_o)
    assert_victims_match(vic.cpu().numpy(), s_o, t_o, offs, k, gpu_scores=s_g)
    return A, sc, vic


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
    # A new block that no table entry names is still written; only the new slots change.
    d = W.Dims(1, 32, 8, 128, 32, 16, 600)
    x = make(d, [500], 1, 2, seed=99)
    in_table = set(x["table"].tolist())
    outside = next(b for b in range(d.max_blocks) if b not in in_table)
    x["new_ids"] = torch.tensor([int(x["table"][7]), outside], dtype=torch.int32, device=DEV)
    inline_vs_oracle(d, x, 0, 32)


@pytest.mark.parametrize("first,n_new", [(8, 3), (2040, 2), (0, 8), (100, 9)])
def test_layer_step_several_new_blocks(first, n_new):
    # The decode layer (8 table entries per scoring CTA): n_new new blocks at consecutive
    # table positions, so several warps of one CTA wait for the projection of their block.
    d = W.Dims(2, 32, 8, 128, 32, 16, 2100)
    x = make(d, [2048], 1, n_new, seed=first + n_new)
    x["new_ids"] = x["table"][first:first + n_new].contiguous()
    x["K_new"] = W.bf16_normal(torch.Generator().manual_seed(first),
                               (n_new, 16, 8, 128)).to(DEV)
    inline_vs_oracle(d, x, 1, 256)


def test_layer_step_new_block_named_twice():
    # One new block at two table positions far apart (scored by different CTAs, each of which
    # projects it) and a second new block at the next position: every copy scores alike.
    d = W.Dims(2, 32, 8, 128, 32, 16, 2100)
    x = make(d, [2048], 1, 2, seed=77)
    x["table"][1500] = x["table"][3]
    x["new_ids"] = x["table"][3:5].contiguous()
    A, sc, _ = inline_vs_oracle(d, x, 1, 256)
    assert float(sc[3]) == float(sc[1500])


@pytest.mark.parametrize("shape,lengths,n_new", [
    ((1, 16, 4, 64, 32, 32, 1200), [1000], 3),   # 4 kv heads x 2 tiles of 16 tokens, hd 64
    ((1, 32, 8, 128, 32, 32, 1200), [1000], 2),  # 16 tiles per block
    ((1, 8, 1, 64, 16, 16, 400), [1, 300, 2], 8),  # one tile per block, r 16
])
def test_layer_step_new_blocks_other_shapes(shape, lengths, n_new):
    d = W.Dims(*shape)
    x = make(d, lengths, 1, n_new, seed=sum(shape) + n_new)
    inline_vs_oracle(d, x, 0, 16)


def test_layer_step_bad_new_id():
    # A new id outside the pool is skipped and reported; the call's other results stand.
    d = W.Dims(1, 32, 8, 128, 32, 16, 2100)
    x = make(d, [2048], 1, 2, seed=31)
    x["new_ids"] = torch.tensor([int(x["table"][5]), d.max_blocks + 7], dtype=torch.int32,
                                device=DEV)
    x["bad_new"] = True
    inline_vs_oracle(d, x, 0, 256, status=hss.HSS_ERR_OUT_OF_RANGE)
    assert hss.hss_read_device_error() == hss.HSS_ERR_OUT_OF_RANGE


def _with_ties(x, d, groups, seed):
    """Replace the table by `groups` distinct blocks, each named several times: equal scores,
    which the ranking must order by table position."""
    g = torch.Generator().manual_seed(seed)
    total = x["total"]
    base = torch.randperm(d.max_blocks, generator=g)[:groups].to(torch.int32)
    table = base[torch.randint(0, groups, (total,), generator=g)]
    x["table"] = table.to(DEV)
    if x["n_new"]:
        x["new_ids"] = table[:x["n_new"]].unique().contiguous().to(DEV)
        x["n_new"] = int(x["new_ids"].numel())
    return x


# One sequence of at most 4096 entries: every CTA of the decode scorer ranks its own entries
# once the sequence's count is complete.  Past 4096 the last CTA ranks the whole sequence.
@pytest.mark.parametrize("shape,n,k,ties,inline", [
    ((2, 32, 8, 128, 32, 16, 2100), 2048, 256, 0, True),     # the decode layer
    ((2, 32, 8, 128, 32, 16, 2100), 2048, 256, 97, True),    # many equal scores
    ((1, 32, 8, 128, 32, 16, 5000), 4096, 4096, 0, False),   # the longest spread sequence
    ((1, 32, 8, 128, 32, 16, 5000), 4097, 300, 0, True),     # one entry past it
    ((1, 32, 8, 128, 32, 16, 500), 100, 256, 0, True),       # fewer entries than victims
    ((1, 32, 8, 128, 32, 16, 500), 1, 8, 0, False),          # a single entry
    ((1, 8, 2, 64, 16, 16, 900), 777, 777, 5, True),         # r 16, k == n, ties
])
def test_layer_step_one_sequence_ranking(shape, n, k, ties, inline):
    d = W.Dims(*shape)
    x = make(d, [n], 1, 1, seed=n + k + ties)
    if ties:
        x = _with_ties(x, d, ties, seed=n)
    layer = d.num_layers - 1
    A1, _, sc1, vic1 = separate(d, x, layer, k)
    A = x["A"].clone()
    sc = torch.empty(n, dtype=torch.float32, device=DEV)
    vic = torch.full((1, k), 12345, dtype=torch.int32, device=DEV)
    nb = hss.hss_layer_step_workspace_bytes(1)
    ws = torch.zeros(max(nb, 4) // 4, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    Qp = None if inline else torch.empty(1, 1, d.num_q_heads, d.r, dtype=torch.bfloat16,
                                         device=DEV)
    for _ in range(3):  # the workspace is reused: each call must leave it zeroed
        vic.fill_(12345)
        hss.hss_layer_step(d, x["P"], x["K_new"], x["new_ids"], x["n_new"], x["Q"], 1, Qp, A,
                           layer, x["table"], x["offs"], 1, n, sc, k, vic, ws, nb, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert counters_zero(ws, 1), "the counters must be left zeroed"
        if inline:
            # The scorer projected the queries and the new block itself (within 1 ulp of the
            # separate projections): its ranking must be exactly the ranking kernel's on the
            # call's own scores, and the scores stay within the score tolerance.
            ref = torch.empty(1, k, dtype=torch.int32, device=DEV)
            hss.hss_rank_victims(sc, x["offs"], 1, n, k, ref)
            torch.cuda.synchronize()
            assert torch.equal(vic, ref)
            assert torch.allclose(sc, sc1, rtol=2e-3, atol=1e-2)
        else:
            assert torch.equal(sc, sc1)
            assert torch.equal(vic, vic1)
    if ties:
        s = sc1.cpu().numpy()
        assert len(np.unique(s)) <= ties
    v = vic1[0].cpu().numpy()
    assert (v[min(n, k):] == -1).all()
    assert sorted(v[:min(n, k)].tolist()) == sorted(set(v[:min(n, k)].tolist()))


def test_layer_step_one_sequence_bad_id():
    # A table entry outside the pool scores +inf and raises the status; the ranking still
    # places it (last) exactly as the separate ranking call does.
    d = W.Dims(1, 32, 8, 128, 32, 16, 3000)
    n, k = 2048, 2048
    x = make(d, [n], 1, 1, seed=5)
    x["table"][777] = d.max_blocks + 3
    layer = 0
    Qp = torch.empty(1, 1, d.num_q_heads, d.r, dtype=torch.bfloat16, device=DEV)
    A = x["A"].clone()
    hss.hss_project_kv_blocks(d, x["P"], x["K_new"], layer, x["new_ids"], 1, A)
    hss.hss_project_q(d, x["P"], x["Q"], 1, Qp)
    sc1 = torch.empty(n, dtype=torch.float32, device=DEV)
    st1 = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_score_blocks(d, Qp, 1, A, layer, x["table"], x["offs"], 1, n, sc1,
                         dev_status=st1)
    vic1 = torch.empty(1, k, dtype=torch.int32, device=DEV)
    hss.hss_rank_victims(sc1, x["offs"], 1, n, k, vic1)
    sc = torch.empty(n, dtype=torch.float32, device=DEV)
    vic = torch.full((1, k), 12345, dtype=torch.int32, device=DEV)
    nb = hss.hss_layer_step_workspace_bytes(1)
    ws = torch.zeros(max(nb, 4) // 4, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_layer_step(d, x["P"], x["K_new"], x["new_ids"], 1, x["Q"], 1, None, x["A"].clone(),
                       layer, x["table"], x["offs"], 1, n, sc, k, vic, ws, nb, st)
    torch.cuda.synchronize()
    assert int(st1.item()) == hss.HSS_ERR_OUT_OF_RANGE
    assert int(st.item()) == hss.HSS_ERR_OUT_OF_RANGE
    assert float(sc[777]) == float("inf")
    assert torch.equal(sc, sc1)
    assert torch.equal(vic, vic1)
    assert int(vic[0, -1]) == 777
    assert counters_zero(ws, 1)
    assert hss.hss_read_device_error() == hss.HSS_ERR_OUT_OF_RANGE


def test_layer_step_one_workspace_for_every_sequence_count():
    # One workspace sized for the largest batch serves calls with one sequence (spread
    # ranking: call number and tagged keys) and with many (per-sequence counters, the last
    # CTA ranks), in any order.
    d = W.Dims(1, 32, 8, 128, 32, 16, 3000)
    ws = torch.zeros(hss.hss_layer_step_workspace_bytes(80) // 4, dtype=torch.int32, device=DEV)
    for i, lengths in enumerate(([2048], [30] * 80, [1500], [10] * 70 + [5], [700], [2048])):
        x = make(d, lengths, 1, 1, seed=100 + i)
        _, _, sc1, vic1 = separate(d, x, 0, 16)
        _, _, sc2, vic2, _ = fused(d, x, 0, 16, ws=ws)
        assert torch.equal(sc1, sc2)
        assert torch.equal(vic1, vic2), f"call {i}: {len(lengths)} sequences"
        assert counters_zero(ws, 80)


@pytest.mark.parametrize("inline", [True, False])
def test_prepared_layer_step_equals_the_plain_call(inline):
    # hss.LayerStep binds the arguments that stay fixed across calls; each call must give
    # exactly what hss_layer_step gives (the decode layer, 32 layers of one step).
    d = W.Dims(4, 32, 8, 128, 32, 16, 2100)
    x = make(d, [2048], 1, 1, seed=11)
    k = 256
    nb = hss.hss_layer_step_workspace_bytes(1)
    Qp = None if inline else torch.empty(1, 1, d.num_q_heads, d.r, dtype=torch.bfloat16,
                                         device=DEV)
    out = []
    for prepared in (False, True):
        A = x["A"].clone()
        ws = torch.zeros(nb // 4, dtype=torch.int32, device=DEV)
        sc = torch.empty(d.num_layers, 2048, dtype=torch.float32, device=DEV)
        vic = torch.full((d.num_layers, 1, k), 12345, dtype=torch.int32, device=DEV)
        step = hss.LayerStep(d, x["P"], x["new_ids"], 1, 1, Qp, A, x["table"], x["offs"], 1,
                             2048, k, ws, nb)
        for layer in range(d.num_layers):
            if prepared:
                step(layer, x["K_new"], x["Q"], sc[layer].data_ptr(), vic[layer])
            else:
                hss.hss_layer_step(d, x["P"], x["K_new"], x["new_ids"], 1, x["Q"], 1, Qp, A,
                                   layer, x["table"], x["offs"], 1, 2048, sc[layer], k,
                                   vic[layer], ws, nb)
        torch.cuda.synchronize()
        out.append((A, sc, vic))
    assert torch.equal(out[0][0].view(torch.int16), out[1][0].view(torch.int16))
    assert torch.equal(out[0][1], out[1][1])
    assert torch.equal(out[0][2], out[1][2])


# Up to 8 sequences and 4096 entries in all: the scorer's CTAs rank every sequence together
# (one word per entry, sequence index inside the word).  Victims must equal the ranking
# kernel's bit for bit, over three calls on one workspace.
@pytest.mark.parametrize("lengths,k,ties,inline", [
    ([1024, 1024], 256, 0, True),                       # two halves of the decode layer
    ([500, 0, 1300, 7], 64, 0, True),                   # an empty sequence, one shorter than k
    ([600] * 6 + [300, 96], 128, 0, False),             # eight sequences, Qp given
    ([2000, 2000, 96], 300, 0, True),                   # 4096 entries in all (the limit)
    ([2000, 2097], 64, 0, True),                        # 4097: the last CTA ranks instead
    ([700, 700, 700], 700, 13, True),                   # k == n, many equal scores
    ([1, 1, 1, 1, 1], 8, 0, True),                      # five one-block sequences
])
def test_layer_step_few_sequences_ranking(lengths, k, ties, inline):
    d = W.Dims(1, 32, 8, 128, 32, 16, 6000)
    x = make(d, lengths, 1, 1, seed=sum(lengths) + k + ties)
    if ties:
        x = _with_ties(x, d, ties, seed=k)
    S, n = len(lengths), sum(lengths)
    _, _, sc1, vic1 = separate(d, x, 0, k)
    A = x["A"].clone()
    sc = torch.empty(n, dtype=torch.float32, device=DEV)
    vic = torch.full((S, k), 12345, dtype=torch.int32, device=DEV)
    nb = hss.hss_layer_step_workspace_bytes(S)
    ws = torch.zeros(max(nb, 4) // 4, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    Qp = None if inline else torch.empty(S, 1, d.num_q_heads, d.r, dtype=torch.bfloat16,
                                         device=DEV)
    for _ in range(3):
        vic.fill_(12345)
        hss.hss_layer_step(d, x["P"], x["K_new"], x["new_ids"], x["n_new"], x["Q"], 1, Qp, A, 0,
                           x["table"], x["offs"], S, n, sc, k, vic, ws, nb, st)
        ref = torch.empty(S, k, dtype=torch.int32, device=DEV)
        hss.hss_rank_victims(sc, x["offs"], S, n, k, ref)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert counters_zero(ws, S), "the counters must be left zeroed"
        assert torch.equal(vic, ref)
        if inline:
            assert torch.allclose(sc, sc1, rtol=2e-3, atol=1e-2)
        else:
            assert torch.equal(sc, sc1) and torch.equal(vic, vic1)
