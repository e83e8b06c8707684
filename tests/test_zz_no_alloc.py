"""hss_layer_step_static: the layer call for callers that cannot allocate device memory.

Such a caller (an engine whose arena already owns the GPU's memory, a host process that
gives the library no allocator) cannot hand hss_layer_step a workspace; this entry point
keeps its completion counters in a fixed array inside the library instead.  It runs the
same kernels as hss_layer_step, so on the same inputs its outputs must agree exactly --
inside every tolerance the other tests use.  Each case makes two calls in a row, so the
second call runs on the array as the first one left it.

This file is collected last on purpose: it must pass on its own in a fresh process and
after every other test.
"""
import pytest
import torch

import kv_cache_block_lowrank_gb300 as hss
import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_block_lowrank_gb300 import _build

    _build.build()
    hss.load()


def inputs(dims, lengths, rows, n_new, seed):
    g = torch.Generator().manual_seed(seed)
    total = sum(lengths)
    P = W.projection(g, dims.head_dim, dims.r).to(DEV)
    A = W.bf16_normal(g, dims.a_g_shape).to(DEV)
    table = torch.randperm(dims.max_blocks, generator=g)[:total].to(torch.int32)
    new_ids = table[torch.randperm(total, generator=g)[:n_new]].contiguous()
    K_new = W.bf16_normal(g, (n_new, dims.block_size, dims.num_kv_heads, dims.head_dim))
    Q = W.bf16_normal(g, (len(lengths), rows, dims.num_q_heads, dims.head_dim))
    return dict(P=P, A=A, table=table.to(DEV), offs=W.identity_offsets(lengths).to(DEV),
                new_ids=new_ids.to(DEV), K_new=K_new.to(DEV), Q=Q.to(DEV), S=len(lengths),
                rows=rows, total=total, n_new=n_new)


def outputs(dims, x, k):
    A = x["A"].clone()
    Qp = torch.empty(x["S"], x["rows"], dims.num_q_heads, dims.r, dtype=torch.bfloat16,
                     device=DEV)
    sc = torch.empty(x["total"], dtype=torch.float32, device=DEV)
    vic = torch.full((x["S"], k), 777, dtype=torch.int32, device=DEV)
    return A, Qp, sc, vic


def with_workspace(dims, x, layer, k):
    A, Qp, sc, vic = outputs(dims, x, k)
    nb = hss.hss_layer_step_workspace_bytes(x["S"])
    ws = torch.zeros(nb // 4, dtype=torch.int32, device=DEV)
    hss.hss_layer_step(dims, x["P"], x["K_new"], x["new_ids"], x["n_new"], x["Q"], x["rows"],
                       Qp, A, layer, x["table"], x["offs"], x["S"], x["total"], sc, k, vic, ws, nb)
    torch.cuda.synchronize()
    return A, Qp, sc, vic


def without_allocation(dims, x, layer, k):
    A, Qp, sc, vic = outputs(dims, x, k)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_layer_step_static(dims, x["P"], x["K_new"], x["new_ids"], x["n_new"], x["Q"],
                              x["rows"], Qp, A, layer, x["table"], x["offs"], x["S"], x["total"],
                              sc, k, vic, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return A, Qp, sc, vic


@pytest.mark.parametrize("shape,lengths,rows,n_new,k", [
    ((2, 32, 8, 128, 32, 16, 2100), [2048], 1, 1, 256),                   # the decode layer
    ((1, 8, 2, 128, 32, 16, 900), [0, 5, 300, 1, 0, 77, 400], 2, 3, 8),   # many sequences
])
def test_static_counters_match_workspace_twice(shape, lengths, rows, n_new, k):
    dims = W.Dims(*shape)
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        x = inputs(dims, lengths, rows, n_new, seed=seed + sum(shape))
        layer = call % dims.num_layers
        ref = with_workspace(dims, x, layer, k)
        got = without_allocation(dims, x, layer, k)
        for name, a, b in zip(("A_g", "Qp", "scores", "victims"), ref, got):
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b), f"call {call}: {name} differs"


def test_static_limit_is_enforced():
    limit = hss.hss_layer_step_static_max_seqs()
    assert limit == 4096
    dims = W.Dims(1, 8, 2, 128, 32, 16, 64)
    with pytest.raises(hss.HssError) as e:
        hss.hss_layer_step_static(dims, 0x10000, None, None, 0, 0x10000, 1, 0x10000, 0x10000, 0,
                                  0x10000, 0x10000, limit + 1, limit + 1, 0x10000, 4, 0x10000,
                                  None, 0)
    assert e.value.status == hss.HSS_ERR_WORKSPACE_TOO_SMALL


def test_static_null_qp_is_rejected():
    # This entry point needs the caller's Qp buffer; NULL comes back as an error, not a launch.
    dims = W.Dims(2, 32, 8, 128, 32, 16, 2100)
    x = inputs(dims, [2048], 1, 1, seed=3)
    A, _, sc, vic = outputs(dims, x, 256)
    with pytest.raises(hss.HssError) as e:
        hss.hss_layer_step_static(dims, x["P"], x["K_new"], x["new_ids"], 1, x["Q"], 1, None, A,
                                  0, x["table"], x["offs"], 1, x["total"], sc, 256, vic)
    assert e.value.status == hss.HSS_ERR_NULL_POINTER


def test_static_failed_call_then_valid_call():
    # A call that fails its checks enqueues nothing; the valid call after it is still exact.
    dims = W.Dims(2, 32, 8, 128, 32, 16, 2100)
    x = inputs(dims, [2048], 1, 1, seed=5)
    A, Qp, sc, vic = outputs(dims, x, 256)
    with pytest.raises(hss.HssError) as e:  # layer out of range
        hss.hss_layer_step_static(dims, x["P"], x["K_new"], x["new_ids"], 1, x["Q"], 1, Qp, A, 7,
                                  x["table"], x["offs"], 1, x["total"], sc, 256, vic)
    assert e.value.status == hss.HSS_ERR_OUT_OF_RANGE
    torch.cuda.synchronize()
    assert (vic == 777).all(), "a failed call must not have run anything"
    ref = with_workspace(dims, x, 1, 256)
    got = without_allocation(dims, x, 1, 256)
    for name, a, b in zip(("A_g", "Qp", "scores", "victims"), ref, got):
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), f"{name} differs after a failed call"


def test_static_calls_back_to_back_with_different_batches():
    # Static calls in a row, no workspace call between them: one sequence (the one-sequence
    # ranking's part of the array), then 80 (the per-sequence counters), then one again.
    dims = W.Dims(1, 32, 8, 128, 32, 16, 3000)
    cases = [([2048], 256, 21), ([30] * 80, 16, 22), ([1500], 64, 23)]
    got = []
    for lengths, k, seed in cases:
        x = inputs(dims, lengths, 1, 1, seed=seed)
        got.append((x, k, without_allocation(dims, x, 0, k)))
    for x, k, out in got:
        ref = with_workspace(dims, x, 0, k)
        for name, a, b in zip(("A_g", "Qp", "scores", "victims"), ref, out):
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b), f"{x['S']} sequences: {name} differs"
