"""Failure detection on the GPU without a fault: a pipeline wait that runs out reports
HSS_ERR_DEVICE_TIMEOUT and the context stays usable."""
import time

import pytest
import torch

import kv_cache_block_lowrank_gb300 as hss
import workloads as W
from test_gpu_layer_step import make

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_block_lowrank_gb300 import _build

    _build.build()
    hss.load()


def test_wait_that_runs_out_reports_timeout_and_the_gpu_stays_usable():
    hss.hss_read_device_error()  # start from a clear library word
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.perf_counter()
    hss.hss_self_test_wait_timeout(st, 2_000_000)  # 2 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(st.item()) == hss.HSS_ERR_DEVICE_TIMEOUT
    assert elapsed < 5.0
    assert hss.hss_read_device_error() == hss.HSS_ERR_DEVICE_TIMEOUT
    assert hss.hss_read_device_error() == hss.HSS_OK
    # The context still works: a small projection right after.
    g = torch.Generator().manual_seed(1)
    d = W.Dims(1, 8, 2, 128, 32, 16, 4)
    P = W.projection(g, 128, 32).to(DEV)
    Q = W.bf16_normal(g, (3, 8, 128)).to(DEV)
    Qp = torch.empty(3, 8, 32, dtype=torch.bfloat16, device=DEV)
    hss.hss_project_q(d, P, Q, 3, Qp)
    ref = (Q.float() @ P.float()).to(torch.bfloat16)
    torch.cuda.synchronize()
    assert (Qp.float() - ref.float()).abs().max().item() <= 0.1
    with pytest.raises(hss.HssError):
        hss.hss_self_test_wait_timeout(st, 10)  # below the allowed range: refused on the host


def test_spread_ranking_wait_runs_out_then_the_next_call_is_exact():
    # The decode layer (one sequence of 2048 blocks): the scorer's CTAs rank the sequence
    # together, each waiting for every other CTA's keys.  With the last CTA withholding its
    # keys the wait runs out after 2 ms and reports HSS_ERR_DEVICE_TIMEOUT; after the
    # workspace is zeroed again the next layer call is exact.
    d = W.Dims(2, 32, 8, 128, 32, 16, 2100)
    x = make(d, [2048], 1, 0, seed=17)
    n, k = 2048, 256
    nb = hss.hss_layer_step_workspace_bytes(1)
    ws = torch.zeros(nb // 4, dtype=torch.int32, device=DEV)
    sc = torch.empty(n, dtype=torch.float32, device=DEV)
    vic = torch.empty(1, k, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hss.hss_read_device_error()
    t0 = time.perf_counter()
    hss.hss_self_test_spread_wait(d, x["P"], x["Q"], x["A"], 1, x["table"], x["offs"], n, sc, k,
                                  vic, ws, nb, 2_000_000, st)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    assert int(st.item()) == hss.HSS_ERR_DEVICE_TIMEOUT
    assert hss.hss_read_device_error() == hss.HSS_ERR_DEVICE_TIMEOUT
    # Recovery as documented: zero the workspace, then an ordinary call.
    ws.zero_()
    st.zero_()
    hss.hss_layer_step(d, x["P"], None, None, 0, x["Q"], 1, None, x["A"], 1, x["table"],
                       x["offs"], 1, n, sc, k, vic, ws, nb, st)
    ref = torch.empty(1, k, dtype=torch.int32, device=DEV)
    hss.hss_rank_victims(sc, x["offs"], 1, n, k, ref)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and hss.hss_read_device_error() == hss.HSS_OK
    assert torch.equal(vic, ref)
    # A shape that does not take the one-sequence ranking is refused before any launch.
    big = W.Dims(1, 32, 8, 128, 32, 16, 5000)
    y = make(big, [4097], 1, 0, seed=19)
    sc2 = torch.empty(4097, dtype=torch.float32, device=DEV)
    with pytest.raises(hss.HssError) as e:
        hss.hss_self_test_spread_wait(big, y["P"], y["Q"], y["A"], 0, y["table"], y["offs"],
                                      4097, sc2, k, vic, ws, nb, 2_000_000, st)
    assert e.value.status == hss.HSS_ERR_UNSUPPORTED_SHAPE
