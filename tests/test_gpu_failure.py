"""Failure detection on the GPU without a fault: a pipeline wait that runs out reports
HSS_ERR_DEVICE_TIMEOUT and the context stays usable."""
import time

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
