"""bench.py's host logic on the CPU: max-over-ranks timing with two gloo ranks, clock-log
parsing, defaults."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [1.5, 2.5][rank]
    units = [1000.0, 3000.0][rank]
    bench.barrier(world)
    t, u = bench.aggregate(elapsed, units, world, "cpu")
    q.put((rank, t, u))
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, u in out:
        assert t == 2.5 and u == 4000.0  # the job's time is the slowest rank's; work adds up


def test_aggregate_single_rank_is_identity():
    assert bench.aggregate(1.25, 10.0, 1) == (1.25, 10.0)


def test_clock_summary_parsing():
    c = bench.ClockSampler("GPU-abc")
    c.lines = [
        "GPU-abc, 1980, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, "
        "Not Active",
        "GPU-abc, 1900, 2070, 1300.0, 0x0000000000000004, Not Active, Not Active, Not Active, "
        "Active",
        "GPU-zzz, 100, 2070, 10.0, 0x0, Active, Active, Active, Active",  # another GPU
    ]
    s = c.summary()
    assert s["sm_mhz"] == 1940.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 2


def test_defaults_and_peaks():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps > 0 and a.impl == "hss"
    p = bench.measured_peaks()
    assert p["hbm_gbs"] > 1000 and p["bf16_tflops"] > 100


def test_reference_arm_prints_one_contract_line():
    # `bench.py --impl reference` times the oracle (the CPU restatement of the method) on the
    # host; its single JSON line carries the contract's keys with the decode workload's
    # metric, and an e2e entry that moves no bytes between host and device.
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], cwd=root, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "blocks/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
