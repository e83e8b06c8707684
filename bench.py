#!/usr/bin/env python3
"""Throughput benchmark of the GB300 low-rank KV-block predictor.

Default workload (one "step" = one model decode step = 32 layer calls): the
Llama-3-8B-like decode layer -- 32 query heads / 8 kv heads, head_dim 128, r 32,
block_size 16, one sequence of 32768 tokens (2048 blocks), one query row,
bottom-256 victims.  Each layer call runs the whole predictor path through the
C ABI: project the block being written this step into A_g, project the query,
score all 2048 blocks through the (permuted) block table, rank the victims.
The 32 layers' A_g (512 MiB) exceed the 129 MB L2, so every layer call reads
its 16 MiB of A_g from HBM.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle
instead (on this workload's layer call, a bounded sample of blocks per step).
Under torchrun each rank runs an independent replica on its own GPU (the path
has no exchange step); the elapsed time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "blocks scored/s and A_g GB/s (fraction of GB300 HBM peak) per layer call"


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["hss", "reference"], default="hss")
    p.add_argument("--workload", choices=["decode"], default="decode")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true",
                   help="launch every call from the host instead of replaying a CUDA graph")
    return p.parse_args(argv)


# ----------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, use_cuda: bool):
    if world <= 1:
        return None
    import torch.distributed as dist

    if not dist.is_initialized():
        dist.init_process_group("nccl" if use_cuda else "gloo")
    return dist


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist

        if device is not None and str(device).startswith("cuda"):
            dist.barrier(device_ids=[int(str(device).split(":")[-1])])
        else:
            dist.barrier()


def aggregate(elapsed_s: float, units: float, world: int, device="cpu"):
    """(max elapsed over ranks, sum of units over ranks): the job's wall time and work."""
    if world <= 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist

    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ----------------------------------------------------------------------------- clocks

CLOCK_FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    def __init__(self, uuid: str | None):
        self.uuid = (uuid or "").lower()
        self.lines = []
        self.proc = None
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.25)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            if self.uuid and self.uuid not in f[0].lower():
                continue
            rows.append(f)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


def device_uuid(index: int):
    import torch

    try:
        return str(torch.cuda.get_device_properties(index).uuid)
    except Exception:
        return None


# ----------------------------------------------------------------------------- peaks

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------------------- decode workload

class DecodeWorkload:
    """The decode layer, all 32 layers projected; one step = 32 layer calls."""

    name = "decode"

    def __init__(self, device, seed: int):
        import torch

        import kv_cache_block_lowrank_gb300 as hss
        import workloads as W

        self.hss = hss
        self.torch = torch
        self.device = device
        self.case = c = W.decode(seed=seed, device=device)
        self.dims = d = c.dims
        self.L = d.num_layers
        self.n = c.total_blocks
        self.k = c.k_victims
        self.P = c.P.to(device)
        self.A = torch.empty(d.a_g_shape, dtype=torch.bfloat16, device=device)
        self.ids = c.block_ids.to(device)
        self.table = c.table.to(device)
        self.offs = c.seq_offsets.to(device)
        for layer in range(self.L):  # the context already in the cache (untimed)
            hss.hss_project_kv_blocks(d, self.P, c.K[layer], layer, self.ids, self.n, self.A)
        # The block being written this step: the sequence's last table entry.
        self.new_id = int(c.table[-1])
        self.new_ids = torch.tensor([self.new_id], dtype=torch.int32, device=device)
        self.K_new = [c.K[l][self.new_id:self.new_id + 1] for l in range(self.L)]
        self.Q = [c.Q[l] for l in range(self.L)]  # [1, 1, nq, hd] each
        self.Qp = torch.empty(self.L, 1, 1, d.num_q_heads, d.r, dtype=torch.bfloat16,
                              device=device)
        self.scores = torch.empty(self.L, self.n, dtype=torch.float32, device=device)
        self.victims = torch.empty(self.L, 1, self.k, dtype=torch.int32, device=device)
        torch.cuda.synchronize()

    # Work units and algorithmic bytes of the dominant kernel (the scorer).
    units_per_step = property(lambda self: self.L * self.n)
    launches_per_step = property(lambda self: self.L * 4)

    @property
    def score_bytes_per_launch(self):
        d = self.dims
        slot = d.num_kv_heads * d.block_size * d.r * 2
        return self.n * (slot + 4 + 4) + d.num_q_heads * d.r * 2 + 8

    def layer_call(self, l: int, K_new=None, Q=None):
        hss, d = self.hss, self.dims
        hss.hss_project_kv_blocks(d, self.P, self.K_new[l] if K_new is None else K_new, l,
                                  self.new_ids, 1, self.A)
        hss.hss_project_q(d, self.P, self.Q[l] if Q is None else Q, 1, self.Qp[l])
        hss.hss_score_blocks(d, self.Qp[l], 1, self.A, l, self.table, self.offs, 1, self.n,
                             self.scores[l])
        hss.hss_rank_victims(self.scores[l], self.offs, 1, self.n, self.k, self.victims[l])

    def step(self):
        for l in range(self.L):
            self.layer_call(l)

    def score_only(self, l: int):
        self.hss.hss_score_blocks(self.dims, self.Qp[l], 1, self.A, l, self.table, self.offs, 1,
                                  self.n, self.scores[l])

    def describe(self):
        d = self.dims
        return (f"decode layer x {self.L} layers per step: {d.num_q_heads} q heads / "
                f"{d.num_kv_heads} kv heads, head_dim {d.head_dim}, r {d.r}, block_size "
                f"{d.block_size}, 1 sequence of {self.n * d.block_size} tokens ({self.n} blocks, "
                f"permuted table), 1 query row, bottom-{self.k}; per layer call: project the "
                f"block being written, project Q, score, rank")

    # ---- end to end through the API with host buffers
    def e2e_setup(self):
        torch = self.torch
        self.h_Q = [q.cpu().pin_memory() for q in self.Q]
        self.h_K = [k.cpu().pin_memory() for k in self.K_new]
        self.h_vic = torch.empty(self.L, 1, self.k, dtype=torch.int32).pin_memory()
        self.d_Q = torch.empty_like(self.Q[0])
        self.d_K = torch.empty_like(self.K_new[0])

    def e2e_step(self):
        for l in range(self.L):
            self.d_Q.copy_(self.h_Q[l], non_blocking=True)
            self.d_K.copy_(self.h_K[l], non_blocking=True)
            self.layer_call(l, K_new=self.d_K, Q=self.d_Q)
            self.h_vic[l].copy_(self.victims[l], non_blocking=True)
        self.torch.cuda.current_stream().synchronize()

    @property
    def e2e_bytes(self):
        h2d = self.L * (self.Q[0].numel() * 2 + self.K_new[0].numel() * 2)
        d2h = self.L * self.k * 4
        return h2d, d2h


# ----------------------------------------------------------------------------- oracle timing

def oracle_decode_sample(case, max_seconds: float, nthreads: int, blocks_per_call=None,
                         max_calls=None):
    """Time the oracle on decode layer calls; returns (blocks scored, seconds, calls, blocks)."""
    import numpy as np

    import oracle

    def bits(t):
        return t.detach().cpu().contiguous().view(__import__("torch").int16).numpy().view(
            np.uint16)

    d = case.dims
    layer = 0
    n = case.total_blocks if blocks_per_call is None else min(blocks_per_call, case.total_blocks)
    table = case.table.numpy()[:n].astype(np.int32)
    P = bits(case.P)
    K = bits(case.K[layer])
    A = np.zeros((1, d.max_blocks, d.num_kv_heads, d.block_size, d.r), dtype=np.uint16)
    ids = table  # pool position == block id in this workload
    oracle.project_kv_blocks(P, K[ids], 0, ids, A, nthreads=nthreads)  # context (untimed)
    Q = bits(case.Q[layer])
    offs = np.array([0, n], dtype=np.int64)
    new = np.array([int(case.table[-1])], dtype=np.int32)
    Knew = K[new]
    calls, scored = 0, 0
    t0 = time.perf_counter()
    while True:
        oracle.project_kv_blocks(P, Knew, 0, new, A, nthreads=nthreads)
        Qp = oracle.project_q(Q, P, nthreads=nthreads)
        s, _, _ = oracle.score_blocks(Qp, A, 0, table, offs, nthreads=nthreads)
        oracle.rank_victims(s.astype(np.float32), offs, min(case.k_victims, n))
        calls += 1
        scored += n
        el = time.perf_counter() - t0
        if el >= max_seconds or (max_calls is not None and calls >= max_calls):
            return scored, el, calls, n


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- arms

def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    import workloads as W

    case = W.decode(seed=args.seed, device="cpu", layers=1)
    threads = cpu_threads()
    # Per-block cost, to size each step's sample so the whole run takes about a minute.
    scored, el, _, _ = oracle_decode_sample(case, 0.0, threads, blocks_per_call=64, max_calls=1)
    per_block = el / max(scored, 1)
    total_steps = args.steps + args.warmup
    sample = int(max(16, min(case.total_blocks, 60.0 / max(total_steps * per_block, 1e-12))))
    for _ in range(args.warmup):
        oracle_decode_sample(case, 0.0, threads, blocks_per_call=sample, max_calls=1)
    t0 = time.perf_counter()
    blocks = 0
    for _ in range(args.steps):
        b, _, _, _ = oracle_decode_sample(case, 0.0, threads, blocks_per_call=sample, max_calls=1)
        blocks += b
    el = time.perf_counter() - t0
    value = blocks / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "blocks/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "decode layer call (oracle): project the new block, project Q, "
                               f"score the first {sample} blocks of the table, rank"},
        "cpu_baseline": {"value": value, "unit": "blocks/s", "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} layer calls of {sample} blocks each"},
        "e2e": {"value": value, "unit": "blocks/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_hss(args):
    import torch

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the predictor has no CPU path)")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    dist_init(world, True)
    import __graft_entry__

    __graft_entry__.build()
    import kv_cache_block_lowrank_gb300 as hss

    wl = DecodeWorkload(device, args.seed + rank)
    peaks = measured_peaks()
    stream = torch.cuda.Stream(device=device)
    torch.cuda.synchronize()

    # ---- warm-up, then capture one step into a CUDA graph
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            wl.step()
    stream.synchronize()
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            wl.step()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
    run_step = graph.replay if graph is not None else wl.step

    # ---- timed region
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    torch.cuda.synchronize()
    with ClockSampler(device_uuid(local)) as clocks:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                run_step()
            ev1.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    barrier(world, device)
    elapsed = ev0.elapsed_time(ev1) / 1e3
    elapsed_max, units = aggregate(elapsed, wl.units_per_step * args.steps, world, device)
    value = units / elapsed_max

    # ---- dominant kernel (the scorer): 32 back-to-back launches (cold layers) per replay
    reps = max(20, min(400, args.steps // 4))
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        for l in range(wl.L):
            wl.score_only(l)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g2.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g2.replay()
        e1.record(stream)
    stream.synchronize()
    score_s = e0.elapsed_time(e1) / 1e3 / (reps * wl.L)
    achieved = wl.score_bytes_per_launch / score_s / 1e9

    # ---- end to end through the API with host buffers
    e2e = None
    if args.e2e_steps > 0:
        wl.e2e_setup()
        with torch.cuda.stream(stream):
            for _ in range(3):
                wl.e2e_step()
            torch.cuda.synchronize()
            barrier(world, device)
            t0 = time.perf_counter()
            for _ in range(args.e2e_steps):
                wl.e2e_step()
            t1 = time.perf_counter()
        el_e2e, units_e2e = aggregate(t1 - t0, wl.units_per_step * args.e2e_steps, world, device)
        h2d, d2h = wl.e2e_bytes
        e2e = {"value": units_e2e / el_e2e, "unit": "blocks/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
               "how": "every layer call from the host through the C ABI (no graph): pinned "
                      "H2D of Q and the new K block, D2H of the victims, one sync per step"}

    err = hss.hss_read_device_error()
    if err != 0:
        raise SystemExit(f"device error raised during the benchmark: {hss.status_string(err)}")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import workloads as W

        threads = cpu_threads()
        case_cpu = W.decode(seed=args.seed, device="cpu", layers=1)
        scored, el, calls, n = oracle_decode_sample(case_cpu, 10.0, threads)
        cpu = {"value": scored / el, "unit": "blocks/s", "cores": threads, "kind": "oracle",
               "sample": f"{calls} decode layer calls ({n} blocks each: project the new block, "
                         f"project Q, score, rank) on layer 0, ~10 s"}

    if rank == 0:
        d = wl.dims
        slot = d.num_kv_heads * d.block_size * d.r * 2
        line = {
            "metric": METRIC, "value": value, "unit": "blocks/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed_max / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "a_g_gbs": value * slot / 1e9,
            "a_g_hbm_frac": value * slot / 1e9 / peaks["hbm_gbs"],
            "config": {"workload": wl.describe(),
                       "l2": "no flush: each step reads 32 x 16 MiB = 512 MiB of A_g, above "
                             "the 129 MB L2, so every layer call reads cold A_g",
                       "graph": graph is not None, "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": "score_decode", "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                         "peak_source": peaks["source"] + " hbm_gbs (burst copy)",
                         "launch_us": score_s * 1e6,
                         "bytes_per_launch": wl.score_bytes_per_launch,
                         "how": "CUDA events around graphs of 32 back-to-back scorer launches "
                                "(one per layer) on the launching stream; duration per launch "
                                "includes the gap between graph nodes"},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": wl.launches_per_step * args.steps,
            "clocks": clocks.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_hss(args)


if __name__ == "__main__":
    sys.exit(main())
