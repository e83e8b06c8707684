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
    p.add_argument("--workload", choices=["decode", "batched", "prefill", "ingest",
                                          "ingest_tokens", "prefill_rows"],
                   default="decode")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true",
                   help="launch every call from the host instead of replaying a CUDA graph")
    p.add_argument("--unfused", action="store_true",
                   help="decode: four separate calls per layer instead of hss_layer_step")
    p.add_argument("--cpu-threads", type=int, default=0,
                   help="threads for the oracle's CPU legs (0: every core this process may use)")
    p.add_argument("--layers", type=int, default=32,
                   help="ingest workloads: layers written per step (1: a small case for ncu)")
    p.add_argument("--no-extras", action="store_true",
                   help="decode: skip the short passes of the batched, prefill and ingest "
                        "workloads reported under 'workloads'")
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


# ----------------------------------------------------------------------------- traffic
# DRAM bytes per launch of each workload's dominant kernel (dram__bytes_read.sum +
# dram__bytes_write.sum) from the ncu captures summarised in profiles/, or None when the
# kernel has changed since its capture.
TRAFFIC = {
    "decode": (16886656 + 0, "profiles/score_decode_layer_step.md"),
    "batched": (283582976 + 3016448, "profiles/score_decode_batched.md"),
    "prefill": (139942144 + 3391488, "profiles/score_tc_prefill.md"),
    # captured on a 40000-block launch; traffic grows with the blocks, so scaled to 4096
    "ingest": (round((1310975000 + 303530240) * 4096 / 40000),
               "profiles/project_ingest_40000_blocks.md, scaled from 40000 to 4096 blocks"),
    "ingest_tokens": (134840576 + 112052480, "profiles/project_tokens_65536.md"),
    "prefill_rows": (157091328 + 3819520, "profiles/score_tc_prefill_rows.md"),
}


# ----------------------------------------------------------------------------- workloads

class _Base:
    """Shared plumbing: binding handle, device buffers, graph-capturable steps."""

    def __init__(self, device):
        import torch

        import kv_cache_block_lowrank_gb300 as hss

        self.hss = hss
        self.torch = torch
        self.device = device

    def slot_bytes(self):
        d = self.dims
        return d.num_kv_heads * d.block_size * d.r * 2

    def score_bytes(self, n):
        d = self.dims
        return n * (self.slot_bytes() + 4 + 4) + d.num_q_heads * d.r * 2 + 8


class DecodeWorkload(_Base):
    """The decode layer, all 32 layers projected; one step = 32 layer calls."""

    name = "decode"

    def __init__(self, device, seed: int, unfused: bool = False):
        super().__init__(device)
        import workloads as W

        torch, hss = self.torch, self.hss
        self.unfused = unfused
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
        self.ws_bytes = hss.hss_layer_step_workspace_bytes(1)
        self.hdims = hss.hss_dims.of(d)
        self.ws = torch.zeros(self.ws_bytes // 4, dtype=torch.int32, device=device)
        # The layer call with its fixed arguments bound once (Qp = NULL: the caller wants
        # scores and victims, not the projected queries, so the decode scorer projects them).
        self.step_call = hss.LayerStep(self.hdims, self.P, self.new_ids, 1, 1, None, self.A,
                                       self.table, self.offs, 1, self.n, self.k, self.ws,
                                       self.ws_bytes)
        self.score_ptrs = [self.scores[l].data_ptr() for l in range(self.L)]
        self.victim_ptrs = [self.victims[l].data_ptr() for l in range(self.L)]
        torch.cuda.synchronize()

    units_per_step = property(lambda self: self.L * self.n)
    # hss_layer_step with Qp = NULL: the new block's projection, then the scorer (which
    # projects the query, scores and ranks), two launches per layer call.
    launches_per_step = property(lambda self: self.L * (4 if self.unfused else 2))

    def layer_call(self, l: int, K_new=None, Q=None, stream=None):
        hss, d = self.hss, self.dims
        K_new = self.K_new[l] if K_new is None else K_new
        Q = self.Q[l] if Q is None else Q
        if not self.unfused:
            self.step_call(l, K_new, Q, self.score_ptrs[l], self.victim_ptrs[l], stream=stream)
            return
        hss.hss_project_kv_blocks(d, self.P, K_new, l, self.new_ids, 1, self.A)
        hss.hss_project_q(d, self.P, Q, 1, self.Qp[l])
        hss.hss_score_blocks(d, self.Qp[l], 1, self.A, l, self.table, self.offs, 1, self.n,
                             self.scores[l])
        hss.hss_rank_victims(self.scores[l], self.offs, 1, self.n, self.k, self.victims[l])

    def step(self):
        for l in range(self.L):
            self.layer_call(l)

    # The dominant kernel: the decode scorer as the step runs it, timed per layer call (the
    # scorer, which projects the query, scores and ranks, after the small kernel projecting
    # the new block), 32 calls per replay.  Algorithmic bytes of one layer call: every entry's
    # A_g slot, table id and score; the query, P and the new key block read; the new slot and
    # the victims written; the sequence offsets.
    dominant_bound = "hbm"
    dominant_launches = property(lambda self: self.L)

    @property
    def dominant_kernel(self):
        return ("score_decode (the plain scorer, hss_score_blocks)" if self.unfused else
                "score_decode as hss_layer_step runs it, per layer call (the new block's "
                "projection kernel, then the scorer: query projected, 2048 blocks scored by "
                "bulk copies into shared memory, bottom-256 ranked)")

    @property
    def dominant_units(self):
        if self.unfused:
            return self.score_bytes(self.n)
        d = self.dims
        return (self.n * (self.slot_bytes() + 4 + 4) + d.num_q_heads * d.head_dim * 2 +
                d.head_dim * d.r * 2 + d.block_size * d.num_kv_heads * d.head_dim * 2 +
                self.slot_bytes() + self.k * 4 + 8)

    def dominant(self):
        if self.unfused:
            self.plain_scorer()
        else:
            self.step()

    def plain_scorer(self):
        for l in range(self.L):
            self.hss.hss_score_blocks(self.dims, self.Qp[l], 1, self.A, l, self.table, self.offs,
                                      1, self.n, self.scores[l])

    def secondary(self):
        """The plain scorer (hss_score_blocks on a stored Qp), timed the same way:
        (name, function, launches per replay, algorithmic bytes per launch)."""
        for l in range(self.L):
            self.hss.hss_project_q(self.dims, self.P, self.Q[l], 1, self.Qp[l])
        return ("plain_scorer", self.plain_scorer, self.L, self.score_bytes(self.n))

    def describe(self):
        d = self.dims
        return (f"decode layer x {self.L} layers per step: {d.num_q_heads} q heads / "
                f"{d.num_kv_heads} kv heads, head_dim {d.head_dim}, r {d.r}, block_size "
                f"{d.block_size}, 1 sequence of {self.n * d.block_size} tokens ({self.n} blocks, "
                f"permuted table), 1 query row, bottom-{self.k}; per layer call: project the "
                f"block being written, project Q, score, rank"
                + (" (four calls)" if self.unfused else
                   " (hss_layer_step, queries projected in the scorer: 2 launches)"))

    l2_note = ("no flush: each step reads 32 x 16 MiB = 512 MiB of A_g, above the 129 MB L2, "
               "so every layer call reads cold A_g")

    # ---- end to end through the API with host buffers: one pinned H2D copy of the step's
    # inputs (every layer's query and new key block), 32 layer calls, one D2H of the victims.
    def e2e_setup(self):
        torch = self.torch
        q_el = self.Q[0].numel()
        k_el = self.K_new[0].numel()
        host = torch.empty(self.L * (q_el + k_el), dtype=torch.bfloat16).pin_memory()
        for l in range(self.L):
            host[l * q_el:(l + 1) * q_el].copy_(self.Q[l].reshape(-1))
            o = self.L * q_el + l * k_el
            host[o:o + k_el].copy_(self.K_new[l].reshape(-1))
        self.h_in = host
        self.d_in = torch.empty_like(host, device=self.device)
        self.d_Q = [self.d_in[l * q_el:(l + 1) * q_el].view(self.Q[0].shape)
                    for l in range(self.L)]
        self.d_K = [self.d_in[self.L * q_el + l * k_el:self.L * q_el + (l + 1) * k_el]
                    .view(self.K_new[0].shape) for l in range(self.L)]
        self.d_Q_ptrs = [t.data_ptr() for t in self.d_Q]
        self.d_K_ptrs = [t.data_ptr() for t in self.d_K]
        self.h_vic = torch.empty(self.L, 1, self.k, dtype=torch.int32).pin_memory()

    def e2e_step(self):
        self.d_in.copy_(self.h_in, non_blocking=True)
        stream = self.torch.cuda.current_stream().cuda_stream  # one lookup per step
        for l in range(self.L):
            self.layer_call(l, K_new=self.d_K_ptrs[l], Q=self.d_Q_ptrs[l], stream=stream)
        self.h_vic.copy_(self.victims, non_blocking=True)
        self.torch.cuda.current_stream().synchronize()

    @property
    def e2e_bytes(self):
        return self.h_in.numel() * 2, self.L * self.k * 4

    def oracle_case(self, seed):
        import workloads as W

        return W.decode(seed=seed, device="cpu", layers=1)


class BatchedWorkload(_Base):
    """64 sequences over a 40000-block pool; one step = one layer call for the batch."""

    name = "batched"

    def __init__(self, device, seed: int):
        super().__init__(device)
        import workloads as W

        torch, hss = self.torch, self.hss
        self.case = c = W.batched(seed=seed, device=device)
        self.dims = d = c.dims
        self.S = c.num_seqs
        self.n = c.total_blocks
        self.k = c.k_victims
        self.P = c.P.to(device)
        self.A = torch.empty(d.a_g_shape, dtype=torch.bfloat16, device=device)
        ids = c.block_ids.to(device)
        hss.hss_project_kv_blocks(d, self.P, c.K[0], 0, ids, ids.numel(), self.A)
        self.table = c.table.to(device)
        self.offs = c.seq_offsets.to(device)
        self.Q = c.Q[0]
        self.Qp = torch.empty(self.S, 1, d.num_q_heads, d.r, dtype=torch.bfloat16, device=device)
        self.scores = torch.empty(self.n, dtype=torch.float32, device=device)
        self.victims = torch.empty(self.S, self.k, dtype=torch.int32, device=device)
        torch.cuda.synchronize()

    units_per_step = property(lambda self: self.n)
    launches_per_step = 3

    def step(self, Q=None):
        hss, d = self.hss, self.dims
        hss.hss_project_q(d, self.P, self.Q if Q is None else Q, self.S, self.Qp)
        hss.hss_score_blocks(d, self.Qp, 1, self.A, 0, self.table, self.offs, self.S, self.n,
                             self.scores)
        hss.hss_rank_victims(self.scores, self.offs, self.S, self.n, self.k, self.victims)

    dominant_kernel = "score_decode"
    dominant_bound = "hbm"
    dominant_launches = 1
    dominant_units = property(lambda self: self.score_bytes(self.n))

    def dominant(self):
        self.hss.hss_score_blocks(self.dims, self.Qp, 1, self.A, 0, self.table, self.offs,
                                  self.S, self.n, self.scores)

    def describe(self):
        return (f"batched decode: {self.S} sequences (contexts U{{1024..16384}} tokens, "
                f"{self.n} blocks in all) from a 40000-block pool, 32 q / 8 kv heads, hd 128, "
                f"r 32, bottom-{self.k} per sequence; per step: project Q, score, rank")

    l2_note = "no flush: each step reads ~285 MB of A_g, above the 129 MB L2"

    def e2e_setup(self):
        torch = self.torch
        self.h_Q = self.Q.cpu().pin_memory()
        self.h_vic = torch.empty(self.S, self.k, dtype=torch.int32).pin_memory()
        self.d_Q = torch.empty_like(self.Q)

    def e2e_step(self):
        self.d_Q.copy_(self.h_Q, non_blocking=True)
        self.step(Q=self.d_Q)
        self.h_vic.copy_(self.victims, non_blocking=True)
        self.torch.cuda.current_stream().synchronize()

    @property
    def e2e_bytes(self):
        return self.Q.numel() * 2, self.S * self.k * 4


class PrefillWorkload(_Base):
    """A 512-row prefill chunk against 8192 blocks (tcgen05 scorer).  Two copies of the
    context's A_g alternate between steps so each step reads it cold (2 x 128 MiB > L2)."""

    name = "prefill"

    def __init__(self, device, seed: int):
        super().__init__(device)
        import workloads as W

        torch, hss = self.torch, self.hss
        self.case = c = W.prefill(seed=seed, device=device)
        base = c.dims
        self.dims = d = W.Dims(2, base.num_q_heads, base.num_kv_heads, base.head_dim, base.r,
                               base.block_size, base.max_blocks)
        self.n = c.total_blocks
        self.k = c.k_victims
        self.R = c.rows_per_seq
        self.P = c.P.to(device)
        self.A = torch.empty(d.a_g_shape, dtype=torch.bfloat16, device=device)
        ids = c.block_ids.to(device)
        for layer in range(2):
            hss.hss_project_kv_blocks(d, self.P, c.K[0], layer, ids, ids.numel(), self.A)
        self.table = c.table.to(device)
        self.offs = c.seq_offsets.to(device)
        # The chunk's own keys: its 512 tokens are the last 32 blocks of the table.
        nb = self.R // d.block_size
        self.new_ids = self.table[-nb:].contiguous()
        self.K_new = c.K[0][self.new_ids.long()].contiguous()
        self.Q = c.Q[0]
        self.Qp = torch.empty(1, self.R, d.num_q_heads, d.r, dtype=torch.bfloat16, device=device)
        self.scores = torch.empty(2, self.n, dtype=torch.float32, device=device)
        self.victims = torch.empty(2, 1, self.k, dtype=torch.int32, device=device)
        self.parity = 0
        torch.cuda.synchronize()

    units_per_step = property(lambda self: self.n)
    launches_per_step = 5  # ingest, project Q, fill, score, rank

    def step(self, Q=None, K_new=None):
        hss, d, l = self.hss, self.dims, self.parity
        hss.hss_project_kv_blocks(d, self.P, self.K_new if K_new is None else K_new, l,
                                  self.new_ids, self.new_ids.numel(), self.A)
        hss.hss_project_q(d, self.P, self.Q if Q is None else Q, self.R, self.Qp)
        hss.hss_score_blocks(d, self.Qp, self.R, self.A, l, self.table, self.offs, 1, self.n,
                             self.scores[l])
        hss.hss_rank_victims(self.scores[l], self.offs, 1, self.n, self.k, self.victims[l])
        self.parity ^= 1

    def steps_for_graph(self):
        # A graph holds both parities so replays alternate the A_g copy.
        self.step()
        self.step()

    graph_steps = 2
    dominant_kernel = "score_tc"
    dominant_bound = "tensor"
    dominant_launches = 2

    @property
    def dominant_units(self):
        d = self.dims
        return 2.0 * self.R * d.num_q_heads * d.block_size * d.r * self.n  # flop per launch

    def dominant(self):
        for l in range(2):
            self.hss.hss_score_blocks(self.dims, self.Qp, self.R, self.A, l, self.table,
                                      self.offs, 1, self.n, self.scores[l])

    def describe(self):
        d = self.dims
        return (f"prefill chunk: {self.R} query rows x {d.num_q_heads} q heads (g "
                f"{d.num_q_heads // d.num_kv_heads}) against {self.n} blocks "
                f"({self.n * d.block_size} tokens), hd {d.head_dim}, r {d.r}, bottom-{self.k}; "
                f"per step: project the chunk's {self.new_ids.numel()} blocks, project Q, "
                f"score (tcgen05), rank")

    l2_note = ("no flush: steps alternate between two 128 MiB copies of the context's A_g "
               "(256 MiB > 129 MB L2)")

    def e2e_setup(self):
        torch = self.torch
        self.h_Q = self.Q.cpu().pin_memory()
        self.h_K = self.K_new.cpu().pin_memory()
        self.h_vic = torch.empty(self.k, dtype=torch.int32).pin_memory()
        self.d_Q = torch.empty_like(self.Q)
        self.d_K = torch.empty_like(self.K_new)

    def e2e_step(self):
        self.d_Q.copy_(self.h_Q, non_blocking=True)
        self.d_K.copy_(self.h_K, non_blocking=True)
        l = self.parity
        self.step(Q=self.d_Q, K_new=self.d_K)
        self.h_vic.copy_(self.victims[l][0], non_blocking=True)
        self.torch.cuda.current_stream().synchronize()

    @property
    def e2e_bytes(self):
        return self.Q.numel() * 2 + self.K_new.numel() * 2, self.k * 4


class PrefillRowsWorkload(PrefillWorkload):
    """The prefill chunk with per-row selection (QSA-style): every query row scores the
    8192 blocks on its own and takes the 128 it has seen whole with the largest scores.
    The chunk is the context's last 512 tokens (first_pos = 131072 - 512), so every row has
    seen between 8160 and 8191 blocks whole."""

    name = "prefill_rows"
    topk = 128

    def __init__(self, device, seed: int):
        super().__init__(device, seed)
        torch = self.torch
        self.row_scores = torch.empty(2, self.R, self.n, dtype=torch.float32, device=device)
        self.lists = torch.empty(2, self.R, self.topk, dtype=torch.int32, device=device)
        self.first_pos = self.n * self.dims.block_size - self.R
        torch.cuda.synchronize()

    launches_per_step = 5  # ingest, project Q, fill, score rows, select rows

    def step(self, Q=None, K_new=None):
        hss, d, l = self.hss, self.dims, self.parity
        hss.hss_project_kv_blocks(d, self.P, self.K_new if K_new is None else K_new, l,
                                  self.new_ids, self.new_ids.numel(), self.A)
        hss.hss_project_q(d, self.P, self.Q if Q is None else Q, self.R, self.Qp)
        hss.hss_score_rows(d, self.Qp, self.R, self.A, l, self.table, self.n, self.row_scores[l])
        hss.hss_select_rows(self.row_scores[l], self.R, self.n, self.first_pos, d.block_size,
                            self.topk, self.lists[l])
        self.parity ^= 1

    dominant_kernel = "score_tc (per-row)"

    def dominant(self):
        for l in range(2):
            self.hss.hss_score_rows(self.dims, self.Qp, self.R, self.A, l, self.table, self.n,
                                    self.row_scores[l])

    def describe(self):
        d = self.dims
        return (f"prefill chunk, per-row selection: {self.R} query rows x {d.num_q_heads} q "
                f"heads (g {d.num_q_heads // d.num_kv_heads}) against {self.n} blocks, hd "
                f"{d.head_dim}, r {d.r}; per step: project the chunk's "
                f"{self.new_ids.numel()} blocks, project Q, per-row scores (tcgen05), per-row "
                f"top-{self.topk} of the blocks each row has seen whole")

    def e2e_step(self):
        self.d_Q.copy_(self.h_Q, non_blocking=True)
        self.d_K.copy_(self.h_K, non_blocking=True)
        l = self.parity
        self.step(Q=self.d_Q, K_new=self.d_K)
        self.h_lists.copy_(self.lists[l], non_blocking=True)
        self.torch.cuda.current_stream().synchronize()

    def e2e_setup(self):
        super().e2e_setup()
        self.h_lists = self.torch.empty(self.R, self.topk, dtype=self.torch.int32).pin_memory()

    @property
    def e2e_bytes(self):
        return self.Q.numel() * 2 + self.K_new.numel() * 2, self.R * self.topk * 4


class IngestWorkload(_Base):
    """4096 new blocks projected into each of 32 layers, then one layer's 65536 blocks
    scored and ranked; skewed keys.  One step = 32 ingest calls + project Q + score + rank."""

    name = "ingest"

    def __init__(self, device, seed: int, layers: int = 32):
        super().__init__(device)
        import workloads as W

        torch, hss = self.torch, self.hss
        self.case = c = W.ingest(seed=seed, device=device, layers=layers,
                                 score_layer=min(17, layers - 1))
        self.dims = d = c.dims
        self.L = d.num_layers
        self.n = c.total_blocks
        self.k = c.k_victims
        self.P = c.P.to(device)
        self.A = torch.empty(d.a_g_shape, dtype=torch.bfloat16, device=device)
        self.new_ids = c.block_ids.to(device)
        self.K = c.K
        self.layer = c.score_layer
        fill = c.fill_ids.to(device)
        hss.hss_project_kv_blocks(d, self.P, c.K_fill, self.layer, fill, fill.numel(), self.A)
        self.table = c.table.to(device)
        self.offs = c.seq_offsets.to(device)
        self.Q = c.Q[0]
        self.Qp = torch.empty(1, 1, d.num_q_heads, d.r, dtype=torch.bfloat16, device=device)
        self.scores = torch.empty(self.n, dtype=torch.float32, device=device)
        self.victims = torch.empty(1, self.k, dtype=torch.int32, device=device)
        torch.cuda.synchronize()

    units_per_step = property(lambda self: self.n)
    launches_per_step = property(lambda self: self.L + 3)

    def step(self):
        hss, d = self.hss, self.dims
        nb = self.new_ids.numel()
        for l in range(self.L):
            hss.hss_project_kv_blocks(d, self.P, self.K[l], l, self.new_ids, nb, self.A)
        hss.hss_project_q(d, self.P, self.Q, 1, self.Qp)
        hss.hss_score_blocks(d, self.Qp, 1, self.A, self.layer, self.table, self.offs, 1, self.n,
                             self.scores)
        hss.hss_rank_victims(self.scores, self.offs, 1, self.n, self.k, self.victims)

    dominant_kernel = "project (ingest)"
    dominant_bound = "hbm"
    dominant_launches = property(lambda self: self.L)

    @property
    def dominant_units(self):
        d = self.dims
        nb = self.new_ids.numel()
        return nb * d.block_size * d.num_kv_heads * (d.head_dim * 2 + d.r * 2) + d.head_dim * d.r * 2

    def dominant(self):
        nb = self.new_ids.numel()
        for l in range(self.L):
            self.hss.hss_project_kv_blocks(self.dims, self.P, self.K[l], l, self.new_ids, nb,
                                           self.A)

    def secondary(self):
        """The score of the whole step's layer (65536 blocks, one hss_score_blocks launch),
        timed on its own."""
        self.hss.hss_project_q(self.dims, self.P, self.Q, 1, self.Qp)

        def score():
            self.hss.hss_score_blocks(self.dims, self.Qp, 1, self.A, self.layer, self.table,
                                      self.offs, 1, self.n, self.scores)
        return ("c5_score", score, 1, self.score_bytes(self.n))

    def describe(self):
        return (f"ingest + score under skew: {self.new_ids.numel()} new blocks projected into "
                f"each of {self.L} layers (K with 4 outlier channels x20 and log-normal token "
                f"norms), then layer {self.layer}'s {self.n} blocks scored, bottom-{self.k}")

    l2_note = "no flush: each step reads 4 GiB of K and 512 MiB of A_g, far above the 129 MB L2"

    def e2e_setup(self):
        # Every step's new key blocks (all 32 layers, 4 GiB) and the query come from pinned
        # host memory, layer by layer, into the device buffers the step projects from.
        torch = self.torch
        self.h_K = [k.cpu().pin_memory() for k in self.K]
        self.h_Q = self.Q.cpu().pin_memory()
        self.h_vic = torch.empty(1, self.k, dtype=torch.int32).pin_memory()

    def e2e_step(self):
        hss, d = self.hss, self.dims
        nb = self.new_ids.numel()
        for l in range(self.L):
            self.K[l].copy_(self.h_K[l], non_blocking=True)
            hss.hss_project_kv_blocks(d, self.P, self.K[l], l, self.new_ids, nb, self.A)
        self.Q.copy_(self.h_Q, non_blocking=True)
        hss.hss_project_q(d, self.P, self.Q, 1, self.Qp)
        hss.hss_score_blocks(d, self.Qp, 1, self.A, self.layer, self.table, self.offs, 1, self.n,
                             self.scores)
        hss.hss_rank_victims(self.scores, self.offs, 1, self.n, self.k, self.victims)
        self.h_vic.copy_(self.victims, non_blocking=True)
        self.torch.cuda.current_stream().synchronize()

    @property
    def e2e_bytes(self):
        return sum(k.numel() for k in self.K) * 2 + self.Q.numel() * 2, self.k * 4


class IngestTokensWorkload(IngestWorkload):
    """The ingest workload through the cache-write path: each layer's keys of the 4096 new
    blocks arrive as 65536 tokens (block * 16 + position slots) and one hss_write_kv_tokens
    call per layer writes them into the paged key cache and their projections into A_g."""

    name = "ingest_tokens"

    def __init__(self, device, seed: int, layers: int = 32):
        super().__init__(device, seed, layers)
        torch, d = self.torch, self.dims
        bs, nkv, hd = d.block_size, d.num_kv_heads, d.head_dim
        ids = self.new_ids.to(torch.int64)
        self.slots = (ids[:, None] * bs + torch.arange(bs, device=device)[None, :]).reshape(-1)
        self.n_tok = self.slots.numel()
        self.K_tok = [k.view(self.n_tok, nkv, hd) for k in self.K]
        # One paged key cache (2 GiB) that every layer writes: the same bytes per call as a
        # cache per layer.
        self.cache = torch.empty(d.max_blocks, bs, nkv, hd, dtype=torch.bfloat16, device=device)
        torch.cuda.synchronize()

    def ingest(self, l):
        self.hss.hss_write_kv_tokens(self.dims, self.P, self.K_tok[l], self.slots, self.n_tok,
                                     self.cache, self.A, l)

    def step(self):
        hss, d = self.hss, self.dims
        for l in range(self.L):
            self.ingest(l)
        hss.hss_project_q(d, self.P, self.Q, 1, self.Qp)
        hss.hss_score_blocks(d, self.Qp, 1, self.A, self.layer, self.table, self.offs, 1, self.n,
                             self.scores)
        hss.hss_rank_victims(self.scores, self.offs, 1, self.n, self.k, self.victims)

    dominant_kernel = "project (cache write + A_g, tokens)"

    @property
    def dominant_units(self):
        d = self.dims
        # key row read, key row written to the cache, A_g row written; P once; slots
        return (self.n_tok * d.num_kv_heads * (2 * d.head_dim * 2 + d.r * 2) +
                d.head_dim * d.r * 2 + self.n_tok * 8)

    def dominant(self):
        for l in range(self.L):
            self.ingest(l)

    def describe(self):
        return (f"ingest + score under skew through the cache write: {self.n_tok} new tokens "
                f"({self.new_ids.numel()} blocks) written into the paged key cache and A_g of "
                f"each of {self.L} layers (one call per layer), then layer {self.layer}'s "
                f"{self.n} blocks scored, bottom-{self.k}")

    l2_note = ("no flush: each step reads 4 GiB of keys and writes 4 GiB of cache and 1 GiB of "
               "A_g, far above the 129 MB L2")

    def e2e_step(self):
        hss, d = self.hss, self.dims
        for l in range(self.L):
            self.K[l].copy_(self.h_K[l], non_blocking=True)
            self.ingest(l)
        self.Q.copy_(self.h_Q, non_blocking=True)
        hss.hss_project_q(d, self.P, self.Q, 1, self.Qp)
        hss.hss_score_blocks(d, self.Qp, 1, self.A, self.layer, self.table, self.offs, 1, self.n,
                             self.scores)
        hss.hss_rank_victims(self.scores, self.offs, 1, self.n, self.k, self.victims)
        self.h_vic.copy_(self.victims, non_blocking=True)
        self.torch.cuda.current_stream().synchronize()


WORKLOADS = {"decode": DecodeWorkload, "batched": BatchedWorkload, "prefill": PrefillWorkload,
             "ingest": IngestWorkload, "ingest_tokens": IngestTokensWorkload,
             "prefill_rows": PrefillRowsWorkload}


# ----------------------------------------------------------------------------- oracle timing

def _bits(t):
    import numpy as np
    import torch

    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


SAMPLE_BLOCKS = {"decode": 2048, "batched": 544, "prefill": 8, "ingest": 256,
                 "ingest_tokens": 256, "prefill_rows": 8}


class OracleSample:
    """The CPU oracle on a sample of one workload's step, in the GPU step's proportions.

    Each call projects the query rows, projects `ingest_per_block` new blocks per scored
    block (the decode workloads project one block per layer call; the ingest workload two
    per scored block), scores `m` table entries and ranks them.  Unit: blocks scored/s.
    """

    def __init__(self, name: str, seed: int, threads: int):
        import numpy as np

        import oracle
        import workloads as W

        self.np, self.oracle, self.threads = np, oracle, threads
        self.tokens = name == "ingest_tokens"  # ingest through the oracle's cache write
        self.rows = name == "prefill_rows"    # per-row scores and per-row selection
        if self.tokens:
            name = "ingest"
        if self.rows:
            name = "prefill"
        one = lambda d, mb=None: W.Dims(1, d.num_q_heads, d.num_kv_heads, d.head_dim, d.r,
                                        d.block_size, mb or d.max_blocks)
        # (dims, query rows, key distribution, blocks drawn, ingest per call, ingest per scored)
        spec = {"decode": (one(W.DECODE), 1, "normal", 2048, 1, 0.0),
                "batched": (W.BATCHED, 1, "normal", 1024, 0, 0.0),
                "prefill": (W.PREFILL, 512, "normal", 64, 32, 0.0),
                "ingest": (one(W.INGEST, 1024 if self.tokens else None), 1, "skewed", 1024, 0,
                           2.0)}[name]
        dims, rows, kind, pool, self.extra_ingest, self.ingest_ratio = spec
        m = SAMPLE_BLOCKS[name]
        c = W.generic(name, dims, num_seqs=1, rows_per_seq=rows, lengths=[min(m, pool)],
                      k_victims={"decode": 256, "batched": 64, "prefill": 1024,
                                 "ingest": 4096}[name],
                      seed=seed, key_kind=kind, pool=pool)
        self.case = c
        d = c.dims
        self.P = _bits(c.P)
        self.Q = _bits(c.Q[0])
        self.K = _bits(c.K[0])
        self.table = c.table.numpy()
        self.pool = self.K.shape[0]
        self.A = np.zeros((1, d.max_blocks, d.num_kv_heads, d.block_size, d.r), dtype=np.uint16)
        if self.tokens:
            self.cache = np.zeros((d.max_blocks, d.block_size, d.num_kv_heads, d.head_dim),
                                  dtype=np.uint16)

    def call(self, m: int):
        """One sampled call scoring m entries; returns m."""
        np, oracle, c = self.np, self.oracle, self.case
        ids = (self.table[:m] % self.pool).astype(np.int32)
        n_ing = self.extra_ingest + int(round(self.ingest_ratio * m))
        if n_ing > 0:
            pos = np.arange(n_ing) % self.pool
            bid = ids[pos % m] if m else pos.astype(np.int32)
            if self.tokens:
                d = c.dims
                slots = (bid.astype(np.int64)[:, None] * d.block_size +
                         np.arange(d.block_size)[None, :]).reshape(-1)
                oracle.write_kv_tokens(self.P, self.K[pos].reshape(-1, d.num_kv_heads,
                                                                   d.head_dim),
                                       slots, 0, self.A, K_cache=self.cache,
                                       nthreads=self.threads)
            else:
                oracle.project_kv_blocks(self.P, self.K[pos], 0, bid, self.A,
                                         nthreads=self.threads)
        Qp = oracle.project_q(self.Q, self.P, nthreads=self.threads)
        if self.rows:
            d = c.dims
            s, _, _ = oracle.score_rows(Qp.reshape(-1, d.num_q_heads, d.r), self.A, 0, ids,
                                        nthreads=self.threads)
            oracle.select_rows(s.astype(np.float32), m, m * d.block_size, d.block_size,
                               min(128, max(1, m)))
            return m
        offs = np.array([0, m], dtype=np.int64)
        s, _, _ = oracle.score_blocks(Qp, self.A, 0, ids, offs, nthreads=self.threads)
        oracle.rank_victims(s.astype(np.float32), offs, max(1, min(c.k_victims, m)))
        return m

    def prepare(self, m: int):
        """Project the sampled blocks' context (untimed)."""
        ids = (self.table[:m] % self.pool).astype(self.np.int32)
        pos = self.np.arange(m) % self.pool
        self.oracle.project_kv_blocks(self.P, self.K[pos], 0, ids, self.A,
                                      nthreads=self.threads)

    def time(self, m: int, seconds: float, max_calls=None):
        self.prepare(m)
        calls, scored = 0, 0
        t0 = time.perf_counter()
        while True:
            scored += self.call(m)
            calls += 1
            el = time.perf_counter() - t0
            if el >= seconds or (max_calls is not None and calls >= max_calls):
                return scored, el, calls


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
    threads = args.cpu_threads or cpu_threads()
    orc = OracleSample(args.workload, args.seed, threads)
    m_full = SAMPLE_BLOCKS[args.workload]
    # Per-block cost, to size each step's sample so the whole run takes about a minute.
    scored, el, _ = orc.time(min(16, m_full), 0.0, max_calls=1)
    per_block = el / max(scored, 1)
    total_steps = args.steps + args.warmup
    m = int(max(1, min(m_full, 60.0 / max(total_steps * per_block, 1e-12))))
    orc.prepare(m)
    for _ in range(args.warmup):
        orc.call(m)
    t0 = time.perf_counter()
    blocks = 0
    for _ in range(args.steps):
        blocks += orc.call(m)
    el = time.perf_counter() - t0
    value = blocks / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "blocks/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload} (CPU oracle, {m} blocks scored per step)"},
        "cpu_baseline": {"value": value, "unit": "blocks/s", "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} sampled {args.workload} calls of {m} blocks"},
        "e2e": {"value": value, "unit": "blocks/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def time_launches(fn, stream, reps: int, launches: int) -> float:
    """Seconds per launch: a CUDA graph of `fn` (`launches` back-to-back launches) replayed
    `reps` times, timed with CUDA events on the launching stream (gaps between graph nodes
    included)."""
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) / 1e3 / (reps * launches)


def roofline_of(bound: str, units: float, sec: float, peaks: dict) -> dict:
    if bound == "hbm":
        return {"bound": "hbm", "achieved": units / sec / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": units / sec / 1e9 / peaks["hbm_gbs"],
                "peak_source": peaks["source"] + " hbm_gbs (copy)"}
    return {"bound": "tensor", "achieved": units / sec / 1e12, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": units / sec / 1e12 / peaks["bf16_tflops"],
            "peak_source": peaks["source"] + " bf16_tflops (burst, cuBLAS)"}


def run_timed(wl, stream, steps: int, warmup: int, use_graph: bool, world: int, device,
              min_seconds: float = 0.0):
    """Warm up, capture the step into a graph, time `steps` steps (rounded to whole replays;
    with min_seconds > 0, as many more as that many seconds take).  Returns
    (steps timed, max elapsed over ranks, total units, clock summary)."""
    import torch

    per_replay = getattr(wl, "graph_steps", 1)
    capture = getattr(wl, "steps_for_graph", wl.step)
    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 3)):
            capture()
    stream.synchronize()
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            capture()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
    run_replay = graph.replay if graph is not None else capture
    replays = max(1, steps // per_replay)
    if min_seconds > 0:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(3):
                run_replay()
            e1.record(stream)
        stream.synchronize()
        per = e0.elapsed_time(e1) / 1e3 / 3
        replays = max(replays, int(min_seconds / max(per, 1e-9)) + 1)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    torch.cuda.synchronize()
    with ClockSampler(device_uuid(torch.cuda.current_device())) as clocks:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(replays):
                run_replay()
            ev1.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    barrier(world, device)
    elapsed = ev0.elapsed_time(ev1) / 1e3
    n_steps = replays * per_replay
    elapsed_max, units = aggregate(elapsed, wl.units_per_step * n_steps, world, device)
    return n_steps, elapsed_max, units, clocks.summary()


def dominant_roofline(wl, stream, peaks, reps: int, traffic=None) -> dict:
    sec = time_launches(wl.dominant, stream, reps, wl.dominant_launches)
    r = roofline_of(wl.dominant_bound, wl.dominant_units, sec, peaks)
    r.update({"kernel": wl.dominant_kernel, "traffic": traffic[0] if traffic else None,
              "traffic_source": traffic[1] if traffic else "not captured since the kernel "
                                                               "changed",
              "launch_us": sec * 1e6,
              "work_per_launch": wl.dominant_units,
              "how": "CUDA events around graph replays of back-to-back launches of this kernel "
                     "on its launching stream (gaps between graph nodes included)"})
    return r


def secondary_roofline(wl, stream, peaks, reps: int):
    if not hasattr(wl, "secondary"):
        return None
    name, fn, launches, units = wl.secondary()
    sec = time_launches(fn, stream, reps, launches)
    r = roofline_of("hbm", units, sec, peaks)
    r.update({"launch_us": sec * 1e6, "work_per_launch": units})
    return name, r


def run_extras(args, device, stream, peaks) -> dict:
    """Short passes of the batched, prefill and ingest workloads (one GPU, no e2e, no oracle):
    value, per-step time, the dominant kernel's roofline and the clocks of each, so that
    their fractions are measured in the default run.  Each timed region lasts ~1 s."""
    import torch

    out = {}
    for name in ("batched", "prefill", "ingest"):
        wl = WORKLOADS[name](device, args.seed)
        n_steps, el, units, clk = run_timed(wl, stream, 20, 5, True, 1, device, min_seconds=1.0)
        entry = {"value": units / el, "unit": "blocks/s", "steps": n_steps,
                 "ms_per_step": el / n_steps * 1e3, "workload": wl.describe(),
                 "l2": wl.l2_note, "clocks": clk,
                 "roofline": dominant_roofline(wl, stream, peaks, 50,
                                               TRAFFIC.get(name))}
        sec = secondary_roofline(wl, stream, peaks, 50)
        if sec is not None:
            out[sec[0]] = sec[1]
        out[name] = entry
        del wl
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


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

    if args.workload == "decode":
        wl = DecodeWorkload(device, args.seed + rank, unfused=args.unfused)
    elif args.workload in ("ingest", "ingest_tokens"):
        wl = WORKLOADS[args.workload](device, args.seed + rank, layers=args.layers)
    else:
        wl = WORKLOADS[args.workload](device, args.seed + rank)
    peaks = measured_peaks()
    stream = torch.cuda.Stream(device=device)
    torch.cuda.synchronize()
    per_replay = getattr(wl, "graph_steps", 1)
    describe, l2_note = wl.describe(), wl.l2_note
    launches, slot = wl.launches_per_step, wl.slot_bytes()

    # ---- timed region: exactly the requested steps
    steps, elapsed_max, units, clocks = run_timed(wl, stream, args.steps, args.warmup,
                                                  not args.no_graph, world, device)
    value = units / elapsed_max

    # ---- dominant kernel: graphs of back-to-back launches timed with events on its stream
    reps = max(20, min(400, args.steps // 4))
    roofline = dominant_roofline(wl, stream, peaks, reps, TRAFFIC.get(args.workload))
    secondary = secondary_roofline(wl, stream, peaks, reps)

    # ---- end to end through the API with host buffers
    e2e = None
    if args.e2e_steps > 0:
        wl.e2e_setup()
        n_e2e = max(1, args.e2e_steps // per_replay) * per_replay
        with torch.cuda.stream(stream):
            for _ in range(3 * per_replay):
                wl.e2e_step()
            torch.cuda.synchronize()
            barrier(world, device)
            t0 = time.perf_counter()
            for _ in range(n_e2e):
                wl.e2e_step()
            t1 = time.perf_counter()
        el_e2e, units_e2e = aggregate(t1 - t0, wl.units_per_step * n_e2e, world, device)
        h2d, d2h = wl.e2e_bytes
        e2e = {"value": units_e2e / el_e2e, "unit": "blocks/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "how": "every call from the host through the C ABI (no graph): pinned H2D of the "
                      "step's new inputs, D2H of the victims, one sync per step"}

    err = hss.hss_read_device_error()
    if err != 0:
        raise SystemExit(f"device error raised during the benchmark: {hss.status_string(err)}")

    extras = None
    if args.workload == "decode" and not args.no_extras and world == 1:
        del wl
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        extras = run_extras(args, device, stream, peaks)
        err = hss.hss_read_device_error()
        if err != 0:
            raise SystemExit(f"device error raised during the extra workloads: "
                             f"{hss.status_string(err)}")
        wl = None

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        threads = args.cpu_threads or cpu_threads()
        orc = OracleSample(args.workload, args.seed, threads)
        m = SAMPLE_BLOCKS[args.workload]
        scored, el, calls = orc.time(m, 10.0)
        cpu = {"value": scored / el, "unit": "blocks/s", "cores": threads, "kind": "oracle",
               "sample": f"{calls} oracle calls on the {args.workload} workload, {m} blocks "
                         f"scored per call in the GPU step's proportions, ~10 s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "blocks/s", "n_gpus": world,
            "steps": steps, "warmup": args.warmup,
            "ms_per_step": elapsed_max / steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "a_g_gbs": value * slot / 1e9,
            "a_g_hbm_frac": value * slot / 1e9 / peaks["hbm_gbs"],
            "config": {"workload": describe, "l2": l2_note, "graph": not args.no_graph,
                       "parallelism": f"replicas x{world}"},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches * steps,
            "clocks": clocks,
        }
        if secondary is not None:
            line[secondary[0]] = secondary[1]
        if extras is not None:
            line["workloads"] = extras
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
