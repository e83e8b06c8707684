"""Seeded synthetic inputs for the low-rank KV-block predictor.

This module only draws inputs; it holds none of the predictor's arithmetic.
Both the CUDA path and the CPU oracle are fed the bytes it produces, so the
two sides always see identical inputs.

Draw discipline (one seed per case):
  * a CPU ``torch.Generator`` draws everything small and structural, in this
    order: P, then the block-table structure (sequence lengths, permutation,
    sampled block ids, outlier channels);
  * a generator on the target device draws the large bf16 tensors in this
    order: Q, then K (layer by layer).
Values are drawn in fp32 and rounded to bf16 (round to nearest even) by
PyTorch's dtype conversion.

Workload shapes follow the pages' predictor (page "metrale_storage/predictor.rs",
`PredictorDims`): num_layers, num_q_heads, num_kv_heads, head_dim, r,
block_size, max_blocks.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass(frozen=True)
class Dims:
    """The seven predictor dimensions (PredictorDims on the predictor page)."""

    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    r: int
    block_size: int
    max_blocks: int

    @property
    def gqa(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def slot_elems(self) -> int:
        return self.num_kv_heads * self.block_size * self.r

    @property
    def a_g_shape(self):
        return (self.num_layers, self.max_blocks, self.num_kv_heads, self.block_size, self.r)


@dataclass
class Case:
    """One seeded input set.

    P            [head_dim, r] bf16
    Q            [num_q_layers, num_seqs, rows_per_seq, num_q_heads, head_dim] bf16
    K            [num_k_layers, n, block_size, num_kv_heads, head_dim] bf16
                 (K[l] is projected into A_g layer ingest_layers[l])
    block_ids    [n] int32, the slots K[l] is written to
    table        [total] int32 physical block ids, CSR order
    seq_offsets  [num_seqs + 1] int32
    """

    name: str
    dims: Dims
    num_seqs: int
    rows_per_seq: int
    k_victims: int
    P: torch.Tensor
    Q: torch.Tensor
    K: torch.Tensor
    block_ids: torch.Tensor
    ingest_layers: list
    table: torch.Tensor
    seq_offsets: torch.Tensor
    score_layer: int = 0
    K_fill: Optional[torch.Tensor] = None
    fill_ids: Optional[torch.Tensor] = None
    notes: dict = field(default_factory=dict)

    @property
    def total_blocks(self) -> int:
        return int(self.table.numel())


def _cpu_gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _dev_gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed + 0x9E3779B1)
    return g


def bf16_normal(gen: torch.Generator, shape, std: float = 1.0, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32, rounded to bf16."""
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def projection(gen: torch.Generator, head_dim: int, r: int) -> torch.Tensor:
    """P [head_dim, r] with entries N(0, 1/r), as bf16 (drawn on the CPU)."""
    return bf16_normal(gen, (head_dim, r), std=1.0 / math.sqrt(r))


def skewed_keys(gen: torch.Generator, shape, channels: torch.Tensor, outlier_scale: float = 20.0,
                device="cpu") -> torch.Tensor:
    """Keys with outlier channels and log-normal per-token norms.

    shape is [..., block_size, num_kv_heads, head_dim].  Every key vector starts
    as N(0, 1) per channel; the listed channels (the same for all heads and
    tokens) are multiplied by outlier_scale; then every token (all of its kv
    heads together) is multiplied by exp(N(0, 1)).
    """
    z = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    z[..., channels.to(device)] *= outlier_scale
    tok = torch.randn(tuple(shape[:-2]) + (1, 1), generator=gen, device=device,
                      dtype=torch.float32)
    z.mul_(torch.exp(tok))
    return z.to(torch.bfloat16)


def identity_offsets(lengths) -> torch.Tensor:
    offs = [0]
    for n in lengths:
        offs.append(offs[-1] + int(n))
    return torch.tensor(offs, dtype=torch.int32)


def batched_lengths(gen: torch.Generator, num_seqs: int, lo_tokens: int, hi_tokens: int,
                    block_size: int, pool: int):
    """Context lengths ~ U{lo..hi} tokens, in blocks; redrawn until they fit the pool."""
    for _ in range(1000):
        ctx = torch.randint(lo_tokens, hi_tokens + 1, (num_seqs,), generator=gen)
        nblk = (ctx + block_size - 1) // block_size
        if int(nblk.sum()) <= pool:
            return [int(x) for x in nblk]
    raise RuntimeError("could not draw lengths that fit the block pool")


def generic(name: str, dims: Dims, *, num_seqs: int, rows_per_seq: int, lengths, k_victims: int,
            seed: int = 0, device="cpu", key_kind: str = "normal", ingest_layers=None,
            score_layer: int = 0, permute: bool = True, pool: Optional[int] = None,
            q_layers: int = 1, q_std: float = 1.0) -> Case:
    """A case of arbitrary shape: every block of the pool is written once.

    The pool is the first `pool` ids (default: the sum of lengths); the table
    lists a seeded permutation of the pool (or the identity), cut into
    sequences of the given lengths.
    """
    cg = _cpu_gen(seed)
    dg = _dev_gen(seed, device)
    P = projection(cg, dims.head_dim, dims.r)
    total = sum(int(n) for n in lengths)
    pool = total if pool is None else pool
    if total > pool or pool > dims.max_blocks:
        raise ValueError("lengths exceed the pool, or the pool exceeds max_blocks")
    perm = torch.randperm(pool, generator=cg) if permute else torch.arange(pool)
    table = perm[:total].to(torch.int32)
    channels = torch.randperm(dims.head_dim, generator=cg)[:4]
    ingest_layers = list(ingest_layers) if ingest_layers is not None else [score_layer]
    Q = bf16_normal(dg, (q_layers, num_seqs, rows_per_seq, dims.num_q_heads, dims.head_dim),
                    std=q_std, device=device)
    kshape = (len(ingest_layers), pool, dims.block_size, dims.num_kv_heads, dims.head_dim)
    if key_kind == "normal":
        K = bf16_normal(dg, kshape, device=device)
    elif key_kind == "skewed":
        K = skewed_keys(dg, kshape, channels, device=device)
    else:
        raise ValueError(key_kind)
    return Case(name=name, dims=dims, num_seqs=num_seqs, rows_per_seq=rows_per_seq,
                k_victims=k_victims, P=P, Q=Q, K=K,
                block_ids=torch.arange(pool, dtype=torch.int32), ingest_layers=ingest_layers,
                table=table, seq_offsets=identity_offsets(lengths), score_layer=score_layer,
                notes={"channels": channels.tolist(), "key_kind": key_kind})


# ----------------------------------------------------------------------------- configs
#
# The five workloads, with the sizes of their descriptions.  "tiny" is small
# enough for the oracle to run in full; the others are run in full on the GPU
# and checked against the oracle on sampled outputs.

TINY = Dims(num_layers=1, num_q_heads=4, num_kv_heads=2, head_dim=64, r=16, block_size=16,
            max_blocks=64)
DECODE = Dims(num_layers=32, num_q_heads=32, num_kv_heads=8, head_dim=128, r=32, block_size=16,
              max_blocks=2048)
BATCHED = Dims(num_layers=1, num_q_heads=32, num_kv_heads=8, head_dim=128, r=32, block_size=16,
               max_blocks=40000)
PREFILL = Dims(num_layers=1, num_q_heads=64, num_kv_heads=8, head_dim=128, r=64, block_size=16,
               max_blocks=8192)
INGEST = Dims(num_layers=32, num_q_heads=32, num_kv_heads=8, head_dim=128, r=32, block_size=16,
              max_blocks=65536)


def tiny(seed: int = 0, device="cpu") -> Case:
    """1 layer, 4 q heads / 2 kv heads, hd 64, r 16, 64 blocks, identity table, bottom-8."""
    return generic("tiny", TINY, num_seqs=1, rows_per_seq=1, lengths=[64], k_victims=8,
                   seed=seed, device=device, permute=False)


def decode(seed: int = 0, device="cpu", layers: int = 32) -> Case:
    """Llama-3-8B-like decode layer: 2048 blocks (32768 tokens), 1 row, bottom-256.

    All `layers` A_g layers are projected (one K per layer) so that successive
    layer calls read data that is not in L2.
    """
    d = Dims(num_layers=layers, **{k: getattr(DECODE, k) for k in
                                   ("num_q_heads", "num_kv_heads", "head_dim", "r",
                                    "block_size", "max_blocks")})
    return generic("decode", d, num_seqs=1, rows_per_seq=1, lengths=[2048], k_victims=256,
                   seed=seed, device=device, ingest_layers=range(layers), q_layers=layers)


def batched(seed: int = 0, device="cpu") -> Case:
    """64 sequences, contexts U{1024..16384} tokens, tables from a 40000-block pool, bottom-64."""
    cg = _cpu_gen(seed + 7)
    lengths = batched_lengths(cg, 64, 1024, 16384, BATCHED.block_size, BATCHED.max_blocks)
    return generic("batched", BATCHED, num_seqs=64, rows_per_seq=1, lengths=lengths,
                   k_victims=64, seed=seed, device=device, pool=BATCHED.max_blocks)


def prefill(seed: int = 0, device="cpu") -> Case:
    """512 query rows against 8192 blocks (131072 tokens), g = 8, r = 64, bottom-1024."""
    return generic("prefill", PREFILL, num_seqs=1, rows_per_seq=512, lengths=[8192],
                   k_victims=1024, seed=seed, device=device)


def ingest(seed: int = 0, device="cpu", layers: int = 32, new_blocks: int = 4096,
           score_layer: int = 17) -> Case:
    """Skewed keys: 4096 new blocks projected into each of 32 layers, then one layer scored.

    The scored layer's other slots are filled (untimed) from the same key
    distribution; its table is a permutation of all 65536 slots; bottom-4096.
    """
    d = Dims(num_layers=layers, **{k: getattr(INGEST, k) for k in
                                   ("num_q_heads", "num_kv_heads", "head_dim", "r",
                                    "block_size", "max_blocks")})
    cg = _cpu_gen(seed)
    dg = _dev_gen(seed, device)
    P = projection(cg, d.head_dim, d.r)
    table = torch.randperm(d.max_blocks, generator=cg).to(torch.int32)
    new_ids = torch.randperm(d.max_blocks, generator=cg)[:new_blocks].to(torch.int32)
    channels = torch.randperm(d.head_dim, generator=cg)[:4]
    mask = torch.ones(d.max_blocks, dtype=torch.bool)
    mask[new_ids.long()] = False
    fill_ids = torch.nonzero(mask).flatten().to(torch.int32)
    Q = bf16_normal(dg, (1, 1, 1, d.num_q_heads, d.head_dim), device=device)
    K = skewed_keys(dg, (layers, new_blocks, d.block_size, d.num_kv_heads, d.head_dim), channels,
                    device=device)
    K_fill = skewed_keys(dg, (int(fill_ids.numel()), d.block_size, d.num_kv_heads, d.head_dim),
                         channels, device=device)
    return Case(name="ingest", dims=d, num_seqs=1, rows_per_seq=1, k_victims=4096, P=P, Q=Q,
                K=K, block_ids=new_ids, ingest_layers=list(range(layers)), table=table,
                seq_offsets=identity_offsets([d.max_blocks]), score_layer=score_layer,
                K_fill=K_fill, fill_ids=fill_ids,
                notes={"channels": channels.tolist(), "key_kind": "skewed"})


CONFIGS = {"tiny": tiny, "decode": decode, "batched": batched, "prefill": prefill,
           "ingest": ingest}


def random_scores(seed: int, lengths, *, ties: float = 0.0, device="cpu") -> tuple:
    """f32 block scores per sequence (for the victim ranking alone), with optional exact ties.

    A fraction `ties` of the entries copy another entry of the same sequence,
    and signed zeros are planted, so that the (score, index) order is exercised.
    """
    g = _cpu_gen(seed)
    total = sum(int(n) for n in lengths)
    s = torch.randn(total, generator=g, dtype=torch.float32) * 8.0
    offs = identity_offsets(lengths)
    if ties > 0 and total > 1:
        nt = int(total * ties)
        for _ in range(nt):
            seq = int(torch.randint(0, len(lengths), (1,), generator=g))
            a, b = int(offs[seq]), int(offs[seq + 1])
            if b - a < 2:
                continue
            i = a + int(torch.randint(0, b - a, (1,), generator=g))
            j = a + int(torch.randint(0, b - a, (1,), generator=g))
            s[i] = s[j]
        z = torch.randint(0, total, (max(2, total // 50),), generator=g)
        s[z[::2]] = 0.0
        s[z[1::2]] = -0.0
    return s.to(device), offs.to(device)
