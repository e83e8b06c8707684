"""CPU oracle for the high-speed-swap low-rank block predictor.

TEST INFRASTRUCTURE ONLY.  The oracle is the plain fp64 statement of what the
predictor computes (page "metrale_storage/predictor.rs": `Predictor::project_q`,
`Predictor::project_kv_block`, `Predictor::score_blocks`; victim order from
"metrale_model_layers/layers/qsa_select.rs", host top-k).  It shares no code
with the CUDA library and never imports it.  Only the tests, the smoke check
and the benchmark's CPU-baseline leg may use it.

The arithmetic lives in ``hss_oracle.c`` (plain loops, fp64).  This module
builds it with gcc and marshals numpy arrays into it.  bf16 tensors travel as
``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hss_oracle.c")
_LIB = os.path.join(_HERE, "libhss_oracle.so")
_lock = threading.Lock()
_lib = None

_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64
_int = ctypes.c_int


def build(force: bool = False, src: str | None = None, out: str | None = None) -> str:
    """Compile the oracle into a shared library with gcc; return its path."""
    src = src or _SRC
    out = out or _LIB
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-o", tmp, src, "-lm",
           "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.orc_bf16_from_double.restype = ctypes.c_uint16
    lib.orc_bf16_from_double.argtypes = [ctypes.c_double]
    lib.orc_bf16_to_double.restype = ctypes.c_double
    lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_from_double_n.restype = None
    lib.orc_bf16_from_double_n.argtypes = [_f64p, _i64, _u16p]
    lib.orc_bf16_to_double_n.restype = None
    lib.orc_bf16_to_double_n.argtypes = [_u16p, _i64, _f64p]
    lib.orc_project_q.restype = None
    lib.orc_project_q.argtypes = [_u16p, _i64, _int, _u16p, _int, _u16p, _int]
    lib.orc_project_kv_blocks.restype = _i64
    lib.orc_project_kv_blocks.argtypes = [_u16p, _u16p, _i64, _i32p, _i64, _i64, _i64, _int,
                                          _int, _int, _int, _u16p, _int]
    lib.orc_write_kv_tokens.restype = _i64
    lib.orc_write_kv_tokens.argtypes = [_u16p, _u16p, _i64p, _i64, _i64, _i64, _int, _int, _int,
                                        _int, _i64, ctypes.c_void_p, _u16p, _int]
    lib.orc_score_rows.restype = _i64
    lib.orc_score_rows.argtypes = [_u16p, _i64, _int, _int, _int, _int, _u16p, _i64, _i64, _i32p,
                                   _i64, _f64p, _f64p, _int]
    lib.orc_select_rows.restype = _int
    lib.orc_select_rows.argtypes = [_f32p, _i64, _i64, _i64, _i64, _int, _int, _i32p]
    lib.orc_score_blocks.restype = _i64
    lib.orc_score_blocks.argtypes = [_u16p, _i64, _int, _int, _int, _int, _int, _u16p, _i64,
                                     _i64, _i32p, _i64p, _f64p, _f64p, _int]
    lib.orc_score_entries.restype = _i64
    lib.orc_score_entries.argtypes = [_u16p, _i64, _int, _int, _int, _int, _int, _u16p, _i64,
                                      _i64, _i32p, _i64p, _i64p, _i64, _f64p, _f64p]
    lib.orc_score_blocks_masked.restype = _i64
    lib.orc_score_blocks_masked.argtypes = [_u16p, _i64, _int, _int, _int, _int, _int, _u16p,
                                            _i64, _i64, _i32p, _i64p, ctypes.c_void_p,
                                            ctypes.c_void_p, _f64p, _f64p, _int]
    lib.orc_rank_victims.restype = _int
    lib.orc_rank_victims.argtypes = [_f32p, _i64p, _i64, _int, _i32p]
    return lib


def lib():
    """The loaded oracle library (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def load_from(path: str):
    """Bind an oracle library at an explicit path (used to test mutated copies)."""
    return _bind(path)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else
               (os.cpu_count() or 1))


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns as uint16, got {a.dtype}")
    return a


# --------------------------------------------------------------------------- bf16


def bf16_from_double(x, L=None) -> np.ndarray:
    """Round each double to the nearest bf16 (ties to even); return the bit patterns."""
    L = L or lib()
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, dtype=np.uint16)
    L.orc_bf16_from_double_n(x.reshape(-1), x.size, out.reshape(-1))
    return out


def bf16_to_double(b, L=None) -> np.ndarray:
    L = L or lib()
    b = _u16(b)
    out = np.empty(b.shape, dtype=np.float64)
    L.orc_bf16_to_double_n(b.reshape(-1), b.size, out.reshape(-1))
    return out


# --------------------------------------------------------------------------- method


def project_q(Q: np.ndarray, P: np.ndarray, nthreads: int = 1, L=None) -> np.ndarray:
    """Qp = bf16(Q . P) for Q [..., head_dim] and P [head_dim, r]; returns [..., r]."""
    L = L or lib()
    Q = _u16(Q)
    P = _u16(P)
    hd, r = P.shape
    if Q.shape[-1] != hd:
        raise ValueError("Q's last dimension must equal head_dim")
    nv = Q.size // hd
    out = np.empty(Q.shape[:-1] + (r,), dtype=np.uint16)
    L.orc_project_q(Q.reshape(-1), nv, hd, P.reshape(-1), r, out.reshape(-1), nthreads)
    return out


def project_kv_blocks(P: np.ndarray, K: np.ndarray, layer: int, block_ids: np.ndarray,
                      A_g: np.ndarray, nthreads: int = 1, L=None) -> int:
    """Write bf16(K . P) of each block into its A_g slot, in place.

    K is [n, block_size, num_kv_heads, head_dim]; A_g is
    [num_layers, max_blocks, num_kv_heads, block_size, r].  Returns the oracle's
    status (0 ok, -1 bad layer, i+1 = first bad block id at position i).
    """
    L = L or lib()
    P = _u16(P)
    K = _u16(K)
    if not A_g.flags.c_contiguous or A_g.dtype != np.uint16:
        raise TypeError("A_g must be a C-contiguous uint16 array")
    ids = np.ascontiguousarray(block_ids, dtype=np.int32)
    nl, mb, nkv, bs, r = A_g.shape
    n, kbs, knkv, hd = K.shape
    if (kbs, knkv) != (bs, nkv) or P.shape != (hd, r) or ids.shape != (n,):
        raise ValueError("inconsistent shapes")
    return int(L.orc_project_kv_blocks(P.reshape(-1), K.reshape(-1), layer, ids, n, nl, mb, nkv,
                                       bs, hd, r, A_g.reshape(-1), nthreads))


def write_kv_tokens(P: np.ndarray, K_tok: np.ndarray, slots: np.ndarray, layer: int,
                    A_g: np.ndarray, K_cache=None, nthreads: int = 1, L=None) -> int:
    """Token-granular ingest: copy each new token's keys into the paged cache (if given) and
    write bf16(K . P) into its A_g row, both in place.

    K_tok is [n, num_kv_heads, head_dim]; slots [n] int64 (block * block_size + position,
    negative = padding); K_cache [max_blocks, block_size, num_kv_heads, head_dim] or None;
    A_g as in project_kv_blocks.  Returns 0, -1 (bad layer) or i+1 (first slot past the end).
    """
    L = L or lib()
    P = _u16(P)
    K = _u16(K_tok)
    for a in (A_g,) + ((K_cache,) if K_cache is not None else ()):
        if not a.flags.c_contiguous or a.dtype != np.uint16:
            raise TypeError("A_g and K_cache must be C-contiguous uint16 arrays")
    sl = np.ascontiguousarray(slots, dtype=np.int64)
    nl, mb, nkv, bs, r = A_g.shape
    n, knkv, hd = K.shape
    if knkv != nkv or P.shape != (hd, r) or sl.shape != (n,):
        raise ValueError("inconsistent shapes")
    if K_cache is not None and K_cache.shape != (mb, bs, nkv, hd):
        raise ValueError("K_cache shape")
    cache_ptr = None if K_cache is None else K_cache.ctypes.data_as(ctypes.c_void_p)
    return int(L.orc_write_kv_tokens(P.reshape(-1), K.reshape(-1), sl, n, nl, mb, nkv, bs, hd, r,
                                     layer, cache_ptr, A_g.reshape(-1), nthreads))


def score_rows(Qp: np.ndarray, A_g: np.ndarray, layer: int, table: np.ndarray,
               nthreads: int = 1, L=None):
    """Per-row block scores of one sequence's chunk, in fp64.

    Qp is [rows, num_q_heads, r]; table [n] physical ids.  Returns (score [rows, n] f64,
    tsum [rows, n] f64, bad_entries).
    """
    L = L or lib()
    Qp = _u16(Qp)
    if not A_g.flags.c_contiguous or A_g.dtype != np.uint16:
        raise TypeError("A_g must be a C-contiguous uint16 array")
    rows, nq, r = Qp.shape
    nl, mb, nkv, bs, ar = A_g.shape
    if ar != r:
        raise ValueError("inconsistent shapes")
    t = np.ascontiguousarray(table, dtype=np.int32)
    n = t.size
    score = np.empty((rows, n), dtype=np.float64)
    tsum = np.empty((rows, n), dtype=np.float64)
    bad = L.orc_score_rows(Qp.reshape(-1), rows, nq, nkv, r, bs, A_g.reshape(-1), layer, mb, t, n,
                           score.reshape(-1), tsum.reshape(-1), nthreads)
    return score, tsum, int(bad)


def select_rows(scores: np.ndarray, n: int, first_pos: int, block_size: int, topk: int,
                L=None) -> np.ndarray:
    """Per-row top-k (larger score first, lower index on ties) over the blocks each row has
    seen whole.  scores is [rows, stride] f32 with stride >= n; returns [rows, topk] int32."""
    L = L or lib()
    sc = np.ascontiguousarray(scores, dtype=np.float32)
    rows, stride = sc.shape
    if stride < n:
        raise ValueError("stride < n")
    out = np.empty((rows, topk), dtype=np.int32)
    if L.orc_select_rows(sc.reshape(-1), rows, n, stride, first_pos, block_size, topk,
                         out.reshape(-1)) != 0:
        raise MemoryError("oracle allocation failed")
    return out


def score_blocks(Qp: np.ndarray, A_g: np.ndarray, layer: int, block_table: np.ndarray,
                 seq_offsets: np.ndarray, nthreads: int = 1, L=None):
    """Block scores in fp64 and their tolerance scale.

    Qp is [num_seqs, rows_per_seq, num_q_heads, r]; A_g as in project_kv_blocks;
    block_table holds physical ids in CSR order, seq_offsets has num_seqs + 1
    entries.  Returns (score [total] f64, tsum [total] f64, bad_entries).
    """
    L = L or lib()
    Qp = _u16(Qp)
    S, R, nq, r = Qp.shape
    nl, mb, nkv, bs, r2 = A_g.shape
    if r2 != r:
        raise ValueError("r mismatch")
    table = np.ascontiguousarray(block_table, dtype=np.int32)
    offs = np.ascontiguousarray(seq_offsets, dtype=np.int64)
    total = int(offs[-1])
    score = np.empty(total, dtype=np.float64)
    tsum = np.empty(total, dtype=np.float64)
    bad = L.orc_score_blocks(Qp.reshape(-1), S, R, nq, nkv, r, bs, _u16(A_g).reshape(-1), layer,
                             mb, table, offs, score, tsum, nthreads)
    return score, tsum, int(bad)


def score_entries(Qp: np.ndarray, A_g: np.ndarray, layer: int, block_table: np.ndarray,
                  seq_offsets: np.ndarray, entries: np.ndarray, L=None):
    """Like score_blocks, for the listed table entries only."""
    L = L or lib()
    Qp = _u16(Qp)
    S, R, nq, r = Qp.shape
    nl, mb, nkv, bs, r2 = A_g.shape
    table = np.ascontiguousarray(block_table, dtype=np.int32)
    offs = np.ascontiguousarray(seq_offsets, dtype=np.int64)
    ent = np.ascontiguousarray(entries, dtype=np.int64)
    score = np.empty(ent.size, dtype=np.float64)
    tsum = np.empty(ent.size, dtype=np.float64)
    bad = L.orc_score_entries(Qp.reshape(-1), S, R, nq, nkv, r, bs, _u16(A_g).reshape(-1), layer,
                              mb, table, offs, ent, ent.size, score, tsum)
    return score, tsum, int(bad)


def score_blocks_masked(Qp: np.ndarray, A_g: np.ndarray, layer: int, block_table: np.ndarray,
                        seq_offsets: np.ndarray, ctx_len=None, row_pos0=None, nthreads: int = 1,
                        L=None):
    """score_blocks restricted to visible candidates.

    Token t of table position j (within its sequence) sits at p = j * block_size + t.
    ctx_len[s] (optional): only tokens with p < ctx_len[s] count.  row_pos0[s] (optional,
    causal): query row `row` sees tokens with p <= row_pos0[s] + row.  A block with no
    visible candidate scores -inf.
    """
    L = L or lib()
    Qp = _u16(Qp)
    S, R, nq, r = Qp.shape
    nl, mb, nkv, bs, r2 = A_g.shape
    table = np.ascontiguousarray(block_table, dtype=np.int32)
    offs = np.ascontiguousarray(seq_offsets, dtype=np.int64)
    cl = None if ctx_len is None else np.ascontiguousarray(ctx_len, dtype=np.int64)
    rp = None if row_pos0 is None else np.ascontiguousarray(row_pos0, dtype=np.int64)
    total = int(offs[-1])
    score = np.empty(total, dtype=np.float64)
    tsum = np.empty(total, dtype=np.float64)
    bad = L.orc_score_blocks_masked(Qp.reshape(-1), S, R, nq, nkv, r, bs, _u16(A_g).reshape(-1),
                                    layer, mb, table, offs,
                                    None if cl is None else cl.ctypes.data,
                                    None if rp is None else rp.ctypes.data, score, tsum, nthreads)
    return score, tsum, int(bad)


def rank_victims(scores: np.ndarray, seq_offsets: np.ndarray, k: int, L=None) -> np.ndarray:
    """Per sequence, the k entries with the smallest (score, index), ascending; -1 pad."""
    L = L or lib()
    sc = np.ascontiguousarray(scores, dtype=np.float32)
    offs = np.ascontiguousarray(seq_offsets, dtype=np.int64)
    S = offs.size - 1
    out = np.empty((S, k), dtype=np.int32)
    if L.orc_rank_victims(sc, offs, S, k, out.reshape(-1)) != 0:
        raise MemoryError("oracle rank_victims ran out of memory")
    return out


def score_tolerance(tsum: np.ndarray) -> np.ndarray:
    """Allowed |GPU - oracle| per block score: 2e-3 * sum|terms| + 1e-6."""
    return 2e-3 * np.asarray(tsum, dtype=np.float64) + 1e-6
