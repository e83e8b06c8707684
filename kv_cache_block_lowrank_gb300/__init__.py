"""GB300 (sm_103a) low-rank KV-block predictor: Python binding of libhss.so.

The predictor ("high-speed swap" block predictor; page "metrale_storage/predictor.rs")
projects query rows and key tokens through a fixed P [head_dim, r], keeps the projected
keys of every paged KV block in A_g [num_layers, max_blocks, num_kv_heads, block_size, r]
(bf16), scores each block as the max over query heads, query rows and tokens of Qp . A_g,
and ranks eviction victims by ascending score.

Every step runs in the CUDA kernels of libhss.so (include/hss.h).  This module only
marshals arguments: torch tensors become device pointers, the current torch stream becomes
the cudaStream_t, and a non-zero status becomes an HssError.  There is no CPU fallback: if
the library is missing, importing a compute function raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libhss.so")

HSS_OK = 0
HSS_ERR_INVALID_DIMS = 1
HSS_ERR_OUT_OF_RANGE = 2
HSS_ERR_NULL_POINTER = 3
HSS_ERR_MISALIGNED = 4
HSS_ERR_WORKSPACE_TOO_SMALL = 5
HSS_ERR_UNSUPPORTED_SHAPE = 6
HSS_ERR_CUDA = 7
HSS_ERR_DEVICE_TIMEOUT = 8
HSS_ERR_INVALID_ARGUMENT = 9

HSS_PATH_AUTO = 0
HSS_PATH_DECODE = 1
HSS_PATH_TCGEN05 = 2
HSS_MAX_VICTIMS = 8192

EXPORTED = (
    "hss_status_string", "hss_version", "hss_validate_dims", "hss_a_g_bytes", "hss_project_q",
    "hss_project_kv_blocks", "hss_score_blocks", "hss_rank_victims", "hss_read_device_error",
    "hss_layer_step", "hss_layer_step_workspace_bytes", "hss_layer_step_static",
    "hss_score_blocks_masked",
    "hss_layer_step_static_max_seqs", "hss_write_kv_tokens", "hss_score_rows",
    "hss_select_rows", "hss_self_test_wait_timeout", "hss_self_test_spread_wait",
    "hss_layer_step_bound",
)


class hss_dims(ctypes.Structure):
    """The seven predictor dimensions (PredictorDims on the predictor page)."""

    _fields_ = [
        ("num_layers", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("r", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("max_blocks", ctypes.c_int64),
    ]

    @classmethod
    def of(cls, d) -> "hss_dims":
        """From any object with the seven attributes (or an hss_dims)."""
        if isinstance(d, cls):
            return d
        return cls(int(d.num_layers), int(d.num_q_heads), int(d.num_kv_heads), int(d.head_dim),
                   int(d.r), int(d.block_size), int(d.max_blocks))


class HssError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib: Optional[ctypes.CDLL] = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libhss.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    dp = ctypes.POINTER(hss_dims)
    lib.hss_status_string.restype = ctypes.c_char_p
    lib.hss_status_string.argtypes = [i32]
    lib.hss_version.restype = i32
    lib.hss_version.argtypes = []
    lib.hss_validate_dims.restype = i32
    lib.hss_validate_dims.argtypes = [dp]
    lib.hss_a_g_bytes.restype = sz
    lib.hss_a_g_bytes.argtypes = [dp]
    lib.hss_project_q.restype = i32
    lib.hss_project_q.argtypes = [dp, vp, vp, i64, vp, vp]
    lib.hss_project_kv_blocks.restype = i32
    lib.hss_project_kv_blocks.argtypes = [dp, vp, vp, i32, vp, i64, vp, vp, vp]
    lib.hss_write_kv_tokens.restype = i32
    lib.hss_write_kv_tokens.argtypes = [dp, vp, vp, vp, i64, vp, vp, i32, vp, vp]
    lib.hss_score_rows.restype = i32
    lib.hss_score_rows.argtypes = [dp, vp, i32, vp, i32, vp, i64, vp, vp, vp]
    lib.hss_select_rows.restype = i32
    lib.hss_select_rows.argtypes = [vp, i32, i64, i64, i32, i32, vp, vp]
    lib.hss_score_blocks.restype = i32
    lib.hss_score_blocks.argtypes = [dp, vp, i32, vp, i32, vp, vp, i32, i64, vp, i32, vp, vp]
    lib.hss_score_blocks_masked.restype = i32
    lib.hss_score_blocks_masked.argtypes = [dp, vp, i32, vp, i32, vp, vp, i32, i64, vp, vp, vp,
                                            i32, vp, vp]
    lib.hss_self_test_wait_timeout.restype = i32
    lib.hss_self_test_wait_timeout.argtypes = [vp, i64, vp]
    lib.hss_self_test_spread_wait.restype = i32
    lib.hss_self_test_spread_wait.argtypes = [dp, vp, vp, vp, i32, vp, vp, i64, vp, i32, vp, vp,
                                              sz, i64, vp, vp]
    lib.hss_rank_victims.restype = i32
    lib.hss_rank_victims.argtypes = [vp, vp, i32, i64, i32, vp, vp]
    lib.hss_read_device_error.restype = i32
    lib.hss_read_device_error.argtypes = [ctypes.POINTER(i32), vp]
    lib.hss_layer_step_workspace_bytes.restype = sz
    lib.hss_layer_step_workspace_bytes.argtypes = [i32]
    lib.hss_layer_step_static_max_seqs.restype = i32
    lib.hss_layer_step_static_max_seqs.argtypes = []
    lib.hss_layer_step_static.restype = i32
    lib.hss_layer_step_static.argtypes = [dp, vp, vp, vp, i64, vp, i32, vp, vp, i32, vp, vp, i32,
                                          i64, vp, i32, vp, vp, vp]
    lib.hss_layer_step.restype = i32
    lib.hss_layer_step.argtypes = [dp, vp, vp, vp, i64, vp, i32, vp, vp, i32, vp, vp, i32, i64,
                                   vp, i32, vp, vp, sz, vp, vp]
    lib.hss_layer_step_bound.restype = i32
    lib.hss_layer_step_bound.argtypes = [ctypes.POINTER(hss_layer_step_args), i32, vp, vp, vp,
                                         vp, vp]
    _lib = lib
    return lib


# ----------------------------------------------------------------------------- marshalling

def _ptr(x) -> Optional[int]:
    """Device pointer of a tensor (or an int address, or None for NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        # The raw handle of the current stream: the same value as
        # torch.cuda.current_stream().cuda_stream without building a Stream object.
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return raw(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str) -> None:
    if status != HSS_OK:
        raise HssError(status, what)


def status_string(status: int) -> str:
    return load().hss_status_string(status).decode()


def hss_version() -> int:
    return load().hss_version()


def hss_validate_dims(dims) -> int:
    """Status of the dims (HSS_OK when valid and supported); never raises."""
    return load().hss_validate_dims(ctypes.byref(hss_dims.of(dims)))


def hss_a_g_bytes(dims) -> int:
    return load().hss_a_g_bytes(ctypes.byref(hss_dims.of(dims)))


def hss_project_q(dims, P, Q, num_rows: int, Qp, stream=None) -> None:
    """Qp [num_rows, num_q_heads, r] = bf16(Q [num_rows, num_q_heads, head_dim] . P)."""
    st = load().hss_project_q(ctypes.byref(hss_dims.of(dims)), _ptr(P), _ptr(Q), int(num_rows),
                              _ptr(Qp), _stream(stream))
    _check(st, "hss_project_q")


def hss_project_kv_blocks(dims, P, K, layer: int, block_ids, num_blocks: int, A_g,
                          dev_status=None, stream=None) -> None:
    """A_g[layer][block_ids[i]] = bf16(K[i] . P), head-major slots."""
    st = load().hss_project_kv_blocks(ctypes.byref(hss_dims.of(dims)), _ptr(P), _ptr(K),
                                      int(layer), _ptr(block_ids), int(num_blocks), _ptr(A_g),
                                      _ptr(dev_status), _stream(stream))
    _check(st, "hss_project_kv_blocks")


def hss_write_kv_tokens(dims, P, K_tok, slots, num_tokens: int, K_cache, A_g, layer: int,
                        dev_status=None, stream=None) -> None:
    """K_cache[slot] = K_tok[i] and A_g[layer][slot's block][h][slot's position] =
    bf16(K_tok[i][h] . P) for every new token i (K_cache may be None)."""
    st = load().hss_write_kv_tokens(ctypes.byref(hss_dims.of(dims)), _ptr(P), _ptr(K_tok),
                                    _ptr(slots), int(num_tokens), _ptr(K_cache), _ptr(A_g),
                                    int(layer), _ptr(dev_status), _stream(stream))
    _check(st, "hss_write_kv_tokens")


def hss_score_rows(dims, Qp, rows: int, A_g, layer: int, block_table, num_blocks: int, scores,
                   dev_status=None, stream=None) -> None:
    """scores[row, j] = max over heads and tokens of block_table[j] of Qp[row] . A_g."""
    st = load().hss_score_rows(ctypes.byref(hss_dims.of(dims)), _ptr(Qp), int(rows), _ptr(A_g),
                               int(layer), _ptr(block_table), int(num_blocks), _ptr(scores),
                               _ptr(dev_status), _stream(stream))
    _check(st, "hss_score_rows")


def hss_select_rows(scores, rows: int, num_blocks: int, first_pos: int, block_size: int,
                    topk: int, lists, stream=None) -> None:
    """lists[r] = the topk blocks row r has seen whole, largest score first."""
    st = load().hss_select_rows(_ptr(scores), int(rows), int(num_blocks), int(first_pos),
                                int(block_size), int(topk), _ptr(lists), _stream(stream))
    _check(st, "hss_select_rows")


def hss_score_blocks(dims, Qp, rows_per_seq: int, A_g, layer: int, block_table, seq_offsets,
                     num_seqs: int, total_blocks: int, scores, path: int = HSS_PATH_AUTO,
                     dev_status=None, stream=None) -> None:
    """scores[i] = max over rows, heads and tokens of Qp . A_g[layer][block_table[i]]."""
    st = load().hss_score_blocks(ctypes.byref(hss_dims.of(dims)), _ptr(Qp), int(rows_per_seq),
                                 _ptr(A_g), int(layer), _ptr(block_table), _ptr(seq_offsets),
                                 int(num_seqs), int(total_blocks), _ptr(scores), int(path),
                                 _ptr(dev_status), _stream(stream))
    _check(st, "hss_score_blocks")


def hss_score_blocks_masked(dims, Qp, rows_per_seq: int, A_g, layer: int, block_table,
                            seq_offsets, num_seqs: int, total_blocks: int, ctx_len, row_pos0,
                            scores, path: int = HSS_PATH_AUTO, dev_status=None,
                            stream=None) -> None:
    """hss_score_blocks over visible tokens only (length mask ctx_len, causal row_pos0)."""
    st = load().hss_score_blocks_masked(ctypes.byref(hss_dims.of(dims)), _ptr(Qp),
                                        int(rows_per_seq), _ptr(A_g), int(layer),
                                        _ptr(block_table), _ptr(seq_offsets), int(num_seqs),
                                        int(total_blocks), _ptr(ctx_len), _ptr(row_pos0),
                                        _ptr(scores), int(path), _ptr(dev_status),
                                        _stream(stream))
    _check(st, "hss_score_blocks_masked")


def hss_rank_victims(scores, seq_offsets, num_seqs: int, total_blocks: int, k: int, victims,
                     stream=None) -> None:
    """victims[s, :] = the min(k, n_s) smallest (score, index) entries of sequence s; -1 pad."""
    st = load().hss_rank_victims(_ptr(scores), _ptr(seq_offsets), int(num_seqs),
                                 int(total_blocks), int(k), _ptr(victims), _stream(stream))
    _check(st, "hss_rank_victims")


def hss_layer_step_workspace_bytes(num_seqs: int) -> int:
    return load().hss_layer_step_workspace_bytes(int(num_seqs))


def hss_layer_step(dims, P, K_new, new_ids, num_new: int, Q, rows_per_seq: int, Qp, A_g,
                   layer: int, block_table, seq_offsets, num_seqs: int, total_blocks: int,
                   scores, k: int, victims, workspace, workspace_bytes: int, dev_status=None,
                   stream=None) -> None:
    """One layer call: project new blocks and queries, score, rank (fused where possible)."""
    st = load().hss_layer_step(ctypes.byref(hss_dims.of(dims)), _ptr(P), _ptr(K_new),
                               _ptr(new_ids), int(num_new), _ptr(Q), int(rows_per_seq), _ptr(Qp),
                               _ptr(A_g), int(layer), _ptr(block_table), _ptr(seq_offsets),
                               int(num_seqs), int(total_blocks), _ptr(scores), int(k),
                               _ptr(victims), _ptr(workspace), int(workspace_bytes),
                               _ptr(dev_status), _stream(stream))
    _check(st, "hss_layer_step")


class hss_layer_step_args(ctypes.Structure):
    """The bound arguments of hss_layer_step_bound (hss_layer_step_args in hss.h)."""

    _fields_ = [
        ("dims", hss_dims),
        ("P", ctypes.c_void_p),
        ("new_ids", ctypes.c_void_p),
        ("num_new", ctypes.c_int64),
        ("rows_per_seq", ctypes.c_int32),
        ("Qp", ctypes.c_void_p),
        ("A_g", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("seq_offsets", ctypes.c_void_p),
        ("num_seqs", ctypes.c_int32),
        ("total_blocks", ctypes.c_int64),
        ("k", ctypes.c_int32),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("dev_status", ctypes.c_void_p),
    ]


class LayerStep:
    """hss_layer_step with the arguments that stay the same from call to call bound once.

    A serving loop makes one layer call per layer and step with the same dims, P, A_g,
    block table, offsets, workspace and sizes; they are bound once in an
    hss_layer_step_args struct and each call passes only the per-call ones (layer, the new
    key blocks, the queries, the score and victim buffers, the stream) to
    hss_layer_step_bound, which is exactly hss_layer_step.  Tensors or integer device
    addresses are accepted for those.
    """

    def __init__(self, dims, P, new_ids, num_new: int, rows_per_seq: int, Qp, A_g,
                 block_table, seq_offsets, num_seqs: int, total_blocks: int, k: int,
                 workspace, workspace_bytes: int, dev_status=None):
        self._fn = load().hss_layer_step_bound
        self._args = hss_layer_step_args(
            hss_dims.of(dims), _ptr(P), _ptr(new_ids), int(num_new), int(rows_per_seq),
            _ptr(Qp), _ptr(A_g), _ptr(block_table), _ptr(seq_offsets), int(num_seqs),
            int(total_blocks), int(k), _ptr(workspace), int(workspace_bytes), _ptr(dev_status))
        self._ref = ctypes.byref(self._args)  # kept alive with the struct

    def __call__(self, layer: int, K_new, Q, scores, victims, stream=None) -> None:
        st = self._fn(self._ref, int(layer), _ptr(K_new), _ptr(Q), _ptr(scores), _ptr(victims),
                      _stream(stream))
        _check(st, "hss_layer_step_bound")


def hss_layer_step_static_max_seqs() -> int:
    return load().hss_layer_step_static_max_seqs()


def hss_layer_step_static(dims, P, K_new, new_ids, num_new: int, Q, rows_per_seq: int, Qp, A_g,
                          layer: int, block_table, seq_offsets, num_seqs: int, total_blocks: int,
                          scores, k: int, victims, dev_status=None, stream=None) -> None:
    """hss_layer_step without a workspace, for callers that cannot allocate device memory.

    The completion counters live in a fixed array inside the library (at most
    hss_layer_step_static_max_seqs() sequences per call).  Calls share that array, so they
    must not overlap on the GPU.  The first call on a device must come before any stream
    capture on it.
    """
    st = load().hss_layer_step_static(ctypes.byref(hss_dims.of(dims)), _ptr(P), _ptr(K_new),
                                      _ptr(new_ids), int(num_new), _ptr(Q), int(rows_per_seq),
                                      _ptr(Qp), _ptr(A_g), int(layer), _ptr(block_table),
                                      _ptr(seq_offsets), int(num_seqs), int(total_blocks),
                                      _ptr(scores), int(k), _ptr(victims), _ptr(dev_status),
                                      _stream(stream))
    _check(st, "hss_layer_step_static")


def hss_self_test_wait_timeout(dev_status, limit_ns: int, stream=None) -> None:
    """Launch a kernel whose bounded pipeline wait runs out (it sets dev_status)."""
    st = load().hss_self_test_wait_timeout(_ptr(dev_status), int(limit_ns), _stream(stream))
    _check(st, "hss_self_test_wait_timeout")


def hss_self_test_spread_wait(dims, P, Q, A_g, layer: int, block_table, seq_offsets,
                              total_blocks: int, scores, k: int, victims, workspace,
                              workspace_bytes: int, limit_ns: int, dev_status=None,
                              stream=None) -> None:
    """Run the layer call's one-sequence ranking with one CTA withholding its keys, so that
    the other CTAs' bounded waits run out after limit_ns (they set dev_status)."""
    st = load().hss_self_test_spread_wait(ctypes.byref(hss_dims.of(dims)), _ptr(P), _ptr(Q),
                                          _ptr(A_g), int(layer), _ptr(block_table),
                                          _ptr(seq_offsets), int(total_blocks), _ptr(scores),
                                          int(k), _ptr(victims), _ptr(workspace),
                                          int(workspace_bytes), int(limit_ns), _ptr(dev_status),
                                          _stream(stream))
    _check(st, "hss_self_test_spread_wait")


def hss_read_device_error(stream=None) -> int:
    """Synchronise the stream; return and clear the library's device error word."""
    out = ctypes.c_int32(0)
    st = load().hss_read_device_error(ctypes.byref(out), _stream(stream))
    _check(st, "hss_read_device_error")
    return out.value


# ----------------------------------------------------------------------------- host helpers

def check_a_g_budget(dims, free_bytes: int, margin: float = 0.05) -> int:
    """Refuse an A_g that would not fit in (1 - margin) of the free HBM.

    Mirrors the budget check of Predictor::new (predictor page): the error names the
    settings that shrink A_g.  Returns the A_g size in bytes when it fits.
    """
    d = hss_dims.of(dims)
    need = (d.num_layers * d.max_blocks * d.num_kv_heads * d.block_size * d.r * 2)
    budget = int(free_bytes * (1.0 - margin))
    if need > budget:
        raise MemoryError(
            f"A_g would need {need / 2**30:.2f} GiB but only {budget / 2**30:.2f} GiB of HBM "
            f"may be used ({margin:.0%} of the free memory is left for other buffers). "
            f"Shrink one of: r (now {d.r}; r/2 halves A_g), max_blocks (now {d.max_blocks}; "
            f"set by the longest context), num_layers kept ({d.num_layers}). "
            f"A_g = num_layers x max_blocks x num_kv_heads x block_size x r x 2 bytes.")
    return need
