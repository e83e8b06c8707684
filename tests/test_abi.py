"""The C ABI on the host: the library loads, exports what include/hss.h declares, and
rejects bad arguments before touching the GPU.  No call here reaches a kernel launch
(every call fails validation first), so these tests are safe on any machine."""
import ctypes
import os
import re

import pytest

import kv_cache_block_lowrank_gb300 as hss

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hss.h")


@pytest.fixture(scope="module")
def lib():
    from kv_cache_block_lowrank_gb300 import _build

    _build.build()
    return hss.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hss_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("hss_project_q", "hss_project_kv_blocks", "hss_score_blocks", "hss_rank_victims"):
        assert n in names
    assert set(names) == set(hss.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_dims_struct_layout():
    assert ctypes.sizeof(hss.hss_dims) == 32
    assert hss.hss_dims.max_blocks.offset == 24


def test_layer_step_args_struct_layout(tmp_path):
    # The binding's struct against the header's, field by field, as the C compiler lays it out.
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f for f, _ in hss.hss_layer_step_args._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "hss.h"\nint main(void) {\n'
                   '  printf("%zu\\n", sizeof(hss_layer_step_args));\n' +
                   "".join(f'  printf("%zu\\n", offsetof(hss_layer_step_args, {f}));\n'
                           for f in fields) + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [ctypes.sizeof(hss.hss_layer_step_args)] + [
        getattr(hss.hss_layer_step_args, f).offset for f in fields]
    assert got == want


def test_layer_step_bound_null_args(lib):
    st = lib.hss_layer_step_bound(None, 0, None, None, None, None, None)
    assert st == hss.HSS_ERR_NULL_POINTER


D = dict(num_layers=32, num_q_heads=32, num_kv_heads=8, head_dim=128, r=32, block_size=16,
         max_blocks=2048)


def dims(**kw):
    d = dict(D)
    d.update(kw)
    return hss.hss_dims(*[d[k] for k in ("num_layers", "num_q_heads", "num_kv_heads", "head_dim",
                                          "r", "block_size", "max_blocks")])


def test_status_strings(lib):
    assert hss.status_string(0) == "HSS_OK"
    assert hss.status_string(hss.HSS_ERR_DEVICE_TIMEOUT) == "HSS_ERR_DEVICE_TIMEOUT"
    assert hss.status_string(12345) == "HSS_ERR_UNKNOWN"
    assert hss.hss_version() >= 100


@pytest.mark.parametrize("kw,code", [
    ({}, hss.HSS_OK),
    ({"num_q_heads": 30}, hss.HSS_ERR_INVALID_DIMS),    # 30 % 8 != 0 (PredictorDims::validate)
    ({"num_kv_heads": 0}, hss.HSS_ERR_INVALID_DIMS),
    ({"r": 24}, hss.HSS_ERR_UNSUPPORTED_SHAPE),
    ({"r": 48}, hss.HSS_ERR_UNSUPPORTED_SHAPE),
    ({"r": 256}, hss.HSS_ERR_UNSUPPORTED_SHAPE),
    ({"r": 512}, hss.HSS_ERR_UNSUPPORTED_SHAPE),
    ({"block_size": 8}, hss.HSS_ERR_UNSUPPORTED_SHAPE),
    ({"head_dim": 96}, hss.HSS_ERR_UNSUPPORTED_SHAPE),
    ({"max_blocks": 2 ** 31}, hss.HSS_ERR_UNSUPPORTED_SHAPE),
    ({"num_layers": -1}, hss.HSS_ERR_INVALID_DIMS),
])
def test_validate_dims(lib, kw, code):
    assert hss.hss_validate_dims(dims(**kw)) == code


def test_a_g_bytes(lib):
    assert hss.hss_a_g_bytes(dims()) == 32 * 2048 * 8 * 16 * 32 * 2
    assert hss.hss_a_g_bytes(dims(num_layers=32, max_blocks=65536)) == 16 * 2 ** 30
    assert hss.hss_a_g_bytes(dims(num_q_heads=7)) == 0


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def status_of(fn, *args, **kw):
    with pytest.raises(hss.HssError) as e:
        fn(*args, **kw)
    return e.value.status


def test_project_q_validation(lib):
    assert status_of(hss.hss_project_q, dims(num_q_heads=9), FAKE, FAKE, 1, FAKE, 0) == \
        hss.HSS_ERR_INVALID_DIMS
    assert status_of(hss.hss_project_q, dims(), None, FAKE, 1, FAKE, 0) == hss.HSS_ERR_NULL_POINTER
    assert status_of(hss.hss_project_q, dims(), FAKE + 2, FAKE, 1, FAKE, 0) == \
        hss.HSS_ERR_MISALIGNED
    assert status_of(hss.hss_project_q, dims(), FAKE, FAKE, -1, FAKE, 0) == \
        hss.HSS_ERR_INVALID_ARGUMENT
    hss.hss_project_q(dims(), FAKE, FAKE, 0, FAKE, 0)  # zero rows: nothing to do, HSS_OK


def test_project_kv_validation(lib):
    assert status_of(hss.hss_project_kv_blocks, dims(), FAKE, FAKE, 32, FAKE, 4, FAKE, None, 0) \
        == hss.HSS_ERR_OUT_OF_RANGE                        # layer >= num_layers
    assert status_of(hss.hss_project_kv_blocks, dims(), FAKE, FAKE, -1, FAKE, 4, FAKE, None, 0) \
        == hss.HSS_ERR_OUT_OF_RANGE
    assert status_of(hss.hss_project_kv_blocks, dims(), FAKE, FAKE, 0, None, 4, FAKE, None, 0) \
        == hss.HSS_ERR_NULL_POINTER
    assert status_of(hss.hss_project_kv_blocks, dims(), FAKE, FAKE + 8, 0, FAKE, 4, FAKE, None,
                     0) == hss.HSS_ERR_MISALIGNED
    assert status_of(hss.hss_project_kv_blocks, dims(), FAKE, FAKE, 0, FAKE, -4, FAKE, None, 0) \
        == hss.HSS_ERR_INVALID_ARGUMENT


def test_score_validation(lib):
    args = lambda **o: [o.get("d", dims()), FAKE, o.get("rows", 1), FAKE, o.get("layer", 0),
                        FAKE, FAKE, o.get("S", 1), o.get("total", 10), o.get("scores", FAKE),
                        o.get("path", 0), None, 0]
    assert status_of(hss.hss_score_blocks, *args(layer=40)) == hss.HSS_ERR_OUT_OF_RANGE
    assert status_of(hss.hss_score_blocks, *args(rows=0)) == hss.HSS_ERR_INVALID_ARGUMENT
    assert status_of(hss.hss_score_blocks, *args(path=7)) == hss.HSS_ERR_INVALID_ARGUMENT
    assert status_of(hss.hss_score_blocks, *args(S=0)) == hss.HSS_ERR_INVALID_ARGUMENT
    assert status_of(hss.hss_score_blocks, *args(scores=None)) == hss.HSS_ERR_NULL_POINTER
    assert status_of(hss.hss_score_blocks, *args(d=dims(r=48))) == hss.HSS_ERR_UNSUPPORTED_SHAPE


def test_rank_validation(lib):
    assert status_of(hss.hss_rank_victims, FAKE, FAKE, 1, 10, 0, FAKE, 0) == \
        hss.HSS_ERR_INVALID_ARGUMENT
    assert status_of(hss.hss_rank_victims, FAKE, FAKE, 1, 10, hss.HSS_MAX_VICTIMS + 1, FAKE, 0) \
        == hss.HSS_ERR_INVALID_ARGUMENT
    assert status_of(hss.hss_rank_victims, FAKE, None, 1, 10, 4, FAKE, 0) == \
        hss.HSS_ERR_NULL_POINTER


def test_a_g_budget_message():
    d = dims(num_layers=32, max_blocks=65536)
    assert hss.check_a_g_budget(d, free_bytes=100 * 2 ** 30) == 16 * 2 ** 30
    with pytest.raises(MemoryError, match="r/2 halves A_g"):
        hss.check_a_g_budget(d, free_bytes=10 * 2 ** 30)


def test_missing_library_fails_loudly(tmp_path):
    import importlib

    mod = importlib.import_module("kv_cache_block_lowrank_gb300")
    with pytest.raises(RuntimeError, match="missing"):
        mod.load.__wrapped__(str(tmp_path / "nope.so")) if hasattr(mod.load, "__wrapped__") \
            else _load_fresh(mod, str(tmp_path / "nope.so"))


def _load_fresh(mod, path):
    saved = mod._lib
    mod._lib = None
    try:
        return mod.load(path)
    finally:
        mod._lib = saved


def test_layer_step_validation(lib):
    assert hss.hss_layer_step_workspace_bytes(0) == 0
    assert hss.hss_layer_step_workspace_bytes(1) == 33024 + 256
    assert hss.hss_layer_step_workspace_bytes(65) == 33024 + 512
    base = lambda **o: [o.get("d", dims()), FAKE, FAKE, FAKE, o.get("num_new", 1), FAKE, 1, FAKE,
                        FAKE, o.get("layer", 0), FAKE, FAKE, o.get("S", 1), 10, FAKE,
                        o.get("k", 4), FAKE, o.get("ws", FAKE), o.get("wsb", 65536), None, 0]
    assert status_of(hss.hss_layer_step, *base(wsb=16)) == hss.HSS_ERR_WORKSPACE_TOO_SMALL
    assert status_of(hss.hss_layer_step, *base(ws=None)) == hss.HSS_ERR_NULL_POINTER
    assert status_of(hss.hss_layer_step, *base(layer=99)) == hss.HSS_ERR_OUT_OF_RANGE
    assert status_of(hss.hss_layer_step, *base(k=0)) == hss.HSS_ERR_INVALID_ARGUMENT
    assert status_of(hss.hss_layer_step, *base(num_new=-1)) == hss.HSS_ERR_INVALID_ARGUMENT
    assert status_of(hss.hss_layer_step, *base(d=dims(num_kv_heads=3))) == \
        hss.HSS_ERR_INVALID_DIMS
    # Qp may be NULL only where the decode scorer projects the queries itself.
    qnull = lambda **o: [x if i != 7 else None for i, x in enumerate(base(**o))]
    assert status_of(hss.hss_layer_step, *qnull(S=9)) == hss.HSS_ERR_NULL_POINTER
    wide = dims(num_q_heads=64, num_kv_heads=2)  # 32 query vectors per kv head: tcgen05 path
    assert status_of(hss.hss_layer_step, *qnull(d=wide)) == hss.HSS_ERR_NULL_POINTER


def test_static_layer_step_checks_before_anything(lib):
    # The allocation-free variant runs every check of hss_layer_step before it looks up its
    # array or enqueues the clear: the same statuses come back on a machine without a GPU.
    base = lambda **o: [o.get("d", dims()), FAKE, FAKE, FAKE, o.get("num_new", 1), FAKE, 1,
                        o.get("Qp", FAKE), FAKE, o.get("layer", 0), FAKE, FAKE, o.get("S", 1), 10,
                        FAKE, o.get("k", 4), FAKE, None, 0]
    st = lambda **o: status_of(hss.hss_layer_step_static, *base(**o))
    assert st(layer=99) == hss.HSS_ERR_OUT_OF_RANGE
    assert st(k=0) == hss.HSS_ERR_INVALID_ARGUMENT
    assert st(num_new=-1) == hss.HSS_ERR_INVALID_ARGUMENT
    assert st(Qp=None) == hss.HSS_ERR_NULL_POINTER
    assert st(d=dims(num_kv_heads=3)) == hss.HSS_ERR_INVALID_DIMS
    assert st(S=hss.hss_layer_step_static_max_seqs() + 1) == hss.HSS_ERR_WORKSPACE_TOO_SMALL
    wide = dims(num_q_heads=64, num_kv_heads=2, head_dim=128, r=16, block_size=48)
    assert st(d=wide) == hss.HSS_ERR_UNSUPPORTED_SHAPE  # tcgen05 path: block size 16 or 32


def test_self_test_validation(lib):
    assert status_of(hss.hss_self_test_wait_timeout, None, 1_000_000, 0) == hss.HSS_ERR_NULL_POINTER
    assert status_of(hss.hss_self_test_wait_timeout, FAKE, 10, 0) == hss.HSS_ERR_INVALID_ARGUMENT
    assert status_of(hss.hss_self_test_wait_timeout, FAKE, 3 * 10 ** 9, 0) == \
        hss.HSS_ERR_INVALID_ARGUMENT


def test_layer_step_prepared_call_marshals_like_the_plain_call(lib):
    # The bound-arguments form reaches the same C entry point with the same arguments: each
    # validation error of the plain call comes back from it too (argument positions included).
    def both(layer=0, k=4, wsb=65536, num_new=1, ws=FAKE):
        plain = status_of(hss.hss_layer_step, dims(), FAKE, FAKE, FAKE, num_new, FAKE, 1, FAKE,
                          FAKE, layer, FAKE, FAKE, 1, 10, FAKE, k, FAKE, ws, wsb, None, 0)
        step = hss.LayerStep(dims(), FAKE, FAKE, num_new, 1, FAKE, FAKE, FAKE, FAKE, 1, 10, k,
                             ws, wsb)
        return plain, status_of(step, layer, FAKE, FAKE, FAKE, FAKE, 0)

    for kw, want in [({"layer": 99}, hss.HSS_ERR_OUT_OF_RANGE),
                     ({"k": 0}, hss.HSS_ERR_INVALID_ARGUMENT),
                     ({"num_new": -1}, hss.HSS_ERR_INVALID_ARGUMENT),
                     ({"wsb": 16}, hss.HSS_ERR_WORKSPACE_TOO_SMALL),
                     ({"ws": None}, hss.HSS_ERR_NULL_POINTER)]:
        assert both(**kw) == (want, want), kw
