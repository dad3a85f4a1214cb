"""The C-ABI library on the host: it loads, exports every declared symbol, and
rejects bad arguments before touching CUDA (no GPU needed)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def sef():
    from sparse_expert_ffn_gb300 import build
    build.build()
    import sparse_expert_ffn_gb300
    return sparse_expert_ffn_gb300


def _declared_functions():
    names = []
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            src = open(os.path.join(HEADER_DIR, fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[\w]+\**\s+\**(colibri_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("colibri_init", "colibri_forward", "colibri_forward_host", "colibri_free",
              "colibri_forward_host_async", "colibri_host_wait",
              "colibri_get_routing", "colibri_forward_stack_layer", "colibri_status_str",
              "colibri_check", "colibri_init_int8", "colibri_quantize_int8_block64"):
        assert n in names


def test_library_exports_every_declared_symbol(sef):
    lib = ctypes.CDLL(sef.LIB_PATH)
    for n in _declared_functions():
        assert hasattr(lib, n), n
        assert getattr(sef, n) is not None


def test_status_strings(sef):
    for s in range(6):
        assert sef.colibri_status_str(s)
    assert sef.colibri_status_str(99) == "unknown status"


def _cfg(sef, **kw):
    base = dict(n_experts=8, top_k=2, d_model=128, d_ff=256, max_tokens=16,
                dtype=sef.DTYPE_FP32, device=0, executor=sef.EXEC_AUTO)
    base.update(kw)
    return sef.ColibriConfig(**base)


@pytest.mark.parametrize("kw,expect", [
    (dict(n_experts=0), 1), (dict(top_k=0), 1), (dict(top_k=9, n_experts=8), 1),
    (dict(d_model=-64), 1), (dict(max_tokens=0), 1), (dict(dtype=7), 1), (dict(executor=5), 1),
    (dict(device=-1), 1),
    (dict(n_experts=300), 4), (dict(top_k=9, n_experts=16), 4), (dict(d_model=96), 4),
    (dict(d_ff=200), 4), (dict(executor=2, dtype=0), 4),
])
def test_init_rejects_bad_config_before_cuda(sef, kw, expect):
    h = ctypes.c_void_p(123)
    buf = (ctypes.c_float * 4)()
    p = ctypes.cast(buf, ctypes.c_void_p)
    st = sef.colibri_init(ctypes.byref(_cfg(sef, **kw)), p, None, p, p, p, 0, ctypes.byref(h))
    assert st == expect
    assert h.value is None


def test_init_rejects_null_pointers(sef):
    h = ctypes.c_void_p()
    buf = (ctypes.c_float * 4)()
    p = ctypes.cast(buf, ctypes.c_void_p)
    assert sef.colibri_init(ctypes.byref(_cfg(sef)), None, None, p, p, p, 0, ctypes.byref(h)) == 1
    assert sef.colibri_init(ctypes.byref(_cfg(sef)), p, None, p, p, p, 3, ctypes.byref(h)) == 1
    assert sef.colibri_init(None, p, None, p, p, p, 0, ctypes.byref(h)) == 1
    assert sef.colibri_init(ctypes.byref(_cfg(sef)), p, None, p, p, p, 0, None) == 1


def test_calls_on_null_handle_are_invalid(sef):
    assert sef.colibri_forward(None, None, 1, None, None) == 1
    assert sef.colibri_forward_host(None, None, 1, None, None) == 1
    assert sef.colibri_forward_host_async(None, None, 1, None, None) == 1
    assert sef.colibri_host_wait(None) == 1
    assert sef.colibri_get_routing(None, None, None, None, None, None) == 1
    assert sef.colibri_set_executor(None, 0) == 1
    assert sef.colibri_check(None, None) == 1
    n = ctypes.c_uint64()
    assert sef.colibri_launch_count(None, ctypes.byref(n)) == 1
    sef.colibri_free(None)   # NULL-safe


def _aligned(buf, offset=0):
    """An address inside `buf` on a 16-byte boundary, plus `offset` bytes."""
    a = ctypes.addressof(buf)
    return ctypes.c_void_p(((a + 15) & ~15) + offset)


def test_handle_free_calls_check_arguments_before_cuda(sef):
    buf = (ctypes.c_uint8 * 4096)()
    p, odd = _aligned(buf), _aligned(buf, 8)
    F32, BF16 = sef.DTYPE_FP32, sef.DTYPE_BF16
    # gather_rows(x, x_rows, perm, k, npairs, d_model, dtype, xp, stream)
    g = sef.colibri_gather_rows
    assert g(None, 4, p, 2, 8, 64, F32, p, None) == 1
    assert g(p, -1, p, 2, 8, 64, F32, p, None) == 1
    assert g(p, 4, p, 0, 8, 64, F32, p, None) == 1
    assert g(p, 4, p, 2, -1, 64, F32, p, None) == 1
    assert g(p, 4, p, 2, 8, 64, 7, p, None) == 1
    assert g(odd, 4, p, 2, 8, 64, F32, p, None) == 1
    assert g(p, 4, p, 2, 8, 2, F32, p, None) == 1          # 8-byte rows
    assert g(p, 1 << 30, p, 4, 8, 64, F32, p, None) == 1   # x_rows * k overflows
    assert g(p, 4, p, 2, 0, 64, BF16, p, None) == 0        # nothing to gather
    # combine_rows(rows, rows_dtype, topk_w, perm, T, k, d_model, dtype, inv, y, stream)
    c = sef.colibri_combine_rows
    assert c(None, F32, p, p, 4, 2, 64, F32, p, p, None) == 1
    assert c(p, F32, p, p, 4, 2, 64, F32, None, p, None) == 1
    assert c(p, F32, p, p, -1, 2, 64, F32, p, p, None) == 1
    assert c(p, BF16, p, p, 4, 2, 64, F32, p, p, None) == 1  # bf16 rows need bf16 y
    assert c(p, F32, p, p, 4, 2, 60, F32, p, p, None) == 1   # d_model % 8
    assert c(p, F32, p, p, 4, 2, 64, F32, p, odd, None) == 1
    assert c(p, BF16, p, p, 0, 2, 64, BF16, p, p, None) == 0  # no tokens
    # forward_routed needs a handle
    assert sef.colibri_forward_routed(None, p, 4, 2, p, p, p, None) == 1
    # route_static: the configuration limits
    r = sef.colibri_route_static
    assert r(p, p, None, 4, 64, 8, 9, F32, p, p, p, p, None) == 1   # k > E
    assert r(p, p, None, 4, 64, 300, 2, F32, p, p, p, p, None) == 4
    assert r(p, p, None, 4, 96, 8, 2, F32, p, p, p, p, None) == 4   # d % 64
    assert r(p, p, None, 0, 64, 8, 2, F32, p, p, p, p, None) == 0   # T = 0
