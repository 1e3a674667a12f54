"""The C-ABI library loads and exports every function include/moe.h declares,
and the Python binding covers the same names (no GPU needed: nothing is
called that touches the device)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "for", "while", "sizeof")))


@pytest.fixture(scope="module")
def libmoe():
    from routed_expert_layer_router_gb300 import build, moe
    if not os.path.exists(moe.LIB_PATH):
        build()
    return ctypes.CDLL(moe.LIB_PATH)


def test_header_declares_the_calls():
    names = _declared_functions()
    for want in ("moe_route", "moe_permute", "moe_expert_ffn", "moe_combine", "expcache_lookup",
                 "expcache_fill", "moe_layer_forward", "expcache_create", "moe_layer_create"):
        assert want in names


def test_library_exports_every_declared_symbol(libmoe):
    for name in _declared_functions():
        assert hasattr(libmoe, name), name


def test_binding_covers_the_header(libmoe):
    from routed_expert_layer_router_gb300 import moe
    assert sorted(moe.SIGNATURES) == _declared_functions()
    L = moe.lib()
    assert L.moe_abi_version() == 6
    assert L.moe_record_bytes(6144, 2048, 0) == 21233664
    assert L.moe_record_bytes(6144, 2048, 1) == 20054016
    assert L.moe_record_bytes(6144, 2048, 7) == 0
    assert L.moe_status_string(6) == b"MOE_ERR_DEVICE"
    # the router weights' three bf16 pieces, expert rows padded to multiples of 32
    assert L.moe_route_split_bytes(288, 6144) == 3 * 288 * 6144 * 2
    assert L.moe_route_split_bytes(100, 512) == 3 * 128 * 512 * 2
    assert L.moe_route_split_bytes(16, 256) == 3 * 32 * 256 * 2
    assert L.moe_route_split_bytes(0, 256) == 0 and L.moe_route_split_bytes(16, 0) == 0


def test_argument_errors_return_before_touching_the_device(libmoe):
    from routed_expert_layer_router_gb300 import moe
    L = moe.lib()
    assert L.moe_route(None, None) == moe.MOE_ERR_INVALID_ARG
    a = moe.moe_route_args()
    a.x = a.w_router = a.ids = a.w = 16
    a.T, a.H, a.E, a.k = 1, 6144, 288, 300  # k > E
    assert L.moe_route(ctypes.byref(a), None) == moe.MOE_ERR_INVALID_ARG
    a.k, a.H = 8, 100  # H not a multiple of 256
    assert L.moe_route(ctypes.byref(a), None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_nvfp4_quantize(16, 0, 4, 100, 16, 16, 16, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_nvfp4_quantize(16, 1, 4, 8192, 16, 16, 16, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_nvfp4_quantize(16, 2, 4, 256, 16, 16, 16, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_nvfp4_quantize(None, 0, 4, 256, 16, 16, 16, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_permute(None, 1, 8, 2000, 16, 16, 16, 16, None, 128, None, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert L.expcache_create(None, None) == moe.MOE_ERR_INVALID_ARG
    d = moe.expcache_desc()
    d.L, d.E, d.H, d.I = 1, 16, 200, 128
    h = ctypes.c_void_p()
    assert L.expcache_create(ctypes.byref(d), ctypes.byref(h)) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_combine(None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_layer_forward(None, None, 1, None, None) == moe.MOE_ERR_INVALID_ARG
    # slot planner: floors that do not fit, a floor above E, oversized shapes
    assert L.expcache_plan_slots(16, 2, 4, 3, 2, 16, 16, None) == moe.MOE_ERR_INVALID_ARG
    assert L.expcache_plan_slots(16, 2, 4, 10, 5, 16, 16, None) == moe.MOE_ERR_INVALID_ARG
    assert L.expcache_plan_slots(None, 2, 4, 10, 1, 16, 16, None) == moe.MOE_ERR_INVALID_ARG
    assert L.expcache_plan_slots(16, 2, 2000, 10, 1, 16, 16, None) == moe.MOE_ERR_UNSUPPORTED
