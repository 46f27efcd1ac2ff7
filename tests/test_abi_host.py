"""Host-side checks of the C ABI that need no GPU: the library builds for sm_103a,
loads, exports every entry point include/moe_w4a16.h declares, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

from moe_layer_bit_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe_w4a16.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ["moe_route_topk", "moe_permute", "moe_w4a16_gate_up_swiglu", "moe_w4a16_down",
              "moe_unpermute_combine", "moe_layer_forward", "moe_layer_forward_host", "moe_workspace_bytes",
              "moe_prepack_w4", "moe_get_device_status", "moe_status_string"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), n
    assert set(_declared()) <= set(_lib.exported_symbols())


def test_status_strings(lib):
    assert _lib.status_string(0) == "MOE_OK"
    assert _lib.status_string(6) == "MOE_ERR_DEVICE_TIMEOUT"
    assert _lib.status_string(99) == "MOE_ERR_UNKNOWN"


def test_workspace_sizes(lib):
    d = _lib.dims(32, 2048, 768, 128, 8)
    full = _lib.moe_workspace_bytes(d)
    stage = _lib.moe_stage_workspace_bytes(d)
    n = 32 * 8
    assert stage > 0 and full > stage
    # x_perm + h + y_perm dominate the workspace
    assert full >= n * 2048 * 2 + n * 768 * 2 + n * 2048 * 4
    assert _lib.moe_packed_w4_bytes(128, 1536, 2048) == 128 * 1536 * 2048 * 9 // 16


@pytest.mark.parametrize("dims,code", [
    ((4, 100, 64, 8, 2), _lib.MOE_ERR_UNSUPPORTED_SHAPE),   # H % 128
    ((4, 128, 96, 8, 2), _lib.MOE_ERR_UNSUPPORTED_SHAPE),   # I % 64
    ((4, 128, 64, 8, 9), _lib.MOE_ERR_INVALID_ARG),         # k > E
    ((4, 128, 64, 64, 33), _lib.MOE_ERR_INVALID_ARG),       # k > 32
    ((4, 128, 64, 2048, 2), _lib.MOE_ERR_INVALID_ARG),      # E > 1024
    ((-1, 128, 64, 8, 2), _lib.MOE_ERR_INVALID_ARG),        # T < 0
    ((4, 128, 64, 8, 0), _lib.MOE_ERR_INVALID_ARG),         # k < 1
])
def test_bad_dims_are_rejected_before_launch(lib, dims, code):
    d = _lib.dims(*dims)
    fake = ctypes.c_void_p(0x10000)     # never dereferenced: validation fails first
    assert lib.moe_route_topk(fake, d, fake, fake, None) == code
    assert lib.moe_unpermute_combine(fake, fake, fake, d, fake, None) == code
    assert _lib.moe_workspace_bytes(d) == 0
    assert _lib.moe_layer_kernel_launches(d) == -code


@pytest.mark.parametrize("dims,launches,fused", [
    ((0, 2048, 768, 128, 8), 0, False),     # nothing to do
    ((32, 2048, 768, 128, 8), 3, True),     # routing + grouping block; both projections in one GEMM launch
    ((64, 256, 128, 1024, 4), 4, True),     # T*E too large for the fused block: routing, then grouping
    ((800, 2048, 512, 256, 8), 8, False),   # chunked grouping (4 launches), row gather, two 64-row-tile GEMMs
    ((16, 128, 64, 8, 2), 3, True),         # narrow tiles at any K
    ((2048, 256, 128, 64, 2), 8, False),    # 128-row tiles read a permuted copy: row gather kernel
])
def test_layer_kernel_launch_count(lib, dims, launches, fused):
    # host-only queries; the bench reports the launches it timed
    d = _lib.dims(*dims)
    assert _lib.moe_layer_kernel_launches(d) == launches
    assert _lib.moe_layer_projections_fused(d) == fused


def test_null_misaligned_and_small_workspace(lib):
    d = _lib.dims(4, 128, 64, 8, 2)
    ok = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    assert lib.moe_route_topk(None, d, ok, ok, None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_route_topk(odd, d, ok, ok, None) == _lib.MOE_ERR_MISALIGNED
    w = _lib.W4(0x10000, 0x10000)
    small = _lib.moe_workspace_bytes(d) - 1
    assert lib.moe_layer_forward(ok, ok, w, w, d, ok, None, None, ok, small, None) == \
        _lib.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_w4a16_gate_up_swiglu(ok, ok, _lib.W4(0, 0x10000), d, ok, ok, 1 << 20, None) == \
        _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_permute(ok, ok, d, ok, ok, ok, ok, ok, ok, 1, None) == _lib.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_prepack_w4(ok, ok, 2, 100, 64, 0, ok, None) == _lib.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_prepack_w4(ok, ok, 2, 128, 64, 7, ok, None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_get_device_status(None, None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward_host(None, ok, w, w, d, ok, ok, 1 << 30, None) == _lib.MOE_ERR_INVALID_ARG
    # router logits: weights required, bias optional but 4-byte aligned
    assert lib.moe_router_logits(ok, None, None, d, ok, None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_router_logits(ok, odd, None, d, ok, None) == _lib.MOE_ERR_MISALIGNED
    assert lib.moe_router_logits(ok, ok, ctypes.c_void_p(0x10002), d, ok, None) == _lib.MOE_ERR_MISALIGNED
    assert lib.moe_layer_forward_router(ok, ok, None, w, w, d, ok, None, None, None, ok, small, None) == \
        _lib.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_layer_forward_router(ok, ok, None, w, w, d, ok, odd, None, None, ok, 1 << 30, None) == \
        _lib.MOE_ERR_MISALIGNED


def test_host_plan_argument_checks(lib):
    # rejected before any CUDA call: no plan pointer, null host buffers, small workspace
    d = _lib.dims(4, 128, 64, 8, 2)
    ok = ctypes.c_void_p(0x10000)
    w = _lib.W4(0x10000, 0x10000)
    plan = ctypes.c_void_p(0x1234)
    big = _lib.moe_workspace_bytes(d)
    assert lib.moe_host_plan_create(ok, ok, w, w, d, ok, ok, big, ok, None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_host_plan_create(None, ok, w, w, d, ok, ok, big, ok, ctypes.byref(plan)) == \
        _lib.MOE_ERR_INVALID_ARG
    assert plan.value is None                       # cleared on every failure
    assert lib.moe_host_plan_create(ok, ok, w, w, d, ok, ok, big - 1, ok, ctypes.byref(plan)) == \
        _lib.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_host_plan_create(ok, ok, w, w, _lib.dims(4, 100, 64, 8, 2), ok, ok, big, ok,
                                    ctypes.byref(plan)) == _lib.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_host_plan_run(None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_host_plan_destroy(None) == _lib.MOE_OK


@pytest.mark.parametrize("dims,launches", [
    ((0, 2048, 768, 128, 8), 0),
    ((32, 2048, 768, 128, 8), 5),       # routing + grouping block, quantize + gather, gate_up, down, combine
    ((800, 2048, 512, 256, 8), 8),      # chunked grouping (4 launches) + 4
    ((16, 256, 128, 8, 2), -_lib.MOE_ERR_UNSUPPORTED_SHAPE),  # I below the W4A4 stage of 256
])
def test_w4a4_kernel_launch_count(lib, dims, launches):
    assert _lib.moe_w4a4_kernel_launches(_lib.dims(*dims)) == launches
