"""The C ABI without a GPU: the library loads, exports every symbol that
include/moe_ffn.h declares, and rejects bad shapes and arguments on the host
before touching CUDA."""
import ctypes as C
import os
import re

import pytest

import mxfp4_expert_ffn_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _library():
    # the checks load the compiled library: build it (nvcc cross-compiles for
    # sm_103a without a GPU) if this checkout has not, a no-op when up to date
    from mxfp4_expert_ffn_gb300 import build as b
    b.build()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe_ffn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src))


def test_header_declares_the_binding_exports():
    assert _declared() == set(m.EXPORTS)


def test_library_exports_every_declared_symbol():
    L = m.lib()
    for name in _declared():
        assert hasattr(L, name), name


def test_abi_version_and_status_strings():
    assert m.moe_abi_version() == 1
    for s in range(7):
        assert m.status_string(s)
    assert m.status_string(99) == "unknown status"


def _weights(fake=0x1000):
    w = m.MoeWeights()
    for name in ("gate", "up", "down", "s_gate", "s_up", "s_down"):
        setattr(w, name, m.MxMat(fake, fake))
    w.router_w = fake
    return w


@pytest.mark.parametrize("cfg", [
    (200, 128, 16, 2, 1, 4),      # hidden not a multiple of 128
    (256, 100, 16, 2, 1, 4),      # inter not a multiple of 128
    (256, 128, 600, 2, 1, 4),     # too many experts
    (256, 128, 16, 9, 1, 4),      # k > 8
    (256, 128, 4, 6, 1, 4),       # k > E
    (256, 128, 16, 2, 5, 4),      # too many shared experts
    (256, 128, 16, 2, 1, 0),      # no tokens
    (32768, 128, 16, 2, 1, 4),    # hidden too large
    (256, 32768, 16, 2, 1, 4),    # inter too large
    (256, 128, 0, 1, 1, 4),       # no experts
    (256, 128, 16, 0, 1, 4),      # k = 0
    (256, 128, 16, 2, -1, 4),     # negative shared count
    (256, 128, 16, 2, 1, 65537),  # more tokens than the workspace limit
    (-256, 128, 16, 2, 1, 4),     # negative hidden
])
def test_create_rejects_unsupported_shapes(cfg):
    h = C.c_void_p()
    rc = m.lib().moe_layer_create(C.byref(m.MoeConfig(*cfg)), C.byref(_weights()), 0, C.byref(h))
    assert rc == m.MOE_ERR_UNSUPPORTED and not h.value


def test_create_rejects_null_and_misaligned_weights():
    h = C.c_void_p()
    cfg = m.MoeConfig(256, 128, 16, 2, 1, 4)
    w = _weights()
    w.down = m.MxMat(None, 0x1000)
    assert m.lib().moe_layer_create(C.byref(cfg), C.byref(w), 0, C.byref(h)) == m.MOE_ERR_INVALID_ARG
    w = _weights(0x1008)  # 8-byte aligned only
    assert m.lib().moe_layer_create(C.byref(cfg), C.byref(w), 0, C.byref(h)) == m.MOE_ERR_INVALID_ARG
    assert m.lib().moe_layer_create(None, C.byref(w), 0, C.byref(h)) == m.MOE_ERR_INVALID_ARG
    assert m.lib().moe_layer_create_range(None, C.byref(w), 0, 0, 8, C.byref(h)) == m.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("lo,hi", [(-1, 8), (0, 17), (8, 8), (9, 4)])
def test_create_range_rejects_bad_ranges(lo, hi):
    h = C.c_void_p()
    cfg = m.MoeConfig(256, 128, 16, 2, 1, 4)
    assert m.lib().moe_layer_create_range(C.byref(cfg), C.byref(_weights()), 0, lo, hi, C.byref(h)) == \
        m.MOE_ERR_INVALID_ARG
    assert not h.value


def test_combine_partials_rejects_bad_arguments():
    L = m.lib()
    buf = (C.c_float * 64)()
    assert L.moe_combine_partials(buf, 0, 1, 8, None, buf, None) == m.MOE_ERR_INVALID_ARG   # no parts
    assert L.moe_combine_partials(buf, 1, 1, 6, None, buf, None) == m.MOE_ERR_INVALID_ARG   # H % 4
    assert L.moe_combine_partials(None, 1, 1, 8, None, buf, None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_combine_partials(buf, 1, 0, 8, None, None, None) == m.MOE_OK                # T = 0
    assert L.moe_forward_partial(None, buf, 1, buf, buf, buf, None) == m.MOE_ERR_INVALID_ARG


def test_fault_injection_alloc(monkeypatch):
    monkeypatch.setenv("MOE_FAULT", "alloc")
    h = C.c_void_p()
    cfg = m.MoeConfig(256, 128, 16, 2, 1, 4)
    assert m.lib().moe_layer_create(C.byref(cfg), C.byref(_weights()), 0, C.byref(h)) == m.MOE_ERR_OOM
    assert not h.value


def test_null_handle_is_rejected():
    L = m.lib()
    assert L.moe_route(None, None, 1, None, None, None, None, None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_forward(None, None, 1, None, None, None, None, None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_sync(None, None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_destroy(None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_layer_destroy(None) == m.MOE_ERR_INVALID_ARG
    buf = (C.c_uint16 * 8)()
    assert L.moe_stack_forward_host(None, 1, buf, 1, C.c_float(1e-6), buf, None) == m.MOE_ERR_INVALID_ARG
    arr = (C.c_void_p * 1)(None)
    assert L.moe_stack_forward_host(arr, 1, buf, 1, C.c_float(1e-6), buf, None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_stack_forward_host(arr, 0, buf, 1, C.c_float(1e-6), buf, None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_rmsnorm(None, 1, 100, 1e-6, None, None) == m.MOE_ERR_INVALID_ARG  # H % 8
