"""The C-ABI library builds, loads and exports every symbol include/moe.h
declares; host-side argument checks work without a GPU."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


def _lib():
    import moe_expert_layer_sorted_gb300 as m
    if not os.path.exists(m.LIB_PATH):
        from moe_expert_layer_sorted_gb300 import _build
        _build.build()
    return m


def _declared():
    hdr = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"^(?:moe_status|const char\*)\s+(moe_\w+)\(", hdr, re.M)))


def test_header_declares_what_the_binding_names():
    m = _lib()
    assert _declared() == sorted(m.EXPORTS)


def test_library_exports_every_declared_symbol():
    m = _lib()
    L = m.lib()
    for name in _declared():
        assert hasattr(L, name), name


def test_status_strings():
    m = _lib()
    L = m.lib()
    for code, name in m.STATUS.items():
        assert L.moe_status_string(code).decode() == name


def test_bad_descriptors_rejected_on_the_host():
    m = _lib()
    L = m.lib()
    d = m.PlanDesc()
    d.struct_size = 3  # wrong ABI size
    h = ctypes.c_void_p()
    assert L.moe_plan_create(ctypes.byref(d), ctypes.byref(h)) == 1
    assert b"struct_size" in L.moe_last_error(None)
    d.struct_size = ctypes.sizeof(m.PlanDesc)
    d.num_layers, d.num_experts, d.hidden, d.inter, d.top_k = 1, 16, 300, 128, 2
    d.weight_bits, d.group_size, d.scale_dtype, d.max_tokens = 4, 32, 0, 8
    assert L.moe_plan_create(ctypes.byref(d), ctypes.byref(h)) == 1   # H % 256 != 0
    d.hidden = 256
    d.top_k = 9
    assert L.moe_plan_create(ctypes.byref(d), ctypes.byref(h)) == 1   # k > 8
    d.top_k = 2
    d.reserved[0] = 1
    assert L.moe_plan_create(ctypes.byref(d), ctypes.byref(h)) == 1
    assert L.moe_plan_destroy(None) == 1
    assert L.moe_update_router_biases(None, 0, 1, None, None) == 1
    assert L.moe_debug_fail_next_forward(None) == 1
    assert L.moe_quantize(None, 4, 4, 4, 4, 0, None, None, None) == 1
    assert L.moe_layer_forward_residual(None, 0, None, 1, None, None, None, None) == 1
    assert L.moe_layer_forward_host(None, 0, None, 1, None, None) == 1


def test_no_device_is_an_error_not_a_crash():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("has a GPU")
    m = _lib()
    L = m.lib()
    d = m.PlanDesc()
    d.struct_size = ctypes.sizeof(m.PlanDesc)
    d.num_layers, d.num_experts, d.hidden, d.inter, d.top_k = 1, 16, 256, 128, 2
    d.weight_bits, d.group_size, d.scale_dtype, d.max_tokens = 4, 32, 0, 8
    d.hbm_experts = 16
    h = ctypes.c_void_p()
    rc = L.moe_plan_create(ctypes.byref(d), ctypes.byref(h))
    assert rc in (1, 3) and not h.value
