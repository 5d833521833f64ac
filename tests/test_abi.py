"""The C ABI: library loads, exports what include/moe.h declares, host-side checks.

No compute call is made here (these tests run without a GPU).
"""
import ctypes
import os
import re

import pytest

from conftest import ROOT, golden_path


@pytest.fixture(scope="module")
def L():
    from mxfp4_routed_expert_03_gb300 import build
    build.build()
    import mxfp4_routed_expert_03_gb300 as m
    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    decl = _declared()
    assert set(decl) == set(L.EXPORTS)
    lib = L.lib()
    for name in decl:
        assert hasattr(lib, name), name


def test_expert_bytes_match_the_k3_store(L):
    g = {}
    with open(golden_path("k3_layer_bytes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                g[k] = float(v) if "." in v else int(v)
    assert g["routed_experts"] == g["routed_layers"] * g["experts_per_layer"]
    per_expert = g["canonical_routed_bytes"] // g["routed_experts"]
    assert per_expert * g["routed_experts"] == g["canonical_routed_bytes"]
    assert L.moe_expert_bytes(7168, 1536) == per_expert == 17547264
    assert round(per_expert / 2**20, 3) == g["slot_mib_printed"]
    assert L.moe_expert_bytes(256, 128) == 3 * (256 * 128 // 2 + 256 * 128 // 32)
    assert L.moe_expert_bytes(100, 128) == -1


def test_strerror(L):
    assert L.moe_strerror(0) == "ok"
    assert "workspace" in L.moe_strerror(L.MOE_ERR_WORKSPACE)
    assert L.moe_strerror(-99) == "unknown status code"


def test_create_rejects_bad_descriptors_on_the_host(L):
    w = L.moe_weights(*([16] * 6 + [None] * 4))
    cases = [
        (L.moe_desc(7168, 1536, 896, 0, 0, 0), L.MOE_ERR_INVALID_ARG),
        (L.moe_desc(7168, 1536, 8, 16, 0, 0), L.MOE_ERR_INVALID_ARG),
        (L.moe_desc(7168, 1536, 896, 16, 5, 0), L.MOE_ERR_INVALID_ARG),
        (L.moe_desc(7200, 1536, 896, 16, 0, 0), L.MOE_ERR_UNSUPPORTED),
        (L.moe_desc(7168, 1536, 2048, 16, 0, 0), L.MOE_ERR_UNSUPPORTED),
        (L.moe_desc(7168, 1536, 896, 33, 0, 0), L.MOE_ERR_UNSUPPORTED),
        (L.moe_desc(7168, 1536, 896, 16, 0, 0, 2), L.MOE_ERR_INVALID_ARG),   # act_mode
    ]
    for d, code in cases:
        h = ctypes.c_void_p()
        assert L.lib().moe_create(ctypes.byref(d), ctypes.byref(w), ctypes.byref(h)) == code
        assert h.value is None
    assert L.lib().moe_create(None, None, None) == L.MOE_ERR_INVALID_ARG
    bad_w = L.moe_weights(*([16] * 5 + [None] * 5))
    h = ctypes.c_void_p()
    assert L.lib().moe_create(ctypes.byref(L.moe_desc(256, 128, 32, 4, 0, 0)), ctypes.byref(bad_w),
                              ctypes.byref(h)) == L.MOE_ERR_INVALID_ARG


def test_null_handle_calls_are_rejected(L):
    plan = L.moe_plan_buf()
    assert L.moe_plan(None, 1, None, None, plan, None, 0) == L.MOE_ERR_INVALID_ARG
    assert L.moe_decode(None, 1, None, plan, None, None, 0) == L.MOE_ERR_INVALID_ARG
    assert L.moe_forward(None, 1, None, plan, None, None, 0) == L.MOE_ERR_INVALID_ARG
    assert L.moe_router_logits(None, 1, None, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_workspace_bytes(None, 16, L.MOE_OP_DECODE) == 0
    L.moe_destroy(None)


def test_store_entry_points_check_arguments_on_the_host(L):
    """Argument errors of the compressed-store calls come back before anything
    reaches the device (these run without a GPU)."""
    w = L.moe_weights()
    st = L.moe_store(None, 0, None, None)
    # decode: null status, bad shape, negative count; zero items is a no-op
    assert L.moe_store_decode(4, 256, 128, st, None, None, 1, w, 1, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_store_decode(4, 256, 100, st, None, None, 1, w, 1, 1) == L.MOE_ERR_INVALID_ARG
    assert L.moe_store_decode(4, 256, 128, st, None, None, -1, w, 1, 1) == L.MOE_ERR_INVALID_ARG
    assert L.moe_store_decode(0, 256, 128, st, None, None, 1, w, 1, 1) == L.MOE_ERR_INVALID_ARG
    assert L.moe_store_decode(4, 256, 128, st, None, None, 0, w, 1, 1) == L.MOE_OK
    assert L.moe_store_decode(4, 256, 128, st, None, None, 1, w, 1, 1) == L.MOE_ERR_INVALID_ARG
    # streaming from a store: null store arrays, bad slot counts
    desc = L.moe_desc(256, 128, 8, 2, 0, 0)
    with pytest.raises(L.MoeError):
        L.moe_create_streaming_store(desc, st, w, 4, 16)
    for n_slots in (0, 9):
        with pytest.raises(L.MoeError):
            L.moe_create_streaming_store(desc, st, w, n_slots, 16)
    assert L.moe_strerror(L.MOE_ERR_CORRUPT_TILE) == "a compressed-store tile failed its checks"
