"""The C-ABI library loads and exports every symbol include/ftmoe.h declares.

Only host-side behaviour is exercised here, with no GPU: the version, the
status strings, the workspace-size queries, and argument checks that return
before any CUDA call.
"""
import ctypes
import os
import re
import subprocess

import pytest

import sparse_moe_expert_sorted_b300 as ft
from sparse_moe_expert_sorted_b300 import build as ftbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ftmoe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(ftmoe_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def L():
    ftbuild.build()
    return ft.lib()


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 18
    out = subprocess.run(["nm", "-D", "--defined-only", ft.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (ftmoe_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    assert sorted(ft.EXPORTS) == names
    for n in names:
        assert hasattr(L, n)


def test_host_only_calls(L):
    assert L.ftmoe_version() == 100
    assert L.ftmoe_status_string(0) == b"ok"
    assert L.ftmoe_status_string(4) == b"workspace too small"
    d = ft.desc(128, 8, 2048, 768, ft.NVFP4)
    # workspace sizes: header + logits [T,E] fp32; permute header only for one chunk
    assert L.ftmoe_route_workspace_size(ctypes.byref(d), 16) == 256 + 16 * 128 * 4
    assert L.ftmoe_permute_workspace_size(ctypes.byref(d), 16) == 256
    assert L.ftmoe_permute_workspace_size(ctypes.byref(d), 8192) == 256 + 64 * 128 * 4
    assert L.ftmoe_expert_ffn_workspace_size(ctypes.byref(d), 1) == 256 + 8 * 768 * 4
    assert L.ftmoe_layer_workspace_size(ctypes.byref(d), 1) > 0


@pytest.mark.parametrize("bad", [dict(E=0), dict(k=0), dict(k=200), dict(d=100), dict(ffn=100), dict(fmt=9),
                                 dict(renorm=2), dict(E=2000)])
def test_invalid_descriptors_are_rejected_on_the_host(L, bad):
    f = dict(E=8, k=2, d=256, ffn=512, fmt=ft.BF16, renorm=1)
    f.update(bad)
    d = ft.LayerDesc(**f)
    assert L.ftmoe_route_workspace_size(ctypes.byref(d), 4) == 0
    # invalid descriptors return FTMOE_ERR_INVALID_ARG before touching any pointer
    st = L.ftmoe_route(ctypes.byref(d), 16, 16, None, 4, 16, 16, None, 16, 1 << 20, None)
    assert st == 1
    st = L.ftmoe_permute(ctypes.byref(d), 16, 4, 16, 16, 16, 16, 1 << 20, None)
    assert st == 1


def test_short_workspace_and_null_pointers(L):
    d = ft.desc(8, 2, 256, 512, ft.BF16)
    need = L.ftmoe_route_workspace_size(ctypes.byref(d), 16)
    st = L.ftmoe_route(ctypes.byref(d), 16, 16, None, 16, 16, 16, None, 16, need - 1, None)
    assert st == 4                                          # FTMOE_ERR_WORKSPACE
    st = L.ftmoe_route(ctypes.byref(d), None, 16, None, 16, 16, 16, None, 16, need, None)
    assert st == 1
    st = L.ftmoe_route(ctypes.byref(d), 8, 16, None, 16, 16, 16, None, 16, need, None)
    assert st == 1                                          # x not 16-byte aligned
    assert L.ftmoe_lru_create(0, 8, 4, ctypes.byref(ctypes.c_void_p())) == 1
    assert L.ftmoe_lru_create(1, 1 << 16, 1 << 12, ctypes.byref(ctypes.c_void_p())) == 2   # state too large
    assert L.ftmoe_slot_lru(None, 0, 16, 1, 1, 16, 16, 16, 16, None) == 1
    w = ft.WeightsStruct(ft.NVFP4, 4, 256, 512, 16, 16, 16, 16, 16, 16, None)   # NVFP4 needs tensor scales
    d2 = ft.desc(8, 2, 256, 512, ft.NVFP4)
    st = L.ftmoe_expert_ffn(ctypes.byref(d2), ctypes.byref(w), None, 16, 4, 16, 16, None, 16, 16, 1 << 30, None)
    assert st == 1


def _fake_weights(fmt, C, d, f, prepared):
    # aligned fake device addresses: ftmoe_layer_path only checks them, never reads them
    return ft.WeightsStruct(fmt, C, d, f, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000,
                            0x8000 if prepared else None)


def test_layer_path_choice_on_the_host(L):
    """Which form ftmoe_layer_forward takes: one kernel for few tokens with 4-bit prepared
    weights, separate steps otherwise, -1 for invalid arguments (host logic only)."""
    dec = ft.desc(128, 8, 2048, 768, ft.NVFP4)
    w = _fake_weights(ft.NVFP4, 128, 2048, 768, True)
    for T in range(1, 9):                                                        # the slice form (NVFP4)
        assert L.ftmoe_layer_path(ctypes.byref(dec), ctypes.byref(w), T) == 2, T
    assert L.ftmoe_layer_path(ctypes.byref(dec), ctypes.byref(w), 9) == 0
    assert L.ftmoe_layer_path(ctypes.byref(dec), ctypes.byref(w), 8192) == 0
    wn = _fake_weights(ft.NVFP4, 128, 2048, 768, False)
    assert L.ftmoe_layer_path(ctypes.byref(dec), ctypes.byref(wn), 1) == 0      # not prepared
    stack = ft.desc(256, 6, 4096, 2048, ft.MXFP4)
    ws = _fake_weights(ft.MXFP4, 225, 4096, 2048, True)
    assert L.ftmoe_layer_path(ctypes.byref(stack), ctypes.byref(ws), 1) == 1   # d 4096: no slice layout
    small = ft.desc(32, 6, 512, 256, ft.MXFP4)
    wsm = _fake_weights(ft.MXFP4, 32, 512, 256, True)
    assert L.ftmoe_layer_path(ctypes.byref(small), ctypes.byref(wsm), 1) == 2   # MXFP4: slice form for one token
    assert L.ftmoe_layer_path(ctypes.byref(small), ctypes.byref(wsm), 2) == 1   # and the merge form beyond
    fp8 = ft.desc(256, 6, 4096, 2048, ft.FP8_B128)
    w8 = _fake_weights(ft.FP8_B128, 256, 4096, 2048, True)
    assert L.ftmoe_layer_path(ctypes.byref(fp8), ctypes.byref(w8), 1) == 0       # no 4-bit decode layout
    assert L.ftmoe_layer_path(ctypes.byref(dec), ctypes.byref(w), 0) == -1
    wrong = _fake_weights(ft.MXFP4, 128, 2048, 768, True)                       # format differs from the layer
    assert L.ftmoe_layer_path(ctypes.byref(dec), ctypes.byref(wrong), 1) == -1
