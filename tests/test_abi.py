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
