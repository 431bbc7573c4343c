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


# Fake, 256-byte aligned device addresses: every case below fails a host check before any
# pointer is dereferenced or any CUDA call is made.
A = 0x10000


def _w(fmt, C=4, d=256, f=512, prepared=False, **over):
    w = _fake_weights(fmt, C, d, f, prepared)
    for k, v in over.items():
        setattr(w, k, v)
    return w


def test_quantize_act_argument_checks(L):
    d = ft.desc(8, 2, 256, 512, ft.NVFP4)
    q = L.ftmoe_quantize_act
    assert q(ctypes.byref(d), A, 0, A, A, None) == 1                 # T < 1
    assert q(ctypes.byref(d), A, (1 << 20) + 1, A, A, None) == 1     # T above 2^20
    assert q(ctypes.byref(d), None, 4, A, A, None) == 1
    assert q(ctypes.byref(d), A + 8, 4, A, A, None) == 1             # x not 16-byte aligned
    assert q(ctypes.byref(d), A, 4, A + 4, A, None) == 1             # codes not 8-byte aligned
    assert q(ctypes.byref(d), A, 4, A, None, None) == 1
    d8 = ft.desc(8, 2, 256, 512, ft.FP8_B128)
    assert q(ctypes.byref(d8), A, 4, A, A + 2, None) == 1            # fp32 scales not 4-byte aligned


def test_combine_argument_checks(L):
    d = ft.desc(8, 2, 256, 512, ft.BF16)
    c = L.ftmoe_combine
    #        desc           T  y  pair_pos w  ids slot_of partial_b out_f32 out_bf16
    assert c(ctypes.byref(d), 4, A, A, A, A, None, None, None, None, None) == 1       # no output
    assert c(ctypes.byref(d), 0, A, A, A, A, None, None, A, None, None) == 1          # T < 1
    assert c(ctypes.byref(d), 4, A, None, A, A, None, None, A, None, None) == 1       # y without pair_pos
    assert c(ctypes.byref(d), 4, A, A, None, A, None, None, A, None, None) == 1       # y without weights
    assert c(ctypes.byref(d), 4, A, A, A, None, A, None, A, None, None) == 1          # slot_of without ids
    assert c(ctypes.byref(d), 4, A + 4, A, A, A, None, None, A, None, None) == 1      # y misaligned
    assert c(ctypes.byref(d), 4, None, None, None, None, None, A + 4, A, None, None) == 1   # partial_b misaligned
    assert c(ctypes.byref(d), 4, A, A, A, A, None, None, A + 8, None, None) == 1      # out_f32 misaligned
    assert c(ctypes.byref(d), 4, A, A, A, A, None, None, None, A + 2, None) == 1      # out_bf16 misaligned


def test_prepare_weights_argument_checks(L):
    dn = ft.desc(8, 2, 256, 512, ft.NVFP4)
    p = L.ftmoe_prepare_weights
    need = L.ftmoe_prepare_weights_size(ctypes.byref(dn), 4)
    assert need > 0
    assert p(ctypes.byref(dn), None, A, need, None) == 1
    assert p(ctypes.byref(dn), ctypes.byref(_w(ft.MXFP4)), A, need, None) == 1          # format differs
    assert p(ctypes.byref(dn), ctypes.byref(_w(ft.NVFP4, d=512)), A, need, None) == 1   # d differs
    assert p(ctypes.byref(dn), ctypes.byref(_w(ft.NVFP4, tensor_scale=None)), A, need, None) == 1
    assert p(ctypes.byref(dn), ctypes.byref(_w(ft.NVFP4, gate=A + 8)), A, need, None) == 1
    assert p(ctypes.byref(dn), ctypes.byref(_w(ft.NVFP4)), None, need, None) == 1
    assert p(ctypes.byref(dn), ctypes.byref(_w(ft.NVFP4)), A + 8, need, None) == 1
    assert p(ctypes.byref(dn), ctypes.byref(_w(ft.NVFP4)), A, need - 1, None) == 4
    # BF16 and FP8 need no prepared layout: size 0 and a no-op
    for fmt in (ft.BF16, ft.FP8_B128):
        df = ft.desc(8, 2, 256, 512, fmt)
        assert L.ftmoe_prepare_weights_size(ctypes.byref(df), 4) == 0
        assert p(ctypes.byref(df), ctypes.byref(_w(fmt)), None, 0, None) == 0
    assert L.ftmoe_prepare_weights_size(ctypes.byref(dn), 0) == 0


def test_prepared_size_grows_with_the_slots(L):
    for fmt in (ft.NVFP4, ft.MXFP4):
        d = ft.desc(128, 8, 2048, 768, fmt)
        one = L.ftmoe_prepare_weights_size(ctypes.byref(d), 1)
        assert one > 0
        # each slot's prepared layout is at least as large as its canonical packed weights
        canonical = 3 * 2048 * 768 // 2
        assert one >= canonical
        assert L.ftmoe_prepare_weights_size(ctypes.byref(d), 47) >= 47 * canonical


def test_expert_ffn_argument_checks(L):
    d = ft.desc(8, 2, 256, 512, ft.BF16)
    f = L.ftmoe_expert_ffn
    need = L.ftmoe_expert_ffn_workspace_size(ctypes.byref(d), 4)
    w = ctypes.byref(_w(ft.BF16))
    #        desc           weights slot_of x  T  off sp topk_w out ws  bytes
    assert f(ctypes.byref(d), w, None, A, 0, A, A, None, A, A, need, None) == 1
    assert f(ctypes.byref(d), w, None, A, 4, None, A, None, A, A, need, None) == 1
    assert f(ctypes.byref(d), w, None, A, 4, A, None, None, A, A, need, None) == 1
    assert f(ctypes.byref(d), w, None, A, 4, A, A, None, None, A, need, None) == 1
    assert f(ctypes.byref(d), w, None, A, 4, A, A, None, A + 4, A, need, None) == 1    # out misaligned
    assert f(ctypes.byref(d), w, None, A + 2, 4, A, A, None, A, A, need, None) == 1    # x misaligned
    assert f(ctypes.byref(d), w, None, A, 4, A, A, None, A, None, need, None) == 1
    assert f(ctypes.byref(d), w, None, A, 4, A, A, None, A, A, need - 1, None) == 4
    assert f(ctypes.byref(d), None, None, A, 4, A, A, None, A, A, need, None) == 1


def test_expert_ffn_path_choice(L):
    path = L.ftmoe_expert_ffn_path
    for fmt in (ft.BF16, ft.NVFP4, ft.MXFP4, ft.FP8_B128):
        d = ft.desc(128, 8, 2048, 768, fmt)
        assert path(ctypes.byref(d), 1) == 0                          # decode: weight-only streaming
        assert path(ctypes.byref(d), 255) == 0
    big = {ft.BF16: 0, ft.NVFP4: 1, ft.MXFP4: 0, ft.FP8_B128: 2}
    for fmt, want in big.items():
        d = ft.desc(128, 8, 2048, 768, fmt)
        assert path(ctypes.byref(d), 256) == want
        assert path(ctypes.byref(d), 8192) == want
    assert path(ctypes.byref(ft.desc(128, 8, 2048, 768, ft.NVFP4)), 0) == -1
    assert path(ctypes.byref(ft.desc(128, 8, 2048, 700, ft.NVFP4)), 256) == -1       # ffn % 128 != 0


def test_layer_forward_argument_checks(L):
    d = ft.desc(8, 2, 256, 512, ft.NVFP4)
    lf = L.ftmoe_layer_forward
    need = L.ftmoe_layer_workspace_size(ctypes.byref(d), 4)
    assert need > 0
    w = ctypes.byref(_w(ft.NVFP4, prepared=True))
    #          desc          weights slot_of x  w_router bias T ids tw out_f32 out_bf16 ws bytes
    assert lf(ctypes.byref(d), w, None, A, A, None, 0, A, A, A, None, A, need, None) == 1
    assert lf(ctypes.byref(d), w, None, A, A, None, 4, A, None, A, None, A, need, None) == 1    # ids without tw
    assert lf(ctypes.byref(d), w, None, A, A, None, 4, None, A, A, None, A, need, None) == 1    # tw without ids
    assert lf(ctypes.byref(d), w, None, A, A, None, 4, A, A, None, None, A, need, None) == 1    # no out_f32
    assert lf(ctypes.byref(d), w, None, A, None, None, 4, A, A, A, None, A, need, None) == 1    # no router
    assert lf(ctypes.byref(d), w, None, A + 8, A, None, 4, A, A, A, None, A, need, None) == 1
    assert lf(ctypes.byref(d), w, None, A, A, None, 4, A, A, A, A + 2, A, need, None) == 1     # out_bf16 misaligned
    assert lf(ctypes.byref(d), ctypes.byref(_w(ft.MXFP4)), None, A, A, None, 4, A, A, A, None, A, need, None) == 1
    assert lf(ctypes.byref(d), w, None, A, A, None, 4, A, A, A, None, A, need - 1, None) == 4
    assert lf(ctypes.byref(d), w, None, A, A, None, 4, A, A, A, None, None, need, None) == 1


def test_route_noalloc_argument_checks(L):
    d = ft.desc(128, 8, 2048, 768, ft.NVFP4)
    r = L.ftmoe_route_noalloc
    assert r(ctypes.byref(d), A, A, None, 0, A, A, None) == 1
    assert r(ctypes.byref(d), None, A, None, 4, A, A, None) == 1
    assert r(ctypes.byref(d), A, A, None, 4, None, A, None) == 1
    assert r(ctypes.byref(d), A + 8, A, None, 4, A, A, None) == 1
    # the library's fixed logits array holds FTMOE_NOALLOC_MAX_LOGITS = 262144 entries
    assert r(ctypes.byref(d), A, A, None, 262144 // 128 + 1, A, A, None) == 4


def test_lru_argument_checks(L):
    s = L.ftmoe_slot_lru
    assert s(None, 0, A, 4, 2, A, A, A, A, None) == 1
    assert L.ftmoe_slot_lru_replay(None, A, 4, 1, 2, A, A, A, 16, A, None) == 1
    assert L.ftmoe_lru_reset(None, None) == 1
    assert L.ftmoe_lru_destroy(None) == 1
    assert L.ftmoe_lru_copy_slot_of(None, A, None) == 1
    assert L.ftmoe_lru_slot_of(None) is None
    assert L.ftmoe_get_device_error(None, None) == 1
    for Lyr, E, C in [(0, 8, 4), (1, 0, 4), (1, 8, 0), (-1, 8, 4)]:
        assert L.ftmoe_lru_create(Lyr, E, C, ctypes.byref(ctypes.c_void_p())) == 1
    assert L.ftmoe_lru_create(1, 8, 4, None) == 1
    # the state must fit in shared memory: (L*E + 3C + ceil(E/32)) * 4 bytes <= 200 KiB
    assert L.ftmoe_lru_create(200, 256, 225, ctypes.byref(ctypes.c_void_p())) == 2
    assert L.ftmoe_lru_create(1, 32, 17056, ctypes.byref(ctypes.c_void_p())) == 2    # 51201 ints, one too many


def test_status_strings_cover_every_code(L):
    seen = set()
    for code in range(7):
        s = L.ftmoe_status_string(code)
        assert s and s != b"unknown status"
        seen.add(s)
    assert len(seen) == 7
    assert L.ftmoe_status_string(99) == b"unknown status"


def test_layer_workspace_holds_only_what_the_call_can_use(L):
    """The one-kernel forms' scratch (the slice form keeps one partial output per SM) is
    reserved only where those forms can run: a few tokens with 4-bit weights."""
    dec = ft.desc(128, 8, 2048, 768, ft.NVFP4)
    ffn = L.ftmoe_expert_ffn_workspace_size
    lay = L.ftmoe_layer_workspace_size
    assert lay(ctypes.byref(dec), 1) >= 148 * 2048 * 4                 # one fp32 partial per SM
    assert lay(ctypes.byref(dec), 8192) < ffn(ctypes.byref(dec), 8192) + (8 << 20)   # prefill: FFN scratch + pairs
    fp8 = ft.desc(256, 6, 4096, 2048, ft.FP8_B128)
    assert lay(ctypes.byref(fp8), 16384) < ffn(ctypes.byref(fp8), 16384) + (8 << 20)
    stack = ft.desc(256, 6, 4096, 2048, ft.MXFP4)                      # d 4096: no slice form
    assert lay(ctypes.byref(stack), 1) < 148 * 4096 * 4


def test_streaming_path_refuses_calls_beyond_its_item_range(L):
    """Path 0 indexes (pairs / 8 + E) x max(d, ffn) work items in 32-bit arithmetic; calls
    beyond 2^28 of them return FTMOE_ERR_UNSUPPORTED before any launch."""
    big = ft.desc(1024, 32, 8192, 8192, ft.BF16)
    T = 1 << 20                                      # (2^25 / 8 + 1024) x 8192 > 2^28
    assert L.ftmoe_expert_ffn_path(ctypes.byref(big), T) == 0
    w = ctypes.byref(_w(ft.BF16, C=1024, d=8192, f=8192))
    assert L.ftmoe_expert_ffn(ctypes.byref(big), w, None, A, T, A, A, None, A, A, 1 << 62, None) == 2
    assert L.ftmoe_layer_forward(ctypes.byref(big), w, None, A, A, None, T, A, A, A, None, A, 1 << 62, None) == 2
    mx = ft.desc(256, 6, 4096, 2048, ft.MXFP4)       # MXFP4 streams at every T: up to 87040 tokens here
    wm = ctypes.byref(_w(ft.MXFP4, C=256, d=4096, f=2048))
    assert L.ftmoe_expert_ffn(ctypes.byref(mx), wm, None, A, 400000, A, A, None, A, A, 1 << 62, None) == 2


def test_size_queries_are_consistent(L):
    """Host-side size queries over a sweep of layers: the layer workspace covers each step's
    own workspace; within one form of the call (the same FFN path, up to 8 tokens or more)
    sizes never shrink as T grows; the tensor-core paths start at FTMOE_PREFILL_MIN_T = 256;
    the prepared size grows with the slots."""
    import itertools
    shapes = [(8, 2, 256, 512), (128, 8, 2048, 768), (256, 6, 4096, 2048), (300, 2, 256, 128), (1024, 32, 512, 256)]
    for (E, k, d, f), fmt in itertools.product(shapes, [ft.BF16, ft.NVFP4, ft.MXFP4, ft.FP8_B128]):
        dsc = ctypes.byref(ft.desc(E, k, d, f, fmt))
        prev = {}
        for T in (1, 2, 7, 8, 9, 64, 255, 256, 1000, 8192):
            lay = L.ftmoe_layer_workspace_size(dsc, T)
            assert lay >= L.ftmoe_route_workspace_size(dsc, T) - 256
            assert lay >= L.ftmoe_permute_workspace_size(dsc, T)
            assert lay >= L.ftmoe_expert_ffn_workspace_size(dsc, T)
            p = L.ftmoe_expert_ffn_path(dsc, T)
            assert p in (0, 1, 2) and (p == 0 or T >= 256)
            form = (p, T <= 8)
            assert lay >= prev.get(form, 0), (E, k, d, f, fmt, T)
            prev[form] = lay
        one, two = L.ftmoe_prepare_weights_size(dsc, 1), L.ftmoe_prepare_weights_size(dsc, 2)
        assert (one == 0) == (fmt in (ft.BF16, ft.FP8_B128)) and two >= 2 * one - 2048


# --- expert cache calls: q*, slot copies, the split, resize (host checks only) -----------
def test_qstar_host_arithmetic(L):
    assert abs(L.ftmoe_qstar(8, 52.7, 77.3) - 8 * 52.7 / 77.3) == 0.0
    assert L.ftmoe_qstar_fill_count(8, 52.7, 77.3) == 5
    assert L.ftmoe_qstar_fill_count(8, 11.8, 47.5) == 2
    assert L.ftmoe_qstar_fill_count(1, 1.0, 2.0) == 1          # 0.5 rounds half up
    assert L.ftmoe_qstar_fill_count(5, 100.0, 1.0) == 5        # clamped to m
    for bad in [(-1, 1.0, 1.0), (3, 0.0, 1.0), (3, 1.0, 0.0), (3, float("nan"), 1.0), (3, 1.0, float("inf"))]:
        assert L.ftmoe_qstar(*bad) == -1.0
        assert L.ftmoe_qstar_fill_count(*bad) == -1


def _ws(C, fmt=ft.NVFP4, d=256, f=256, prepared=None):
    return ft.WeightsStruct(fmt, C, d, f, 16, 16, 16, 16, 16, 16, 16, prepared)


def test_copy_slots_checks_its_arguments_on_the_host(L):
    d = ft.desc(8, 2, 256, 256, ft.NVFP4)
    src, dst = _ws(8), _ws(4)
    assert L.ftmoe_copy_slots(ctypes.byref(d), ctypes.byref(src), ctypes.byref(dst), 16, None, 0, None) == 0
    assert L.ftmoe_copy_slots(ctypes.byref(d), ctypes.byref(src), ctypes.byref(dst), None, None, 3, None) == 1
    assert L.ftmoe_copy_slots(ctypes.byref(d), ctypes.byref(src), ctypes.byref(dst), 16, None, -1, None) == 1
    assert L.ftmoe_copy_slots(ctypes.byref(d), None, ctypes.byref(dst), 16, None, 1, None) == 1
    other = ft.desc(8, 2, 512, 256, ft.NVFP4)                 # arenas of another shape
    assert L.ftmoe_copy_slots(ctypes.byref(other), ctypes.byref(src), ctypes.byref(dst), 16, None, 1, None) == 1
    # prepared layouts must be on both sides or on neither
    assert L.ftmoe_copy_slots(ctypes.byref(d), ctypes.byref(_ws(8, prepared=256)), ctypes.byref(dst), 16, None, 1,
                              None) == 1


def test_miss_split_and_resize_check_their_arguments_on_the_host(L):
    assert L.ftmoe_miss_split(None, 0, 16, 1, 8, 16, 1.0, 2.0, -1, 16, 16, 16, 16, 16, None) == 1
    assert L.ftmoe_lru_resize(None, 4, None, None, None) == 1
    assert L.ftmoe_lru_capacity(None) == -1


def test_host_buffer_layer_call_checks(L):
    d = ft.desc(128, 8, 2048, 768, ft.NVFP4)
    need = L.ftmoe_layer_host_workspace_size(ctypes.byref(d), 4)
    assert need >= L.ftmoe_layer_workspace_size(ctypes.byref(d), 4) + 2 * 4 * 2048 * 2
    w = _ws(8, d=2048, f=768)
    args = [ctypes.byref(d), ctypes.byref(w), None, 16, 16, None, 4, 16, 16, 16, 16, 16]
    assert L.ftmoe_layer_forward_host(*args, need - 1, None) == 4             # workspace too small
    bad = list(args)
    bad[3] = None                                                             # no host input
    assert L.ftmoe_layer_forward_host(*bad, need, None) == 1
    bad = list(args)
    bad[10] = None                                                            # no host output
    assert L.ftmoe_layer_forward_host(*bad, need, None) == 1


def test_layer_graph_checks_its_arguments_on_the_host(L):
    """ftmoe_layer_graph_create refuses before any CUDA call: no output handle, no stream
    (the legacy default stream cannot be captured), the host call's own checks; launch and
    destroy take NULL as the header says."""
    d = ft.desc(128, 8, 2048, 768, ft.NVFP4)
    need = L.ftmoe_layer_host_workspace_size(ctypes.byref(d), 1)
    w = _ws(8, d=2048, f=768)
    h = ctypes.c_void_p(123)
    args = [ctypes.byref(d), ctypes.byref(w), None, 16, 16, None, 1, 16, 16, 16, 16, 16]
    assert L.ftmoe_layer_graph_create(*args, need, 16, None) == 1                    # no handle output
    assert L.ftmoe_layer_graph_create(*args, need, None, ctypes.byref(h)) == 1       # no stream
    assert h.value is None                                                            # *out cleared
    assert L.ftmoe_layer_graph_create(*args, need - 1, 16, ctypes.byref(h)) == 4     # workspace too small
    for i, v in ((3, None), (10, None), (9, None), (4, None)):                        # x, out_host, out_f32, router
        bad = list(args)
        bad[i] = v
        assert L.ftmoe_layer_graph_create(*bad, need, 16, ctypes.byref(h)) == 1
    bad = list(args)
    bad[8] = None                                                                     # topk_w without topk_ids
    assert L.ftmoe_layer_graph_create(*bad, need, 16, ctypes.byref(h)) == 1
    assert L.ftmoe_layer_graph_launch(None, None) == 1
    assert L.ftmoe_layer_graph_destroy(None) == 0


def test_streamed_layers_check_their_arguments_on_the_host(L):
    d = ft.desc(16, 4, 256, 256, ft.NVFP4)
    pool, arena = _ws(48), _ws(16)
    arenas = (ft.WeightsStruct * 2)(arena, arena)
    P3 = ctypes.c_void_p * 3
    xs, wr, of = P3(16, 16, 16), P3(16, 16, 16), P3(16, 16, 16)
    ws = L.ftmoe_layer_workspace_size(ctypes.byref(d), 300)
    call = lambda **kw: L.ftmoe_layers_streamed(
        ctypes.byref(d), kw.get("L", 3), ctypes.byref(kw.get("pool", pool)), arenas, kw.get("n", 2), kw.get("xs", xs),
        wr, None, 300, of, None, 16, kw.get("ws", ws), None, None)
    assert call(n=3) == 1                                   # one or two arenas
    assert call(n=0) == 1
    assert call(pool=_ws(47)) == 1                          # the pool holds fewer than L*E slots
    assert call(xs=P3(16, None, 16)) == 1                   # a chained layer without bf16 outputs
    assert call(xs=P3(None, 16, 16)) == 1                   # the first layer needs an input
    assert call(ws=ws - 1) == 4
