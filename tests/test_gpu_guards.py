"""Out-of-bounds writes, checked from the host: every output buffer and workspace a call gets
is the middle of a larger allocation whose 256-byte margins hold a sentinel.  After the call
(and a synchronise) the margins must be unchanged, on every path of every call: route,
permute, the activation quantiser, the expert FFN (each path, y and fused out), combine,
the layer call (each form, decode and prefill), and the LRU (call by call and replay).
The input buffers are read-only to the library and get no margins."""
import numpy as np
import pytest
import torch

import synth

from gpu_helpers import ensure_built
import sparse_moe_expert_sorted_b300 as ft

pytestmark = pytest.mark.gpu
MARGIN = 256                 # bytes on each side (keeps every buffer 256-byte aligned)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


class Guarded:
    """n elements of dtype between two MARGIN-byte sentinel regions."""

    def __init__(self, n, dtype, fill=0):
        es = torch.empty(0, dtype=dtype).element_size()
        self.g = MARGIN // es
        self.n = n
        self.buf = torch.empty(n + 2 * self.g, dtype=dtype, device="cuda")
        self.buf.view(torch.uint8).fill_(0xA5)                        # sentinel bytes
        self.t = self.buf[self.g:self.g + n]
        if fill is not None:
            self.t.fill_(fill)

    def intact(self):
        raw = self.buf.view(torch.uint8)
        b = MARGIN
        return bool((raw[:b] == 0xA5).all()) and bool((raw[raw.numel() - b:] == 0xA5).all())


def _ws(nbytes):
    return Guarded(max(int(nbytes), ft.WS_ZERO_BYTES), torch.uint8, fill=0)


def _check(*bufs):
    torch.cuda.synchronize()
    bad = [i for i, b in enumerate(bufs) if not b.intact()]
    assert not bad, f"margins overwritten around buffers {bad}"
    assert ft.get_device_error() == 0


def _weights(fmt, E, d, f, seed, prepare=True):
    W = synth.make_experts(fmt, E, d, f, seed, device="cuda")
    if prepare:
        ft.prepare_weights(ft.desc(E, 2, d, f, fmt), W)
    return W


def _route_permute(dsc, x, wr):
    T = x.shape[0]
    P = T * dsc.k
    ids, w, lg = Guarded(P, torch.int32), Guarded(P, torch.float32), Guarded(T * dsc.E, torch.float32)
    ws = _ws(ft.route_workspace_size(dsc, T))
    ft.route(dsc, x, wr, None, ids.t, w.t, lg.t, ws.t)
    off, sp, pp = Guarded(dsc.E + 1, torch.int32), Guarded(P, torch.int32), Guarded(P, torch.int32)
    ws2 = _ws(ft.permute_workspace_size(dsc, T))
    ft.permute(dsc, ids.t.view(T, dsc.k), off.t, sp.t, pp.t, ws2.t)
    _check(ids, w, lg, ws, off, sp, pp, ws2)
    return ids.t.view(T, dsc.k), w.t.view(T, dsc.k), off.t, sp.t, pp.t


@pytest.mark.parametrize("E,k,d,T", [(8, 2, 256, 16), (128, 8, 2048, 1), (128, 8, 2048, 70), (256, 6, 512, 3000)])
def test_route_and_permute(E, k, d, T):
    dsc = ft.desc(E, k, d, 512, synth.BF16)
    _route_permute(dsc, synth.make_x(T, d, T, device="cuda"), synth.make_router(E, d, T, device="cuda"))


@pytest.mark.parametrize("fmt", [synth.NVFP4, synth.FP8_B128])
def test_quantize_act(fmt):
    T, d = 37, 512
    dsc = ft.desc(8, 2, d, 256, fmt)
    x = synth.make_x(T, d, 3, device="cuda")
    fp8 = fmt == synth.FP8_B128
    codes = Guarded(T * d if fp8 else T * d // 2, torch.uint8)
    scales = Guarded(T * (d // 128) * 4 if fp8 else T * d // 16, torch.uint8)
    ft.quantize_act(dsc, x, codes.t, scales.t)
    _check(codes, scales)


FFN_CASES = [
    # fmt, E, k, d, f, T, prepare: every path of ftmoe_expert_ffn
    (synth.BF16, 8, 2, 256, 512, 13, True),
    (synth.FP8_B128, 16, 6, 256, 256, 9, True),        # FP8 weights, CUDA-core streaming
    (synth.NVFP4, 16, 8, 512, 256, 3, True),           # 4-bit decode kernel, prepared layout
    (synth.MXFP4, 32, 6, 256, 512, 13, True),
    (synth.NVFP4, 16, 8, 512, 256, 5, False),          # 4-bit decode kernel, canonical arena
    (synth.NVFP4, 16, 8, 512, 256, 300, True),         # tcgen05, NVFP4 activations
    (synth.FP8_B128, 8, 2, 768, 384, 300, True),       # tcgen05, FP8 activations
]


@pytest.mark.parametrize("fmt,E,k,d,f,T,prepare", FFN_CASES)
def test_expert_ffn_and_combine(fmt, E, k, d, f, T, prepare):
    dsc = ft.desc(E, k, d, f, fmt)
    W = _weights(fmt, E, d, f, 5, prepare)
    x = synth.make_x(T, d, 6, device="cuda")
    ids, w, off, sp, pp = _route_permute(dsc, x, synth.make_router(E, d, 6, device="cuda"))
    P = T * k
    slot = torch.arange(E, dtype=torch.int32, device="cuda")
    st = ft.weights_struct(W)
    y = Guarded(P * d, torch.float32, fill=float("nan"))
    ws = _ws(ft.expert_ffn_workspace_size(dsc, T))
    ft.expert_ffn(dsc, st, slot, x, off, sp, None, y.t, ws.t)
    out = Guarded(T * d, torch.float32)
    ws2 = _ws(ft.expert_ffn_workspace_size(dsc, T))
    ft.expert_ffn(dsc, st, slot, x, off, sp, w, out.t, ws2.t)
    of, ob = Guarded(T * d, torch.float32), Guarded(T * d, torch.bfloat16)
    ft.combine(dsc, T, y.t, pp, w, ids, slot, None, of.t, ob.t)
    _check(y, ws, out, ws2, of, ob)
    assert torch.isfinite(y.t).all() and torch.isfinite(of.t).all()


LAYER_CASES = [
    # fmt, E, k, d, f, T: each form of ftmoe_layer_forward
    (synth.BF16, 8, 2, 256, 512, 16),          # separate steps, y and the combine call
    (synth.NVFP4, 16, 8, 512, 256, 12),        # separate steps, decode kernel with fused combine
    (synth.MXFP4, 32, 6, 256, 512, 5),         # one kernel, merge form
    (synth.NVFP4, 16, 8, 512, 256, 1),         # one kernel, slice form
    (synth.NVFP4, 24, 4, 256, 384, 6),
    (synth.NVFP4, 16, 8, 512, 256, 300),       # prefill, tcgen05
    (synth.FP8_B128, 8, 2, 768, 384, 300),
]


@pytest.mark.parametrize("fmt,E,k,d,f,T", LAYER_CASES)
def test_layer_forward(fmt, E, k, d, f, T):
    dsc = ft.desc(E, k, d, f, fmt)
    W = _weights(fmt, E, d, f, 8)
    x = synth.make_x(T, d, 9, device="cuda")
    wr = synth.make_router(E, d, 9, device="cuda")
    P = T * k
    ids, tw = Guarded(P, torch.int32), Guarded(P, torch.float32)
    of, ob = Guarded(T * d, torch.float32, fill=float("nan")), Guarded(T * d, torch.bfloat16)
    ws = _ws(ft.layer_workspace_size(dsc, T))
    for _ in range(2):                                  # the second call reuses the workspace
        ft.layer_forward(dsc, ft.weights_struct(W), None, x, wr, None, ids.t, tw.t, of.t, ob.t, ws.t)
    _check(ids, tw, of, ob, ws)
    assert torch.isfinite(of.t).all()


def test_lru_step_and_replay():
    L, E, C, B, k, steps = 2, 16, 5, 3, 2, 40
    trace = synth.make_trace(steps, L, B, k, E, 1.1, seed=4)
    lru = ft.LRU(L, E, C)
    n = min(B * k, E)
    hit, slot, ev = Guarded(n, torch.uint8), Guarded(n, torch.int32), Guarded(n, torch.int32)
    cnt = Guarded(2, torch.int64)
    for s in range(steps):
        for layer in range(L):
            ids = torch.from_numpy(np.ascontiguousarray(trace[s, layer])).cuda()
            lru.step(layer, ids, hit.t, slot.t, ev.t, cnt.t)
    _check(hit, slot, ev, cnt)
    lru.reset()
    cap = steps * L * n
    hit2, slot2, ev2 = Guarded(cap, torch.uint8), Guarded(cap, torch.int32), Guarded(cap, torch.int32)
    lru.replay(torch.from_numpy(np.ascontiguousarray(trace)).cuda(), hit2.t, slot2.t, ev2.t, cnt.t)
    _check(hit2, slot2, ev2, cnt)
    lru.close()
