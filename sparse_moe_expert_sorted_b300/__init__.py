"""Python binding of the ftmoe C ABI (include/ftmoe.h).

Argument marshalling only: every step of the layer runs in the CUDA kernels
of libftmoe.so.  Each tensor argument is checked for its type and size first,
since the library sees only its address.  Tensors are torch CUDA tensors (device memory); streams are
torch CUDA streams.  Nothing here computes the layer: there is no CPU or
PyTorch fallback.  If the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

__all__ = [
    "BF16", "NVFP4", "MXFP4", "FP8_B128", "LayerDesc", "FtmoeError", "lib", "route", "permute", "expert_ffn",
    "combine", "layer_forward", "LRU", "weights_struct", "workspace", "get_device_error", "prepare_weights",
    "quantize_act", "copy_slots", "qstar", "qstar_fill_count", "miss_split", "LayerHostCall", "layers_streamed",
]

BF16, NVFP4, MXFP4, FP8_B128 = 0, 1, 2, 3
WS_ZERO_BYTES = 256

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libftmoe.so")

# Symbols declared in include/ftmoe.h (checked by the ABI test).
EXPORTS = [
    "ftmoe_route_workspace_size", "ftmoe_route", "ftmoe_route_noalloc", "ftmoe_permute_workspace_size", "ftmoe_permute",
    "ftmoe_prepare_weights_size", "ftmoe_prepare_weights", "ftmoe_quantize_act",
    "ftmoe_expert_ffn_workspace_size", "ftmoe_expert_ffn_path", "ftmoe_expert_ffn", "ftmoe_combine", "ftmoe_lru_create", "ftmoe_lru_reset",
    "ftmoe_lru_destroy", "ftmoe_lru_slot_of", "ftmoe_lru_copy_slot_of", "ftmoe_slot_lru", "ftmoe_slot_lru_replay",
    "ftmoe_layer_workspace_size", "ftmoe_layer_path", "ftmoe_layer_forward", "ftmoe_status_string", "ftmoe_get_device_error",
    "ftmoe_version", "ftmoe_copy_slots", "ftmoe_qstar", "ftmoe_qstar_fill_count", "ftmoe_miss_split",
    "ftmoe_lru_capacity", "ftmoe_lru_resize", "ftmoe_layer_host_workspace_size", "ftmoe_layer_forward_host",
    "ftmoe_layers_streamed", "ftmoe_set_wait_limit", "ftmoe_layer_graph_create", "ftmoe_layer_graph_launch",
    "ftmoe_layer_graph_destroy",
]


class FtmoeError(RuntimeError):
    pass


class LayerDesc(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("k", ctypes.c_int), ("d", ctypes.c_int), ("ffn", ctypes.c_int),
                ("fmt", ctypes.c_int), ("renorm", ctypes.c_int)]


class WeightsStruct(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("C", ctypes.c_int), ("d", ctypes.c_int), ("ffn", ctypes.c_int),
                ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p),
                ("gate_scale", ctypes.c_void_p), ("up_scale", ctypes.c_void_p), ("down_scale", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_void_p), ("prepared", ctypes.c_void_p)]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


def lib() -> ctypes.CDLL:
    """The loaded libftmoe.so (raises FtmoeError if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise FtmoeError(f"libftmoe.so is missing ({LIB_PATH}); run `python -m sparse_moe_expert_sorted_b300.build`")
    L = ctypes.CDLL(LIB_PATH)
    sig = {
        "ftmoe_route_workspace_size": (_SZ, [_P, _I]),
        "ftmoe_route": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _P, _SZ, _P]),
        "ftmoe_route_noalloc": (_I, [_P, _P, _P, _P, _I, _P, _P, _P]),
        "ftmoe_prepare_weights_size": (_SZ, [_P, _I]),
        "ftmoe_prepare_weights": (_I, [_P, _P, _P, _SZ, _P]),
        "ftmoe_quantize_act": (_I, [_P, _P, _I, _P, _P, _P]),
        "ftmoe_permute_workspace_size": (_SZ, [_P, _I]),
        "ftmoe_permute": (_I, [_P, _P, _I, _P, _P, _P, _P, _SZ, _P]),
        "ftmoe_expert_ffn_workspace_size": (_SZ, [_P, _I]),
        "ftmoe_expert_ffn_path": (_I, [_P, _I]),
        "ftmoe_expert_ffn": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _SZ, _P]),
        "ftmoe_combine": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
        "ftmoe_lru_create": (_I, [_I, _I, _I, ctypes.POINTER(_P)]),
        "ftmoe_lru_reset": (_I, [_P, _P]),
        "ftmoe_lru_destroy": (_I, [_P]),
        "ftmoe_lru_slot_of": (_P, [_P]),
        "ftmoe_lru_copy_slot_of": (_I, [_P, _P, _P]),
        "ftmoe_slot_lru": (_I, [_P, _I, _P, _I, _I, _P, _P, _P, _P, _P]),
        "ftmoe_slot_lru_replay": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, ctypes.c_int64, _P, _P]),
        "ftmoe_layer_workspace_size": (_SZ, [_P, _I]),
        "ftmoe_layer_path": (_I, [_P, _P, _I]),
        "ftmoe_layer_forward": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _SZ, _P]),
        "ftmoe_status_string": (ctypes.c_char_p, [_I]),
        "ftmoe_get_device_error": (_I, [ctypes.POINTER(_I), _P]),
        "ftmoe_version": (_I, []),
        "ftmoe_copy_slots": (_I, [_P, _P, _P, _P, _P, _I, _P]),
        "ftmoe_qstar": (ctypes.c_double, [_I, ctypes.c_double, ctypes.c_double]),
        "ftmoe_qstar_fill_count": (_I, [_I, ctypes.c_double, ctypes.c_double]),
        "ftmoe_miss_split": (_I, [_P, _I, _P, _I, _I, _P, ctypes.c_double, ctypes.c_double, _I, _P, _P, _P, _P, _P,
                                  _P]),
        "ftmoe_lru_capacity": (_I, [_P]),
        "ftmoe_lru_resize": (_I, [_P, _I, _P, _P, _P]),
        "ftmoe_layer_host_workspace_size": (_SZ, [_P, _I]),
        "ftmoe_layer_forward_host": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _SZ, _P]),
        "ftmoe_layers_streamed": (_I, [_P, _I, _P, _P, _I, _P, _P, _P, _I, _P, _P, _P, _SZ, _P, _P]),
        "ftmoe_set_wait_limit": (_I, [ctypes.c_ulonglong]),
        "ftmoe_layer_graph_create": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _SZ, _P,
                                          ctypes.POINTER(_P)]),
        "ftmoe_layer_graph_launch": (_I, [_P, _P]),
        "ftmoe_layer_graph_destroy": (_I, [_P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(status: int, what: str):
    if status != 0:
        msg = lib().ftmoe_status_string(status).decode()
        raise FtmoeError(f"{what}: {msg} (status {status})")


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda and not t.is_pinned():
        raise FtmoeError("ftmoe takes CUDA tensors (device memory) or pinned host tensors the device can address")
    if not t.is_contiguous():
        raise FtmoeError("ftmoe takes contiguous tensors")
    return t.data_ptr()


def _need(t, name, dtype=None, count=None, nbytes=None, optional=False):
    """Check one tensor argument before its pointer crosses the C ABI: the library sees only
    the address, so a tensor of the wrong type or too small for what the call reads or writes
    would be read or written past its end.  Raw integer addresses are the caller's to size."""
    if t is None:
        if optional:
            return
        raise FtmoeError(f"{name} is required")
    if isinstance(t, int):
        return
    if not isinstance(t, torch.Tensor):
        raise FtmoeError(f"{name}: expected a torch tensor, got {type(t).__name__}")
    if dtype is not None and t.dtype != dtype:
        raise FtmoeError(f"{name}: expected {dtype}, got {t.dtype}")
    if count is not None and t.numel() < count:
        raise FtmoeError(f"{name}: needs {count} elements, has {t.numel()}")
    if nbytes is not None and t.numel() * t.element_size() < nbytes:
        raise FtmoeError(f"{name}: needs {nbytes} bytes, has {t.numel() * t.element_size()}")


def _tokens(x, dsc, name="x"):
    """T of a [T, d] bf16 activation tensor."""
    if not isinstance(x, torch.Tensor) or x.dim() != 2 or x.shape[1] != dsc.d:
        raise FtmoeError(f"{name}: expected a [T, {dsc.d}] tensor")
    _need(x, name, torch.bfloat16)
    return x.shape[0]


def _ws_bytes(ws):
    return ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 0


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def desc(E, k, d, ffn, fmt, renorm=1) -> LayerDesc:
    return LayerDesc(E, k, d, ffn, fmt, renorm)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A workspace buffer: zero-filled, so its counter header starts at zero."""
    return torch.zeros(max(int(nbytes), WS_ZERO_BYTES), dtype=torch.uint8, device=device)


@dataclass
class Weights:
    """Expert slot arena tensors (any object with these attributes works)."""
    fmt: int
    d: int
    f: int
    gate: torch.Tensor
    up: torch.Tensor
    down: torch.Tensor
    gate_s: torch.Tensor | None
    up_s: torch.Tensor | None
    down_s: torch.Tensor | None
    glob: torch.Tensor


def _check_arena(W):
    """The arena's tensors hold C slots of their matrices in W.fmt (C = W.gate.shape[0])."""
    C, n = W.gate.shape[0], W.d * W.f
    per = {BF16: 2 * n, NVFP4: n // 2, MXFP4: n // 2, FP8_B128: n}
    if W.fmt not in per:
        raise FtmoeError(f"unknown weight format {W.fmt}")
    for name in ("gate", "up", "down"):
        _need(getattr(W, name), name, nbytes=C * per[W.fmt])
    sc = {NVFP4: n // 16, MXFP4: n // 32, FP8_B128: 4 * (n // (128 * 128))}.get(W.fmt)
    for name in ("gate_s", "up_s", "down_s"):
        _need(getattr(W, name), name, nbytes=C * sc if sc else None, optional=not sc)
    if W.fmt == NVFP4:
        _need(W.glob, "glob", torch.float32, 3 * C)


def weights_struct(W, prepared=None) -> WeightsStruct:
    """ftmoe_weights view of an arena with attributes fmt, d, f, gate, up, down,
    gate_s, up_s, down_s, glob (tensor scale [C, 3], NVFP4 only).  `prepared` is
    the buffer filled by prepare_weights (needed by the NVFP4 tensor-core path);
    by default the one prepare_weights attached to W, if any."""
    if prepared is None:
        prepared = getattr(W, "ftmoe_prepared", None)
    _check_arena(W)
    return WeightsStruct(W.fmt, W.gate.shape[0], W.d, W.f, _ptr(W.gate), _ptr(W.up), _ptr(W.down),
                         _ptr(W.gate_s), _ptr(W.up_s), _ptr(W.down_s), _ptr(W.glob) if W.fmt == NVFP4 else None,
                         _ptr(prepared))


def prepare_weights_size(dsc: LayerDesc, C: int) -> int:
    return lib().ftmoe_prepare_weights_size(ctypes.byref(dsc), C)


def prepare_weights(dsc: LayerDesc, W, stream=None):
    """Repack the arena's block scales for the tensor-core path (ftmoe_prepare_weights).
    The buffer is attached to W (W.ftmoe_prepared) and returned; None when the
    format needs no repack."""
    C = W.gate.shape[0]
    n = prepare_weights_size(dsc, C)
    if n == 0:
        return None
    if W.gate.is_cuda:
        buf = torch.empty(n, dtype=torch.uint8, device=W.gate.device)
    else:   # a host pool in pinned memory: the prepare kernels write it over the host link
        buf = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    ws = weights_struct(W, prepared=0)
    _check(lib().ftmoe_prepare_weights(ctypes.byref(dsc), ctypes.byref(ws), _ptr(buf), n, _stream(stream)),
           "ftmoe_prepare_weights")
    W.ftmoe_prepared = buf
    return buf


def quantize_act(dsc, x, codes, scales, stream=None):
    """ftmoe_quantize_act: x [T, d] bf16 -> NVFP4 codes uint8 [T, d/2] + E4M3 scales uint8 [T, d/16]
    (FP8_B128 layers: codes [T, d] + fp32 scales [T, d/128], any tensor type of that many bytes)."""
    T = _tokens(x, dsc)
    fp8 = dsc.fmt == FP8_B128
    _need(codes, "codes", nbytes=T * dsc.d if fp8 else T * dsc.d // 2)
    _need(scales, "scales", nbytes=T * (dsc.d // 128) * 4 if fp8 else T * dsc.d // 16)
    _check(lib().ftmoe_quantize_act(ctypes.byref(dsc), _ptr(x), T, _ptr(codes), _ptr(scales), _stream(stream)),
           "ftmoe_quantize_act")


def route_workspace_size(dsc: LayerDesc, T: int) -> int:
    return lib().ftmoe_route_workspace_size(ctypes.byref(dsc), T)


def _route_args(dsc, x, w_router, bias, ids, w):
    T = _tokens(x, dsc)
    _need(w_router, "w_router", torch.bfloat16, dsc.E * dsc.d)
    _need(bias, "logit_bias", torch.float32, dsc.E, optional=True)
    _need(ids, "topk_ids", torch.int32, T * dsc.k)
    _need(w, "topk_w", torch.float32, T * dsc.k)
    return T


def route(dsc, x, w_router, bias, ids, w, logits, ws, stream=None):
    T = _route_args(dsc, x, w_router, bias, ids, w)
    _need(logits, "logits", torch.float32, T * dsc.E, optional=True)
    _need(ws, "ws")
    _check(lib().ftmoe_route(ctypes.byref(dsc), _ptr(x), _ptr(w_router), _ptr(bias), T, _ptr(ids), _ptr(w),
                             _ptr(logits), _ptr(ws), _ws_bytes(ws), _stream(stream)), "ftmoe_route")


def route_noalloc(dsc, x, w_router, bias, ids, w, stream=None):
    """ftmoe_route without a workspace: for callers that cannot allocate device memory.
    Calls sharing the library's fixed scratch must not overlap on the GPU."""
    T = _route_args(dsc, x, w_router, bias, ids, w)
    _check(lib().ftmoe_route_noalloc(ctypes.byref(dsc), _ptr(x), _ptr(w_router), _ptr(bias), T, _ptr(ids), _ptr(w),
                                     _stream(stream)), "ftmoe_route_noalloc")


def permute_workspace_size(dsc: LayerDesc, T: int) -> int:
    return lib().ftmoe_permute_workspace_size(ctypes.byref(dsc), T)


def permute(dsc, ids, offsets, sorted_pair, pair_pos, ws, stream=None):
    if not isinstance(ids, torch.Tensor) or ids.dim() != 2 or ids.shape[1] != dsc.k:
        raise FtmoeError(f"topk_ids: expected a [T, {dsc.k}] tensor")
    _need(ids, "topk_ids", torch.int32)
    T = ids.shape[0]
    _need(offsets, "expert_offsets", torch.int32, dsc.E + 1)
    _need(sorted_pair, "sorted_pair", torch.int32, T * dsc.k)
    _need(pair_pos, "pair_pos", torch.int32, T * dsc.k)
    _need(ws, "ws")
    _check(lib().ftmoe_permute(ctypes.byref(dsc), _ptr(ids), T, _ptr(offsets), _ptr(sorted_pair), _ptr(pair_pos),
                               _ptr(ws), _ws_bytes(ws), _stream(stream)), "ftmoe_permute")


def expert_ffn_workspace_size(dsc: LayerDesc, T: int) -> int:
    return lib().ftmoe_expert_ffn_workspace_size(ctypes.byref(dsc), T)


def expert_ffn_path(dsc: LayerDesc, T: int) -> int:
    """0 = weight-only streaming path, 1 = tensor cores with NVFP4 activations, 2 = with FP8 activations."""
    return lib().ftmoe_expert_ffn_path(ctypes.byref(dsc), T)


def expert_ffn(dsc, wstruct, slot_of, x, offsets, sorted_pair, topk_w, y_or_out, ws, stream=None):
    T = _tokens(x, dsc)
    P = T * dsc.k
    _need(slot_of, "slot_of", torch.int32, dsc.E, optional=True)
    _need(offsets, "expert_offsets", torch.int32, dsc.E + 1)
    _need(sorted_pair, "sorted_pair", torch.int32, P)
    _need(topk_w, "topk_w", torch.float32, P, optional=True)
    _need(y_or_out, "y_or_out", torch.float32, (P if topk_w is None else T) * dsc.d)
    _need(ws, "ws")
    _check(lib().ftmoe_expert_ffn(ctypes.byref(dsc), ctypes.byref(wstruct), _ptr(slot_of), _ptr(x), T,
                                  _ptr(offsets), _ptr(sorted_pair), _ptr(topk_w), _ptr(y_or_out), _ptr(ws),
                                  _ws_bytes(ws), _stream(stream)), "ftmoe_expert_ffn")


def combine(dsc, T, y, pair_pos, topk_w, topk_ids, slot_of, partial_b, out_f32, out_bf16, stream=None):
    P = T * dsc.k
    _need(y, "y", torch.float32, P * dsc.d, optional=True)
    _need(pair_pos, "pair_pos", torch.int32, P, optional=y is None)
    _need(topk_w, "topk_w", torch.float32, P, optional=y is None)
    _need(topk_ids, "topk_ids", torch.int32, P, optional=y is None or slot_of is None)
    _need(slot_of, "slot_of", torch.int32, dsc.E, optional=True)
    _need(partial_b, "partial_b", torch.float32, T * dsc.d, optional=True)
    _need(out_f32, "out_f32", torch.float32, T * dsc.d, optional=True)
    _need(out_bf16, "out_bf16", torch.bfloat16, T * dsc.d, optional=True)
    _check(lib().ftmoe_combine(ctypes.byref(dsc), T, _ptr(y), _ptr(pair_pos), _ptr(topk_w), _ptr(topk_ids),
                               _ptr(slot_of), _ptr(partial_b), _ptr(out_f32), _ptr(out_bf16), _stream(stream)),
           "ftmoe_combine")


def layer_workspace_size(dsc: LayerDesc, T: int) -> int:
    return lib().ftmoe_layer_workspace_size(ctypes.byref(dsc), T)


def layer_path(dsc: LayerDesc, wstruct, T: int) -> int:
    """1 = ftmoe_layer_forward runs as one kernel (router + expert FFN + merge), 0 = as separate steps."""
    return lib().ftmoe_layer_path(ctypes.byref(dsc), ctypes.byref(wstruct), T)


def layer_forward(dsc, wstruct, slot_of, x, w_router, bias, ids, topk_w, out_f32, out_bf16, ws, stream=None):
    T = _tokens(x, dsc)
    _need(slot_of, "slot_of", torch.int32, dsc.E, optional=True)
    _need(w_router, "w_router", torch.bfloat16, dsc.E * dsc.d)
    _need(bias, "logit_bias", torch.float32, dsc.E, optional=True)
    _need(ids, "topk_ids", torch.int32, T * dsc.k, optional=True)
    _need(topk_w, "topk_w", torch.float32, T * dsc.k, optional=True)
    _need(out_f32, "out_f32", torch.float32, T * dsc.d)
    _need(out_bf16, "out_bf16", torch.bfloat16, T * dsc.d, optional=True)
    _need(ws, "ws")
    _check(lib().ftmoe_layer_forward(ctypes.byref(dsc), ctypes.byref(wstruct), _ptr(slot_of), _ptr(x),
                                     _ptr(w_router), _ptr(bias), T, _ptr(ids), _ptr(topk_w), _ptr(out_f32),
                                     _ptr(out_bf16), _ptr(ws), _ws_bytes(ws), _stream(stream)), "ftmoe_layer_forward")


def set_wait_limit(ns: int = 0):
    """ftmoe_set_wait_limit: the time (ns) after which a bounded device wait gives up; 0 = 2 s."""
    _check(lib().ftmoe_set_wait_limit(int(ns)), "ftmoe_set_wait_limit")


def get_device_error(stream=None) -> int:
    code = ctypes.c_int(0)
    _check(lib().ftmoe_get_device_error(ctypes.byref(code), _stream(stream)), "ftmoe_get_device_error")
    return code.value


class LRU:
    """Global LRU slot map handle (device state owned by the library)."""

    def __init__(self, L: int, E: int, C: int):
        self.L, self.E, self.C = L, E, C
        h = ctypes.c_void_p()
        _check(lib().ftmoe_lru_create(L, E, C, ctypes.byref(h)), "ftmoe_lru_create")
        self._h = h

    def reset(self, stream=None):
        _check(lib().ftmoe_lru_reset(self._h, _stream(stream)), "ftmoe_lru_reset")

    def slot_of_ptr(self) -> int:
        return lib().ftmoe_lru_slot_of(self._h)

    def slot_of(self, stream=None) -> torch.Tensor:
        """A copy of the slot_of table [L, E] (device)."""
        out = torch.empty(self.L, self.E, dtype=torch.int32, device="cuda")
        _check(lib().ftmoe_lru_copy_slot_of(self._h, _ptr(out), _stream(stream)), "ftmoe_lru_copy_slot_of")
        return out

    def step(self, layer, ids, hit, slot, evicted, counters, stream=None):
        if not isinstance(ids, torch.Tensor) or ids.dim() != 2:
            raise FtmoeError("topk_ids: expected a [B, k] tensor")
        _need(ids, "topk_ids", torch.int32)
        B, k = ids.shape
        n = min(B * k, self.E)
        _need(hit, "hit", torch.uint8, n)
        _need(slot, "slot", torch.int32, n)
        _need(evicted, "evicted_key", torch.int32, n)
        _need(counters, "counters", torch.int64, 2, optional=True)
        _check(lib().ftmoe_slot_lru(self._h, layer, _ptr(ids), B, k, _ptr(hit), _ptr(slot), _ptr(evicted),
                                    _ptr(counters), _stream(stream)), "ftmoe_slot_lru")

    def replay(self, trace, hit, slot, evicted, counters, stream=None):
        if not isinstance(trace, torch.Tensor) or trace.dim() != 4:
            raise FtmoeError("trace: expected a [steps, L, B, k] tensor")
        _need(trace, "trace", torch.int32)
        steps, L, B, k = trace.shape
        _need(hit, "hit", torch.uint8)
        _need(slot, "slot", torch.int32, hit.numel())
        _need(evicted, "evicted_key", torch.int32, hit.numel())
        _need(counters, "counters", torch.int64, 2, optional=True)
        if L != self.L:
            raise FtmoeError("trace layer count differs from the handle's")
        _check(lib().ftmoe_slot_lru_replay(self._h, _ptr(trace), steps, B, k, _ptr(hit), _ptr(slot), _ptr(evicted),
                                           hit.numel(), _ptr(counters), _stream(stream)), "ftmoe_slot_lru_replay")

    @property
    def capacity(self) -> int:
        return lib().ftmoe_lru_capacity(self._h)

    def resize(self, C_new, moves=None, n_moves=None, stream=None):
        """ftmoe_lru_resize: new capacity at a safe point; moves [min(C_old, C_new), 2] int32 and
        n_moves [1] int32 receive the (old slot, new slot) pairs of the kept keys."""
        _need(moves, "moves", torch.int32, 2 * min(self.C, C_new), optional=True)
        _need(n_moves, "n_moves", torch.int32, 1, optional=True)
        _check(lib().ftmoe_lru_resize(self._h, int(C_new), _ptr(moves), _ptr(n_moves), _stream(stream)),
               "ftmoe_lru_resize")
        self.C = int(C_new)

    def close(self):
        if getattr(self, "_h", None):
            lib().ftmoe_lru_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def copy_slots(dsc, src, dst, pairs, n_pairs=None, max_pairs=None, stream=None):
    """ftmoe_copy_slots: slot pairs[i][0] of the arena `src` -> slot pairs[i][1] of `dst`
    (WeightsStruct views; the source may be a pinned host pool)."""
    if max_pairs is None:
        max_pairs = pairs.numel() // 2 if isinstance(pairs, torch.Tensor) else 0
    _need(pairs, "pairs", torch.int32, 2 * max_pairs, optional=max_pairs == 0)
    _need(n_pairs, "n_pairs", torch.int32, 1, optional=True)
    _check(lib().ftmoe_copy_slots(ctypes.byref(dsc), ctypes.byref(src), ctypes.byref(dst), _ptr(pairs),
                                  _ptr(n_pairs), int(max_pairs), _stream(stream)), "ftmoe_copy_slots")


def qstar(m: int, link_gbs: float, host_gbs: float) -> float:
    return lib().ftmoe_qstar(int(m), float(link_gbs), float(host_gbs))


def qstar_fill_count(m: int, link_gbs: float, host_gbs: float) -> int:
    return lib().ftmoe_qstar_fill_count(int(m), float(link_gbs), float(host_gbs))


def miss_split(lru, layer, ids, hit, link_gbs, host_gbs, fill_override, slot_of_a, slot_of_b, fill_now, fill_later,
               counts, stream=None):
    """ftmoe_miss_split right after lru.step(layer, ids, hit, ...) on the same stream."""
    if not isinstance(ids, torch.Tensor) or ids.dim() != 2:
        raise FtmoeError("topk_ids: expected a [B, k] tensor")
    _need(ids, "topk_ids", torch.int32)
    B, k = ids.shape
    n = min(B * k, lru.E)
    _need(hit, "hit", torch.uint8, n)
    for t, name in ((slot_of_a, "slot_of_a"), (slot_of_b, "slot_of_b")):
        _need(t, name, torch.int32, lru.E)
    for t, name in ((fill_now, "fill_now"), (fill_later, "fill_later")):
        _need(t, name, torch.int32, 2 * n)
    _need(counts, "counts", torch.int32, 4)
    _check(lib().ftmoe_miss_split(lru._h, int(layer), _ptr(ids), B, k, _ptr(hit), float(link_gbs), float(host_gbs),
                                  int(fill_override), _ptr(slot_of_a), _ptr(slot_of_b), _ptr(fill_now),
                                  _ptr(fill_later), _ptr(counts), _stream(stream)), "ftmoe_miss_split")


def layer_host_workspace_size(dsc: LayerDesc, T: int) -> int:
    return lib().ftmoe_layer_host_workspace_size(ctypes.byref(dsc), T)


class LayerHostCall:
    """ftmoe_layer_forward_host bound once to a set of buffers: x_host and out_host are pinned
    host tensors [T, d] bf16; everything else is device memory.  The arguments are checked and
    packed here, once, so that each call is one ctypes call (the per-step cost of a serving loop)."""

    def __init__(self, dsc, wstruct, slot_of, x_host, w_router, bias, ids, topk_w, out_f32, out_host, ws,
                 stream=None):
        for t, name in ((x_host, "x_host"), (out_host, "out_host")):
            if not isinstance(t, torch.Tensor) or t.is_cuda or t.dim() != 2 or t.shape[1] != dsc.d:
                raise FtmoeError(f"{name}: expected a host [T, {dsc.d}] tensor")
            _need(t, name, torch.bfloat16)
            # the library copies T * d elements from (to) the address in row order, asynchronously
            if not t.is_contiguous():
                raise FtmoeError(f"{name}: expected a contiguous tensor")
            if not t.is_pinned():
                raise FtmoeError(f"{name}: expected pinned host memory (tensor.pin_memory())")
        T = x_host.shape[0]
        if out_host.shape[0] < T:
            raise FtmoeError("out_host: fewer rows than x_host")
        _need(slot_of, "slot_of", torch.int32, dsc.E, optional=True)
        _need(w_router, "w_router", torch.bfloat16, dsc.E * dsc.d)
        _need(bias, "logit_bias", torch.float32, dsc.E, optional=True)
        _need(ids, "topk_ids", torch.int32, T * dsc.k, optional=True)
        _need(topk_w, "topk_w", torch.float32, T * dsc.k, optional=True)
        _need(out_f32, "out_f32", torch.float32, T * dsc.d)
        _need(ws, "ws", nbytes=layer_host_workspace_size(dsc, T))
        self._keep = (dsc, wstruct, slot_of, x_host, w_router, bias, ids, topk_w, out_f32, out_host, ws)
        self._fn = lib().ftmoe_layer_forward_host
        self._args = (ctypes.byref(dsc), ctypes.byref(wstruct), _ptr(slot_of), x_host.data_ptr(), _ptr(w_router),
                      _ptr(bias), T, _ptr(ids), _ptr(topk_w), _ptr(out_f32), out_host.data_ptr(), _ptr(ws),
                      _ws_bytes(ws), _stream(stream))

    def __call__(self):
        st = self._fn(*self._args)
        if st:
            _check(st, "ftmoe_layer_forward_host")


class LayerHostGraph(LayerHostCall):
    """The same call recorded once as a CUDA graph (ftmoe_layer_graph_create) and replayed by
    each call (ftmoe_layer_graph_launch) on `stream`, or on the stream given to the call.
    `stream` is required: the capture needs a stream the caller created."""

    def __init__(self, *args, stream=None, **kw):
        if stream is None:
            raise FtmoeError("LayerHostGraph: a stream is required for the capture")
        super().__init__(*args, stream=stream, **kw)
        h = _P()
        _check(lib().ftmoe_layer_graph_create(*self._args, ctypes.byref(h)), "ftmoe_layer_graph_create")
        self._h = h
        self._launch = lib().ftmoe_layer_graph_launch
        self._st = _stream(stream)

    def __call__(self, stream=None):
        st = self._launch(self._h, self._st if stream is None else _stream(stream))
        if st:
            _check(st, "ftmoe_layer_graph_launch")

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().ftmoe_layer_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def layers_streamed(dsc, pool, arenas, xs, routers, biases, outs_f32, outs_bf16, ws, stream=None, copy_stream=None):
    """ftmoe_layers_streamed over L = len(routers) layers: `pool` and `arenas` are WeightsStruct
    views (the pool in pinned host memory, C >= L * E); xs[l] None (l > 0) chains the previous
    layer's bf16 output.  Returns nothing; outputs land in outs_f32 / outs_bf16."""
    L = len(routers)
    if not (len(xs) == len(outs_f32) == L) or (outs_bf16 is not None and len(outs_bf16) != L):
        raise FtmoeError("one input, router and output per layer")
    if xs[0] is None:
        raise FtmoeError("the first layer needs an input")
    T = _tokens(xs[0], dsc)
    for l in range(L):
        if xs[l] is not None and _tokens(xs[l], dsc) != T:
            raise FtmoeError("every layer input has T rows")
        if xs[l] is None and (outs_bf16 is None or outs_bf16[l - 1] is None):
            raise FtmoeError(f"layer {l} chains the previous bf16 output, which is missing")
        _need(routers[l], "w_router", torch.bfloat16, dsc.E * dsc.d)
        if biases is not None:
            _need(biases[l], "logit_bias", torch.float32, dsc.E, optional=True)
        _need(outs_f32[l], "out_f32", torch.float32, T * dsc.d)
        if outs_bf16 is not None:
            _need(outs_bf16[l], "out_bf16", torch.bfloat16, T * dsc.d, optional=True)
    _need(ws, "ws", nbytes=layer_workspace_size(dsc, T))
    arr = (WeightsStruct * len(arenas))(*arenas)
    vp = lambda ts: (ctypes.c_void_p * L)(*[_ptr(t) for t in ts])
    if copy_stream is None:
        raise FtmoeError("layers_streamed needs a copy stream")
    _check(lib().ftmoe_layers_streamed(ctypes.byref(dsc), L, ctypes.byref(pool), arr, len(arenas), vp(xs), vp(routers),
                                       None if biases is None else vp(biases), T, vp(outs_f32),
                                       None if outs_bf16 is None else vp(outs_bf16), _ptr(ws), _ws_bytes(ws),
                                       _stream(stream), _stream(copy_stream)), "ftmoe_layers_streamed")
