"""Thin drivers of the C ABI for the GPU tests: allocate outputs and workspaces,
call the library, return torch tensors.  No layer arithmetic here."""
import torch

import sparse_moe_expert_sorted_b300 as ft
from sparse_moe_expert_sorted_b300 import build as ftbuild

_built = False


def ensure_built():
    global _built
    if not _built:
        ftbuild.build()
        ft.lib()
        _built = True


def route(dsc, x, wr, bias=None, want_logits=True):
    T = x.shape[0]
    ids = torch.empty(T, dsc.k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, dsc.k, dtype=torch.float32, device="cuda")
    logits = torch.empty(T, dsc.E, dtype=torch.float32, device="cuda") if want_logits else None
    ws = ft.workspace(ft.route_workspace_size(dsc, T))
    ft.route(dsc, x, wr, bias, ids, w, logits, ws)
    return ids, w, logits


def permute(dsc, ids):
    T = ids.shape[0]
    P = T * dsc.k
    off = torch.empty(dsc.E + 1, dtype=torch.int32, device="cuda")
    sp = torch.empty(P, dtype=torch.int32, device="cuda")
    pp = torch.empty(P, dtype=torch.int32, device="cuda")
    ws = ft.workspace(ft.permute_workspace_size(dsc, T))
    ft.permute(dsc, ids, off, sp, pp, ws)
    return off, sp, pp


def expert_ffn(dsc, W, slot_of, x, off, sp, topk_w=None, out=None):
    T = x.shape[0]
    P = T * dsc.k
    ws = ft.workspace(ft.expert_ffn_workspace_size(dsc, T))
    if topk_w is None:
        y = torch.full((P, dsc.d), float("nan"), dtype=torch.float32, device="cuda")
    else:
        y = out if out is not None else torch.zeros(T, dsc.d, dtype=torch.float32, device="cuda")
    ft.expert_ffn(dsc, ft.weights_struct(W), slot_of, x, off, sp, topk_w, y, ws)
    return y


def combine(dsc, T, y, pp, w, ids, slot_of=None, partial_b=None):
    of = torch.empty(T, dsc.d, dtype=torch.float32, device="cuda")
    ob = torch.empty(T, dsc.d, dtype=torch.bfloat16, device="cuda")
    ft.combine(dsc, T, y, pp, w, ids, slot_of, partial_b, of, ob)
    return of, ob


def layer_forward(dsc, W, slot_of, x, wr, bias=None):
    T = x.shape[0]
    ids = torch.empty(T, dsc.k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, dsc.k, dtype=torch.float32, device="cuda")
    of = torch.empty(T, dsc.d, dtype=torch.float32, device="cuda")
    ob = torch.empty(T, dsc.d, dtype=torch.bfloat16, device="cuda")
    ws = ft.workspace(ft.layer_workspace_size(dsc, T))
    ft.layer_forward(dsc, ft.weights_struct(W), slot_of, x, wr, bias, ids, w, of, ob, ws)
    return ids, w, of, ob
