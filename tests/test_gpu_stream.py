"""GPU parity of ftmoe_layers_streamed: layers whose experts stream from a pinned host pool
through one or two device arenas (full-layer double buffering during prefill; asapai.co.kr,
"Running 753B GLM-5.2 on a single workstation GPU", section "Abandoning fixed offloading in
favor of measured bandwidth").

  * Each layer's output equals ftmoe_layer_forward on a device arena holding that layer's
    experts (up to the fused combine's fp32 reassociation), with one arena and with two.
  * Layers with their own inputs match the oracle (the prefill mirror on the tensor-core
    paths, weight-only on the decode path) within 5e-3 relative L2 per sampled token.
  * A chained layer (input = the previous layer's bf16 output) equals the device call on
    that same input.
"""
import numpy as np
import pytest
import torch

import synth
import sparse_moe_expert_sorted_b300 as ft
from oracle import ffn as OF
from oracle.route import route as oracle_route

from gpu_helpers import ensure_built
from helpers import bf16_bits, rel_l2, weights_to_numpy

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _pinned(W):
    pin = lambda t: None if t is None else t.cpu().contiguous().pin_memory()
    return synth.ExpertWeights(W.fmt, W.d, W.f, pin(W.gate), pin(W.up), pin(W.down), pin(W.gate_s), pin(W.up_s),
                               pin(W.down_s), pin(W.glob))


def _slots(W, lo, hi, device):
    cut = lambda t: None if t is None else t[lo:hi].contiguous().to(device)
    return synth.ExpertWeights(W.fmt, W.d, W.f, cut(W.gate), cut(W.up), cut(W.down), cut(W.gate_s), cut(W.up_s),
                               cut(W.down_s), cut(W.glob))


def _empty_arena(W, C):
    z = lambda t: None if t is None else torch.zeros((C,) + tuple(t.shape[1:]), dtype=t.dtype, device="cuda")
    return synth.ExpertWeights(W.fmt, W.d, W.f, z(W.gate), z(W.up), z(W.down), z(W.gate_s), z(W.up_s), z(W.down_s),
                               z(W.glob))


@pytest.mark.parametrize("fmt,T,L", [(synth.NVFP4, 300, 3), (synth.FP8_B128, 260, 2), (synth.NVFP4, 2, 3)])
def test_streamed_layers_match_resident_calls_and_the_oracle(fmt, T, L):
    E, k, d, f = 16, 4, 256, 256
    dsc = ft.desc(E, k, d, f, fmt)
    pool = _pinned(synth.make_experts(fmt, L * E, d, f, 90 + fmt))
    ft.prepare_weights(dsc, pool)
    arenas = []
    for _ in range(2):
        A = _empty_arena(pool, E)
        ft.prepare_weights(dsc, A)
        arenas.append(A)
    routers = [synth.make_router(E, d, 95 + l).cuda() for l in range(L)]
    xs = [synth.make_x(T, d, 97 + l).cuda() for l in range(L)]
    xs_in = list(xs)
    xs_in[L - 1] = None                                   # the last layer chains the previous output
    ws = ft.workspace(ft.layer_workspace_size(dsc, T))
    aq = {0: None, 1: "nvfp4", 2: "fp8"}[ft.expert_ffn_path(dsc, T)]
    comp, copy = torch.cuda.Stream(), torch.cuda.Stream()
    results = {}
    for n_arenas in (2, 1):
        of = [torch.full((T, d), float("nan"), device="cuda") for _ in range(L)]
        ob = [torch.empty(T, d, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
        ft.layers_streamed(dsc, ft.weights_struct(pool), [ft.weights_struct(a) for a in arenas[:n_arenas]], xs_in,
                           routers, None, of, ob, ws, stream=comp, copy_stream=copy)
        torch.cuda.synchronize()
        results[n_arenas] = (of, ob)
    Wn = weights_to_numpy(pool)
    rows = sorted(set(np.random.default_rng(T).choice(T, min(T, 12), replace=False).tolist()))
    for l in range(L):
        # the same layer resident on the device
        Wl = _slots(pool, l * E, (l + 1) * E, "cuda")
        ft.prepare_weights(dsc, Wl)
        x_l = xs[l] if l < L - 1 else results[2][1][l - 1]
        ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
        w = torch.empty(T, k, dtype=torch.float32, device="cuda")
        ref = torch.empty(T, d, device="cuda")
        ft.layer_forward(dsc, ft.weights_struct(Wl), None, x_l, routers[l], None, ids, w, ref, None, ws)
        torch.cuda.synchronize()
        for n_arenas in (2, 1):
            got = results[n_arenas][0][l]
            assert rel_l2(got.cpu().numpy(), ref.cpu().numpy()) < 1e-6, (l, n_arenas)
        if l < L - 1:                                      # the oracle, on the layer's own input
            xb, wb = bf16_bits(xs[l].cpu()), bf16_bits(routers[l].cpu())
            ids_r, w_r, _ = oracle_route(xb, wb, None, k, 1)
            assert np.array_equal(ids.cpu().numpy(), ids_r)
            want = OF.layer_tokens(Wn, l * E + np.arange(E), xb, ids_r, w_r, rows, act_quant=aq)
            got = results[2][0][l].cpu().numpy()[rows]
            for i in range(len(rows)):
                assert np.linalg.norm(got[i] - want[i]) / np.linalg.norm(want[i]) < TOL, (l, rows[i])
    assert ft.get_device_error() == 0
