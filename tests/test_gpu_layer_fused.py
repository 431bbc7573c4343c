"""ftmoe_layer_forward with few tokens and a 4-bit format runs router, sort, expert
FFN and merge in one kernel (ftmoe_layer_path 1), or the slice form that applies the
down projection per gate/up item (path 2: d <= 2048, one token or NVFP4).  Path 1 repeats the
separate calls' arithmetic (route -> permute -> expert_ffn -> combine) and must equal
them bit for bit; path 2 regroups the down projection's sums (fp32 reassociation,
within 1e-5 of the separate calls).  Both match the oracle within the layer's
tolerance (5e-3 relative L2):
  * ids bit-exact with the oracle, weights and outputs within tolerance;
  * T = 1 .. 8, NVFP4 and MXFP4, bias and renorm;
  * skipped experts (slot -1), including a token none of whose experts is
    resident (its output row is zero);
  * repeated calls on one workspace (the kernel's counters start at zero each call), and 200
    back-to-back slice-form calls that must agree bit for bit (its sums have a fixed order);
  * the full decode layer shape (128 experts, top-8, d 2048, ffn 768).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import ffn as OF

from gpu_helpers import combine, ensure_built, expert_ffn, permute, route
from helpers import bf16_bits, rel_l2, weights_to_numpy
import sparse_moe_expert_sorted_b300 as ft

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _layer(dsc, W, slot, x, wr, bias, ws=None, want_bf16=True):
    T = x.shape[0]
    ids = torch.full((T, dsc.k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, dsc.k), float("nan"), dtype=torch.float32, device="cuda")
    of = torch.full((T, dsc.d), float("nan"), dtype=torch.float32, device="cuda")
    ob = torch.empty(T, dsc.d, dtype=torch.bfloat16, device="cuda") if want_bf16 else None
    if ws is None:
        ws = ft.workspace(ft.layer_workspace_size(dsc, T))
    ft.layer_forward(dsc, ft.weights_struct(W), slot, x, wr, bias, ids, w, of, ob, ws)
    return ids, w, of, ob


def _expected_path(fmt, d, T):
    return 2 if d <= 2048 and (T == 1 or fmt == synth.NVFP4) else 1


def _same(path, a, b):
    """Path 1 equals the separate calls bit for bit; path 2 up to fp32 reassociation."""
    if path == 1:
        return torch.equal(a, b)
    return rel_l2(a.float().cpu().numpy(), b.float().cpu().numpy()) < 1e-5


def _separate(dsc, W, slot, x, wr, bias):
    T = x.shape[0]
    ids, w, _ = route(dsc, x, wr, bias)
    off, sp, pp = permute(dsc, ids)
    y = expert_ffn(dsc, W, slot, x, off, sp)
    of, ob = combine(dsc, T, y, pp, w, ids, slot)
    return ids, w, of, ob


CASES = [
    # fmt, E, k, d, f, T, renorm, zipf
    (synth.NVFP4, 16, 8, 512, 256, 1, 0, 0.0),
    (synth.NVFP4, 16, 8, 512, 256, 3, 1, 1.1),
    (synth.NVFP4, 24, 4, 256, 384, 8, 0, 1.1),
    (synth.MXFP4, 32, 6, 512, 256, 1, 1, 1.0),
    (synth.MXFP4, 32, 6, 256, 512, 5, 0, 0.0),
    (synth.NVFP4, 300, 2, 256, 128, 2, 0, 0.0),   # more experts than SMs: two router rows per CTA
    (synth.NVFP4, 1024, 4, 256, 128, 1, 1, 1.1),  # router rows too many for a cluster's share: the grid form
]


@pytest.mark.parametrize("fmt,E,k,d,f,T,renorm,zipf", CASES)
def test_fused_layer_matches_separate_calls_and_oracle(fmt, E, k, d, f, T, renorm, zipf):
    seed = 31 * T + E
    W = synth.make_experts(fmt, E, d, f, seed, device="cuda")
    x = synth.make_x(T, d, seed, device="cuda")
    wr = synth.make_router(E, d, seed, device="cuda")
    bias_np = synth.make_zipf_bias(E, zipf, seed) if zipf else None
    bias = torch.from_numpy(bias_np).cuda() if zipf else None
    dsc = ft.desc(E, k, d, f, fmt, renorm)
    ft.prepare_weights(dsc, W)
    slot_np = ((np.arange(E) * 7 + 1) % E).astype(np.int32)
    if np.gcd(7, E) != 1:
        slot_np = np.arange(E, dtype=np.int32)[::-1].copy()
    slot = torch.from_numpy(slot_np).cuda()
    path = ft.layer_path(dsc, ft.weights_struct(W), T)
    assert path == _expected_path(fmt, d, T)
    ids, w, of, ob = _layer(dsc, W, slot, x, wr, bias)
    ids_s, w_s, of_s, ob_s = _separate(dsc, W, slot, x, wr, bias)
    assert torch.equal(ids, ids_s)
    assert torch.equal(w, w_s)
    diff = (of - of_s).abs()
    assert _same(path, of, of_s), (f"path {path}: rel L2 {rel_l2(of.cpu().numpy(), of_s.cpu().numpy()):.3e}, "
                                   f"max abs {float(diff.max()):.3e} at {divmod(int(diff.argmax()), of.shape[1])}")
    if path == 1:
        assert torch.equal(ob, ob_s)
    ref = OF.layer(weights_to_numpy(W.to("cpu")), slot_np, bf16_bits(x.cpu()), bf16_bits(wr.cpu()), bias_np, k,
                   renorm)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert rel_l2(w.cpu().numpy(), ref["w"]) < 1e-5
    assert rel_l2(of.cpu().numpy(), ref["out"]) < TOL
    assert rel_l2(ob.float().cpu().numpy(), ref["out"]) < TOL
    assert ft.get_device_error() == 0


def test_skipped_experts_and_a_token_with_none_resident():
    fmt, E, k, d, f, T = synth.NVFP4, 16, 2, 256, 256, 4
    W = synth.make_experts(fmt, E, d, f, 5, device="cuda")
    x = synth.make_x(T, d, 5, device="cuda")
    wr = synth.make_router(E, d, 5, device="cuda")
    dsc = ft.desc(E, k, d, f, fmt)
    ft.prepare_weights(dsc, W)
    ref_full = OF.layer(weights_to_numpy(W.to("cpu")), np.arange(E, dtype=np.int32), bf16_bits(x.cpu()),
                        bf16_bits(wr.cpu()), None, k, 1)
    ids0 = ref_full["ids"]
    # token 0 loses both of its experts; every other expert stays resident unless token 0 uses it
    slot_np = np.arange(E, dtype=np.int32)
    slot_np[ids0[0]] = -1
    slot = torch.from_numpy(slot_np).cuda()
    path = ft.layer_path(dsc, ft.weights_struct(W), T)
    assert path == _expected_path(fmt, d, T)
    ids, w, of, ob = _layer(dsc, W, slot, x, wr, None)
    ref = OF.layer(weights_to_numpy(W.to("cpu")), slot_np, bf16_bits(x.cpu()), bf16_bits(wr.cpu()), None, k, 1)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert torch.count_nonzero(of[0]).item() == 0
    assert torch.count_nonzero(ob[0].float()).item() == 0
    assert rel_l2(of.cpu().numpy(), ref["out"]) < TOL
    _, _, of_s, _ = _separate(dsc, W, slot, x, wr, None)
    assert _same(path, of, of_s)
    # the two halves of an exact split merge to the full output
    slot_b = np.where(slot_np < 0, np.arange(E), -1).astype(np.int32)
    _, _, of_b, _ = _layer(dsc, W, torch.from_numpy(slot_b).cuda(), x, wr, None)
    _, _, of_full, _ = _layer(dsc, W, torch.arange(E, dtype=torch.int32, device="cuda"), x, wr, None)
    assert rel_l2((of + of_b).cpu().numpy(), of_full.cpu().numpy()) < 1e-6
    assert ft.get_device_error() == 0


def test_repeated_calls_share_one_workspace():
    fmt, E, k, d, f = synth.NVFP4, 32, 4, 512, 256
    W = synth.make_experts(fmt, E, d, f, 8, device="cuda")
    wr = synth.make_router(E, d, 8, device="cuda")
    dsc = ft.desc(E, k, d, f, fmt)
    ft.prepare_weights(dsc, W)
    slot = torch.arange(E, dtype=torch.int32, device="cuda")
    for T in (2, 7):
        ws = ft.workspace(ft.layer_workspace_size(dsc, T))
        outs = []
        for rep in range(4):
            x = synth.make_x(T, d, 100 + rep, device="cuda")
            path = ft.layer_path(dsc, ft.weights_struct(W), T)
            ids, w, of, ob = _layer(dsc, W, slot, x, wr, None, ws=ws, want_bf16=(rep % 2 == 0))
            _, _, of_s, _ = _separate(dsc, W, slot, x, wr, None)
            assert _same(path, of, of_s)
            outs.append(of)
        assert not torch.equal(outs[0], outs[1])
    assert ft.get_device_error() == 0


def test_full_decode_layer_shape():
    L = synth.DECODE.layer
    dsc = ft.desc(L.E, L.k, L.d, L.f, L.fmt, L.renorm)
    W = synth.make_experts(L.fmt, L.E, L.d, L.f, 11, device="cuda")
    ft.prepare_weights(dsc, W)
    wr = synth.make_router(L.E, L.d, 11, device="cuda")
    bias_np = synth.make_zipf_bias(L.E, synth.DECODE.zipf_s, 11)
    bias = torch.from_numpy(bias_np).cuda()
    slot = torch.arange(L.E, dtype=torch.int32, device="cuda")
    for T in (1, 4):
        path = ft.layer_path(dsc, ft.weights_struct(W), T)
        assert path == 2
        x = synth.make_x(T, L.d, 12 + T, device="cuda")
        ids, w, of, ob = _layer(dsc, W, slot, x, wr, bias)
        _, _, of_s, ob_s = _separate(dsc, W, slot, x, wr, bias)
        assert _same(path, of, of_s)
        ref = OF.layer(weights_to_numpy(W.to("cpu")), np.arange(L.E, dtype=np.int32), bf16_bits(x.cpu()),
                       bf16_bits(wr.cpu()), bias_np, L.k, L.renorm)
        assert np.array_equal(ids.cpu().numpy(), ref["ids"])
        assert rel_l2(of.cpu().numpy(), ref["out"]) < TOL
    assert ft.get_device_error() == 0


def test_layer_path_query():
    L = synth.DECODE.layer
    dsc = ft.desc(L.E, L.k, L.d, L.f, L.fmt, L.renorm)
    W = synth.make_experts(L.fmt, 4, L.d, L.f, 1, device="cuda")
    assert ft.layer_path(dsc, ft.weights_struct(W), 1) == 0       # not prepared: separate steps
    ft.prepare_weights(dsc, W)
    assert ft.layer_path(dsc, ft.weights_struct(W), 1) == 2       # the slice form
    assert ft.layer_path(dsc, ft.weights_struct(W), 2) == 2
    assert ft.layer_path(dsc, ft.weights_struct(W), 8) == 2
    assert ft.layer_path(dsc, ft.weights_struct(W), 9) == 0       # more tokens: separate steps
    assert ft.layer_path(dsc, ft.weights_struct(W), 0) == -1


@pytest.mark.parametrize("fmt", [synth.NVFP4, synth.MXFP4])
def test_slice_form_skipped_experts_and_repeated_calls(fmt):
    """One token, the slice form: a partly and a fully non-resident token, and calls that
    reuse one workspace (its grid-sync word and partial buffer)."""
    E, k, d, f = 24, 6, 512, 384
    W = synth.make_experts(fmt, E, d, f, 21, device="cuda")
    wr = synth.make_router(E, d, 21, device="cuda")
    dsc = ft.desc(E, k, d, f, fmt, 1)
    ft.prepare_weights(dsc, W)
    assert ft.layer_path(dsc, ft.weights_struct(W), 1) == 2
    ws = ft.workspace(ft.layer_workspace_size(dsc, 1))
    for rep_ in range(3):
        x = synth.make_x(1, d, 40 + rep_, device="cuda")
        ref_full = OF.layer(weights_to_numpy(W), np.arange(E, dtype=np.int32), bf16_bits(x.cpu()),
                            bf16_bits(wr.cpu()), None, k, 1)
        slot_np = np.arange(E, dtype=np.int32)
        slot_np[ref_full["ids"][0][::2]] = -1                  # half of the token's experts are not resident
        for sl in (slot_np, np.full(E, -1, np.int32)):
            slot = torch.from_numpy(sl).cuda()
            ids, w, of, ob = _layer(dsc, W, slot, x, wr, None, ws=ws)
            ref = OF.layer(weights_to_numpy(W), sl, bf16_bits(x.cpu()), bf16_bits(wr.cpu()), None, k, 1)
            assert np.array_equal(ids.cpu().numpy(), ref["ids"])
            if (sl < 0).all():
                assert torch.count_nonzero(of).item() == 0 and torch.count_nonzero(ob.float()).item() == 0
            else:
                assert rel_l2(of.cpu().numpy(), ref["out"]) < TOL
                _, _, of_s, _ = _separate(dsc, W, slot, x, wr, None)
                assert _same(2, of, of_s)
    assert ft.get_device_error() == 0


@pytest.mark.parametrize("fmt,T", [(synth.NVFP4, 1), (synth.MXFP4, 3)])
def test_host_buffer_call_equals_the_device_call(fmt, T):
    """ftmoe_layer_forward_host (x from pinned host memory, bf16 output back to it) gives the
    device call's outputs bit for bit, twice in a row on one workspace."""
    E, k, d, f = 32, 4, 512, 256
    W = synth.make_experts(fmt, E, d, f, 77, device="cuda")
    dsc = ft.desc(E, k, d, f, fmt)
    ft.prepare_weights(dsc, W)
    wr = synth.make_router(E, d, 77, device="cuda")
    st = ft.weights_struct(W)
    ws = ft.workspace(ft.layer_host_workspace_size(dsc, T))
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    of = torch.empty(T, d, dtype=torch.float32, device="cuda")
    for seed in (5, 6):
        x = synth.make_x(T, d, seed)
        xh = x.pin_memory()
        oh = torch.full((T, d), float("nan"), dtype=torch.bfloat16).pin_memory()
        call = ft.LayerHostCall(dsc, st, None, xh, wr, None, ids, w, of, oh, ws)
        call()
        torch.cuda.synchronize()
        ids_d, w_d, of_d, ob_d = _layer(dsc, W, None, x.cuda(), wr, None)
        assert torch.equal(ids, ids_d) and torch.equal(w, w_d)
        assert torch.equal(of, of_d)
        assert torch.equal(oh, ob_d.cpu())
    assert ft.get_device_error() == 0


@pytest.mark.parametrize("fmt,E,k,d,f,T", [(synth.NVFP4, 32, 4, 512, 256, 1),     # slice form
                                           (synth.MXFP4, 32, 4, 512, 256, 3),     # one kernel, merge form
                                           (synth.NVFP4, 32, 4, 512, 256, 16),    # separate steps
                                           (synth.NVFP4, 32, 4, 512, 256, 512)])  # tensor-core router and GEMMs
def test_graph_replay_equals_the_host_call(fmt, E, k, d, f, T):
    """ftmoe_layer_graph_create records one host-buffer layer call; each replay reads x_host as
    it is then.  Two replays with different tokens refilled into the same pinned buffer give
    the direct call's outputs: bit for bit where the layer call is deterministic (one kernel,
    T <= 8), within fp32 reassociation where a fused combine adds in arrival order (T > 8).
    The one-token replay also matches the oracle."""
    W = synth.make_experts(fmt, E, d, f, 91, device="cuda")
    dsc = ft.desc(E, k, d, f, fmt)
    ft.prepare_weights(dsc, W)
    wr = synth.make_router(E, d, 91, device="cuda")
    st = ft.weights_struct(W)
    stream = torch.cuda.Stream()
    bufs = []
    for _ in range(2):   # [0]: the graph's buffers, [1]: the direct call's
        bufs.append(dict(ws=ft.workspace(ft.layer_host_workspace_size(dsc, T)),
                         ids=torch.empty(T, k, dtype=torch.int32, device="cuda"),
                         w=torch.empty(T, k, dtype=torch.float32, device="cuda"),
                         of=torch.empty(T, d, dtype=torch.float32, device="cuda"),
                         xh=torch.empty(T, d, dtype=torch.bfloat16).pin_memory(),
                         oh=torch.full((T, d), float("nan"), dtype=torch.bfloat16).pin_memory()))
    g, h = bufs

    def args(b):
        return (dsc, st, None, b["xh"], wr, None, b["ids"], b["w"], b["of"], b["oh"], b["ws"])

    direct = ft.LayerHostCall(*args(h), stream)
    graph = ft.LayerHostGraph(*args(g), stream=stream)
    try:
        for seed in (12, 13):
            x = synth.make_x(T, d, seed)
            g["xh"].copy_(x)
            h["xh"].copy_(x)
            graph()
            direct()
            stream.synchronize()
            assert torch.equal(g["ids"], h["ids"]) and torch.equal(g["w"], h["w"])
            if T > 8:   # the fused combine adds in arrival order
                assert rel_l2(g["of"].cpu().numpy(), h["of"].cpu().numpy()) <= 1e-6
                assert rel_l2(g["oh"].float().numpy(), h["oh"].float().numpy()) <= 1e-4
            else:
                assert torch.equal(g["of"], h["of"]) and torch.equal(g["oh"], h["oh"])
            if T == 1:
                ref = OF.layer(weights_to_numpy(W.to("cpu")), np.arange(E, dtype=np.int32), bf16_bits(x),
                               bf16_bits(wr.cpu()), None, k, 1)
                assert np.array_equal(g["ids"].cpu().numpy(), ref["ids"])
                assert rel_l2(g["oh"].float().numpy(), ref["out"]) < TOL
    finally:
        graph.close()
    assert ft.get_device_error() == 0


@pytest.mark.parametrize("E,k,d,f,T", [(24, 4, 256, 384, 8), (128, 8, 2048, 768, 8), (128, 8, 2048, 768, 5)])
def test_slice_form_is_deterministic_over_many_calls(E, k, d, f, T):
    """The slice form sums every output in a fixed order, so back-to-back calls on the same
    inputs agree bit for bit.  These shapes put the cluster form's partial output [T][d] (fp32,
    written over the ring at the end) across stage 0's down slice, which other consumer warps
    read until their last item is done: a write before every warp is done would show up here as
    a call that differs from the first."""
    fmt = synth.NVFP4
    seed = 7 * T + d
    W = synth.make_experts(fmt, E, d, f, seed, device="cuda")
    x = synth.make_x(T, d, seed, device="cuda")
    wr = synth.make_router(E, d, seed, device="cuda")
    dsc = ft.desc(E, k, d, f, fmt)
    ft.prepare_weights(dsc, W)
    slot = torch.arange(E, dtype=torch.int32, device="cuda")
    assert ft.layer_path(dsc, ft.weights_struct(W), T) == 2
    ws = ft.workspace(ft.layer_workspace_size(dsc, T))
    reps = 200
    outs = torch.full((reps, T, d), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    st = ft.weights_struct(W)
    for r in range(reps):   # back to back on one stream, no host synchronisation between calls
        ft.layer_forward(dsc, st, slot, x, wr, None, ids, w, outs[r], None, ws)
    torch.cuda.synchronize()
    same = np.array([torch.equal(outs[r], outs[0]) for r in range(reps)])
    assert same.all(), f"{int((~same).sum())} of {reps} calls differ from the first (first at {int(np.argmin(same))})"
    _, _, of_s, _ = _separate(dsc, W, slot, x, wr, None)
    assert _same(2, outs[0], of_s)
    ref = OF.layer(weights_to_numpy(W.to("cpu")), np.arange(E, dtype=np.int32), bf16_bits(x.cpu()),
                   bf16_bits(wr.cpu()), None, k, 1)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert rel_l2(outs[0].cpu().numpy(), ref["out"]) < TOL
    assert ft.get_device_error() == 0
