"""Data errors found on the device are reported through the library's device error word,
never by a trap.  The case here: a slot-table entry at or beyond the arena's slot count C.
That expert is skipped, exactly as if its entry were -1 (not resident), and the error word
reads 2 (bad slot).  Each call is compared with the same call whose entry is -1:
  * ftmoe_expert_ffn writing y, on every FFN path (BF16 streaming, the 4-bit decode
    kernels with and without the prepared layout, the NVFP4 and FP8 tensor-core paths):
    bit for bit, rows of the skipped expert left untouched;
  * ftmoe_layer_forward on each of its forms: bit for bit where the combine has a fixed
    order, within fp32 reassociation where it adds with atomics.
"""
import pytest
import torch

import synth

from gpu_helpers import ensure_built, expert_ffn, permute, route
from helpers import rel_l2
import sparse_moe_expert_sorted_b300 as ft

pytestmark = pytest.mark.gpu
BAD_SLOT = 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.int32), b.contiguous().view(torch.int32))


def _inputs(fmt, E, k, d, f, T, seed, prepared=True):
    W = synth.make_experts(fmt, E, d, f, seed, device="cuda")
    x = synth.make_x(T, d, seed, device="cuda")
    wr = synth.make_router(E, d, seed, device="cuda")
    dsc = ft.desc(E, k, d, f, fmt)
    if prepared:
        ft.prepare_weights(dsc, W)
    ids, _, _ = route(dsc, x, wr)
    e_bad = int(ids[0, 0])                                  # an expert token 0 uses
    bad = torch.arange(E, dtype=torch.int32, device="cuda")
    bad[e_bad] = E                                          # C = E slots: one past the last
    skip = bad.clone()
    skip[e_bad] = -1
    return dsc, W, x, wr, bad, skip


FFN_CASES = [
    # fmt, E, k, d, f, T, prepared
    (synth.BF16, 8, 2, 256, 512, 16, True),         # CUDA-core streaming
    (synth.NVFP4, 16, 8, 512, 256, 3, True),        # decode, prepared layout
    (synth.MXFP4, 32, 6, 256, 512, 13, True),
    (synth.NVFP4, 16, 8, 512, 256, 3, False),       # decode, canonical arena
    (synth.NVFP4, 16, 8, 512, 256, 300, True),      # tcgen05, NVFP4 activations
    (synth.FP8_B128, 8, 2, 768, 384, 300, True),    # tcgen05, FP8 activations
]


@pytest.mark.parametrize("fmt,E,k,d,f,T,prepared", FFN_CASES)
def test_expert_ffn_skips_a_slot_beyond_the_arena(fmt, E, k, d, f, T, prepared):
    dsc, W, x, wr, bad, skip = _inputs(fmt, E, k, d, f, T, seed=7 * T + E, prepared=prepared)
    ids, _, _ = route(dsc, x, wr)
    off, sp, _ = permute(dsc, ids)
    ft.get_device_error()                                   # clear
    y_bad = expert_ffn(dsc, W, bad, x, off, sp)
    assert ft.get_device_error() == BAD_SLOT
    y_skip = expert_ffn(dsc, W, skip, x, off, sp)
    assert ft.get_device_error() == 0
    assert _same_bits(y_bad, y_skip)
    # the skipped expert's rows are untouched (NaN-filled by the helper), the rest are written
    e_bad = int(ids[0, 0])
    o = off.cpu().numpy()
    rows = slice(int(o[e_bad]), int(o[e_bad + 1]))
    assert rows.stop > rows.start
    assert torch.isnan(y_bad[rows]).all()
    assert torch.isfinite(y_bad[: rows.start]).all() and torch.isfinite(y_bad[rows.stop:]).all()


def _layer(dsc, W, slot, x, wr):
    T = x.shape[0]
    ids = torch.empty(T, dsc.k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, dsc.k, dtype=torch.float32, device="cuda")
    of = torch.full((T, dsc.d), float("nan"), dtype=torch.float32, device="cuda")
    ob = torch.empty(T, dsc.d, dtype=torch.bfloat16, device="cuda")
    ws = ft.workspace(ft.layer_workspace_size(dsc, T))
    ft.layer_forward(dsc, ft.weights_struct(W), slot, x, wr, None, ids, w, of, ob, ws)
    return ids, w, of, ob


LAYER_CASES = [
    # fmt, E, k, d, f, T, the form ftmoe_layer_path reports
    (synth.BF16, 8, 2, 256, 512, 16, 0),            # separate steps: y, then the combine call
    (synth.NVFP4, 16, 8, 512, 256, 12, 0),          # separate steps: decode kernel, fused combine
    (synth.MXFP4, 32, 6, 256, 512, 5, 1),           # one kernel, merge form
    (synth.NVFP4, 16, 8, 512, 256, 1, 2),           # one kernel, slice form
    (synth.NVFP4, 24, 4, 256, 384, 6, 2),
]


@pytest.mark.parametrize("fmt,E,k,d,f,T,form", LAYER_CASES)
def test_layer_forward_skips_a_slot_beyond_the_arena(fmt, E, k, d, f, T, form):
    dsc, W, x, wr, bad, skip = _inputs(fmt, E, k, d, f, T, seed=11 * T + E)
    assert ft.layer_path(dsc, ft.weights_struct(W), T) == form
    ft.get_device_error()                                   # clear
    ids_b, w_b, of_b, ob_b = _layer(dsc, W, bad, x, wr)
    assert ft.get_device_error() == BAD_SLOT
    ids_s, w_s, of_s, ob_s = _layer(dsc, W, skip, x, wr)
    assert ft.get_device_error() == 0
    assert torch.equal(ids_b, ids_s) and _same_bits(w_b, w_s)
    assert torch.isfinite(of_b).all()
    fused_combine = form == 0 and fmt != synth.BF16          # float atomics: the order of adds varies
    if fused_combine:
        assert rel_l2(of_b.cpu().numpy(), of_s.cpu().numpy()) <= 1e-6
    else:
        assert _same_bits(of_b, of_s)
        assert torch.equal(ob_b.view(torch.int16), ob_s.view(torch.int16))
