"""Parity of ftmoe_expert_ffn, ftmoe_combine and ftmoe_layer_forward with the
oracle: max relative L2 error 5e-3 (the layer's stated tolerance), on
shrunken copies of the five workloads and on edge cases:
  * every weight format;
  * slot indirection;
  * skipped experts;
  * the exact split (A + B = full);
  * the fused combine;
  * T = 1;
  * ragged token tiles.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import ffn as OF
from oracle import permute as OP
from oracle import route as OR

from gpu_helpers import combine, ensure_built, expert_ffn, layer_forward, permute, route
from helpers import bf16_bits, rel_l2, weights_to_numpy
import sparse_moe_expert_sorted_b300 as ft

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _setup(fmt, E, k, d, f, T, seed, C=None, zipf=0.0):
    C = C or E
    W = synth.make_experts(fmt, C, d, f, seed)
    x = synth.make_x(T, d, seed)
    wr = synth.make_router(E, d, seed)
    bias = synth.make_zipf_bias(E, zipf, seed) if zipf else None
    return W, x, wr, bias


CASES = [
    # fmt, E, k, d, f, T
    (synth.BF16, 8, 2, 256, 512, 16),        # the tiny workload itself
    (synth.NVFP4, 16, 8, 512, 256, 1),       # decode-like
    (synth.NVFP4, 16, 8, 512, 256, 16),
    (synth.MXFP4, 32, 6, 512, 256, 64),      # stack-like
    (synth.MXFP4, 32, 6, 256, 512, 13),      # ragged tiles
    (synth.FP8_B128, 16, 6, 256, 256, 40),   # prefill-split-like
    (synth.NVFP4, 16, 8, 512, 256, 300),     # many tokens per expert
]


@pytest.mark.parametrize("fmt,E,k,d,f,T", CASES)
def test_ffn_and_combine_match_oracle(fmt, E, k, d, f, T):
    W, x, wr, bias = _setup(fmt, E, k, d, f, T, seed=T + E)
    dsc = ft.desc(E, k, d, f, fmt)
    Wd = W.to("cuda")
    # slot indirection: expert e lives in slot (e * 5 + 3) % E
    slot_np = ((np.arange(E) * 5 + 3) % E).astype(np.int32)
    if E % 5 == 0:
        slot_np = np.arange(E, dtype=np.int32)[::-1].copy()
    ft.prepare_weights(dsc, Wd)
    aq = {0: None, 1: "nvfp4"}[ft.expert_ffn_path(dsc, T)]   # the oracle mirrors the path's quantiser
    ref = OF.layer(weights_to_numpy(W), slot_np, bf16_bits(x), bf16_bits(wr), bias, k, 1, act_quant=aq)
    xd = x.cuda()
    ids, w, _ = route(dsc, xd, wr.cuda(), None if bias is None else torch.from_numpy(bias).cuda())
    off, sp, pp = permute(dsc, ids)
    slot = torch.from_numpy(slot_np).cuda()
    y = expert_ffn(dsc, Wd, slot, xd, off, sp)
    err_y = rel_l2(y.cpu().numpy(), ref["y"])
    assert err_y < TOL, err_y
    of, ob = combine(dsc, T, y, pp, w, ids, slot)
    err = rel_l2(of.cpu().numpy(), ref["out"])
    assert err < TOL, err
    assert rel_l2(ob.float().cpu().numpy(), ref["out"]) < TOL
    # fused combine: w * y added into out
    out = expert_ffn(dsc, Wd, slot, xd, off, sp, topk_w=w)
    assert rel_l2(out.cpu().numpy(), ref["out"]) < TOL
    # whole layer in one call
    ids2, w2, of2, ob2 = layer_forward(dsc, Wd, slot, xd, wr.cuda(), None if bias is None else torch.from_numpy(bias).cuda())
    assert np.array_equal(ids2.cpu().numpy(), ref["ids"])
    assert rel_l2(of2.cpu().numpy(), ref["out"]) < TOL


@pytest.mark.parametrize("fmt", [synth.NVFP4, synth.FP8_B128, synth.BF16])
def test_exact_split_merges_to_the_full_output(fmt):
    E, k, d, f, T = 16, 6, 256, 256, 48
    W, x, wr, _ = _setup(fmt, E, k, d, f, T, seed=3)
    dsc = ft.desc(E, k, d, f, fmt)
    Wd = W.to("cuda")
    xd = x.cuda()
    ids, w, _ = route(dsc, xd, wr.cuda())
    off, sp, pp = permute(dsc, ids)
    full_slot = torch.arange(E, dtype=torch.int32, device="cuda")
    yf = expert_ffn(dsc, Wd, full_slot, xd, off, sp)
    full, _ = combine(dsc, T, yf, pp, w, ids, full_slot)
    mask = synth.make_split(E, seed=0)
    sa = torch.from_numpy(np.where(mask, np.arange(E), -1).astype(np.int32)).cuda()
    sb = torch.from_numpy(np.where(~mask, np.arange(E), -1).astype(np.int32)).cuda()
    ya = expert_ffn(dsc, Wd, sa, xd, off, sp)
    yb = expert_ffn(dsc, Wd, sb, xd, off, sp)
    a, _ = combine(dsc, T, ya, pp, w, ids, sa)
    merged, _ = combine(dsc, T, yb, pp, w, ids, sb, partial_b=a)
    assert rel_l2(merged.cpu().numpy(), full.cpu().numpy()) <= 1e-6
    ref = OF.layer(weights_to_numpy(W), np.arange(E, dtype=np.int32), bf16_bits(x), bf16_bits(wr), None, k, 1)
    ra = OF.combine(OF.expert_ffn(weights_to_numpy(W), mask_to_slot(mask), bf16_bits(x), k, ref["offsets"],
                                  ref["sorted_pair"]), ref["pair_pos"], ref["w"], ref["ids"], mask_to_slot(mask))
    assert rel_l2(a.cpu().numpy(), ra) < TOL
    assert rel_l2(full.cpu().numpy(), ref["out"]) < TOL
    # fused-combine form of the split: both halves accumulate into one buffer
    out = expert_ffn(dsc, Wd, sa, xd, off, sp, topk_w=w)
    out = expert_ffn(dsc, Wd, sb, xd, off, sp, topk_w=w, out=out)
    assert rel_l2(out.cpu().numpy(), full.cpu().numpy()) <= 1e-6


def mask_to_slot(mask):
    return np.where(mask, np.arange(len(mask)), -1).astype(np.int32)


def test_slot_table_smaller_than_expert_count():
    # 32 experts, 8 slots: only experts with a slot are computed; the rest are skipped
    E, k, d, f, T, C = 32, 4, 256, 256, 24, 8
    W, x, wr, _ = _setup(synth.MXFP4, E, k, d, f, T, seed=9, C=C)
    dsc = ft.desc(E, k, d, f, synth.MXFP4)
    slot_np = np.full(E, -1, np.int32)
    slot_np[[3, 5, 8, 13, 21, 22, 30, 31]] = np.arange(C)
    ref = OF.layer(weights_to_numpy(W), slot_np, bf16_bits(x), bf16_bits(wr), None, k, 1)
    ids2, w2, of2, _ = layer_forward(dsc, W.to("cuda"), torch.from_numpy(slot_np).cuda(), x.cuda(), wr.cuda())
    assert rel_l2(of2.cpu().numpy(), ref["out"]) < TOL
