"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times.  Routing and permutation are compared bit for bit.  Outputs
are compared on token samples the oracle computes one by one (max relative
L2 5e-3).

  * decode 128x8, d=2048, ffn=768, NVFP4, batch 1 / 4 / 16;
  * prefill of the same layer, 8192 tokens;
  * one layer of the 256x6, d=4096, ffn=2048, MXFP4 stack, batch 1 / 16 / 64;
  * prefill 256x6 FP8-B128 over 16384 tokens, with the random resident /
    complement split: the partials sum to the full output.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import ffn as OF
from oracle import permute as OP
from oracle import route as OR

from gpu_helpers import combine, ensure_built, expert_ffn, layer_forward, permute, route
from helpers import bf16_bits, rel_l2, weights_lazy
import sparse_moe_expert_sorted_b300 as ft

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


_cache = {}


def _weights(w: synth.Workload, seed=0):
    key = (w.name, seed)
    if key not in _cache:
        _cache.clear()
        torch.cuda.empty_cache()
        L = w.layer
        W = synth.make_experts(L.fmt, L.E, L.d, L.f, seed, device="cuda")
        ft.prepare_weights(ft.desc(L.E, L.k, L.d, L.f, L.fmt), W)
        _cache[key] = W
    return _cache[key]


def _act_quant_of(dsc, T):
    # the library tells which path a call takes; the oracle mirrors the quantiser it uses
    path = ft.expert_ffn_path(dsc, T)
    return {0: None, 1: "nvfp4", 2: "fp8"}[path]


def _layer_check(w: synth.Workload, T, sample, seed=1):
    L = w.layer
    W = _weights(w)
    dsc = ft.desc(L.E, L.k, L.d, L.f, L.fmt)
    x = synth.make_x(T, L.d, seed)
    wr = synth.make_router(L.E, L.d, seed)
    bias = synth.make_zipf_bias(L.E, w.zipf_s, seed)
    ids, tw, of, ob = layer_forward(dsc, W, None, x.cuda(), wr.cuda(), torch.from_numpy(bias).cuda())
    g_ids = ids.cpu().numpy()
    rows = np.arange(T) if sample >= T else np.sort(np.random.default_rng(seed).choice(T, sample, replace=False))
    xb, wb = bf16_bits(x), bf16_bits(wr)
    o_ids, o_w, _ = OR.route(xb[rows], wb, bias, L.k, L.renorm)
    assert np.array_equal(g_ids[rows], o_ids)
    np.testing.assert_allclose(tw.cpu().numpy()[rows], o_w, rtol=2e-6, atol=1e-7)
    ref = OF.layer_tokens(weights_lazy(W), np.arange(L.E), xb, g_ids, tw.cpu().numpy(), rows,
                          act_quant=_act_quant_of(dsc, T))
    err = rel_l2(of.cpu().numpy()[rows], ref)
    assert err < TOL, err
    assert rel_l2(ob.float().cpu().numpy()[rows], ref) < TOL
    return g_ids


@pytest.mark.parametrize("T", [1, 4, 16])
def test_decode_workload(T):
    _layer_check(synth.DECODE, T, sample=16, seed=T)


def test_prefill_workload_8192_tokens():
    w = synth.PREFILL
    g_ids = _layer_check(w, 8192, sample=48, seed=5)
    # every pair is placed exactly as the oracle's permutation places it
    dsc = ft.desc(w.layer.E, w.layer.k, w.layer.d, w.layer.f, w.layer.fmt)
    off, sp, pp = permute(dsc, torch.from_numpy(g_ids).cuda())
    o_off, o_sp, o_pp = OP.permute(g_ids, w.layer.E)
    assert np.array_equal(off.cpu().numpy(), o_off) and np.array_equal(sp.cpu().numpy(), o_sp)
    assert np.array_equal(pp.cpu().numpy(), o_pp)
    assert (np.diff(o_off) > 0).sum() >= 120                  # nearly every expert touched


@pytest.mark.parametrize("T,sample", [(1, 1), (16, 4), (64, 4)])
def test_stack_layer_workload(T, sample):
    _layer_check(synth.STACK, T, sample=sample, seed=20 + T)


def test_prefill_split_workload_16384_tokens():
    w = synth.PREFILL_SPLIT
    L = w.layer
    T = 16384
    W = _weights(w)
    dsc = ft.desc(L.E, L.k, L.d, L.f, L.fmt)
    x = synth.make_x(T, L.d, 7).cuda()
    wr = synth.make_router(L.E, L.d, 7)
    ids, tw, _ = route(dsc, x, wr.cuda(), torch.zeros(L.E, device="cuda"))
    off, sp, pp = permute(dsc, ids)
    g_ids = ids.cpu().numpy()
    o_off, o_sp, o_pp = OP.permute(g_ids, L.E)
    assert np.array_equal(off.cpu().numpy(), o_off) and np.array_equal(pp.cpu().numpy(), o_pp)
    mask = synth.make_split(L.E, seed=0)
    sa = torch.from_numpy(np.where(mask, np.arange(L.E), -1).astype(np.int32)).cuda()
    sb = torch.from_numpy(np.where(~mask, np.arange(L.E), -1).astype(np.int32)).cuda()
    full = expert_ffn(dsc, W, torch.arange(L.E, dtype=torch.int32, device="cuda"), x, off, sp, topk_w=tw)
    part = expert_ffn(dsc, W, sa, x, off, sp, topk_w=tw)
    part_b = expert_ffn(dsc, W, sb, x, off, sp, topk_w=tw)
    merged, _ = combine(dsc, T, None, None, None, None, None, partial_b=part + 0.0)
    merged = merged + part_b
    assert rel_l2(merged.cpu().numpy(), full.cpu().numpy()) <= 1e-6
    rows = np.sort(np.random.default_rng(3).choice(T, 6, replace=False))
    xb = bf16_bits(x.cpu())
    o_ids, _, _ = OR.route(xb[rows], bf16_bits(wr), np.zeros(L.E, np.float32), L.k, L.renorm)
    assert np.array_equal(g_ids[rows], o_ids)
    aq = _act_quant_of(dsc, T)
    ref = OF.layer_tokens(weights_lazy(W), np.arange(L.E), xb, g_ids, tw.cpu().numpy(), rows, act_quant=aq)
    assert rel_l2(full.cpu().numpy()[rows], ref) < TOL
    ref_a = OF.layer_tokens(weights_lazy(W), np.where(mask, np.arange(L.E), -1), xb, g_ids, tw.cpu().numpy(), rows,
                            act_quant=aq)
    assert rel_l2(part.cpu().numpy()[rows], ref_a) < TOL
