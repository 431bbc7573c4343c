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
from oracle.formats import bf16_to_f64
import sparse_moe_expert_sorted_b300 as ft

pytestmark = pytest.mark.gpu
TOL = 5e-3         # relative L2 over the sampled tokens
TOL_TOKEN = 5e-3   # the same bound on each sampled token's own relative L2


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


def _cover_rows(g_ids, E, k):
    """One token per (expert, 128-row tile of the expert's sorted rows): the first pair of every
    M tile the tensor-core path forms, so every expert and every tile is checked."""
    off, sp, _ = OP.permute(g_ids, E)
    rows = set()
    for e in range(E):
        for pos in range(int(off[e]), int(off[e + 1]), 128):
            rows.add(int(sp[pos]) // k)
    return rows


def _per_token_errors(got, want):
    return np.array([np.linalg.norm(got[i] - want[i]) / max(np.linalg.norm(want[i]), 1e-30) for i in range(len(want))])


def _oracle_rows(Wl, slot_of, xb, ids, w, rows, act_quant):
    """The oracle's layer output for the sampled tokens, expert by expert: the sampled tokens
    routed to an expert go through the oracle's swiglu together (the mirror quantises row by
    row), then each adds w * y in ascending rank."""
    rows = list(rows)
    x = bf16_to_f64(xb)
    k = ids.shape[1]
    ys = {}
    for e in np.unique(ids[rows]):
        if slot_of[e] < 0:
            continue
        sel = [(i, r) for i, t in enumerate(rows) for r in range(k) if ids[t, r] == e]
        Wg, Wu, Wd = OF.expert_matrices(Wl, int(slot_of[e]))
        Y = OF.swiglu(x[[rows[i] for i, _ in sel]], Wg, Wu, Wd, act_quant=act_quant)
        for (i, r), y in zip(sel, Y):
            ys[i, r] = y
    out = np.zeros((len(rows), x.shape[1]))
    for i, t in enumerate(rows):
        for r in range(k):
            if (i, r) in ys:
                out[i] += float(w[t, r]) * ys[i, r]
    return out


def _layer_check(w: synth.Workload, T, sample, seed=1, cover=False):
    L = w.layer
    W = _weights(w)
    dsc = ft.desc(L.E, L.k, L.d, L.f, L.fmt)
    x = synth.make_x(T, L.d, seed)
    wr = synth.make_router(L.E, L.d, seed)
    bias = synth.make_zipf_bias(L.E, w.zipf_s, seed)
    ids, tw, of, ob = layer_forward(dsc, W, None, x.cuda(), wr.cuda(), torch.from_numpy(bias).cuda())
    g_ids = ids.cpu().numpy()
    rows = set(np.random.default_rng(seed).choice(T, min(sample, T), replace=False).tolist())
    if cover:
        rows |= _cover_rows(g_ids, L.E, L.k)
    rows = np.array(sorted(rows))
    xb, wb = bf16_bits(x), bf16_bits(wr)
    o_ids, o_w, _ = OR.route(xb[rows], wb, bias, L.k, L.renorm)
    assert np.array_equal(g_ids[rows], o_ids)
    np.testing.assert_allclose(tw.cpu().numpy()[rows], o_w, rtol=2e-6, atol=1e-7)
    aq = _act_quant_of(dsc, T)
    Wl = weights_lazy(W)
    ref = _oracle_rows(Wl, np.arange(L.E), xb, g_ids, tw.cpu().numpy(), rows, aq)
    got = of.cpu().numpy()[rows]
    err = rel_l2(got, ref)
    tok = _per_token_errors(got, ref)
    msg = f"{w.name} T={T}: {len(rows)} tokens, pooled rel L2 {err:.2e}, max per token {tok.max():.2e}"
    if aq is not None:   # the quantised path against the unquantised oracle: information only
        plain = _oracle_rows(Wl, np.arange(L.E), xb, g_ids, tw.cpu().numpy(), rows[:16], None)
        msg += f", against the unquantised oracle {rel_l2(got[:16], plain):.2e}"
    print(msg)
    assert err < TOL, msg
    assert tok.max() < TOL_TOKEN, msg
    assert rel_l2(ob.float().cpu().numpy()[rows], ref) < TOL
    return g_ids


@pytest.mark.parametrize("T", [1, 4, 16])
def test_decode_workload(T):
    _layer_check(synth.DECODE, T, sample=16, seed=T)


def test_prefill_workload_8192_tokens():
    w = synth.PREFILL
    g_ids = _layer_check(w, 8192, sample=48, seed=5, cover=True)
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
    # the exact merge through the library: the complement's FFN adds its partial into a copy
    # of the resident one (its fused combine accumulates into out)
    merged = expert_ffn(dsc, W, sb, x, off, sp, topk_w=tw, out=part.clone())
    assert rel_l2(merged.cpu().numpy(), full.cpu().numpy()) <= 1e-6
    assert rel_l2((part + part_b).cpu().numpy(), merged.cpu().numpy()) <= 1e-6
    # tokens: six at random, and one routed to each of 24 experts drawn at random
    g = np.random.default_rng(3)
    rows = set(g.choice(T, 6, replace=False).tolist())
    for e in g.choice(L.E, 24, replace=False):
        hit = np.flatnonzero((g_ids == e).any(axis=1))
        if hit.size:
            rows.add(int(hit[0]))
    rows = np.array(sorted(rows))
    xb = bf16_bits(x.cpu())
    o_ids, _, _ = OR.route(xb[rows], bf16_bits(wr), np.zeros(L.E, np.float32), L.k, L.renorm)
    assert np.array_equal(g_ids[rows], o_ids)
    aq = _act_quant_of(dsc, T)
    Wl = weights_lazy(W)
    ref = _oracle_rows(Wl, np.arange(L.E), xb, g_ids, tw.cpu().numpy(), rows, aq)
    got = full.cpu().numpy()[rows]
    tok = _per_token_errors(got, ref)
    print(f"FP8 16384 split: {len(rows)} tokens, pooled {rel_l2(got, ref):.2e}, max per token {tok.max():.2e}")
    assert rel_l2(got, ref) < TOL and tok.max() < TOL_TOKEN
    ref_a = _oracle_rows(Wl, np.where(mask, np.arange(L.E), -1), xb, g_ids, tw.cpu().numpy(), rows, aq)
    got_a = part.cpu().numpy()[rows]
    nz = np.linalg.norm(ref_a, axis=1) > 0          # tokens with at least one resident expert
    assert rel_l2(got_a, ref_a) < TOL and _per_token_errors(got_a[nz], ref_a[nz]).max() < TOL_TOKEN
