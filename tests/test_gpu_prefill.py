"""Parity of the tensor-core prefill paths with the oracle's mirror of them:
path 1 (NVFP4 weights, NVFP4 activations) and path 2 (FP8_B128 weights, E4M3
activations with one fp32 scale per row and 128 columns).

  * ftmoe_quantize_act: activation codes and scales bit for bit, including
    zero blocks, signed zeros, blocks whose scale underflows to 0, exact
    rounding ties and saturation;
  * ftmoe_expert_ffn on path 1: y in sorted order and the fused combine,
    within 5e-3 relative L2 of the oracle with act_quant="nvfp4", over several
    M-tiles with ragged tails, both N tilings of gate/up (96 + 96 and 64 + 64),
    slot indirection, empty experts and skewed routing;
  * the exact split of the resident set (A + B = full, reassociation only);
  * the layer call (route + permute + FFN + fused combine + bf16);
  * the same for path 2: E4M3 activation codes and scales bit for bit, parity
    over several K steps and M tiles with skew, the exact split.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import ffn as OF
from oracle import formats as F

from gpu_helpers import ensure_built, expert_ffn, layer_forward, permute, route
from helpers import bf16_bits, rel_l2, weights_to_numpy
import sparse_moe_expert_sorted_b300 as ft

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)


def test_quantize_act_codes_are_bit_exact():
    d, T = 512, 96
    x = synth.make_x(T, d, 11).float().numpy()
    x[0] = 0.0                                                  # all-zero row
    x[1] = -0.0                                                 # negative zeros keep their sign
    x[2, :16] = 1e-4                                            # amax / 6 below the smallest E4M3 scale
    x[2, 16:32] = -3e-4
    tie = np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -2.5, -5.0, 0.5, 1.0, 3.0, 4.0])
    x[3, :16] = tie                                             # scale exactly 1: every E2M1 rounding tie
    x[3, 16:32] = tie * 2.0 ** -6
    x[4] = 1e4 * np.sign(x[4])                                  # scale saturates at 448
    xb = _bf16(x)
    dsc = ft.desc(8, 2, d, 256, ft.NVFP4)
    codes = torch.empty(T, d // 2, dtype=torch.uint8, device="cuda")
    scales = torch.empty(T, d // 16, dtype=torch.uint8, device="cuda")
    ft.quantize_act(dsc, xb.cuda(), codes, scales)
    q, s = F.quant_act_nvfp4(F.bf16_to_f32(bf16_bits(xb)))
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    assert np.array_equal(scales.cpu().numpy(), s)
    assert np.array_equal(codes.cpu().numpy(), packed)


def _prefill_case(E, k, d, f, T, seed, zipf=0.0, C=None, slot_perm=True):
    C = C or E
    W = synth.make_experts(synth.NVFP4, C, d, f, seed, device="cuda")
    x = synth.make_x(T, d, seed)
    wr = synth.make_router(E, d, seed)
    bias = synth.make_zipf_bias(E, zipf, seed) if zipf else np.zeros(E, np.float32)
    dsc = ft.desc(E, k, d, f, ft.NVFP4)
    ft.prepare_weights(dsc, W)
    rng = np.random.default_rng(seed)
    slot_np = (rng.permutation(C)[:E] if slot_perm else np.arange(E)).astype(np.int32)
    return W, x, wr, bias, dsc, slot_np


CASES = [
    # E, k, d, f, T, zipf
    (16, 4, 512, 768, 512, 0.0),     # gate/up N tile 96 + 96
    (16, 4, 512, 512, 512, 0.0),     # gate/up N tile 64 + 64
    (8, 2, 256, 256, 300, 0.0),      # smallest d and ffn, ragged tail
    (32, 8, 256, 512, 1024, 1.2),    # skewed routing: heavy experts span several M-tiles, some are empty
]


@pytest.mark.parametrize("E,k,d,f,T,zipf", CASES)
def test_prefill_ffn_matches_mirror_oracle(E, k, d, f, T, zipf):
    W, x, wr, bias, dsc, slot_np = _prefill_case(E, k, d, f, T, seed=E + T, zipf=zipf)
    assert ft.expert_ffn_path(dsc, T) == 1
    Wn = weights_to_numpy(W)
    ref = OF.layer(Wn, slot_np, bf16_bits(x), bf16_bits(wr), bias, k, 1, act_quant="nvfp4")
    xd = x.cuda()
    ids, w, _ = route(dsc, xd, wr.cuda(), torch.from_numpy(bias).cuda())
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    off, sp, pp = permute(dsc, ids)
    slot = torch.from_numpy(slot_np).cuda()
    y = expert_ffn(dsc, W, slot, xd, off, sp)
    err_y = rel_l2(y.cpu().numpy(), ref["y"])
    assert err_y < TOL, err_y
    out = expert_ffn(dsc, W, slot, xd, off, sp, topk_w=w)
    err = rel_l2(out.cpu().numpy(), ref["out"])
    assert err < TOL, err
    ids2, w2, of2, ob2 = layer_forward(dsc, W, slot, xd, wr.cuda(), torch.from_numpy(bias).cuda())
    assert np.array_equal(ids2.cpu().numpy(), ref["ids"])
    assert rel_l2(of2.cpu().numpy(), ref["out"]) < TOL
    assert rel_l2(ob2.float().cpu().numpy(), ref["out"]) < TOL
    assert ft.get_device_error() == 0


def test_prefill_exact_split():
    E, k, d, f, T = 16, 4, 512, 768, 512
    W, x, wr, bias, dsc, slot_np = _prefill_case(E, k, d, f, T, seed=5, slot_perm=False)
    xd = x.cuda()
    ids, w, _ = route(dsc, xd, wr.cuda())
    off, sp, pp = permute(dsc, ids)
    mask = synth.make_split(E, seed=1)
    sa = torch.from_numpy(np.where(mask, np.arange(E), -1).astype(np.int32)).cuda()
    sb = torch.from_numpy(np.where(~mask, np.arange(E), -1).astype(np.int32)).cuda()
    full = expert_ffn(dsc, W, torch.from_numpy(slot_np).cuda(), xd, off, sp, topk_w=w)
    a = expert_ffn(dsc, W, sa, xd, off, sp, topk_w=w)
    b = expert_ffn(dsc, W, sb, xd, off, sp, topk_w=w)
    assert rel_l2((a + b).cpu().numpy(), full.cpu().numpy()) <= 1e-6
    ref_a = OF.layer(weights_to_numpy(W), np.where(mask, np.arange(E), -1), bf16_bits(x), bf16_bits(wr), None, k, 1,
                     act_quant="nvfp4")
    assert rel_l2(a.cpu().numpy(), ref_a["out"]) < TOL


def test_prefill_all_tokens_on_k_experts():
    # a large bias sends every token to experts 0..k-1: each spans T/128 M-tiles, the rest are empty
    E, k, d, f, T = 16, 2, 256, 512, 640
    W, x, wr, _, dsc, slot_np = _prefill_case(E, k, d, f, T, seed=8, slot_perm=False)
    bias = np.zeros(E, np.float32)
    bias[:k] = 1e3
    ref = OF.layer(weights_to_numpy(W), slot_np, bf16_bits(x), bf16_bits(wr), bias, k, 1, act_quant="nvfp4")
    assert set(np.unique(ref["ids"])) == set(range(k))
    ids, w, of, ob = layer_forward(dsc, W, None, x.cuda(), wr.cuda(), torch.from_numpy(bias).cuda())
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert rel_l2(of.cpu().numpy(), ref["out"]) < TOL


def test_prefill_path_needs_prepared_scales():
    E, k, d, f, T = 8, 2, 256, 256, 256
    W = synth.make_experts(synth.NVFP4, E, d, f, 1, device="cuda")
    dsc = ft.desc(E, k, d, f, ft.NVFP4)
    x = synth.make_x(T, d, 1).cuda()
    ids, w, _ = route(dsc, x, synth.make_router(E, d, 1).cuda())
    off, sp, pp = permute(dsc, ids)
    with pytest.raises(ft.FtmoeError):
        expert_ffn(dsc, W, None, x, off, sp)


# ---------------------------------------------------------------------------
# FP8_B128 weights: path 2 (E4M3 activations, one fp32 scale per row and 128 columns)
# ---------------------------------------------------------------------------
def test_quantize_act_fp8_is_bit_exact():
    d, T = 512, 40
    x = synth.make_x(T, d, 21).float().numpy()
    x[0] = 0.0
    x[1] = -0.0
    x[2, :128] = 1e-38                                           # scale underflows towards zero
    x[3, :128] = np.linspace(-448.0, 448.0, 128)                 # scale exactly 1
    x[4] = 3e4 * np.sign(x[4])
    xb = _bf16(x)
    dsc = ft.desc(8, 2, d, 256, ft.FP8_B128)
    codes = torch.empty(T, d, dtype=torch.uint8, device="cuda")
    scales = torch.empty(T, d // 128, dtype=torch.float32, device="cuda")
    ft.quantize_act(dsc, xb.cuda(), codes, scales.view(torch.uint8))
    q, s = F.quant_act_fp8(F.bf16_to_f32(bf16_bits(xb)))
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), np.asarray(s, np.float32).view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), q)


FP8_CASES = [
    # E, k, d, f, T, zipf
    (16, 4, 512, 256, 512, 0.0),
    (8, 2, 768, 384, 300, 0.0),      # 6 and 3 K steps, ragged tail
    (32, 6, 256, 512, 700, 1.2),     # skewed: several M tiles per hot expert, empty experts
]


@pytest.mark.parametrize("E,k,d,f,T,zipf", FP8_CASES)
def test_prefill_fp8_matches_mirror_oracle(E, k, d, f, T, zipf):
    W = synth.make_experts(synth.FP8_B128, E, d, f, E + T, device="cuda")
    x = synth.make_x(T, d, E + T)
    wr = synth.make_router(E, d, E + T)
    bias = synth.make_zipf_bias(E, zipf, E + T) if zipf else np.zeros(E, np.float32)
    dsc = ft.desc(E, k, d, f, ft.FP8_B128)
    assert ft.expert_ffn_path(dsc, T) == 2
    slot_np = np.random.default_rng(T).permutation(E).astype(np.int32)
    ref = OF.layer(weights_to_numpy(W), slot_np, bf16_bits(x), bf16_bits(wr), bias, k, 1, act_quant="fp8")
    xd = x.cuda()
    ids, w, _ = route(dsc, xd, wr.cuda(), torch.from_numpy(bias).cuda())
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    off, sp, pp = permute(dsc, ids)
    slot = torch.from_numpy(slot_np).cuda()
    y = expert_ffn(dsc, W, slot, xd, off, sp)
    assert rel_l2(y.cpu().numpy(), ref["y"]) < TOL
    out = expert_ffn(dsc, W, slot, xd, off, sp, topk_w=w)
    assert rel_l2(out.cpu().numpy(), ref["out"]) < TOL
    ids2, w2, of2, ob2 = layer_forward(dsc, W, slot, xd, wr.cuda(), torch.from_numpy(bias).cuda())
    assert rel_l2(of2.cpu().numpy(), ref["out"]) < TOL
    assert rel_l2(ob2.float().cpu().numpy(), ref["out"]) < TOL
    assert ft.get_device_error() == 0


def test_prefill_fp8_exact_split():
    E, k, d, f, T = 16, 4, 512, 256, 512
    W = synth.make_experts(synth.FP8_B128, E, d, f, 3, device="cuda")
    x = synth.make_x(T, d, 3).cuda()
    wr = synth.make_router(E, d, 3)
    dsc = ft.desc(E, k, d, f, ft.FP8_B128)
    ids, w, _ = route(dsc, x, wr.cuda())
    off, sp, pp = permute(dsc, ids)
    mask = synth.make_split(E, seed=2)
    sa = torch.from_numpy(np.where(mask, np.arange(E), -1).astype(np.int32)).cuda()
    sb = torch.from_numpy(np.where(~mask, np.arange(E), -1).astype(np.int32)).cuda()
    full = expert_ffn(dsc, W, None, x, off, sp, topk_w=w)
    a = expert_ffn(dsc, W, sa, x, off, sp, topk_w=w)
    b = expert_ffn(dsc, W, sb, x, off, sp, topk_w=w)
    assert rel_l2((a + b).cpu().numpy(), full.cpu().numpy()) <= 1e-6
