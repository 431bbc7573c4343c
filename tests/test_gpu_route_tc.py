"""The tensor-core router (long batches, renormalised weights) against the CUDA-core router
and the oracle.

ftmoe_route without a logits output takes the tensor-core path for T >= 256 (16..256 experts,
a multiple of 16); with a logits output it keeps the order-R CUDA-core path.  The two must
give the same ids and the same weights bit for bit, at every token.  The tensor-core logits
only narrow the experts to candidates whose value lies within the error bound of the k-th;
the candidates' logits are recomputed in order R and the top-k taken from them.  A token with
more than 32 candidates goes through order R entirely.  The workspace header counts both kinds
of token.  Constructed near-ties (one-ulp-apart router rows) give extra candidates; 40 equal
router rows give tokens with more than 32 candidates.

The bound rests on a reading of the tensor cores' fp32 accumulation (at most two ulps of the
running magnitude per K = 16 step).  The test measures the largest |tensor-core logit -
order-R logit| / (||x|| max ||w_e||) on ordinary and on wide-range inputs and checks that it
stays well below the bound.

Pages: banandre.com, "The 284B Model on a 32GB GPU Trick", section "Sparsity Is a Lie (But a
Useful One)": a small router selects a few experts per token.
"""
import numpy as np
import pytest
import torch

import synth
import sparse_moe_expert_sorted_b300 as ft
from oracle.route import route as oracle_route

from gpu_helpers import ensure_built
from helpers import bf16_bits

pytestmark = pytest.mark.gpu
FALLBACK_WORD = 128 // 4       # the header's uint32 index of the full-fallback count
EXTRA_WORD = 132 // 4          # ... and of the count of tokens with more than k candidates


def _gamma(d):
    """The library's bound (twice the two errors' relative bound), restated."""
    return 2.0 * ((d // 16) * 2.0 ** -22 + (d // 32 + 5) * 2.0 ** -24)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _both(dsc, x, wr, bias):
    T = x.shape[0]
    ws = ft.workspace(ft.route_workspace_size(dsc, T))
    ids_tc = torch.full((T, dsc.k), -7, dtype=torch.int32, device="cuda")
    w_tc = torch.full((T, dsc.k), float("nan"), device="cuda")
    ft.route(dsc, x, wr, bias, ids_tc, w_tc, None, ws)          # tensor cores + candidates
    ids_r = torch.full((T, dsc.k), -7, dtype=torch.int32, device="cuda")
    w_r = torch.full((T, dsc.k), float("nan"), device="cuda")
    logits = torch.empty(T, dsc.E, device="cuda")
    ft.route(dsc, x, wr, bias, ids_r, w_r, logits, ft.workspace(ft.route_workspace_size(dsc, T)))   # order R
    torch.cuda.synchronize()
    words = ws.view(torch.int32)
    fb, extra = int(words[FALLBACK_WORD].item()), int(words[EXTRA_WORD].item())
    a256 = lambda n: (n + 255) // 256 * 256
    part = lambda o: ws[o:o + T * dsc.E * 4].view(torch.float32).view(T, dsc.E).double()
    tc_logits = part(ft.WS_ZERO_BYTES)
    # with fewer 128-token tiles than half the SMs the library splits K in two; the second part
    # follows the expert norms and the fallback list
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if 2 * ((T + 127) // 128) <= sms and (dsc.d // 64) % 2 == 0:
        tc_logits = tc_logits + part(ft.WS_ZERO_BYTES + a256(T * dsc.E * 4) + a256(dsc.E * 4) + a256(T * 4))
    # the largest logit error relative to ||x|| max ||w_e|| (bias removed in fp64)
    lr = logits.double().cpu()
    if bias is not None:
        lr = lr - bias.double().cpu()
    xn = x.double().cpu().norm(dim=1)
    wn = wr.double().cpu().norm(dim=1).max()
    rel = float(((tc_logits.cpu() - lr).abs().max(dim=1).values / (xn * wn)).max())
    return ids_tc, w_tc, ids_r, w_r, fb, extra, rel


def _check_oracle(ids, w, x, wr, bias_np, k, rows):
    o_ids, o_w, _ = oracle_route(bf16_bits(x.cpu())[rows], bf16_bits(wr.cpu()), bias_np, k, 1)
    assert np.array_equal(ids.cpu().numpy()[rows], o_ids)
    np.testing.assert_allclose(w.cpu().numpy()[rows], o_w, rtol=2e-6, atol=1e-7)


# 12288 tokens: 96 tiles, more than half the SMs, so the logits run without the split of K
@pytest.mark.parametrize("E,k,d,T,zipf", [(128, 8, 2048, 8192, 0.0), (128, 8, 2048, 1000, 1.1), (256, 6, 4096, 300, 1.0),
                                          (16, 4, 256, 256, 0.0), (64, 32, 1024, 520, 0.0),
                                          (256, 6, 4096, 12288, 1.0)])
def test_tensor_core_router_equals_order_r_and_the_oracle(E, k, d, T, zipf):
    seed = E + T
    dsc = ft.desc(E, k, d, 256, synth.NVFP4, 1)
    x = synth.make_x(T, d, seed).cuda()
    wr = synth.make_router(E, d, seed).cuda()
    bias_np = synth.make_zipf_bias(E, zipf, seed) if zipf else None
    bias = torch.from_numpy(bias_np).cuda() if zipf else None
    ids_tc, w_tc, ids_r, w_r, fb, extra, rel = _both(dsc, x, wr, bias)
    assert torch.equal(ids_tc, ids_r)
    assert torch.equal(w_tc, w_r)
    print(f"E={E} k={k} d={d} T={T}: {extra} tokens with extra candidates, {fb} in full order R; "
          f"logit error {rel:.3e} of ||x|| ||w|| (bound {_gamma(d) / 2:.3e})")
    assert rel < _gamma(d) / 8
    assert fb < T // 8
    rows = np.sort(np.random.default_rng(seed).choice(T, min(T, 64), replace=False))
    _check_oracle(ids_tc, w_tc, x, wr, bias_np, k, rows)
    assert ft.get_device_error() == 0


def test_near_ties_give_extra_candidates():
    """Rows 16..31 of the router copy rows 0..15 (exact ties, broken by the lower id) and rows
    48..63 differ from rows 32..47 in one element by one bf16 ulp (near ties).  Every expert has
    a twin, so with an odd k the k-th and (k+1)-th values are twins at every token."""
    E, k, d, T = 64, 7, 512, 2048
    dsc = ft.desc(E, k, d, 256, synth.NVFP4, 1)
    wr = synth.make_router(E, d, 3)
    wr[16:32] = wr[0:16]
    wr[48:64] = wr[32:48]
    bits = wr[48:64].contiguous().view(torch.int16).clone()
    bits[:, 7] += 1                                  # one ulp in one element
    wr[48:64] = bits.view(torch.bfloat16)
    wr = wr.cuda()
    x = synth.make_x(T, d, 4).cuda()
    ids_tc, w_tc, ids_r, w_r, fb, extra, rel = _both(dsc, x, wr, None)
    assert torch.equal(ids_tc, ids_r) and torch.equal(w_tc, w_r)
    print(f"near ties: {extra} of {T} tokens with extra candidates, {fb} in full order R")
    assert extra > T // 2
    _check_oracle(ids_tc, w_tc, x, wr, None, k, np.arange(0, T, 37))


def test_forty_equal_rows_send_tokens_to_the_full_order_r_path():
    """Router rows 0..39 are one row: whenever the k-th value falls in that group the token has at
    least 40 candidates, more than a warp holds, and is recomputed entirely in order R."""
    E, k, d, T = 64, 8, 768, 1024
    dsc = ft.desc(E, k, d, 256, synth.NVFP4, 1)
    wr = synth.make_router(E, d, 5)
    wr[1:40] = wr[0:1]
    wr = wr.cuda()
    x = synth.make_x(T, d, 6).cuda()
    bias_np = synth.make_zipf_bias(E, 0.3, 5)
    bias_np[:40] = 0.0                               # keep the 40 rows tied after the bias
    bias = torch.from_numpy(bias_np).cuda()
    ids_tc, w_tc, ids_r, w_r, fb, extra, rel = _both(dsc, x, wr, bias)
    assert torch.equal(ids_tc, ids_r) and torch.equal(w_tc, w_r)
    print(f"40 equal rows: {fb} of {T} tokens in full order R, {extra} with extra candidates")
    assert fb > T // 8
    _check_oracle(ids_tc, w_tc, x, wr, bias_np, k, np.arange(0, T, 29))


def test_wide_range_inputs_stay_inside_the_bound():
    """x and W_r with magnitudes spread over 2^-12 .. 2^12 (random signs): the tensor cores'
    accumulation error relative to ||x|| ||w|| must stay inside the bound the selection uses."""
    E, k, d, T = 128, 8, 2048, 512
    dsc = ft.desc(E, k, d, 256, synth.NVFP4, 1)
    g = torch.Generator().manual_seed(11)

    def wide(n, m):
        sign = torch.randint(0, 2, (n, m), generator=g) * 2 - 1
        mant = 1.0 + torch.rand(n, m, generator=g)
        ex = torch.randint(-12, 13, (n, m), generator=g)
        return (sign * mant * torch.pow(2.0, ex.double())).to(torch.bfloat16)

    x = wide(T, d).cuda()
    wr = wide(E, d).cuda()
    ids_tc, w_tc, ids_r, w_r, fb, extra, rel = _both(dsc, x, wr, None)
    assert torch.equal(ids_tc, ids_r) and torch.equal(w_tc, w_r)
    print(f"wide range: logit error {rel:.3e} of ||x|| ||w|| (bound {_gamma(d) / 2:.3e}); "
          f"{extra} with extra candidates, {fb} in full order R")
    assert rel < _gamma(d) / 8
    _check_oracle(ids_tc, w_tc, x, wr, None, k, np.arange(0, T, 17))
