"""The router entry point that allocates nothing (ftmoe_route_noalloc).

It serves callers that cannot call cudaMalloc or own a workspace: code under a
memory pool that holds the whole device budget, or code inside another
library's callback, where an allocation could fail or synchronise the device
at the wrong moment.  Its scratch is a fixed array inside the library.

The test calls it through the C ABI twice in a row and checks each call
against ftmoe_route, which uses a caller workspace.  The second call reuses the
array the first call left behind.  The two calls have different shapes, so
they cover both selection paths:
  * up to 64 tokens: the last CTA selects;
  * more tokens: a second kernel selects.
Ids must match bit for bit; weights within the router tests' tolerance.
This file is collected last, and passes alone or after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import ensure_built, route
import sparse_moe_expert_sorted_b300 as ft

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _noalloc(dsc, x, wr, bias):
    T = x.shape[0]
    ids = torch.full((T, dsc.k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, dsc.k), float("nan"), dtype=torch.float32, device="cuda")
    ft.route_noalloc(dsc, x, wr, bias, ids, w)
    torch.cuda.synchronize()
    return ids, w


def test_route_noalloc_matches_route_on_two_calls_in_a_row():
    cases = [(synth.DECODE, 16, 1.1, 3), (synth.PREFILL, 600, 0.0, 4)]
    for wl, T, zipf, seed in cases:
        L = wl.layer
        dsc = ft.desc(L.E, L.k, L.d, L.f, L.fmt, L.renorm)
        x = synth.make_x(T, L.d, seed).cuda()
        wr = synth.make_router(L.E, L.d, seed).cuda()
        bias = torch.from_numpy(synth.make_zipf_bias(L.E, zipf, seed)).cuda()
        ids, w = _noalloc(dsc, x, wr, bias)
        r_ids, r_w, _ = route(dsc, x, wr, bias)
        assert np.array_equal(ids.cpu().numpy(), r_ids.cpu().numpy())
        np.testing.assert_allclose(w.cpu().numpy(), r_w.cpu().numpy(), rtol=2e-6, atol=1e-7)


def test_route_noalloc_rejects_sizes_beyond_its_array():
    dsc = ft.desc(1024, 8, 256, 128, synth.BF16)
    T = 257                                   # 257 * 1024 logits > the 262144-entry array
    st = ft.lib().ftmoe_route_noalloc(ctypes.byref(dsc), 16, 16, None, T, 16, 16, None)
    assert st == 4                            # FTMOE_ERR_WORKSPACE, before any device work


def test_route_noalloc_fills_its_array_exactly_and_matches_the_oracle():
    """T * E equal to the array's capacity (256 tokens x 1024 experts, top-32: the path where a
    second kernel selects), twice in a row: ids bit for bit and weights against ftmoe_route and
    against the oracle's router (oracle/route.py)."""
    from oracle.route import route as oracle_route
    from helpers import bf16_bits
    E, k, d, T = 1024, 32, 256, 256
    assert T * E == 262144                    # FTMOE_NOALLOC_MAX_LOGITS
    dsc = ft.desc(E, k, d, 128, synth.BF16, 1)
    for seed in (7, 8):
        x = synth.make_x(T, d, seed).cuda()
        wr = synth.make_router(E, d, seed).cuda()
        ids, w = _noalloc(dsc, x, wr, None)
        r_ids, r_w, _ = route(dsc, x, wr, None)
        assert np.array_equal(ids.cpu().numpy(), r_ids.cpu().numpy())
        np.testing.assert_allclose(w.cpu().numpy(), r_w.cpu().numpy(), rtol=2e-6, atol=1e-7)
        o_ids, o_w, _ = oracle_route(bf16_bits(x.cpu()), bf16_bits(wr.cpu()), None, k, 1)
        assert np.array_equal(ids.cpu().numpy(), o_ids)
        np.testing.assert_allclose(w.cpu().numpy(), o_w, rtol=2e-6, atol=1e-7)
