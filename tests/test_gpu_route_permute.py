"""Parity of ftmoe_route and ftmoe_permute with the oracle (bit-exact ids,
logits and permutation; weights within 1e-6 relative).

Shapes are those of the five workloads (tiny, decode 128x8 at batch 1/4/16,
the 256x6 stack at batch 1/16/64, prefill chunks) plus edge cases:
  * T = 1;
  * ragged token tiles;
  * k = E;
  * exact ties;
  * renorm off;
  * an unscaled N(0,1) router;
  * the largest expert count and top-k (1024, 32);
  * more than one permutation chunk;
  * every pair on one expert.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import permute as OP
from oracle import route as OR

from gpu_helpers import ensure_built, permute, route
from helpers import bf16_bits
import sparse_moe_expert_sorted_b300 as ft

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _check_route(E, k, d, T, seed, zipf=0.0, renorm=1, scaled=True, bias_zero=False):
    dsc = ft.desc(E, k, d, 512, synth.BF16, renorm)
    x = synth.make_x(T, d, seed)
    wr = synth.make_router(E, d, seed, scaled=scaled)
    bias = synth.make_zipf_bias(E, zipf, seed) if zipf else (np.zeros(E, np.float32) if bias_zero else None)
    ids, w, lg = route(dsc, x.cuda(), wr.cuda(), None if bias is None else torch.from_numpy(bias).cuda())
    o_ids, o_w, o_lg = OR.route(bf16_bits(x), bf16_bits(wr), bias, k, renorm)
    g_lg = lg.cpu().numpy()
    assert np.array_equal(g_lg.view(np.uint32), o_lg.view(np.uint32)), "logits differ from order R"
    assert np.array_equal(ids.cpu().numpy(), o_ids)
    np.testing.assert_allclose(w.cpu().numpy(), o_w, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("T", [16, 1, 3])
def test_route_tiny(T):
    _check_route(8, 2, 256, T, seed=0)


@pytest.mark.parametrize("T", [1, 4, 16])
def test_route_decode_shape(T):
    _check_route(128, 8, 2048, T, seed=T, zipf=1.1)


@pytest.mark.parametrize("T", [1, 16, 64])
def test_route_stack_shape(T):
    _check_route(256, 6, 4096, T, seed=10 + T, zipf=1.0)


@pytest.mark.parametrize("T", [65, 300, 1031])
def test_route_prefill_paths_with_ragged_tiles(T):
    _check_route(128, 8, 2048, T, seed=T, bias_zero=True)


@pytest.mark.parametrize("T,renorm", [(1, 1), (5, 0), (70, 1)])
def test_route_largest_expert_count_and_top_k(T, renorm):
    """E = 1024 and k = 32, the largest the descriptor allows: each lane of the selecting
    warp holds 32 experts and every lane ends up holding one rank."""
    _check_route(1024, 32, 256, T, seed=40 + T, renorm=renorm)


def test_route_renorm_off_unscaled_router_and_k_equals_E():
    _check_route(16, 4, 256, 40, seed=5, renorm=0, scaled=False)
    _check_route(8, 8, 256, 9, seed=6)


def test_route_exact_ties_go_to_lowest_id():
    E, k, d, T = 32, 5, 256, 70
    dsc = ft.desc(E, k, d, 512, synth.BF16)
    x = torch.zeros(T, d, dtype=torch.bfloat16)
    x[::2] = 1.0                                           # even tokens: logits = row sums
    wr = torch.zeros(E, d, dtype=torch.bfloat16)
    wr[:, :8] = 0.25                                       # every expert ties
    wr[7, :8] = 0.5                                        # except expert 7
    ids, w, lg = route(dsc, x.cuda(), wr.cuda())
    o_ids, o_w, o_lg = OR.route(bf16_bits(x), bf16_bits(wr), None, k, 1)
    assert np.array_equal(ids.cpu().numpy(), o_ids)
    assert list(o_ids[0]) == [7, 0, 1, 2, 3] and list(o_ids[1]) == [0, 1, 2, 3, 4]


def _check_permute(E, k, ids_np):
    dsc = ft.desc(E, k, 256, 512, synth.BF16)
    off, sp, pp = permute(dsc, torch.from_numpy(ids_np).cuda())
    o_off, o_sp, o_pp = OP.permute(ids_np, E)
    assert np.array_equal(off.cpu().numpy(), o_off)
    assert np.array_equal(sp.cpu().numpy(), o_sp)
    assert np.array_equal(pp.cpu().numpy(), o_pp)


@pytest.mark.parametrize("E,k,T", [(8, 2, 16), (8, 2, 1), (128, 8, 1), (128, 8, 16), (256, 6, 64),
                                   (128, 8, 128), (128, 8, 129), (128, 8, 8192), (256, 6, 16384),
                                   (1024, 4, 3000), (1024, 32, 100)])
def test_permute_matches_oracle(E, k, T):
    g = np.random.default_rng(E * 7 + T)
    ids = np.argsort(g.random((T, E)), axis=1)[:, :k].astype(np.int32)
    _check_permute(E, k, ids)


def test_permute_all_pairs_one_expert_and_empty_experts():
    T, k, E = 3000, 1, 64
    _check_permute(E, k, np.full((T, k), 17, np.int32))


def test_out_of_range_id_sets_the_device_error_without_trapping():
    E, k = 8, 2
    ids = np.array([[0, 1], [2, 9]], np.int32)              # 9 is out of range
    dsc = ft.desc(E, k, 256, 512, synth.BF16)
    ft.get_device_error()                                   # clear
    off, sp, pp = permute(dsc, torch.from_numpy(ids).cuda())
    assert ft.get_device_error() == 1
    assert off.cpu().numpy()[-1] == 4                       # counted as expert E-1, nothing lost
    assert ft.get_device_error() == 0
