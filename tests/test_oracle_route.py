"""Pins of the oracle's router.

The router logits are pinned in three ways:
  * hand-derived golden values that only the fixed order R produces;
  * an error bound against the exact rational dot product;
  * selection that agrees with brute force over all k-subsets.
The softmax weights are pinned against the closed form sigmoid(l1 - l2) for
two experts, against scipy.special.softmax, and against invariants.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import route as R
from oracle.formats import bf16_to_f64
from synth import make_router, make_x

from helpers import bf16_bits

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bits(v):
    return torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLD, "order_r_logits.json")))["cases"],
                         ids=lambda c: c["name"])
def test_order_r_golden(case):
    d = case["d"]
    x = np.zeros((1, d), np.float32)
    for i, v in case["x"]:
        x[0, i] = v
    w = np.full((1, d), case.get("w_scale", 1.0), np.float32)
    lg = R.logits_order_r(_bits(x), _bits(w), np.array([case["bias"]], np.float32))
    assert lg[0, 0] == np.float32(case["expect"])


def test_order_r_within_rounding_bound_of_exact_dot():
    # |fl - exact| <= gamma_n * sum |x_i w_i|, n = d/32 sequential adds + 5 tree levels + bias.
    T, E, d = 3, 5, 512
    x = bf16_bits(make_x(T, d, seed=11))
    w = bf16_bits(make_router(E, d, seed=11))
    bias = np.linspace(-1, 1, E).astype(np.float32)
    lg = R.logits_order_r(x, w, bias)
    xf, wf = bf16_to_f64(x), bf16_to_f64(w)
    n = d // 32 + 5 + 1
    u = 2.0 ** -24
    gamma = n * u / (1 - n * u)
    for t in range(T):
        for e in range(E):
            exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(xf[t], wf[e])) + Fraction(float(bias[e]))
            absum = float(np.sum(np.abs(xf[t] * wf[e]))) + abs(float(bias[e]))
            assert abs(Fraction(float(lg[t, e])) - exact) <= Fraction(gamma * absum)


def test_selection_matches_subset_brute_force():
    g = np.random.default_rng(5)
    for trial in range(60):
        E = int(g.integers(2, 9))
        k = int(g.integers(1, E + 1))
        # small integers make exact ties frequent
        lg = g.integers(-3, 4, (4, E)).astype(np.float32)
        ids, _ = R.select_topk(lg, k, renorm=1)
        for t in range(4):
            best = None
            for sub in itertools.combinations(range(E), k):
                key = (-sum(Fraction(float(lg[t, e])) for e in sub), sub)  # max sum, then lexicographic ids
                if best is None or key < best[0]:
                    best = (key, sub)
            chosen = sorted(best[1], key=lambda e: (-float(lg[t, e]), e))
            assert list(ids[t]) == chosen, (lg[t], k)


def test_two_expert_weight_is_sigmoid():
    lg = np.array([[0.3, -1.1], [2.0, 2.5]], np.float32)
    ids, w = R.select_topk(lg, 1, renorm=0)
    for t in range(2):
        a, b = float(lg[t, ids[t, 0]]), float(lg[t, 1 - ids[t, 0]])
        assert abs(float(w[t, 0]) - 1.0 / (1.0 + math.exp(b - a))) < 1e-7


def test_ties_go_to_lowest_id_and_invariants():
    lg = np.array([[1.0, 2.0, 2.0, 0.5, 2.0, -1.0]], np.float32)
    ids, w = R.select_topk(lg, 3, renorm=1)
    assert list(ids[0]) == [1, 2, 4]
    assert np.allclose(w[0], 1.0 / 3.0)
    ids, w = R.select_topk(lg, 2, renorm=1)
    assert list(ids[0]) == [1, 2]
    # k = E: every id, in logit order
    ids, w = R.select_topk(lg, 6, renorm=0)
    assert list(ids[0]) == [1, 2, 4, 0, 3, 5]
    assert abs(float(w.sum()) - 1.0) < 1e-6


def test_route_invariants_on_random_inputs():
    T, E, d, k = 32, 16, 256, 4
    x = bf16_bits(make_x(T, d, seed=3))
    wr = bf16_bits(make_router(E, d, seed=3))
    ids, w, lg = R.route(x, wr, None, k, renorm=1)
    assert ids.shape == (T, k) and w.shape == (T, k)
    for t in range(T):
        assert len(set(ids[t])) == k and ids[t].min() >= 0 and ids[t].max() < E
        assert np.all(np.diff(lg[t, ids[t]]) <= 0)
        assert lg[t, ids[t]].min() >= np.sort(lg[t])[-k]
    assert np.all(w > 0) and np.allclose(w.sum(1), 1.0, atol=1e-6)
    _, w0, _ = R.route(x, wr, None, k, renorm=0)
    assert np.all(w0.sum(1) < 1.0)


def test_weights_match_scipy_softmax():
    """The weights against scipy.special.softmax (a library routine, computed from the
    fp32 logits in fp64): every expert's probability for k = E, and the renormalised
    share of the chosen experts for k < E."""
    from scipy.special import softmax
    rng = np.random.default_rng(11)
    lg = (rng.standard_normal((6, 12)) * 3.0).astype(np.float32)
    ids, w = R.select_topk(lg, 12, renorm=0)
    p = softmax(lg.astype(np.float64), axis=1)
    for t in range(lg.shape[0]):
        assert np.allclose(w[t], p[t, ids[t]].astype(np.float32), rtol=2 ** -22, atol=0)
    ids, w = R.select_topk(lg, 4, renorm=1)
    for t in range(lg.shape[0]):
        share = p[t, ids[t]] / p[t, ids[t]].sum()
        assert np.allclose(w[t], share.astype(np.float32), rtol=2 ** -22, atol=0)
    ids, w = R.select_topk(lg, 4, renorm=0)
    for t in range(lg.shape[0]):
        assert np.allclose(w[t], p[t, ids[t]].astype(np.float32), rtol=2 ** -22, atol=0)


def test_weights_are_shift_invariant_and_stable_for_large_logits():
    """Softmax ignores a common shift of the logits; large logits neither overflow nor
    lose the winner's share (exp(1000) would overflow without the max shift)."""
    lg = np.array([[0.0, 1.0, -2.0, 0.5]], np.float32)
    ids0, w0 = R.select_topk(lg, 2, renorm=0)
    ids1, w1 = R.select_topk(lg + np.float32(1000.0), 2, renorm=0)
    assert np.array_equal(ids0, ids1)
    assert np.all(np.isfinite(w1))
    assert np.allclose(w0, w1, rtol=1e-4)
