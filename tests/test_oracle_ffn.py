"""Pins of the oracle's expert FFN, combine and whole-layer forward.

  * One expert with k = 1 reduces the layer to a plain SwiGLU MLP.  That MLP
    is computed here by pure-Python loops.
  * A token-major fp64 brute force uses no permutation.  It checks the
    expert-major path end to end, including permute, pair_pos and combine.
  * The exact split: the partials over a resident set and over its
    complement sum to the full output.  The pages state this
    (banandre.com, "The 284B Model on a 32GB GPU Trick", section "The q*
    Policy: Math Instead of Guesses").
  * Linearity in the combine weights, slot indirection, and zero-token experts.
  * SiLU against scipy.special.expit and its closed-form values.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import ffn as O
from oracle.formats import bf16_to_f64
from oracle.permute import permute
from oracle.route import route

from helpers import bf16_bits, rel_l2, weights_to_numpy

FMTS = [synth.BF16, synth.NVFP4, synth.MXFP4, synth.FP8_B128]


def _layer_inputs(fmt, E=8, d=256, f=256, T=16, k=2, seed=0):
    W = weights_to_numpy(synth.make_experts(fmt, E, d, f, seed))
    x = bf16_bits(synth.make_x(T, d, seed))
    wr = bf16_bits(synth.make_router(E, d, seed))
    return W, x, wr


def test_single_expert_is_plain_swiglu_mlp():
    T, d, f = 3, 256, 128
    W, x, wr = _layer_inputs(synth.BF16, E=1, d=d, f=f, T=T, k=1)
    res = O.layer(W, np.zeros(1, np.int32), x, wr, None, k=1, renorm=1)
    assert np.all(res["ids"] == 0) and np.all(res["w"] == 1.0)
    Wg, Wu, Wd = (m.tolist() for m in O.expert_matrices(W, 0))
    xs = bf16_to_f64(x).tolist()
    for t in range(T):
        h = []
        for j in range(f):
            g = sum(xs[t][i] * Wg[j][i] for i in range(d))
            u = sum(xs[t][i] * Wu[j][i] for i in range(d))
            h.append(g / (1.0 + math.exp(-g)) * u)
        for n in range(d):
            y = sum(h[j] * Wd[n][j] for j in range(f))
            assert abs(res["out"][t, n] - y) <= 1e-12 * (1 + abs(y))


@pytest.mark.parametrize("fmt", FMTS)
def test_layer_matches_token_major_brute_force(fmt):
    E, k = 8, 2
    W, x, wr = _layer_inputs(fmt, E=E, k=k)
    slot_of = np.arange(E, dtype=np.int32)[::-1].copy()        # slot indirection
    Wp = dict(W)
    for name in ("gate", "up", "down", "gate_s", "up_s", "down_s", "glob"):
        if W[name] is not None:
            Wp[name] = W[name][::-1].copy()                     # arena reversed to match
    res = O.layer(Wp, slot_of, x, wr, None, k=k, renorm=1)
    xf = bf16_to_f64(x)
    for t in range(x.shape[0]):
        acc = np.zeros(x.shape[1])
        for r in range(k):
            e = int(res["ids"][t, r])
            Wg, Wu, Wd = O.expert_matrices(W, e)
            g = Wg @ xf[t]
            u = Wu @ xf[t]
            acc += float(res["w"][t, r]) * (Wd @ (g / (1 + np.exp(-g)) * u))
        assert rel_l2(res["out"][t], acc) < 1e-13


@pytest.mark.parametrize("fmt", [synth.NVFP4, synth.FP8_B128])
def test_exact_split_and_linearity(fmt):
    E, k = 8, 2
    W, x, wr = _layer_inputs(fmt, E=E, k=k, seed=2)
    full = O.layer(W, np.arange(E, dtype=np.int32), x, wr, None, k=k, renorm=1)
    g = np.random.default_rng(7)
    for trial in range(5):
        mask = g.random(E) < 0.5
        if trial == 3:
            mask[:] = True
        if trial == 4:
            mask[:] = False
        sa = np.where(mask, np.arange(E), -1).astype(np.int32)
        sb = np.where(~mask, np.arange(E), -1).astype(np.int32)
        ya = O.expert_ffn(W, sa, x, k, full["offsets"], full["sorted_pair"])
        yb = O.expert_ffn(W, sb, x, k, full["offsets"], full["sorted_pair"])
        a = O.combine(ya, full["pair_pos"], full["w"], full["ids"], sa)
        merged = O.combine(yb, full["pair_pos"], full["w"], full["ids"], sb, partial_b=a)
        assert rel_l2(merged, full["out"]) <= 1e-12
    out2 = O.combine(full["y"], full["pair_pos"], 4.0 * full["w"], full["ids"], np.arange(E))
    assert rel_l2(out2, 4.0 * full["out"]) < 1e-14   # a power of two keeps w exact


def test_zero_token_experts_and_skipped_slots():
    E, k = 8, 1
    W, x, wr = _layer_inputs(synth.BF16, E=E, k=k, T=4)
    ids = np.full((4, 1), 5, np.int32)
    off, sp, pp = permute(ids, E)
    y = O.expert_ffn(W, np.arange(E, dtype=np.int32), x, k, off, sp)
    assert y.shape == (4, W["d"])
    out = O.combine(y, pp, np.ones((4, 1), np.float32), ids, np.arange(E))
    Wg, Wu, Wd = O.expert_matrices(W, 5)
    assert rel_l2(out, O.swiglu(bf16_to_f64(x), Wg, Wu, Wd)) < 1e-14
    skip = np.arange(E, dtype=np.int32)
    skip[5] = -1
    y0 = O.expert_ffn(W, skip, x, k, off, sp)
    assert np.all(y0 == 0)
    assert np.all(O.combine(y, pp, np.ones((4, 1), np.float32), ids, skip) == 0)


def test_layer_tokens_matches_whole_layer():
    E, k = 8, 2
    W, x, wr = _layer_inputs(synth.MXFP4, E=E, k=k)
    slot_of = np.arange(E, dtype=np.int32)
    res = O.layer(W, slot_of, x, wr, None, k=k, renorm=1, act_quant=None)
    toks = [0, 5, 15]
    part = O.layer_tokens(W, slot_of, x, res["ids"], res["w"], toks)
    assert rel_l2(part, res["out"][toks]) < 1e-13


def test_silu_matches_scipy_expit_and_the_odd_identity():
    """With X = I, W_gate = diag(g), W_up = I and W_down = I one expert's output is
    diag(silu(g)).  silu(g) = g * expit(g) (scipy.special.expit, a library routine),
    silu(0) = 0, and silu(g) - silu(-g) = g for every g.  A transposed operand would
    move the values off the diagonal."""
    from scipy.special import expit
    g = np.array([0.0, 0.5, -0.5, 1.0986122886681098, -3.0, 7.5, -40.0, 30.0])
    n = g.size
    rng = np.random.default_rng(5)
    perm = rng.permutation(n)
    Wg = np.diag(g)[perm]          # hidden unit j: gate g[perm[j]] on input perm[j]
    I = np.eye(n)
    Wu, Wd = I[perm], I[perm].T    # up: input perm[j] -> unit j; down: unit j -> output perm[j]
    Y = O.swiglu(I, Wg, Wu, Wd)
    want = np.diag(g * expit(g))
    assert np.allclose(Y, want, rtol=1e-14, atol=1e-300)
    assert Y[0, 0] == 0.0
    # sigmoid(ln 3) = 3/4
    assert abs(Y[3, 3] - 0.75 * 1.0986122886681098) < 1e-15
    Yn = O.swiglu(I, -Wg, Wu, Wd)
    assert np.allclose(np.diag(Y) - np.diag(Yn), g, rtol=0, atol=1e-13)


def test_silu_saturates_without_overflow():
    """Very negative gate values give 0 (exp overflow in the denominator is harmless);
    very positive ones give the identity."""
    g = np.array([-800.0, -100.0, 100.0, 800.0])
    I = np.eye(4)
    Y = np.diag(O.swiglu(I, np.diag(g), I, I))
    assert np.all(np.isfinite(Y))
    assert Y[0] == 0.0 and abs(Y[1]) < 1e-40
    assert Y[2] == 100.0 and Y[3] == 800.0
