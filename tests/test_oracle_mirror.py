"""Pins of the oracle's prefill mirror: swiglu(act_quant=...) and the activation codecs it uses.

The tensor-core prefill path quantises the gathered x rows before the gate/up product and
h = silu(g) * u before the down product.  The oracle mirrors that in `ffn.swiglu` (through
`ffn._mirror`, `formats.quant_act_*` and `formats.dequant_act_*`).  The pages do not say
how activations reach FP4/FP8 tensor cores (zubnet.ai, "FreeToken, Unsloth GGUF ...
consumer hardware" names the formats only); the rule is the library's stated reading.

The expected values are worked by hand in tests/golden/mirror_examples.json: one expert with a
diagonal gate matrix and permutation up/down matrices, so each step of the mirror can be
followed value by value.  The last tests plant plausible mistakes in a copy of the mirror
(on the CPU, in this file) and check that each one changes the result, so the goldens
would catch them.
"""
import json
import os

import numpy as np
import pytest

from oracle import ffn as O
from oracle import formats as F

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "mirror_examples.json")))


def _hex(v):
    return np.array([int(c, 16) for c in v], np.uint8)


def _sparse(d, n):
    out = np.zeros(n, np.float64)
    for k, v in d.items():
        out[int(k)] = v
    return out


def _nvfp4_case():
    g = GOLD["nvfp4"]
    n = g["d"]
    x = np.array(g["x"], np.float64)[None, :]
    Wg = np.diag([64.0 if j < 16 else 80.0 for j in range(n)])
    Wu = np.zeros((n, n))
    Wd = np.zeros((n, n))
    for j in range(n):
        Wu[j, (j + 17) % n] = 1.0
        Wd[j, (j + 5) % n] = 1.0
    y = np.zeros(n)
    for k, v in g["y_nonzero"].items():
        y[int(k)] = v
    return g, x, Wg, Wu, Wd, y


def _fp8_case():
    g = GOLD["fp8"]
    n = g["d"]
    x = _sparse(g["x_nonzero"], n)[None, :]
    Wg = np.diag(np.full(n, 512.0))
    Wu = np.zeros((n, n))
    Wd = np.zeros((n, n))
    for j in range(n):
        Wu[j, (j + 129) % n] = 1.0
        Wd[j, (j + 3) % n] = 1.0
    return g, x, Wg, Wu, Wd, _sparse(g["y_nonzero"], n)


def test_nvfp4_mirror_steps_match_the_hand_derivation():
    g, x, Wg, Wu, Wd, y = _nvfp4_case()
    codes, s = F.quant_act_nvfp4(x.astype(np.float32))
    assert np.array_equal(codes[0], _hex(g["x_codes"]))
    assert np.array_equal(s[0], _hex(g["x_scale_codes"]))
    xq = F.dequant_act_nvfp4(codes, s)[0]
    assert np.array_equal(xq, np.array(g["xq"]))
    h = np.array(g["h"], np.float32)[None, :]
    hc, hs = F.quant_act_nvfp4(h)
    assert np.array_equal(hc[0], _hex(g["h_codes"]))
    assert np.array_equal(hs[0], _hex(g["h_scale_codes"]))
    hq = F.dequant_act_nvfp4(hc, hs)[0]
    assert np.array_equal(hq, np.array(g["hq"]))
    assert np.array_equal(np.signbit(hq), np.signbit(np.array(g["hq"])))     # -0 stays -0


def test_nvfp4_swiglu_mirror_equals_the_hand_derived_output():
    g, x, Wg, Wu, Wd, y = _nvfp4_case()
    out = O.swiglu(x, Wg, Wu, Wd, act_quant="nvfp4")[0]
    assert np.array_equal(out, y)


def test_fp8_mirror_steps_match_the_hand_derivation():
    g, x, Wg, Wu, Wd, y = _fp8_case()
    n = g["d"]
    codes, s = F.quant_act_fp8(x.astype(np.float32))
    want_codes = np.zeros(n, np.uint8)
    for k, v in g["x_codes_nonzero"].items():
        want_codes[int(k)] = int(v, 16)
    assert np.array_equal(codes[0], want_codes)
    assert np.array_equal(s[0], np.array(g["x_scales"], np.float32))
    # two 128-column blocks with different scales: each block dequantises with its own scale
    xq = F.dequant_act_fp8(codes, s)[0]
    assert np.array_equal(xq, _sparse(g["xq_nonzero"], n))
    h = _sparse(g["h_nonzero"], n).astype(np.float32)
    h[1] = h[129] = np.float32(-0.0)
    hc, hs = F.quant_act_fp8(h[None, :])
    want_h = np.zeros(n, np.uint8)
    for k, v in g["h_codes_nonzero"].items():
        want_h[int(k)] = int(v, 16)
    assert np.array_equal(hc[0], want_h)
    assert np.array_equal(hs[0], np.array(g["h_scales"], np.float32))
    assert np.array_equal(F.dequant_act_fp8(hc, hs)[0], _sparse(g["hq_nonzero"], n))


def test_fp8_swiglu_mirror_equals_the_hand_derived_output():
    g, x, Wg, Wu, Wd, y = _fp8_case()
    out = O.swiglu(x, Wg, Wu, Wd, act_quant="fp8")[0]
    assert np.array_equal(out, y)


def test_dequant_act_fp8_applies_each_block_scale_to_its_own_columns():
    """Codes 0x38 (1.0) in every column of two 128-column blocks with scales 0.5 and 3:
    the first 128 values are 0.5, the next 128 are 3 (a scale repeated along the wrong
    axis, interleaved or divided would give other values)."""
    codes = np.full((1, 256), 0x38, np.uint8)
    v = F.dequant_act_fp8(codes, np.array([[0.5, 3.0]], np.float32))[0]
    assert np.all(v[:128] == 0.5) and np.all(v[128:] == 3.0)
    two = F.dequant_act_fp8(np.full((2, 128), 0x40, np.uint8), np.array([[0.25], [4.0]], np.float32))
    assert np.all(two[0] == 0.5) and np.all(two[1] == 8.0)        # 0x40 is E4M3 2.0


# ---------------------------------------------------------------------------------------
# the mirror through the layer-level oracle calls (weights stored as codes in an arena)
# ---------------------------------------------------------------------------------------
def _nvfp4_arena(Wg, Wu, Wd):
    """One slot in NVFP4 holding the golden matrices exactly: 64 = E2M1 4 x E4M3 16,
    80 = 4 x 20, 1 = 1 x 1; tensor scales 1."""
    n = Wg.shape[0]
    e2m1 = {0.0: 0, 1.0: 2, 4.0: 6}
    e4m3 = {1.0: 0x38, 16.0: 0x58, 20.0: 0x5A}

    def enc(Wm):
        codes = np.zeros((n, n), np.uint8)
        sc = np.zeros((n, n // 16), np.uint8)
        for r in range(n):
            for c in np.nonzero(Wm[r])[0]:
                v = Wm[r, c]
                q, s = (4.0, v / 4.0) if v > 1 else (1.0, 1.0)
                codes[r, c] = e2m1[q]
                sc[r, c // 16] = e4m3[s]
        packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
        return packed[None], sc[None]

    (g, gs), (u, us), (dn, ds) = enc(Wg), enc(Wu), enc(Wd)
    return dict(fmt=F.NVFP4, d=n, f=n, gate=g, up=u, down=dn, gate_s=gs, up_s=us, down_s=ds,
                glob=np.ones((1, 3), np.float32))


def _fp8_arena(Wg, Wu, Wd):
    """One slot in FP8_B128: 512 = E4M3 4 (0x48) x block scale 128; 1 = 0x38 x 1."""
    n = Wg.shape[0]

    def enc(Wm, big):
        codes = np.where(Wm != 0, 0x48 if big else 0x38, 0).astype(np.uint8)
        sc = np.full((n // 128, n // 128), 128.0 if big else 1.0, np.float32)
        return codes[None], sc[None]

    (g, gs), (u, us), (dn, ds) = enc(Wg, True), enc(Wu, False), enc(Wd, False)
    return dict(fmt=F.FP8_B128, d=n, f=n, gate=g, up=u, down=dn, gate_s=gs, up_s=us, down_s=ds,
                glob=np.ones((1, 3), np.float32))


@pytest.mark.parametrize("case,arena,aq", [(_nvfp4_case, _nvfp4_arena, "nvfp4"), (_fp8_case, _fp8_arena, "fp8")])
def test_layer_level_calls_carry_the_mirror(case, arena, aq):
    g, x, Wg, Wu, Wd, y = case()
    W = arena(Wg, Wu, Wd)
    mg, mu, md = O.expert_matrices(W, 0)
    assert np.array_equal(mg, Wg) and np.array_equal(mu, Wu) and np.array_equal(md, Wd)
    xb = F.f64_to_bf16_bits(x)                          # the golden x values are bf16 values
    assert np.array_equal(F.bf16_to_f64(xb), x)
    off = np.array([0, 1], np.int32)
    yy = O.expert_ffn(W, np.zeros(1, np.int32), xb, 1, off, np.array([0], np.int32), act_quant=aq)
    assert np.array_equal(yy[0], y)
    yt = O.layer_tokens(W, np.zeros(1, np.int32), xb, np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32), [0],
                        act_quant=aq)
    assert np.array_equal(yt[0], y)


# ---------------------------------------------------------------------------------------
# planted mistakes: each must change the result on the golden inputs
# ---------------------------------------------------------------------------------------
def _silu(G):
    with np.errstate(over="ignore"):
        return G / (1.0 + np.exp(-G))


def _no_h_quant(X, Wg, Wu, Wd, aq):
    Xq = O._mirror(X, aq)
    return (_silu(Xq @ Wg.T) * (Xq @ Wu.T)) @ Wd.T


def _no_x_quant(X, Wg, Wu, Wd, aq):
    H = O._mirror(_silu(X @ Wg.T) * (X @ Wu.T), aq)
    return H @ Wd.T


def _quant_before_silu(X, Wg, Wu, Wd, aq):
    Xq = O._mirror(X, aq)
    G = O._mirror(Xq @ Wg.T, aq)
    U = O._mirror(Xq @ Wu.T, aq)
    return (_silu(G) * U) @ Wd.T


def _transposed_up(X, Wg, Wu, Wd, aq):
    return O.swiglu(X, Wg, Wu.T, Wd, act_quant=aq)


def _transposed_down(X, Wg, Wu, Wd, aq):
    return O.swiglu(X, Wg, Wu, Wd.T, act_quant=aq)


MUTANTS = {"h not quantised": _no_h_quant, "x not quantised": _no_x_quant,
           "g and u quantised before the SiLU instead of h": _quant_before_silu,
           "W_up transposed": _transposed_up, "W_down transposed": _transposed_down}


@pytest.mark.parametrize("case,aq", [(_nvfp4_case, "nvfp4"), (_fp8_case, "fp8")])
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_change_the_golden_output(case, aq, name):
    g, x, Wg, Wu, Wd, y = case()
    out = MUTANTS[name](x, Wg, Wu, Wd, aq)[0]
    assert not np.array_equal(out, y), name


@pytest.mark.parametrize("case,aq", [(_nvfp4_case, "nvfp4"), (_fp8_case, "fp8")])
@pytest.mark.parametrize("mistake", ["divide by the scale", "scales interleaved"])
def test_planted_dequant_mistakes_change_the_golden_output(monkeypatch, case, aq, mistake):
    g, x, Wg, Wu, Wd, y = case()
    if aq == "nvfp4":
        def bad(codes, s):
            sv = F.E4M3_LUT[s]
            sv = 1.0 / sv if mistake == "divide by the scale" else np.tile(sv, (1, 16))
            if mistake == "divide by the scale":
                sv = np.repeat(sv, 16, axis=1)
            with np.errstate(divide="ignore", invalid="ignore"):
                return np.nan_to_num(F.E2M1_LUT[codes] * sv)
        monkeypatch.setattr(F, "dequant_act_nvfp4", bad)
    else:
        def bad(codes, s):
            s = np.asarray(s, np.float64)
            sv = np.repeat(1.0 / s, 128, axis=1) if mistake == "divide by the scale" else np.tile(s, (1, 128))
            return F.E4M3_LUT[codes] * sv
        monkeypatch.setattr(F, "dequant_act_fp8", bad)
    out = O.swiglu(x, Wg, Wu, Wd, act_quant=aq)[0]
    assert not np.array_equal(out, y), mistake
