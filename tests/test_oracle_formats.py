"""Pins of the oracle's number formats and prefill activation quantiser.

Each check ties the oracle to something other than itself:
  * the OCP value table;
  * torch's own float8 codecs (a library routine);
  * exact rational nearest-value search;
  * hand-derived golden blocks in tests/golden/.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_e2m1_table_matches_ocp_values():
    # OCP MX spec, E2M1 element values for codes 0..7; codes 8..15 are the negatives.
    ocp = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        want = ocp[c & 7] * (-1.0 if c & 8 else 1.0)
        assert F.e2m1_value(c) == want, c


def test_e4m3_all_codes_match_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().double().numpy()
    got = F.E4M3_LUT
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert nan.sum() == 2 and np.isnan(got[0x7F]) and np.isnan(got[0xFF])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_e8m0_all_codes_match_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).float().double().numpy()
    got = F.E8M0_LUT
    for c in range(255):
        # torch's e8m0 -> float goes through fp32, which cannot hold 2^-127 as a normal;
        # compare in exact powers of two where fp32 can, and the exponent otherwise.
        if c >= 1:
            assert got[c] == ref[c], c
        assert got[c] == 2.0 ** (c - 127)
    assert np.isnan(got[255])


def test_bf16_decode_and_round_match_torch():
    g = torch.Generator().manual_seed(1)
    v = torch.randn(4096, generator=g) * torch.exp2(torch.randint(-20, 20, (4096,), generator=g).float())
    bits = v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(F.bf16_to_f64(bits), v.to(torch.bfloat16).double().numpy())
    assert np.array_equal(F.f64_to_bf16_bits(v.numpy()), bits)


def _nearest_exact(a, table_codes):
    """Exact rational nearest search with ties to the even code."""
    best = None
    for c, val in table_codes:
        dist = abs(Fraction(a) - Fraction(val))
        key = (dist, c % 2)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_e2m1_encode_matches_exact_nearest_and_tie_table():
    table = [(c, F.e2m1_value(c)) for c in range(8)]
    g = np.random.default_rng(0)
    vals = np.concatenate([g.uniform(-8, 8, 3000).astype(np.float32),
                           np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0, 100.0], np.float32)])
    got = F.e2m1_encode(vals)
    for v, c in zip(vals, got):
        mag = _nearest_exact(min(abs(float(v)), 6.0), table)
        assert (c & 7) == mag, (v, c)
        assert (c >> 3) == (1 if v < 0 else 0)
    # Tie table: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4.
    ties = F.e2m1_encode(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32))
    assert [F.e2m1_value(int(c)) for c in ties] == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_e4m3_encode_matches_torch_cast():
    g = torch.Generator().manual_seed(2)
    v = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-14, 10, (20000,), generator=g).float())
    # midpoints between neighbouring E4M3 values: exact ties
    pos = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).float()
    mids = 0.5 * (pos[1:] + pos[:-1])
    v = torch.cat([v, mids, -mids, torch.tensor([448.0, 460.0, 1e6, -1e6, 0.0])])
    ref = v.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.e4m3_encode(v.numpy())
    # torch maps -0.0 results to 0x80 as well; compare everything
    assert np.array_equal(got, ref)


def test_dequant_golden_blocks():
    gold = json.load(open(os.path.join(GOLD, "format_examples.json")))
    h = lambda s: int(s, 16)
    nv = gold["nvfp4"]
    got = F.dequant(F.NVFP4, np.array([h(b) for b in nv["bytes"]], np.uint8),
                    np.array([h(s) for s in nv["scales"]], np.uint8), nv["glob"], 1, 32)[0]
    want = np.array([0.5] * 16 + [0.0029296875] * 16)
    want[1] = -3.0
    assert np.array_equal(got, want)
    mx = gold["mxfp4"]
    got = F.dequant(F.MXFP4, np.array([h(b) for b in mx["bytes"]], np.uint8),
                    np.array([h(s) for s in mx["scales"]], np.uint8), 1.0, 1, 32)[0]
    want = np.full(32, 12.0)
    want[31] = -32.0
    assert np.array_equal(got, want)
    f8 = gold["fp8_b128"]
    codes = np.zeros((128, 128), np.uint8)
    for key, c in f8["codes_sparse"].items():
        i, j = map(int, key.split(","))
        codes[i, j] = h(c)
    got = F.dequant(F.FP8_B128, codes, np.array([[f8["scale"]]], np.float32), 1.0, 128, 128)
    want = np.zeros((128, 128))
    for key, v in f8["expect_sparse"].items():
        i, j = map(int, key.split(","))
        want[i, j] = v
    assert np.array_equal(got, want)


def test_dequant_nvfp4_is_exact_product_of_three_factors():
    # fp64 holds e2m1 * e4m3 * fp32 exactly; compare with exact rationals.
    g = np.random.default_rng(3)
    codes = g.integers(0, 256, (4, 16), dtype=np.uint8)
    scales = g.integers(0, 0x7E, (4, 2), dtype=np.uint8)
    glob = float(np.float32(0.0123))
    got = F.dequant(F.NVFP4, codes, scales, glob, 4, 32)
    for n in range(4):
        for k in range(32):
            byte = int(codes[n, k // 2])
            nib = byte & 0xF if k % 2 == 0 else byte >> 4
            want = Fraction(F.e2m1_value(nib)) * Fraction(F.e4m3_value(int(scales[n, k // 16]))) * Fraction(glob)
            assert Fraction(got[n, k]) == want


def test_act_quant_nvfp4_golden():
    gold = json.load(open(os.path.join(GOLD, "act_quant_examples.json")))
    h = lambda s: int(s, 16)
    blocks = gold["nvfp4_blocks"]
    v = np.array([b["v"] for b in blocks], np.float32).reshape(1, -1)
    q, s = F.quant_act_nvfp4(v)
    assert [int(c) for c in s[0]] == [h(b["s_code"]) for b in blocks]
    assert [int(c) for c in q[0]] == [h(c) for b in blocks for c in b["q"]]


def test_act_quant_fp8_golden():
    gold = json.load(open(os.path.join(GOLD, "act_quant_examples.json")))
    h = lambda s: int(s, 16)
    row = gold["fp8_rows"][0]
    v = np.zeros((1, 128), np.float32)
    for i, x in row["v_sparse"].items():
        v[0, int(i)] = x
    q, s = F.quant_act_fp8(v)
    assert s[0, 0] == np.float32(row["s"])
    want = np.zeros(128, np.uint8)
    for i, c in row["q_sparse"].items():
        want[int(i)] = h(c)
    assert np.array_equal(q[0], want)


def test_act_quant_roundtrip_of_representable_blocks_is_exact():
    # A block whose values are E2M1 values times s, with amax = 6 s and s an
    # E4M3 value, quantises back to itself.
    g = np.random.default_rng(4)
    for _ in range(200):
        s = F.e4m3_value(int(g.integers(0x20, 0x60)))
        codes = g.integers(0, 16, 16)
        codes[int(g.integers(0, 16))] = 7                # amax = 6 s
        v = (F.E2M1_LUT[codes] * s).astype(np.float32).reshape(1, 16)
        q, sc = F.quant_act_nvfp4(v)
        assert F.e4m3_value(int(sc[0, 0])) == s
        back = F.dequant_act_nvfp4(q, sc)
        assert np.array_equal(back, v.astype(np.float64))
