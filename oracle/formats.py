"""Number formats of the expert weights, and the prefill activation quantiser.

The pages name four weight formats, MXFP4, NVFP4, FP8 and BF16, and no
layout (zubnet.ai, "FreeToken, Unsloth GGUF ... consumer hardware",
single section).  The bit layouts below follow the public OCP Microscaling
(MX) definitions of E2M1, E4M3 and E8M0 and the NVFP4 block layout:
  * NVFP4: E2M1 values, one E4M3 scale per 16 elements, one fp32 scale per tensor.
  * MXFP4: E2M1 values, one E8M0 scale per 32 elements.
  * FP8_B128: E4M3 values, one fp32 scale per 128x128 block.

Reading: two FP4 codes share a byte, and element 2i sits in the low nibble.
Blocks run along K, the reduction dimension, which is innermost in memory.

Decoding is done in fp64, where every format's value is exact.
"""
from __future__ import annotations

import numpy as np

BF16, NVFP4, MXFP4, FP8_B128 = 0, 1, 2, 3


# ----------------------------------------------------------------------------
# scalar codecs (closed forms)
# ----------------------------------------------------------------------------
def e2m1_value(code: int) -> float:
    """E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; no inf/NaN."""
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * 0.5 * m                       # subnormal: 2^(1-1) * m/2
    return s * 2.0 ** (e - 1) * (1.0 + 0.5 * m)


def e4m3_value(code: int) -> float:
    """E4M3 (fn variant): 1 sign, 4 exponent (bias 7), 3 mantissa; no inf,
    S.1111.111 is NaN; largest finite 448."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * 2.0 ** -6 * (m / 8.0)
    return s * 2.0 ** (e - 7) * (1.0 + m / 8.0)


def e8m0_value(code: int) -> float:
    """E8M0: unsigned power of two 2^(code-127); 0xFF is NaN."""
    if code == 0xFF:
        return float("nan")
    return 2.0 ** (code - 127)


E2M1_LUT = np.array([e2m1_value(c) for c in range(16)], np.float64)
E4M3_LUT = np.array([e4m3_value(c) for c in range(256)], np.float64)
E8M0_LUT = np.array([e8m0_value(c) for c in range(256)], np.float64)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> values: the high half of an fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round to nearest even bf16 (through fp32, as a bf16 output is stored from fp32)."""
    f = np.asarray(v, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(f)
    r[nan] = 0x7FC0
    return r


# ----------------------------------------------------------------------------
# weight dequantisation
# ----------------------------------------------------------------------------
def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] codes; element 2i is the low nibble of byte i."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def dequant(fmt: int, codes: np.ndarray, scales, glob: float, N: int, K: int) -> np.ndarray:
    """One stored weight matrix [N, K] -> fp64 values.

    BF16:     w = bf16 value
    NVFP4:    w = e2m1 * e4m3(scale[n, k // 16]) * glob
    MXFP4:    w = e2m1 * 2^(scale[n, k // 32] - 127)
    FP8_B128: w = e4m3 * scale[n // 128, k // 128]
    """
    if fmt == BF16:
        return bf16_to_f64(codes).reshape(N, K)
    if fmt == NVFP4:
        v = E2M1_LUT[unpack_nibbles(codes).reshape(N, K)]
        s = E4M3_LUT[np.asarray(scales, np.uint8).reshape(N, K // 16)]
        return v * np.repeat(s, 16, axis=1) * float(np.float32(glob))
    if fmt == MXFP4:
        v = E2M1_LUT[unpack_nibbles(codes).reshape(N, K)]
        s = E8M0_LUT[np.asarray(scales, np.uint8).reshape(N, K // 32)]
        return v * np.repeat(s, 32, axis=1)
    if fmt == FP8_B128:
        v = E4M3_LUT[np.asarray(codes, np.uint8).reshape(N, K)]
        s = np.asarray(scales, np.float32).astype(np.float64).reshape(N // 128, K // 128)
        return v * np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)
    raise ValueError(f"unknown format {fmt}")


# ----------------------------------------------------------------------------
# encoders (round to nearest, ties to the even code, saturating)
# ----------------------------------------------------------------------------
_E2M1_POS = E2M1_LUT[:8]                          # codes 0..7, ascending values
_E4M3_POS = E4M3_LUT[:127]                        # codes 0..126, ascending, 448 last


def _nearest_code(a: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Nearest entry of an ascending table of non-negative values (a >= 0);
    a tie goes to the even code; values above the table's end saturate."""
    a = np.asarray(a, np.float64)
    hi = np.searchsorted(table, a, side="left").clip(0, len(table) - 1)
    lo = (hi - 1).clip(0, len(table) - 1)
    dlo = np.abs(a - table[lo])
    dhi = np.abs(table[hi] - a)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    return np.where(pick_hi, hi, lo).astype(np.uint8)


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """fp32 -> E2M1 code (RNE, saturate at +-6).  The sign is kept, so a
    negative value that rounds to zero gives the code of -0 (0x8)."""
    v = np.asarray(v, np.float32)
    mag = _nearest_code(np.abs(v).astype(np.float64), _E2M1_POS)
    return mag | (np.signbit(v).astype(np.uint8) << 3)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """fp32 -> E4M3 code (RNE, saturate at +-448).  The sign is kept."""
    v = np.asarray(v, np.float32)
    mag = _nearest_code(np.abs(v).astype(np.float64), _E4M3_POS)
    return mag | (np.signbit(v).astype(np.uint8) << 7)


# ----------------------------------------------------------------------------
# prefill activation quantisation (mirror of the library's prefill path)
# ----------------------------------------------------------------------------
def quant_act_nvfp4(v: np.ndarray):
    """Rows [n, K] (fp32) -> (codes uint8 [n, K], scale codes uint8 [n, K/16]).

    The pages do not say how activations reach FP4 tensor cores.  This is the
    library's stated rule, evaluated in fp32 exactly as the kernel does it.
    For each block of 16 consecutive elements:
        s_code = E4M3_rn_satfinite(amax / 6)   (IEEE fp32 division)
        s      = value of s_code
        q      = E2M1_rn_satfinite(v / s)       (IEEE fp32 division), or a zero
                 with v's sign bit if s == 0 (so -0.0 gives the code of -0)
    The tensor-level scale is 1.
    """
    v = np.asarray(v, np.float32)
    n, K = v.shape
    blk = v.reshape(n, K // 16, 16)
    amax = np.max(np.abs(blk), axis=-1)
    s_code = e4m3_encode(amax / np.float32(6.0))
    s = E4M3_LUT[s_code].astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = blk / s[..., None]
    ratio = np.where(s[..., None] > 0, ratio, np.copysign(np.float32(0.0), blk))
    q = e2m1_encode(ratio.astype(np.float32))
    return q.reshape(n, K), s_code


def dequant_act_nvfp4(codes: np.ndarray, s_code: np.ndarray) -> np.ndarray:
    n, K = codes.shape
    return E2M1_LUT[codes] * np.repeat(E4M3_LUT[s_code], 16, axis=1)


def quant_act_fp8(v: np.ndarray):
    """Rows [n, K] (fp32) -> (E4M3 codes [n, K], fp32 scales [n, K/128]).

    Per row and per block of 128 consecutive elements:
        s = amax / 448                    (IEEE fp32 division)
        q = E4M3_rn_satfinite(v / s)      (IEEE fp32 division), or a zero with
                                          v's sign bit if s == 0
    """
    v = np.asarray(v, np.float32)
    n, K = v.shape
    blk = v.reshape(n, K // 128, 128)
    amax = np.max(np.abs(blk), axis=-1)
    s = (amax / np.float32(448.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = blk / s[..., None]
    ratio = np.where(s[..., None] > 0, ratio, np.copysign(np.float32(0.0), blk))
    q = e4m3_encode(ratio.astype(np.float32))
    return q.reshape(n, K), s


def dequant_act_fp8(codes: np.ndarray, s: np.ndarray) -> np.ndarray:
    return E4M3_LUT[codes] * np.repeat(np.asarray(s, np.float64), 128, axis=1)
