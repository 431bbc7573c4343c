"""Seeded synthetic inputs for the routed mixture-of-experts layer.

This module only *draws inputs*; it holds none of the layer's arithmetic.
It produces:

* activations x ~ N(0, 1) rounded to bf16;
* router weights W_r ~ N(0, 1) / sqrt(d) rounded to bf16 (or unscaled N(0, 1));
* expert weights drawn N(0, 0.02) and *stored* in one of four checkpoint
  formats (BF16, NVFP4, MXFP4, FP8 with 128x128 fp32 block scales).  The
  storage encoder here is this module's own, independent of the oracle's
  and of the CUDA path's codecs: it only has to produce valid codes with
  realistic statistics, which both sides then read;
* a Zipf routing bias and Zipf routing traces (Gumbel-top-k sampling
  without replacement, Kool et al. 2019);
* a random resident/complement split of the experts.

Both the CUDA path (tests, bench) and the oracle consume what this returns;
neither side regenerates inputs by itself.  Tensors may be drawn on CPU or
on a CUDA device: the same seed gives different numbers on the two, so a
caller draws once and hands the same tensors to both sides.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

# Weight storage formats (values match the C-ABI's ftmoe_wfmt).
BF16, NVFP4, MXFP4, FP8_B128 = 0, 1, 2, 3
FMT_NAMES = {BF16: "bf16", NVFP4: "nvfp4", MXFP4: "mxfp4", FP8_B128: "fp8_b128"}


@dataclass(frozen=True)
class LayerShape:
    E: int          # routed experts
    k: int          # experts per token
    d: int          # model width
    f: int          # expert hidden width (SwiGLU)
    fmt: int        # expert weight storage format
    renorm: int = 1  # top-k weights renormalised to sum 1


@dataclass(frozen=True)
class Workload:
    name: str
    layer: LayerShape
    tokens: tuple          # token counts per call (decode batches or one prefill chunk)
    layers: int = 1        # MoE layers sharing one slot table
    zipf_s: float = 0.0    # Zipf exponent of the routing bias (0 = no bias)
    capacity: int = 0      # slot-table capacity of the LRU replay (0 = all resident)
    trace_steps: int = 0   # steps of the LRU replay trace
    split: bool = False    # random resident/complement split of the experts
    seed: int = 0


# The five workloads of the layer specification.
TINY = Workload("tiny_e8k2_d256_f512_bf16", LayerShape(8, 2, 256, 512, BF16), (16,))
DECODE = Workload("decode_e128k8_d2048_f768_nvfp4", LayerShape(128, 8, 2048, 768, NVFP4),
                  (1, 4, 16), zipf_s=1.1, capacity=int(0.37 * 128), trace_steps=4096)
PREFILL = Workload("prefill_e128k8_d2048_f768_nvfp4_t8192", LayerShape(128, 8, 2048, 768, NVFP4),
                   (8192,))
STACK = Workload("decode_stack_l8_e256k6_d4096_f2048_mxfp4", LayerShape(256, 6, 4096, 2048, MXFP4),
                 (1, 16, 64), layers=8, zipf_s=1.0, capacity=int(0.11 * 8 * 256), trace_steps=2048)
PREFILL_SPLIT = Workload("prefill_split_e256k6_d4096_f2048_fp8b128_t16384",
                         LayerShape(256, 6, 4096, 2048, FP8_B128), (16384,), split=True)
WORKLOADS = {w.name: w for w in (TINY, DECODE, PREFILL, STACK, PREFILL_SPLIT)}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _mix(*parts: int) -> int:
    """Combine integers into one 63-bit seed (splitmix64 finaliser)."""
    h = 0x9E3779B97F4A7C15
    for p in parts:
        h = (h ^ (int(p) & 0xFFFF_FFFF_FFFF_FFFF)) & 0xFFFF_FFFF_FFFF_FFFF
        h = (h + 0x9E3779B97F4A7C15) & 0xFFFF_FFFF_FFFF_FFFF
        z = h
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFF_FFFF_FFFF_FFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFF_FFFF_FFFF_FFFF
        h = z ^ (z >> 31)
    return h & 0x7FFF_FFFF_FFFF_FFFF


# ----------------------------------------------------------------------------
# activations and router
# ----------------------------------------------------------------------------
def make_x(T: int, d: int, seed: int, device="cpu") -> torch.Tensor:
    """Activations ~ N(0, 1), bf16 [T, d]."""
    g = _gen(_mix(seed, 1, T, d), device)
    return torch.randn(T, d, generator=g, device=device).to(torch.bfloat16)


def make_router(E: int, d: int, seed: int, device="cpu", scaled: bool = True) -> torch.Tensor:
    """Router weights bf16 [E, d]: N(0, 1)/sqrt(d) (default) or plain N(0, 1)."""
    g = _gen(_mix(seed, 2, E, d), device)
    w = torch.randn(E, d, generator=g, device=device)
    if scaled:
        w = w / math.sqrt(d)
    return w.to(torch.bfloat16)


def zipf_ranks(E: int, seed: int) -> np.ndarray:
    """rank[e] in 1..E: a seeded random mapping of experts onto Zipf ranks."""
    rng = np.random.default_rng(_mix(seed, 3, E))
    perm = rng.permutation(E)
    rank = np.empty(E, np.int64)
    rank[perm] = np.arange(1, E + 1)
    return rank


def make_zipf_bias(E: int, s: float, seed: int) -> np.ndarray:
    """Router logit bias log p_Zipf(rank(e)) up to a constant: -s * log(rank(e)), fp32 [E]."""
    if s == 0.0:
        return np.zeros(E, np.float32)
    return (-s * np.log(zipf_ranks(E, seed).astype(np.float64))).astype(np.float32)


def make_trace(steps: int, layers: int, B: int, k: int, E: int, s: float, seed: int) -> np.ndarray:
    """Routing trace int32 [steps, layers, B, k]: per token, k distinct experts drawn
    without replacement with probability proportional to rank^-s (Gumbel-top-k)."""
    out = np.empty((steps, layers, B, k), np.int32)
    for l in range(layers):
        logp = -s * np.log(zipf_ranks(E, _mix(seed, 40, l)).astype(np.float64))
        rng = np.random.default_rng(_mix(seed, 41, l))
        chunk = max(1, (1 << 22) // max(1, B * E))
        for s0 in range(0, steps, chunk):
            n = min(chunk, steps - s0)
            gum = rng.gumbel(size=(n, B, E))
            keys = logp[None, None, :] + gum
            idx = np.argpartition(-keys, k - 1, axis=-1)[..., :k]
            out[s0:s0 + n, l] = idx.astype(np.int32)
    return out


def make_split(E: int, seed: int, p: float = 0.5) -> np.ndarray:
    """Resident mask bool [E]: each expert resident with probability p."""
    rng = np.random.default_rng(_mix(seed, 5, E))
    return rng.random(E) < p


# ----------------------------------------------------------------------------
# expert weights in storage formats
# ----------------------------------------------------------------------------
# E2M1 magnitudes by code 0..7 and the tie-to-even rounding thresholds between them.
_E2M1_MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _store_e2m1(v: torch.Tensor) -> torch.Tensor:
    """Nearest E2M1 code (ties to the even code), saturating at 6; uint8 codes 0..15."""
    a = v.abs()
    code = torch.zeros_like(a, dtype=torch.uint8)
    for c in range(7):
        mid = 0.5 * (_E2M1_MAG[c] + _E2M1_MAG[c + 1])
        step = (a >= mid) if (c % 2 == 1) else (a > mid)   # tie goes to the even code
        code += step.to(torch.uint8)
    sign = (v < 0) & (code != 0)
    return code | (sign.to(torch.uint8) << 3)


def _pack_nibbles(codes: torch.Tensor) -> torch.Tensor:
    """[..., K] codes 0..15 -> [..., K/2] bytes, element 2i in the low nibble."""
    c = codes.reshape(*codes.shape[:-1], codes.shape[-1] // 2, 2)
    return (c[..., 0] | (c[..., 1] << 4)).contiguous()


def _store_e4m3(v: torch.Tensor) -> torch.Tensor:
    """fp32 -> E4M3 (fn) code bytes, saturating at +-448."""
    return v.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def _draw(N: int, K: int, seed: int, device, std: float) -> torch.Tensor:
    return torch.randn(N, K, generator=_gen(seed, device), device=device) * std


def _store_matrix(fmt: int, w: torch.Tensor):
    """One weight matrix [N, K] (K innermost) -> (codes, scales, global)."""
    N, K = w.shape
    if fmt == BF16:
        return w.to(torch.bfloat16), None, 1.0
    if fmt == NVFP4:
        amax_t = float(w.abs().max())
        glob = amax_t / (6.0 * 448.0) if amax_t > 0 else 1.0
        glob = float(np.float32(glob))
        blk = w.reshape(N, K // 16, 16)
        s_code = _store_e4m3(blk.abs().amax(-1) / (6.0 * glob))
        s_val = s_code.view(torch.float8_e4m3fn).float() * glob
        q = torch.where(s_val[..., None] > 0, blk / s_val[..., None].clamp_min(1e-30),
                        torch.zeros_like(blk))
        return _pack_nibbles(_store_e2m1(q).reshape(N, K)), s_code.contiguous(), glob
    if fmt == MXFP4:
        blk = w.reshape(N, K // 32, 32)
        amax = blk.abs().amax(-1)
        _, ex = torch.frexp(amax)              # amax = m * 2^ex, m in [0.5, 1)
        shared = torch.where(amax > 0, ex.to(torch.int32) - 1 - 2, torch.full_like(ex, -127, dtype=torch.int32))
        shared = shared.clamp(-127, 127)
        s_code = (shared + 127).to(torch.uint8)
        q = blk / torch.exp2(shared.float())[..., None]
        return _pack_nibbles(_store_e2m1(q).reshape(N, K)), s_code.contiguous(), 1.0
    if fmt == FP8_B128:
        blk = w.reshape(N // 128, 128, K // 128, 128)
        amax = blk.abs().amax(dim=(1, 3))
        s = torch.where(amax > 0, amax / 448.0, torch.zeros_like(amax))
        q = torch.where(s[:, None, :, None] > 0, blk / s[:, None, :, None].clamp_min(1e-30),
                        torch.zeros_like(blk))
        return _store_e4m3(q).reshape(N, K).contiguous(), s.float().contiguous(), 1.0
    raise ValueError(f"unknown format {fmt}")


@dataclass
class ExpertWeights:
    """Expert weights for C slots in one storage format.

    gate/up are [C, f, d], down is [C, d, f] (reduction dim innermost).  For
    the FP4 formats the code tensors hold two codes per byte (element 2i in
    the low nibble); scales are E4M3 [C, N, K/16] (NVFP4), E8M0 [C, N, K/32]
    (MXFP4) or fp32 [C, N/128, K/128] (FP8_B128); `glob` is fp32 [C, 3]
    (NVFP4 per-tensor scales of gate, up, down; ones otherwise).
    """
    fmt: int
    d: int
    f: int
    gate: torch.Tensor
    up: torch.Tensor
    down: torch.Tensor
    gate_s: torch.Tensor | None
    up_s: torch.Tensor | None
    down_s: torch.Tensor | None
    glob: torch.Tensor
    extra: dict = field(default_factory=dict)

    @property
    def C(self) -> int:
        return self.gate.shape[0]

    def to(self, device) -> "ExpertWeights":
        mv = lambda t: None if t is None else t.to(device)
        return ExpertWeights(self.fmt, self.d, self.f, mv(self.gate), mv(self.up), mv(self.down),
                             mv(self.gate_s), mv(self.up_s), mv(self.down_s), mv(self.glob))

    def nbytes_per_expert(self) -> int:
        tot = 0
        for t in (self.gate, self.up, self.down, self.gate_s, self.up_s, self.down_s):
            if t is not None:
                tot += t[0].numel() * t.element_size()
        return tot


def make_experts(fmt: int, C: int, d: int, f: int, seed: int, device="cpu", std: float = 0.02,
                 first_slot: int = 0) -> ExpertWeights:
    """Draw C experts' SwiGLU weights N(0, std) and store them in `fmt`.

    Slot i is drawn from its own seed (seed, first_slot + i), so any subset of
    slots can be regenerated alone."""
    mats = {"gate": [], "up": [], "down": []}
    scl = {"gate": [], "up": [], "down": []}
    glob = torch.ones(C, 3, dtype=torch.float32, device=device)
    for i in range(C):
        for j, (name, (N, K)) in enumerate((("gate", (f, d)), ("up", (f, d)), ("down", (d, f)))):
            w = _draw(N, K, _mix(seed, 7, first_slot + i, j), device, std)
            c, s, g = _store_matrix(fmt, w)
            mats[name].append(c)
            scl[name].append(s)
            glob[i, j] = g
    st = lambda xs: None if xs[0] is None else torch.stack(xs).contiguous()
    return ExpertWeights(fmt, d, f, st(mats["gate"]), st(mats["up"]), st(mats["down"]),
                         st(scl["gate"]), st(scl["up"]), st(scl["down"]), glob)


def expert_bytes(fmt: int, d: int, f: int) -> int:
    """Bytes one expert occupies in its storage format (codes + scales)."""
    n = 3 * d * f
    if fmt == BF16:
        return 2 * n
    if fmt == NVFP4:
        return n // 2 + n // 16
    if fmt == MXFP4:
        return n // 2 + n // 32
    if fmt == FP8_B128:
        return n + 4 * (n // (128 * 128))
    raise ValueError(fmt)
