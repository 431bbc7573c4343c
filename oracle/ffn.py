"""Grouped SwiGLU expert FFN, the weighted combine and the whole layer forward.

The pages say each routed expert is a small feed-forward network.  They say
GPU tensor cores compute the resident experts (zubnet.ai, "FreeToken, Unsloth
GGUF ... consumer hardware"; banandre.com, "The 284B Model on a 32GB GPU
Trick", section "Sparsity Is a Lie").  They also state that the partial sums
over a split of the selected experts add up to the full output once the layer completes (same
banandre.com page, section "The q* Policy: Math Instead of Guesses").

Reading, per expert e with weights W_g, W_u [f, d] and W_d [d, f]:
    g = x W_g^T,  u = x W_u^T,  h = silu(g) * u = g / (1 + exp(-g)) * u,
    y = h W_d^T
and per token t, over the ranks r whose expert is resident (slot_of >= 0):
    out_t = sum_r w[t, r] * y[t, r],  summed in ascending r.
All of this is fp64, from exactly dequantised weights.

Prefill mirror: with act_quant set to "nvfp4" or "fp8", the gathered x rows
and the h rows are first quantised by the library's stated rule (see
formats.quant_act_*) and then dequantised.  That is what FP4/FP8 tensor cores
need.
"""
from __future__ import annotations

import numpy as np

from . import formats as F


def expert_matrices(W: dict, slot: int):
    """fp64 (W_g [f,d], W_u [f,d], W_d [d,f]) of one slot of a weight arena.

    W holds numpy arrays: fmt, d, f, gate, up, down ([C, ...] codes),
    gate_s, up_s, down_s ([C, ...] scales or None), glob ([C, 3] fp32).
    """
    fmt, d, f = W["fmt"], W["d"], W["f"]
    sc = lambda name: None if W[name] is None else W[name][slot]
    g = F.dequant(fmt, W["gate"][slot], sc("gate_s"), W["glob"][slot][0], f, d)
    u = F.dequant(fmt, W["up"][slot], sc("up_s"), W["glob"][slot][1], f, d)
    dn = F.dequant(fmt, W["down"][slot], sc("down_s"), W["glob"][slot][2], d, f)
    return g, u, dn


def _mirror(rows: np.ndarray, act_quant):
    if act_quant is None:
        return rows
    r32 = rows.astype(np.float32)
    if act_quant == "nvfp4":
        return F.dequant_act_nvfp4(*F.quant_act_nvfp4(r32))
    if act_quant == "fp8":
        return F.dequant_act_fp8(*F.quant_act_fp8(r32))
    raise ValueError(act_quant)


def swiglu(X: np.ndarray, Wg, Wu, Wd, act_quant=None) -> np.ndarray:
    """Rows X [n, d] (fp64) through one expert -> Y [n, d] (fp64)."""
    X = _mirror(X, act_quant)
    G = X @ Wg.T
    U = X @ Wu.T
    with np.errstate(over="ignore"):
        H = G / (1.0 + np.exp(-G)) * U
    H = _mirror(H, act_quant)
    return H @ Wd.T


def expert_ffn(W: dict, slot_of: np.ndarray, x_bits: np.ndarray, k: int,
               offsets: np.ndarray, sorted_pair: np.ndarray, act_quant=None) -> np.ndarray:
    """y [P, d] fp64 in expert-sorted order: row j is pair sorted_pair[j].
    Rows of experts with slot_of[e] < 0 stay zero (not computed)."""
    x = F.bf16_to_f64(x_bits)
    E = len(offsets) - 1
    P = int(offsets[E])
    y = np.zeros((P, x.shape[1]), np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo or slot_of[e] < 0:
            continue
        Wg, Wu, Wd = expert_matrices(W, int(slot_of[e]))
        tok = np.asarray(sorted_pair[lo:hi]) // k
        y[lo:hi] = swiglu(x[tok], Wg, Wu, Wd, act_quant)
    return y


def combine(y: np.ndarray, pair_pos: np.ndarray, w: np.ndarray, ids: np.ndarray,
            slot_of: np.ndarray, partial_b=None) -> np.ndarray:
    """out [T, d] fp64: out_t = sum over resident ranks r (ascending) of w[t,r] * y[pair_pos[t*k+r]],
    plus partial_b when given (the exact merge of two partial outputs)."""
    T, k = ids.shape
    out = np.zeros((T, y.shape[1]), np.float64)
    for r in range(k):
        res = np.asarray(slot_of)[ids[:, r]] >= 0
        rows = y[pair_pos.reshape(T, k)[:, r]]
        out += np.where(res[:, None], w[:, r].astype(np.float64)[:, None] * rows, 0.0)
    if partial_b is not None:
        out = out + np.asarray(partial_b, np.float64)
    return out


def layer(W: dict, slot_of, x_bits, wr_bits, bias, k: int, renorm: int, act_quant=None):
    """The whole layer forward.  Returns a dict with ids, w, logits, offsets,
    sorted_pair, pair_pos, y (sorted order) and out (fp64 [T, d])."""
    from .route import route
    from .permute import permute
    ids, w, lg = route(x_bits, wr_bits, bias, k, renorm)
    E = wr_bits.shape[0]
    off, sp, pp = permute(ids, E)
    y = expert_ffn(W, slot_of, x_bits, k, off, sp, act_quant)
    out = combine(y, pp, w, ids, slot_of)
    return dict(ids=ids, w=w, logits=lg, offsets=off, sorted_pair=sp, pair_pos=pp, y=y, out=out)


def layer_tokens(W: dict, slot_of, x_bits, ids, w, tokens, act_quant=None) -> np.ndarray:
    """out rows [len(tokens), d] for a sample of tokens, given their routing.
    Token-major: each sampled token runs its own k experts, so it costs work
    proportional to the sample, not to the whole batch."""
    x = F.bf16_to_f64(x_bits)
    k = ids.shape[1]
    cache = {}
    out = np.zeros((len(tokens), x.shape[1]), np.float64)
    for i, t in enumerate(tokens):
        for r in range(k):
            e = int(ids[t, r])
            if slot_of[e] < 0:
                continue
            if e not in cache:
                cache[e] = expert_matrices(W, int(slot_of[e]))
            y = swiglu(x[t:t + 1], *cache[e], act_quant=act_quant)[0]
            out[i] += float(w[t, r]) * y
    return out
