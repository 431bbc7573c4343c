"""Router: logits, top-k expert choice, and the weights of the chosen experts.

The pages: a small router chooses a few experts for each token, six out of
256 in their example model (banandre.com, "The 284B Model on a 32GB
GPU Trick", section "Sparsity Is a Lie (But a Useful One)").  The pages do not
give the function.  The library's reading is:
  * softmax over all E logits, then top-k;
  * the k ids are ordered by (logit descending, id ascending), so a tie goes
    to the lower id;
  * selection uses the logits, not the probabilities, because fp32 softmax can
    create ties the logits do not have;
  * with renorm the k weights are divided by their sum.

Logits decide integers (the ids), so they are defined bit for bit as an fp32
dot product in one fixed order ("order R"):
  * Split the d inputs into chunks of 8 consecutive elements.  Chunk c belongs
    to lane c mod 32.
  * Each lane starts from 0.0f.  It visits its chunks in ascending order and,
    within a chunk, its elements in ascending order.  Each step is
    acc = fl32(acc + fl32(x_i * w_i)).  Each bf16*bf16 product is exact in fp32.
  * The 32 lane sums are then combined by an xor butterfly with offsets
    16, 8, 4, 2, 1: p[j] <- fl32(p[j] + p[j ^ off]).
  * The logit is fl32(p[0] + bias[e]).
The softmax weights are computed in fp64 and rounded to fp32.
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_to_f32


def logits_order_r(x_bits: np.ndarray, wr_bits: np.ndarray, bias=None) -> np.ndarray:
    """x bf16 bits [T, d], W_r bf16 bits [E, d], bias fp32 [E] or None -> logits fp32 [T, E]."""
    x = bf16_to_f32(x_bits)
    w = bf16_to_f32(wr_bits)
    T, d = x.shape
    E = w.shape[0]
    assert d % 256 == 0, "order R needs d to be a multiple of 256 (32 lanes x 8)"
    S = d // 256
    xs = x.reshape(T, S, 32, 8)
    ws = w.reshape(E, S, 32, 8)
    acc = np.zeros((T, E, 32), np.float32)
    for s in range(S):                 # a lane's chunks, ascending
        for u in range(8):             # elements inside a chunk, ascending
            prod = xs[:, None, s, :, u] * ws[None, :, s, :, u]   # fp32, exact
            acc = (acc + prod).astype(np.float32)
    lanes = np.arange(32)
    for off in (16, 8, 4, 2, 1):
        acc = (acc + acc[:, :, lanes ^ off]).astype(np.float32)
    out = acc[:, :, 0]
    if bias is not None:
        out = (out + np.asarray(bias, np.float32)[None, :]).astype(np.float32)
    return out


def select_topk(logits: np.ndarray, k: int, renorm: int):
    """logits fp32 [T, E] -> ids int32 [T, k], w fp32 [T, k].

    ids are the k largest logits ordered by (logit desc, id asc).  w is the
    softmax probability of each chosen expert (fp64, rounded to fp32), divided
    by the chosen experts' probability sum when renorm is set.
    """
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    eid = np.arange(E)
    for t in range(T):
        lt = logits[t].astype(np.float64)
        order = np.lexsort((eid, -lt))          # primary: logit desc; secondary: id asc
        sel = order[:k]
        ids[t] = sel
        p = np.exp(lt - lt.max())
        p = p / p.sum()
        ps = p[sel]
        if renorm:
            ps = ps / ps.sum()
        w[t] = ps.astype(np.float32)
    return ids, w


def route(x_bits, wr_bits, bias, k: int, renorm: int):
    """Whole router: (ids int32 [T,k], w fp32 [T,k], logits fp32 [T,E])."""
    lg = logits_order_r(x_bits, wr_bits, bias)
    ids, w = select_topk(lg, k, renorm)
    return ids, w, lg
