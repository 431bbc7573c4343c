"""Expert-sorted permutation of the (token, rank) pairs.

The pages never describe this step; it is what "compute each selected expert
once" implies for a batch: every pair p = t*k + r that selected expert e must
be gathered next to the other pairs of e (banandre.com, "The 284B Model on a
32GB GPU Trick", section "Sparsity Is a Lie (But a Useful One)").

Definition (a stable counting sort by expert id):
  counts[e]      = number of pairs with ids[p] == e
  offsets        = exclusive prefix sum of counts, offsets[E] = P
  sorted_pair    = pair indices ordered by (expert id, pair index)
  pair_pos[p]    = position of pair p in sorted_pair
"""
from __future__ import annotations

import numpy as np


def permute(ids: np.ndarray, E: int):
    """ids int32 [T, k] -> (offsets int32 [E+1], sorted_pair int32 [P], pair_pos int32 [P])."""
    flat = np.asarray(ids, np.int64).reshape(-1)
    P = flat.size
    order = np.argsort(flat, kind="stable")      # stable: ties keep ascending pair index
    counts = np.bincount(flat, minlength=E)[:E]
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    pair_pos = np.empty(P, np.int64)
    pair_pos[order] = np.arange(P)
    return offsets.astype(np.int32), order.astype(np.int32), pair_pos.astype(np.int32)
