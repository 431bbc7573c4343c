"""The decode-time expert cache around the LRU: the q* split of a step's misses and slot copies.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages:
  * when a selected expert is not resident, the engine either copies its weights
    over the host link and runs it on the GPU, or runs it where the weights are;
    for a step with m misses it fills q* ~= m * B_P / B_H of them, where B_P is
    the measured link (PCIe) bandwidth and B_H the measured host-memory
    bandwidth, and the two partial sums merge exactly after the layer
    (banandre.com, "The 284B Model on a 32GB GPU Trick", section "The q* Policy:
    Math Instead of Guesses");
  * the cache is a global LRU that admits every missed expert (asapai.co.kr,
    "Running 753B GLM-5.2 on a single workstation GPU", section "Abandoning fixed
    offloading in favor of measured bandwidth").

Reading (the pages leave these open):
  * the second executor is the complement partial of the exact merge; on this
    library both executors are GPU work: executor A reads experts from their
    HBM slots, executor B streams the weights of the other experts straight from
    the host pool;
  * m counts the misses of the call (accesses with hit = 0); the fill count is
    q* rounded to the nearest integer (halves up), at most the misses that are
    still resident when the call's accesses are done;
  * an expert of the call is computed by A when its key is resident after the
    call (slot_of >= 0): every resident hit, and the first n_fill resident misses
    in access order (ascending expert id), whose slots are filled first
    ("fill now"); every other expert of the call is computed by B from pool slot
    layer * E + e; the other resident misses are filled after the step ("fill
    later"), so that the slot map stays true;
  * a slot copy moves every byte of one slot of a weight arena to a slot of
    another (or the same) arena: codes, scales, tensor scales, prepared layouts.
"""
from __future__ import annotations

import math

import numpy as np


def qstar(m: int, B_P: float, B_H: float) -> float:
    """q* = m * B_P / B_H (fp64)."""
    return float(m) * float(B_P) / float(B_H)


def fill_count(m: int, B_P: float, B_H: float) -> int:
    """Experts of a step's m misses to fill: q* rounded half up, within [0, m]."""
    q = qstar(m, B_P, B_H)
    return int(max(0, min(m, math.floor(q + 0.5))))


def miss_split(slot_of_after: np.ndarray, layer: int, ids: np.ndarray, hit: np.ndarray, n_fill: int):
    """Split one LRU call's experts between the two executors.

    slot_of_after: the LRU's slot table [L, E] after the call; ids: the call's top-k ids;
    hit: the call's per-access hit flags (accesses = unique ids, ascending).
    Returns dict with slot_of_a [E] (arena slot or -1), slot_of_b [E] (pool slot
    layer * E + e or -1), fill_now and fill_later int32 [n, 2] of (pool slot, arena slot),
    and the counts m (misses) and n_fill (filled now)."""
    L, E = slot_of_after.shape
    experts = np.unique(np.asarray(ids).reshape(-1))
    assert len(experts) == len(hit)
    a = np.full(E, -1, np.int32)
    b = np.full(E, -1, np.int32)
    now, later = [], []
    m = int(np.sum(np.asarray(hit) == 0))
    filled = 0
    for i, e in enumerate(experts):
        e = int(e)
        s = int(slot_of_after[layer, e])
        pool = layer * E + e
        if s < 0:
            b[e] = pool
        elif hit[i]:
            a[e] = s
        elif filled < n_fill:
            a[e] = s
            now.append((pool, s))
            filled += 1
        else:
            b[e] = pool
            later.append((pool, s))
    as_pairs = lambda v: np.array(v, np.int32).reshape(-1, 2)
    return dict(slot_of_a=a, slot_of_b=b, fill_now=as_pairs(now), fill_later=as_pairs(later), m=m, n_fill=filled)


def copy_slots(src: dict, dst: dict, pairs: np.ndarray) -> dict:
    """dst with slot t replaced by slot s of src for every (s, t) in pairs (arrays of the
    oracle's weight dict: gate, up, down, *_s, glob; slot-major)."""
    out = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in dst.items()}
    for s, t in np.asarray(pairs).reshape(-1, 2):
        for name in ("gate", "up", "down", "gate_s", "up_s", "down_s", "glob"):
            if out.get(name) is not None:
                out[name][t] = src[name][s]
    return out
