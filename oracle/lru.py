"""Global LRU slot map over (layer, expert) keys.

The pages:
  * in decode the expert cache is one global LRU that admits every missed expert
    (asapai.co.kr, "Running 753B GLM-5.2 on a single workstation GPU",
    section "Abandoning fixed offloading in favor of measured bandwidth");
  * the LRU is shared by all MoE layers (banandre.com, "The 284B Model on a
    32GB GPU Trick", section "Semantic-Aware Caching: Because Agents Lie");
  * the first request is served from a cold cache (same page, section
    "Elastic Memory: The VRAM Budget Is a Suggestion").

Reading, where the pages are silent:
  * One access per unique (layer, expert) of a decode step.  Within one call
    the experts are visited in ascending id order.
  * A hit refreshes recency.  Every miss admits its key: it takes the lowest
    free slot, else it evicts the least recently used key and reuses that
    key's slot.
  * A key touched earlier in the same step can be evicted by a later miss of
    that step.
  * The key of (layer l, expert e) is l*E + e.

This oracle keeps a last-use timestamp per slot and scans for the minimum.
"""
from __future__ import annotations

import numpy as np


class GlobalLRU:
    def __init__(self, L: int, E: int, C: int):
        self.L, self.E, self.C = L, E, C
        self.reset()

    def reset(self):
        self.slot_of = np.full((self.L, self.E), -1, np.int32)
        self.key_of = np.full(self.C, -1, np.int64)
        self.stamp = np.zeros(self.C, np.int64)
        self.clock = 0
        self.n_access = 0
        self.n_miss = 0

    def access(self, layer: int, e: int):
        """One access of (layer, e) -> (hit, slot, evicted key or -1)."""
        self.clock += 1
        self.n_access += 1
        s = int(self.slot_of[layer, e])
        if s >= 0:
            self.stamp[s] = self.clock
            return 1, s, -1
        self.n_miss += 1
        free = np.flatnonzero(self.key_of < 0)
        if free.size:
            s, ev = int(free[0]), -1
        else:
            s = int(np.argmin(self.stamp))
            ev = int(self.key_of[s])
            self.slot_of[ev // self.E, ev % self.E] = -1
        self.key_of[s] = layer * self.E + e
        self.slot_of[layer, e] = s
        self.stamp[s] = self.clock
        return 0, s, ev

    def step(self, layer: int, ids: np.ndarray):
        """All accesses of one call: the unique experts of ids, ascending.
        Returns int arrays (experts, hit, slot, evicted)."""
        experts = np.unique(np.asarray(ids).reshape(-1))
        res = [self.access(layer, int(e)) for e in experts]
        hit = np.array([r[0] for r in res], np.uint8)
        slot = np.array([r[1] for r in res], np.int32)
        ev = np.array([r[2] for r in res], np.int32)
        return experts.astype(np.int32), hit, slot, ev

    def replay(self, trace: np.ndarray):
        """trace int32 [steps, L, B, k] -> concatenated (hit, slot, evicted) of every access,
        in order step-major, then layer, then expert id."""
        H, S, V = [], [], []
        for t in range(trace.shape[0]):
            for l in range(trace.shape[1]):
                _, h, s, v = self.step(l, trace[t, l])
                H.append(h)
                S.append(s)
                V.append(v)
        cat = lambda xs, dt: np.concatenate(xs).astype(dt) if xs else np.zeros(0, dt)
        return cat(H, np.uint8), cat(S, np.int32), cat(V, np.int32)

    # ------------------------------------------------------------------------------
    # elastic resize at a safe point
    # ------------------------------------------------------------------------------
    def recency(self) -> np.ndarray:
        """Slots of the resident keys, most recently used first."""
        used = np.flatnonzero(self.key_of >= 0)
        return used[np.argsort(-self.stamp[used], kind="stable")]

    def resize(self, C_new: int):
        """Rebuild the slot map under a new capacity C_new, between calls.

        The pages: at scheduler safe points the expert cache is rebuilt under a
        revised VRAM budget, without reloading the host pool (banandre.com, "The
        284B Model on a 32GB GPU Trick", section "Elastic Memory: The VRAM Budget
        Is a Suggestion").

        Reading:
          * the C_new most recently used keys stay resident, in the same recency
            order; the others are evicted;
          * a kept key whose slot is below C_new keeps it; the kept keys in slots
            >= C_new (ascending) move to the freed slots below C_new (ascending),
            so the occupied slots stay 0 .. used-1 and a later miss still takes
            the lowest free slot;
          * growing keeps every key in its slot; the new slots are free.

        Returns (moves int32 [n_kept, 2] of (old slot, new slot) for every kept key
        in ascending old slot, evicted keys int64 in recency order)."""
        if C_new < 1:
            raise ValueError("capacity must be at least 1")
        order = self.recency()
        kept, gone = order[:C_new], order[C_new:]
        evicted = self.key_of[gone].copy()
        for key in evicted:
            self.slot_of[key // self.E, key % self.E] = -1
        keep = np.zeros(self.C, bool)
        keep[kept] = True
        high = [s for s in range(C_new, self.C) if keep[s]]
        free_low = [s for s in range(min(C_new, self.C)) if not keep[s]]
        new_slot = {int(s): int(s) for s in kept if s < C_new}
        for s, t in zip(high, free_low):
            new_slot[s] = t
        key_of = np.full(C_new, -1, np.int64)
        stamp = np.zeros(C_new, np.int64)
        for s, t in new_slot.items():
            key_of[t] = self.key_of[s]
            stamp[t] = self.stamp[s]
            key = int(self.key_of[s])
            self.slot_of[key // self.E, key % self.E] = t
        self.key_of, self.stamp, self.C = key_of, stamp, C_new
        moves = np.array(sorted(new_slot.items()), np.int32).reshape(-1, 2)
        return moves, evicted
