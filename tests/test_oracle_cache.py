"""Pins of the oracle's expert-cache pieces: the q* fill count, the split of a step's
experts between the two executors, slot copies and the elastic resize of the LRU.

  * q*: the pages define it from a balance (banandre.com, "The 284B Model on a 32GB GPU
    Trick", section "The q* Policy"): filling q experts over the link at B_P takes as long
    as computing the other m - q where the weights are, at the residual host bandwidth
    B_H - B_P.  The test checks that balance, the limits, and the fill counts for the
    bandwidth pairs the pages print (52.7 : 77.3 and 11.8 : 47.5 GB/s) at m = 8.
  * The split: invariants that follow from the reading in oracle/cache.py, over many
    LRU calls drawn at random.
  * Resize: (a) Mattson's inclusion property of LRU: after shrinking to C', the hits and
    misses from then on equal those of an LRU of capacity C' run on the whole trace;
    (b) a list-based move-to-front model with a capacity that changes between calls
    (an independent implementation) gives the same hits, misses and resident sets under
    any schedule of resizes; (c) the slot map stays a bijection onto slots 0 .. used-1.
"""
import math

import numpy as np
import pytest

from oracle import cache as Q
from oracle.lru import GlobalLRU


# ------------------------------------------------------------------------------------
# q*
# ------------------------------------------------------------------------------------
def test_qstar_balances_the_fill_against_the_second_executor():
    g = np.random.default_rng(3)
    for _ in range(200):
        m = int(g.integers(1, 64))
        B_H = float(g.uniform(10, 500))
        B_P = float(g.uniform(0.01, 0.999)) * B_H
        q = Q.qstar(m, B_P, B_H)
        # time to fill q experts of size S over the link == time to compute m - q at B_H - B_P
        assert abs(q / B_P - (m - q) / (B_H - B_P)) <= 1e-12 * (m / B_P)
        n = Q.fill_count(m, B_P, B_H)
        assert 0 <= n <= m and abs(n - q) <= 0.5


def test_qstar_at_the_pages_bandwidth_pairs():
    # worked by hand: 8 * 52.7 / 77.3 = 421.6 / 77.3 = 5.4541; 8 * 11.8 / 47.5 = 94.4 / 47.5 = 1.9874
    assert abs(Q.qstar(8, 52.7, 77.3) - 5.4541) < 1e-4
    assert abs(Q.qstar(8, 11.8, 47.5) - 1.9874) < 1e-4
    assert Q.fill_count(8, 52.7, 77.3) == 5
    assert Q.fill_count(8, 11.8, 47.5) == 2


def test_qstar_limits_and_rounding():
    assert Q.fill_count(7, 50.0, 50.0) == 7          # no residual host bandwidth: fill everything
    assert Q.fill_count(7, 1e-9, 50.0) == 0          # no link: fill nothing
    assert Q.fill_count(1, 1.0, 2.0) == 1            # q* = 0.5 rounds half up
    assert Q.fill_count(3, 1.0, 2.0) == 2            # 1.5 -> 2
    assert Q.fill_count(0, 1.0, 2.0) == 0


# ------------------------------------------------------------------------------------
# the split of a call's experts
# ------------------------------------------------------------------------------------
def test_miss_split_invariants_over_random_calls():
    g = np.random.default_rng(11)
    for trial in range(30):
        L, E = int(g.integers(1, 4)), int(g.integers(4, 40))
        C = int(g.integers(1, L * E + 1))
        B, k = int(g.integers(1, 6)), int(g.integers(1, min(E, 6) + 1))
        lru = GlobalLRU(L, E, C)
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        p /= p.sum()
        for step in range(20):
            layer = int(g.integers(0, L))
            ids = np.stack([g.choice(E, k, replace=False, p=p) for _ in range(B)]).astype(np.int32)
            experts, hit, slot, ev = lru.step(layer, ids)
            n_fill = int(g.integers(0, len(experts) + 1))
            r = Q.miss_split(lru.slot_of, layer, ids, hit, n_fill)
            a, b = r["slot_of_a"], r["slot_of_b"]
            in_call = np.zeros(E, bool)
            in_call[experts] = True
            # every expert of the call goes to exactly one executor; nothing else does
            assert np.all((a >= 0) ^ (b >= 0) == in_call)
            # A reads resident slots; B reads pool slot layer * E + e
            assert np.all(a[a >= 0] == lru.slot_of[layer][a >= 0])
            assert np.all(b[b >= 0] == layer * E + np.flatnonzero(b >= 0))
            res_miss = [int(e) for i, e in enumerate(experts) if not hit[i] and lru.slot_of[layer, e] >= 0]
            fills = np.concatenate([r["fill_now"], r["fill_later"]])
            assert sorted(fills[:, 0].tolist()) == sorted(layer * E + e for e in res_miss)
            assert np.all(fills[:, 1] == lru.slot_of[layer][fills[:, 0] - layer * E])
            assert len(set(fills[:, 1].tolist())) == len(fills)
            # fill now: the first n_fill resident misses in ascending expert order, all computed by A
            now = (r["fill_now"][:, 0] - layer * E).tolist()
            assert now == res_miss[:min(n_fill, len(res_miss))]
            assert all(a[e] >= 0 for e in now)
            later = (r["fill_later"][:, 0] - layer * E).tolist()
            assert all(b[e] >= 0 for e in later)
            assert r["m"] == int(np.sum(hit == 0))


def test_copy_slots_moves_whole_slots():
    src = dict(gate=np.arange(12).reshape(4, 3), up=np.arange(12).reshape(4, 3) + 100, down=np.zeros((4, 2)),
               gate_s=None, up_s=None, down_s=None, glob=np.arange(12.0).reshape(4, 3))
    dst = {k: (None if v is None else np.zeros_like(v)) for k, v in src.items()}
    out = Q.copy_slots(src, dst, np.array([[3, 0], [1, 2]]))
    assert np.array_equal(out["gate"][0], src["gate"][3]) and np.array_equal(out["up"][2], src["up"][1])
    assert np.all(out["gate"][1] == 0) and np.array_equal(out["glob"][0], src["glob"][3])
    assert np.all(dst["gate"] == 0)


# ------------------------------------------------------------------------------------
# elastic resize
# ------------------------------------------------------------------------------------
class MtfModel:
    """Move-to-front list of resident keys (most recent first) with a capacity that may
    change between calls.  Independent of the timestamp oracle."""

    def __init__(self, C):
        self.C = C
        self.lst = []

    def access(self, key):
        if key in self.lst:
            self.lst.remove(key)
            self.lst.insert(0, key)
            return 1
        self.lst.insert(0, key)
        if len(self.lst) > self.C:
            self.lst.pop()
        return 0

    def resize(self, C):
        self.C = C
        del self.lst[C:]


def _trace(g, steps, L, E, k):
    p = 1.0 / np.arange(1, E + 1) ** 1.0
    p /= p.sum()
    return [(int(g.integers(0, L)), np.sort(g.choice(E, k, replace=False, p=p))) for _ in range(steps)]


def _check_map(lru):
    used = np.flatnonzero(lru.key_of >= 0)
    assert np.array_equal(used, np.arange(len(used)))              # occupied slots are 0 .. used-1
    for s in used:
        key = int(lru.key_of[s])
        assert lru.slot_of[key // lru.E, key % lru.E] == s
    assert np.sum(lru.slot_of >= 0) == len(used)


def test_shrink_follows_mattson_inclusion():
    g = np.random.default_rng(5)
    for trial in range(20):
        L, E, k = 2, 24, 3
        C, C2 = int(g.integers(6, 30)), None
        C2 = int(g.integers(1, C))
        tr = _trace(g, 120, L, E, k)
        cut = int(g.integers(10, 110))
        big, small = GlobalLRU(L, E, C), GlobalLRU(L, E, C2)
        hits_small = []
        for i, (l, ids) in enumerate(tr):
            if i == cut:
                moves, ev = big.resize(C2)
                # the resident set equals that of the capacity-C2 cache, whatever the history
                assert set(big.key_of[big.key_of >= 0].tolist()) == set(small.key_of[small.key_of >= 0].tolist())
                _check_map(big)
            _, h, _, _ = big.step(l, ids)
            _, hs, _, _ = small.step(l, ids)
            if i >= cut:
                assert np.array_equal(h, hs)


def test_resize_schedules_match_a_move_to_front_list():
    g = np.random.default_rng(9)
    for trial in range(25):
        L, E, k = int(g.integers(1, 4)), int(g.integers(6, 30)), 2
        C = int(g.integers(1, L * E))
        lru, mtf = GlobalLRU(L, E, C), MtfModel(C)
        for i, (l, ids) in enumerate(_trace(g, 150, L, E, min(k, E))):
            if i % 17 == 16:
                C = int(g.integers(1, L * E + 4))
                used_before = int(np.sum(lru.key_of >= 0))
                moves, ev = lru.resize(C)
                mtf.resize(C)
                assert len(moves) == min(used_before, C) and len(ev) == used_before - len(moves)
                assert len(set(moves[:, 1].tolist())) == len(moves) and np.all(moves[:, 1] < C)
                assert np.all(moves[:, 0] == np.sort(moves[:, 0]))
                # keys that stay below the new capacity keep their slot
                stay = moves[moves[:, 0] < C]
                assert np.array_equal(stay[:, 0], stay[:, 1])
                _check_map(lru)
            _, h, _, _ = lru.step(l, ids)
            want = [mtf.access(l * E + int(e)) for e in ids]
            assert h.tolist() == want
            keys = [int(x) for x in lru.key_of[lru.recency()]]
            assert keys == mtf.lst                                   # same keys, same recency order


def test_grow_then_shrink_back_changes_nothing():
    g = np.random.default_rng(2)
    lru = GlobalLRU(2, 20, 9)
    for l, ids in _trace(g, 60, 2, 20, 3):
        lru.step(l, ids)
    before = (lru.slot_of.copy(), lru.key_of.copy(), lru.stamp.copy())
    m1, e1 = lru.resize(15)
    assert len(e1) == 0 and np.array_equal(m1[:, 0], m1[:, 1])
    m2, e2 = lru.resize(9)
    assert len(e2) == 0 and np.array_equal(m2[:, 0], m2[:, 1])
    assert np.array_equal(lru.slot_of, before[0]) and np.array_equal(lru.key_of, before[1])
    assert np.array_equal(lru.stamp, before[2])


def test_resize_rejects_an_empty_cache():
    with pytest.raises(ValueError):
        GlobalLRU(1, 4, 2).resize(0)
