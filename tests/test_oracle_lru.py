"""Pins of the oracle's global LRU slot map.

  * a worked example derived by hand (tests/golden/lru_worked_example.json);
  * Mattson's stack-distance rule: an access hits iff fewer than C distinct
    keys were touched since the key's previous access (LRU inclusion);
  * a move-to-front list that tracks slots and victims (an independent
    implementation of the same policy);
  * closed cases: C >= #keys gives compulsory misses only, C = 1 misses
    iff the key changes, and a cyclic sweep longer than C always misses.
"""
import json
import os

import numpy as np
import pytest

import synth
from oracle.lru import GlobalLRU

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_worked_example():
    g = json.load(open(os.path.join(GOLD, "lru_worked_example.json")))
    lru = GlobalLRU(g["L"], g["E"], g["C"])
    got = []
    for call in g["calls"]:
        ex, h, s, v = lru.step(call["layer"], np.array(call["ids"]))
        got += [dict(key=call["layer"] * g["E"] + int(e), hit=int(a), slot=int(b), evicted=int(c))
                for e, a, b, c in zip(ex, h, s, v)]
    want = [{k: a[k] for k in ("key", "hit", "slot", "evicted")} for a in g["accesses"]]
    assert got == want
    assert lru.n_miss == g["misses"]
    assert lru.slot_of.tolist() == g["final_slot_of"]


def _keys_of_trace(trace, E):
    keys = []
    for t in range(trace.shape[0]):
        for l in range(trace.shape[1]):
            keys += [l * E + int(e) for e in np.unique(trace[t, l])]
    return keys


def stack_distance_hits(keys, C):
    hits, last = [], {}
    for i, key in enumerate(keys):
        if key in last:
            distinct = len(set(keys[last[key] + 1:i]))
            hits.append(1 if distinct < C else 0)
        else:
            hits.append(0)
        last[key] = i
    return hits


def move_to_front(keys, C):
    order, slot_of_key, hits, slots, victims = [], {}, [], [], []
    for key in keys:
        if key in slot_of_key:
            order.remove(key)
            order.insert(0, key)
            hits.append(1)
            slots.append(slot_of_key[key])
            victims.append(-1)
            continue
        if len(order) < C:
            s, v = len(order), -1
        else:
            v = order.pop()
            s = slot_of_key.pop(v)
        order.insert(0, key)
        slot_of_key[key] = s
        hits.append(0)
        slots.append(s)
        victims.append(v)
    return hits, slots, victims


@pytest.mark.parametrize("L,E,B,k,C,s", [(1, 16, 2, 2, 5, 1.1), (2, 16, 4, 3, 7, 1.0), (3, 8, 1, 2, 4, 0.5),
                                         (1, 32, 8, 4, 12, 1.1)])
def test_replay_matches_stack_distance_and_move_to_front(L, E, B, k, C, s):
    trace = synth.make_trace(60, L, B, k, E, s, seed=L * 7 + C)
    lru = GlobalLRU(L, E, C)
    hit, slot, ev = lru.replay(trace)
    keys = _keys_of_trace(trace, E)
    assert list(hit) == stack_distance_hits(keys, C)
    mh, ms, mv = move_to_front(keys, C)
    assert list(hit) == mh and list(slot) == ms and list(ev) == mv
    assert lru.n_access == len(keys) and lru.n_miss == len(keys) - int(hit.sum())


def test_closed_cases():
    trace = synth.make_trace(50, 2, 3, 2, 8, 1.0, seed=9)
    keys = _keys_of_trace(trace, 8)
    lru = GlobalLRU(2, 8, 16)
    hit, _, _ = lru.replay(trace)
    assert lru.n_miss == len(set(keys))                        # C >= keys: compulsory only
    lru = GlobalLRU(1, 8, 1)
    one = np.array([3, 3, 5, 5, 5, 3, 1, 1]).reshape(8, 1, 1, 1)
    hit, slot, _ = lru.replay(one)
    assert list(hit) == [0, 1, 0, 1, 1, 0, 0, 1] and set(slot) == {0}
    lru = GlobalLRU(1, 8, 4)
    cyc = np.array([i % 5 for i in range(40)]).reshape(40, 1, 1, 1)
    hit, _, _ = lru.replay(cyc)
    assert hit.sum() == 0                                     # a sweep of 5 keys through 4 slots
