"""Randomised pins of the oracle (hypothesis): the same independent checks as the fixed
cases in test_oracle_route / test_oracle_permute / test_oracle_lru, over drawn shapes,
seeds and tie patterns.
  * selection: the chosen set maximises the summed logit, ties broken toward the
    lexicographically smallest ids (brute force over every k-subset), ordered by
    (logit desc, id asc); weights non-negative, non-increasing along the ranks, and
    summing to 1 with renorm;
  * permutation: the O(P*E) scan;
  * LRU: Mattson's stack-distance rule and a move-to-front list.
"""
import itertools

import numpy as np
from hypothesis import given, settings
from hypothesis import strategies as st

from oracle import route as R
from oracle.lru import GlobalLRU
from oracle.permute import permute

from test_oracle_lru import _keys_of_trace, move_to_front, stack_distance_hits
from test_oracle_permute import brute_force

SETTINGS = settings(max_examples=40, deadline=None, derandomize=True)   # the same draws every run


@SETTINGS
@given(E=st.integers(1, 8), data=st.data(), seed=st.integers(0, 2 ** 31 - 1),
       levels=st.sampled_from([3, 5, 1000]), renorm=st.integers(0, 1))
def test_selection_is_the_best_subset(E, data, seed, levels, renorm):
    k = data.draw(st.integers(1, E))
    T = 3
    g = np.random.default_rng(seed)
    lg = (g.integers(0, levels, size=(T, E)) / 4.0 - 1.0).astype(np.float32)   # few levels: many ties
    ids, w = R.select_topk(lg, k, renorm)
    for t in range(T):
        best = max(itertools.combinations(range(E), k),
                   key=lambda c: (sum(float(lg[t, e]) for e in c), [-e for e in c]))
        assert sorted(ids[t].tolist()) == sorted(best)
        order = sorted(best, key=lambda e: (-float(lg[t, e]), e))
        assert ids[t].tolist() == order
        assert np.all(w[t] >= 0) and np.all(np.diff(w[t]) <= 0)   # tiny probabilities may round to 0
        if renorm:
            assert abs(float(w[t].astype(np.float64).sum()) - 1.0) < 1e-6


@SETTINGS
@given(T=st.integers(1, 40), E=st.integers(1, 24), data=st.data(), seed=st.integers(0, 2 ** 31 - 1))
def test_permutation_matches_the_scan(T, E, data, seed):
    k = data.draw(st.integers(1, E))
    g = np.random.default_rng(seed)
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    off, sp, pp = permute(ids, E)
    bo, bs, bp = brute_force(ids, E)
    assert np.array_equal(off, bo) and np.array_equal(sp, bs) and np.array_equal(pp, bp)


@SETTINGS
@given(L=st.integers(1, 3), E=st.integers(2, 12), C=st.integers(1, 20), B=st.integers(1, 3),
       data=st.data(), seed=st.integers(0, 2 ** 31 - 1))
def test_lru_matches_stack_distance_and_move_to_front(L, E, C, B, data, seed):
    k = data.draw(st.integers(1, E))
    steps = 30
    g = np.random.default_rng(seed)
    trace = np.stack([np.stack([np.stack([g.permutation(E)[:k] for _ in range(B)]) for _ in range(L)])
                      for _ in range(steps)]).astype(np.int32)
    lru = GlobalLRU(L, E, C)
    hit, slot, ev = lru.replay(trace)
    keys = _keys_of_trace(trace, E)
    assert list(hit) == stack_distance_hits(keys, C)
    mh, ms, mv = move_to_front(keys, C)
    assert list(hit) == mh and list(slot) == ms and list(ev) == mv
    assert lru.n_access == len(keys) and lru.n_miss + int(hit.sum()) == len(keys)
    resident = lru.slot_of.reshape(-1)
    live = resident[resident >= 0]
    assert len(live) == min(C, len(set(keys))) and len(set(live.tolist())) == len(live)
