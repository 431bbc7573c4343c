"""Pins of the oracle's expert-sorted permutation: an O(P*E) brute-force scan
and the invariants of a stable counting sort."""
import numpy as np
import pytest

from oracle.permute import permute


def brute_force(ids, E):
    flat = list(np.asarray(ids).reshape(-1))
    sorted_pair, offsets = [], [0]
    for e in range(E):
        for p, v in enumerate(flat):
            if v == e:
                sorted_pair.append(p)
        offsets.append(len(sorted_pair))
    pair_pos = [0] * len(flat)
    for j, p in enumerate(sorted_pair):
        pair_pos[p] = j
    return np.array(offsets), np.array(sorted_pair, dtype=np.int64), np.array(pair_pos, dtype=np.int64)


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (16, 8, 2), (37, 16, 4), (5, 4, 4), (64, 256, 6)])
def test_permute_matches_brute_force(T, E, k):
    g = np.random.default_rng(T * 100 + E)
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    off, sp, pp = permute(ids, E)
    bo, bs, bp = brute_force(ids, E)
    assert np.array_equal(off, bo) and np.array_equal(sp, bs) and np.array_equal(pp, bp)
    assert off[-1] == T * k
    assert np.array_equal(pp[sp], np.arange(T * k))
    flat = ids.reshape(-1)
    for e in range(E):
        seg = sp[off[e]:off[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


def test_all_pairs_on_one_expert_and_empty_experts():
    ids = np.zeros((10, 1), np.int32) + 3
    off, sp, pp = permute(ids, 8)
    assert list(off) == [0, 0, 0, 0, 10, 10, 10, 10, 10]
    assert list(sp) == list(range(10))
