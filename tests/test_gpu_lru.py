"""Parity of the device global LRU (ftmoe_slot_lru, ftmoe_slot_lru_replay)
with the oracle, bit-exact:
  * the hit / slot / evicted-key sequence;
  * the running access and miss counts;
  * the final slot_of table.
Cases:
  * the hand-worked example;
  * call-by-call use;
  * the full replays of the two decode workloads: 4096 steps over 128 experts
    with 47 slots, and 2048 steps x 8 layers over 256 experts with 225 global
    slots.
"""
import json
import os

import numpy as np
import pytest
import torch

import synth
from oracle.lru import GlobalLRU

from gpu_helpers import ensure_built
import sparse_moe_expert_sorted_b300 as ft

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _replay_device(L, E, C, trace):
    lru = ft.LRU(L, E, C)
    steps, _, B, k = trace.shape
    cap = steps * L * min(B * k, E)
    hit = torch.empty(cap, dtype=torch.uint8, device="cuda")
    slot = torch.empty(cap, dtype=torch.int32, device="cuda")
    ev = torch.empty(cap, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(2, dtype=torch.int64, device="cuda")
    lru.replay(torch.from_numpy(np.ascontiguousarray(trace)).cuda(), hit, slot, ev, cnt)
    n = int(cnt[0])
    out = (hit[:n].cpu().numpy(), slot[:n].cpu().numpy(), ev[:n].cpu().numpy(), cnt.cpu().numpy(),
           lru.slot_of().cpu().numpy())
    lru.close()
    return out


def test_worked_example_call_by_call():
    g = json.load(open(os.path.join(GOLD, "lru_worked_example.json")))
    lru = ft.LRU(g["L"], g["E"], g["C"])
    got = []
    cnt = torch.zeros(2, dtype=torch.int64, device="cuda")
    for call in g["calls"]:
        ids = torch.tensor(call["ids"], dtype=torch.int32, device="cuda")
        n = min(ids.numel(), g["E"])
        hit = torch.empty(n, dtype=torch.uint8, device="cuda")
        slot = torch.empty(n, dtype=torch.int32, device="cuda")
        ev = torch.empty(n, dtype=torch.int32, device="cuda")
        before = int(cnt[0])
        lru.step(call["layer"], ids, hit, slot, ev, cnt)
        m = int(cnt[0]) - before
        got += [dict(hit=int(a), slot=int(b), evicted=int(c)) for a, b, c in
                zip(hit[:m].tolist(), slot[:m].tolist(), ev[:m].tolist())]
    want = [{k: a[k] for k in ("hit", "slot", "evicted")} for a in g["accesses"]]
    assert got == want
    assert int(cnt[1]) == g["misses"]
    assert lru.slot_of().cpu().tolist() == g["final_slot_of"]
    lru.reset()
    assert (lru.slot_of() == -1).all()


@pytest.mark.parametrize("L,E,C,B,k,s,steps", [(1, 16, 5, 2, 2, 1.1, 200), (3, 8, 4, 1, 2, 0.5, 300),
                                               (2, 64, 1, 4, 3, 1.0, 100), (2, 32, 64, 8, 4, 1.0, 50)])
def test_replay_small(L, E, C, B, k, s, steps):
    trace = synth.make_trace(steps, L, B, k, E, s, seed=L + C)
    o = GlobalLRU(L, E, C)
    oh, os_, oe = o.replay(trace)
    h, sl, ev, cnt, slot_of = _replay_device(L, E, C, trace)
    assert np.array_equal(h, oh) and np.array_equal(sl, os_) and np.array_equal(ev, oe)
    assert cnt.tolist() == [o.n_access, o.n_miss]
    assert np.array_equal(slot_of, o.slot_of)


@pytest.mark.parametrize("B", [1, 4, 16])
def test_replay_decode_workload_trace(B):
    w = synth.DECODE
    trace = synth.make_trace(w.trace_steps, 1, B, w.layer.k, w.layer.E, w.zipf_s, seed=w.seed)
    o = GlobalLRU(1, w.layer.E, w.capacity)
    oh, os_, oe = o.replay(trace)
    h, sl, ev, cnt, slot_of = _replay_device(1, w.layer.E, w.capacity, trace)
    assert np.array_equal(h, oh) and np.array_equal(sl, os_) and np.array_equal(ev, oe)
    assert cnt.tolist() == [o.n_access, o.n_miss]
    assert np.array_equal(slot_of, o.slot_of)


@pytest.mark.parametrize("B", [1, 16])
def test_replay_stack_workload_trace(B):
    w = synth.STACK
    trace = synth.make_trace(w.trace_steps, w.layers, B, w.layer.k, w.layer.E, w.zipf_s, seed=w.seed)
    o = GlobalLRU(w.layers, w.layer.E, w.capacity)
    oh, os_, oe = o.replay(trace)
    h, sl, ev, cnt, slot_of = _replay_device(w.layers, w.layer.E, w.capacity, trace)
    assert np.array_equal(h, oh) and np.array_equal(sl, os_) and np.array_equal(ev, oe)
    assert cnt.tolist() == [o.n_access, o.n_miss]
    assert np.array_equal(slot_of, o.slot_of)


def test_replay_output_capacity_is_checked_on_the_device():
    """Output buffers shorter than the trace's accesses: the first `capacity` accesses are
    written, the running counts still cover the whole trace, and the device error word
    reads 3 (output capacity); nothing is written past the buffers."""
    L, E, C, B, k, steps = 1, 16, 5, 2, 2, 50
    trace = synth.make_trace(steps, L, B, k, E, 1.1, seed=3)
    o = GlobalLRU(L, E, C)
    oh, os_, oe = o.replay(trace)
    cap = len(oh) // 2
    lru = ft.LRU(L, E, C)
    guard = 64
    hit = torch.full((cap + guard,), 7, dtype=torch.uint8, device="cuda")
    slot = torch.full((cap + guard,), -9, dtype=torch.int32, device="cuda")
    ev = torch.full((cap + guard,), -9, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(2, dtype=torch.int64, device="cuda")
    ft.get_device_error()                                   # clear
    lru.replay(torch.from_numpy(np.ascontiguousarray(trace)).cuda(), hit[:cap], slot[:cap], ev[:cap], cnt)
    assert ft.get_device_error() == 3
    assert np.array_equal(hit[:cap].cpu().numpy(), oh[:cap])
    assert np.array_equal(slot[:cap].cpu().numpy(), os_[:cap])
    assert np.array_equal(ev[:cap].cpu().numpy(), oe[:cap])
    assert (hit[cap:] == 7).all() and (slot[cap:] == -9).all() and (ev[cap:] == -9).all()
    assert cnt.cpu().tolist() == [o.n_access, o.n_miss]
    assert np.array_equal(lru.slot_of().cpu().numpy(), o.slot_of)
    lru.close()
