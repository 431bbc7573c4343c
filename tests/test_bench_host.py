"""Host logic of bench.py on CPU: the LRU trace report, with the library's handle replaced
by the oracle's LRU and the CUDA events by host clocks.  The device replay itself is
checked against the oracle bit for bit by tests/test_gpu_lru.py."""
import sys
import time

import numpy as np
import torch

import synth
from oracle.lru import GlobalLRU


class _OracleHandle:
    def __init__(self, L, E, C):
        self.args = (L, E, C)
        self.o = GlobalLRU(L, E, C)

    def reset(self, stream=None):
        self.o = GlobalLRU(*self.args)

    def replay(self, trace, hit, slot, ev, cnt, stream=None):
        h, s, e = self.o.replay(trace.numpy())
        n = len(h)
        assert n <= hit.numel()
        hit[:n] = torch.from_numpy(np.asarray(h, np.uint8))
        slot[:n] = torch.from_numpy(np.asarray(s, np.int32))
        ev[:n] = torch.from_numpy(np.asarray(e, np.int32))
        cnt[0], cnt[1] = self.o.n_access, self.o.n_miss

    def close(self):
        pass


class _HostEvent:
    def __init__(self, enable_timing=False):
        self.t = 0.0

    def record(self, stream=None):
        self.t = time.perf_counter()

    def synchronize(self):
        pass

    def elapsed_time(self, other):
        return (other.t - self.t) * 1e3


def test_lru_report_counts_the_whole_trace(monkeypatch):
    import bench
    import sparse_moe_expert_sorted_b300 as ft
    monkeypatch.setattr(ft, "LRU", _OracleHandle)
    monkeypatch.setattr(torch.cuda, "Event", _HostEvent)
    w = synth.DECODE
    rep = bench.lru_replay(w, 4, False, dev="cpu")
    trace = synth.make_trace(w.trace_steps, 1, 4, w.layer.k, w.layer.E, w.zipf_s, seed=w.seed)
    o = GlobalLRU(1, w.layer.E, w.capacity)
    o.replay(trace)
    assert rep["accesses"] == o.n_access and rep["misses"] == o.n_miss
    assert rep["repeatable"] and rep["trace_steps"] == w.trace_steps and rep["capacity"] == 47
    # one access per distinct expert of a step: between k and min(B*k, E) per step
    assert w.trace_steps * w.layer.k <= rep["accesses"] <= w.trace_steps * 4 * w.layer.k
    assert bench.lru_replay(synth.PREFILL, 8192, False, dev="cpu") is None     # no slot table: nothing to replay
