"""GPU parity of the expert cache around the LRU: elastic resize, the q* split, slot copies
from a pinned host pool, and whole decode steps through the two executors.

  * ftmoe_lru_resize: hit / slot / evicted sequences, moves and the final slot table equal
    the oracle's (oracle/lru.py, GlobalLRU.resize) bit for bit over traces with resizes.
  * ftmoe_miss_split: the two slot tables, the fill lists and the counts equal the oracle's
    (oracle/cache.py) bit for bit.
  * ftmoe_copy_slots: a fill from the pinned host pool, an in-place compaction after a
    shrink and a migration to a larger arena leave every resident slot byte-equal to its
    key's pool slot, prepared layouts included.
  * Decode steps with a cache: route, permute, LRU, split, fill, executor A (HBM arena) and
    executor B (host pool), merged by ftmoe_combine: the output equals the oracle's full
    layer (every expert from the pool) within 5e-3 relative L2 per token, ids bit-exact.

The pages: banandre.com, "The 284B Model on a 32GB GPU Trick", sections "The q* Policy" and
"Elastic Memory"; asapai.co.kr, "Running 753B GLM-5.2 on a single workstation GPU", section
"Abandoning fixed offloading in favor of measured bandwidth".
"""
import numpy as np
import pytest
import torch

import synth
import sparse_moe_expert_sorted_b300 as ft
from oracle import cache as OC
from oracle import ffn as OF
from oracle.lru import GlobalLRU
from oracle.route import route as oracle_route

from gpu_helpers import ensure_built
from helpers import bf16_bits, weights_to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _zipf_ids(g, B, k, E, s=1.1):
    p = 1.0 / np.arange(1, E + 1) ** s
    p /= p.sum()
    return np.stack([g.choice(E, k, replace=False, p=p) for _ in range(B)]).astype(np.int32)


def _step_dev(lru, layer, ids_np):
    ids = torch.from_numpy(ids_np).cuda()
    n = min(ids_np.size, lru.E)
    hit = torch.empty(n, dtype=torch.uint8, device="cuda")
    slot = torch.empty(n, dtype=torch.int32, device="cuda")
    ev = torch.empty(n, dtype=torch.int32, device="cuda")
    lru.step(layer, ids, hit, slot, ev, None)
    m = len(np.unique(ids_np))
    return ids, hit, hit[:m].cpu().numpy(), slot[:m].cpu().numpy(), ev[:m].cpu().numpy()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_resize_matches_the_oracle(seed):
    g = np.random.default_rng(seed)
    L, E, k = 2, 64, 4
    C = int(g.integers(8, 60))
    dev, ref = ft.LRU(L, E, C), GlobalLRU(L, E, C)
    try:
        for i in range(160):
            if i % 23 == 22:
                C2 = int(g.integers(1, 100))
                nm = min(C, C2)
                moves = torch.full((nm, 2), -7, dtype=torch.int32, device="cuda")
                n_moves = torch.zeros(1, dtype=torch.int32, device="cuda")
                dev.resize(C2, moves, n_moves)
                want, _ = ref.resize(C2)
                assert dev.capacity == C2
                assert int(n_moves.item()) == len(want)
                assert np.array_equal(moves[:len(want)].cpu().numpy(), want)
                assert np.array_equal(dev.slot_of().cpu().numpy(), ref.slot_of)
                C = C2
            layer = int(g.integers(0, L))
            ids_np = _zipf_ids(g, int(g.integers(1, 5)), k, E)
            _, _, h, s, v = _step_dev(dev, layer, ids_np)
            _, hr, sr, vr = ref.step(layer, ids_np)
            assert np.array_equal(h, hr) and np.array_equal(s, sr) and np.array_equal(v, vr)
        assert np.array_equal(dev.slot_of().cpu().numpy(), ref.slot_of)
    finally:
        dev.close()


@pytest.mark.parametrize("seed", [3, 4])
def test_miss_split_matches_the_oracle(seed):
    g = np.random.default_rng(seed)
    L, E, k = 3, 48, 6
    C = 20
    dev, ref = ft.LRU(L, E, C), GlobalLRU(L, E, C)
    a = torch.empty(E, dtype=torch.int32, device="cuda")
    b = torch.empty(E, dtype=torch.int32, device="cuda")
    cnt = torch.empty(4, dtype=torch.int32, device="cuda")
    try:
        for i in range(60):
            layer = int(g.integers(0, L))
            B = int(g.integers(1, 5))
            ids_np = _zipf_ids(g, B, k, E)
            ids, hit_dev, h, _, _ = _step_dev(dev, layer, ids_np)
            _, hr, _, _ = ref.step(layer, ids_np)
            n = min(B * k, E)
            now = torch.full((n, 2), -9, dtype=torch.int32, device="cuda")
            later = torch.full((n, 2), -9, dtype=torch.int32, device="cuda")
            if i % 2:
                link, host, override = float(g.uniform(5, 60)), float(g.uniform(60, 300)), -1
                n_fill = OC.fill_count(int(np.sum(hr == 0)), link, host)
            else:
                link, host, override = 1.0, 1.0, int(g.integers(0, 8))
                n_fill = override
            ft.miss_split(dev, layer, ids, hit_dev, link, host, override, a, b, now, later, cnt)
            want = OC.miss_split(ref.slot_of, layer, ids_np, hr, n_fill)
            c = cnt.cpu().numpy()
            assert np.array_equal(a.cpu().numpy(), want["slot_of_a"])
            assert np.array_equal(b.cpu().numpy(), want["slot_of_b"])
            assert c[0] == want["m"] and c[1] == len(want["fill_now"]) and c[2] == len(want["fill_later"])
            assert c[3] == int(np.sum(want["slot_of_b"] >= 0))
            assert np.array_equal(now[:c[1]].cpu().numpy(), want["fill_now"])
            assert np.array_equal(later[:c[2]].cpu().numpy(), want["fill_later"])
    finally:
        dev.close()


# ---------------------------------------------------------------------------------------
# slot copies and whole decode steps
# ---------------------------------------------------------------------------------------
def _pinned(W):
    pin = lambda t: None if t is None else t.cpu().contiguous().pin_memory()
    return synth.ExpertWeights(W.fmt, W.d, W.f, pin(W.gate), pin(W.up), pin(W.down), pin(W.gate_s), pin(W.up_s),
                               pin(W.down_s), pin(W.glob))


def _empty_arena(W, C):
    z = lambda t: None if t is None else torch.zeros((C,) + tuple(t.shape[1:]), dtype=t.dtype, device="cuda")
    A = synth.ExpertWeights(W.fmt, W.d, W.f, z(W.gate), z(W.up), z(W.down), z(W.gate_s), z(W.up_s), z(W.down_s),
                            z(W.glob))
    return A


NAMES = ("gate", "up", "down", "gate_s", "up_s", "down_s", "glob")


def _check_slots(pool, arena, pairs, prepared=True, dsc=None):
    """Every (pool slot s, arena slot t): all arrays equal; prepared layouts equal a fresh
    preparation of an arena holding the same slots (unfilled slots zero on both sides)."""
    for name in NAMES:
        P, A = getattr(pool, name), getattr(arena, name)
        if P is None or (name == "glob" and pool.fmt != synth.NVFP4):   # tensor scales: NVFP4 only
            continue
        for s, t in pairs:
            assert torch.equal(A[t].cpu(), P[s].cpu()), (name, s, t)
    if prepared and dsc is not None and getattr(arena, "ftmoe_prepared", None) is not None:
        ref = _empty_arena(arena, arena.gate.shape[0])
        for name in NAMES:
            if getattr(ref, name) is not None:
                getattr(ref, name).copy_(getattr(arena, name))
        ft.prepare_weights(dsc, ref)
        torch.cuda.synchronize()
        assert torch.equal(ref.ftmoe_prepared, arena.ftmoe_prepared)


def test_copy_slots_fill_compact_and_migrate():
    E, L, d, f = 16, 2, 256, 256
    dsc = ft.desc(E, 4, d, f, synth.NVFP4)
    pool = _pinned(synth.make_experts(synth.NVFP4, L * E, d, f, 21))
    ft.prepare_weights(dsc, pool)
    C = 6
    arena = _empty_arena(pool, C)
    ft.prepare_weights(dsc, arena)           # zero slots prepare to zero bytes
    torch.cuda.synchronize()
    assert int(arena.ftmoe_prepared.abs().sum()) == 0
    pairs = np.array([[3, 0], [17, 4], [30, 2], [5, 5]], np.int32)
    pt = torch.from_numpy(pairs).cuda()
    n = torch.tensor([len(pairs)], dtype=torch.int32, device="cuda")
    ft.copy_slots(dsc, ft.weights_struct(pool), ft.weights_struct(arena), pt, n, len(pairs))
    torch.cuda.synchronize()
    _check_slots(pool, arena, pairs.tolist(), dsc=dsc)
    # in-place compaction: slot 4 -> 1, slot 5 -> 3 (as a shrink to 4 slots would move them)
    mv = torch.tensor([[0, 0], [4, 1], [5, 3]], dtype=torch.int32, device="cuda")
    ft.copy_slots(dsc, ft.weights_struct(arena), ft.weights_struct(arena), mv, None, 3)
    torch.cuda.synchronize()
    _check_slots(pool, arena, [[3, 0], [17, 1], [5, 3], [30, 2]], prepared=False)
    # migration to a larger arena (other part offsets of the prepared layout)
    big = _empty_arena(pool, 11)
    ft.prepare_weights(dsc, big)
    keep = torch.tensor([[0, 0], [1, 1], [2, 2], [3, 3]], dtype=torch.int32, device="cuda")
    ft.copy_slots(dsc, ft.weights_struct(arena), ft.weights_struct(big), keep, None, 4)
    torch.cuda.synchronize()
    _check_slots(pool, big, [[3, 0], [17, 1], [30, 2], [5, 3]], dsc=dsc)
    assert ft.get_device_error() == 0
    # a pair outside an arena is skipped and reported
    bad = torch.tensor([[0, 99]], dtype=torch.int32, device="cuda")
    ft.copy_slots(dsc, ft.weights_struct(arena), ft.weights_struct(big), bad, None, 1)
    assert ft.get_device_error() == 2


@pytest.mark.parametrize("fmt,T", [(synth.NVFP4, 1), (synth.NVFP4, 3), (synth.MXFP4, 2)])
def test_cached_decode_steps_merge_to_the_full_layer(fmt, T):
    g = np.random.default_rng(40 + T)
    E, k, d, f, L, C = 32, 4, 256, 256, 2, 9
    dsc = ft.desc(E, k, d, f, fmt)
    pool = _pinned(synth.make_experts(fmt, L * E, d, f, 50 + fmt))
    ft.prepare_weights(dsc, pool)
    arena = _empty_arena(pool, C)
    ft.prepare_weights(dsc, arena)
    routers = [synth.make_router(E, d, 60 + l).cuda() for l in range(L)]
    biases = [torch.from_numpy(synth.make_zipf_bias(E, 1.1, 60 + l)).cuda() for l in range(L)]
    Wn = weights_to_numpy(pool)
    lru = ft.LRU(L, E, C)
    s_pool = ft.weights_struct(pool, prepared=0)      # executor B: plain loads from host memory
    s_fill = ft.weights_struct(pool)
    s_arena = ft.weights_struct(arena)
    P = T * k
    n = min(P, E)
    hit = torch.empty(n, dtype=torch.uint8, device="cuda")
    lslot = torch.empty(n, dtype=torch.int32, device="cuda")
    lev = torch.empty(n, dtype=torch.int32, device="cuda")
    sa = torch.empty(E, dtype=torch.int32, device="cuda")
    sb = torch.empty(E, dtype=torch.int32, device="cuda")
    now = torch.empty(n, 2, dtype=torch.int32, device="cuda")
    later = torch.empty(n, 2, dtype=torch.int32, device="cuda")
    cnt = torch.empty(4, dtype=torch.int32, device="cuda")
    ws_r = ft.workspace(ft.route_workspace_size(dsc, T))
    ws_p = ft.workspace(ft.permute_workspace_size(dsc, T))
    ws_a = ft.workspace(ft.expert_ffn_workspace_size(dsc, T))
    ws_b = ft.workspace(ft.expert_ffn_workspace_size(dsc, T))
    used_b = 0
    try:
        for step in range(14):
            layer = step % L
            x = synth.make_x(T, d, 700 + step).cuda()
            ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
            w = torch.empty(T, k, dtype=torch.float32, device="cuda")
            ft.route(dsc, x, routers[layer], biases[layer], ids, w, None, ws_r)
            off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
            sp = torch.empty(P, dtype=torch.int32, device="cuda")
            pp = torch.empty(P, dtype=torch.int32, device="cuda")
            ft.permute(dsc, ids, off, sp, pp, ws_p)
            lru.step(layer, ids, hit, lslot, lev, None)
            if step % 3 == 0:
                ft.miss_split(lru, layer, ids, hit, 1.0, 1.0, int(g.integers(0, 4)), sa, sb, now, later, cnt)
            else:
                ft.miss_split(lru, layer, ids, hit, 52.7, 77.3, -1, sa, sb, now, later, cnt)
            ft.copy_slots(dsc, s_fill, s_arena, now, cnt[1:2], n)
            y_a = torch.zeros(P, d, dtype=torch.float32, device="cuda")
            ft.expert_ffn(dsc, s_arena, sa, x, off, sp, None, y_a, ws_a)
            out_b = torch.zeros(T, d, dtype=torch.float32, device="cuda")
            ft.expert_ffn(dsc, s_pool, sb, x, off, sp, w, out_b, ws_b)
            of = torch.empty(T, d, dtype=torch.float32, device="cuda")
            ob = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
            ft.combine(dsc, T, y_a, pp, w, ids, sa, out_b, of, ob)
            ft.copy_slots(dsc, s_fill, s_arena, later, cnt[2:3], n)
            torch.cuda.synchronize()
            used_b += int(cnt[3].item())
            # the oracle: the whole layer with every expert taken from the pool
            ids_r, w_r, _ = oracle_route(bf16_bits(x), bf16_bits(routers[layer]), biases[layer].cpu().numpy(), k, 1)
            assert np.array_equal(ids.cpu().numpy(), ids_r)
            want = OF.layer_tokens(Wn, layer * E + np.arange(E), bf16_bits(x), ids_r, w_r, list(range(T)))
            got = of.cpu().numpy()
            for t in range(T):
                err = np.linalg.norm(got[t] - want[t]) / np.linalg.norm(want[t])
                assert err < 5e-3, (step, t, err)
            # every resident key's slot holds its pool slot, byte for byte
            so = lru.slot_of().cpu().numpy()
            pairs = [[l * E + e, int(so[l, e])] for l in range(L) for e in range(E) if so[l, e] >= 0]
            _check_slots(pool, arena, pairs, prepared=False)
        assert used_b > 0                                   # executor B ran on some steps
        assert ft.get_device_error() == 0
    finally:
        lru.close()
