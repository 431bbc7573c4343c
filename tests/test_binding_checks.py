"""The Python binding checks every tensor argument (type, element count, [T, d] shape of the
activations) before its address crosses the C ABI, where the library sees only a pointer:
a tensor too small for what a call reads or writes fails here instead of being accessed
past its end.  Host tensors stand in for device ones: a call whose arguments pass the checks
stops at the device-memory check that follows them."""
import pytest
import torch

import sparse_moe_expert_sorted_b300 as ft
from sparse_moe_expert_sorted_b300 import build as ftbuild

E, k, d, f, T = 16, 4, 256, 512, 5
P = T * k


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ftbuild.build()
    ft.lib()


def _dsc(fmt=ft.BF16):
    return ft.desc(E, k, d, f, fmt)


def t(*shape, dtype=torch.float32):
    return torch.zeros(*shape, dtype=dtype)


def bf(*shape):
    return t(*shape, dtype=torch.bfloat16)


def i32(*shape):
    return t(*shape, dtype=torch.int32)


def _fails(fn, what):
    with pytest.raises(ft.FtmoeError) as e:
        fn()
    assert what in str(e.value), str(e.value)


def _passes_checks(fn):
    _fails(fn, "CUDA tensors")


def test_route_and_route_noalloc():
    ds, ws = _dsc(), t(4096, dtype=torch.uint8)
    args = dict(x=bf(T, d), w_router=bf(E, d), bias=t(E), ids=i32(T, k), w=t(T, k))
    _passes_checks(lambda: ft.route(ds, *args.values(), t(T, E), ws))
    _passes_checks(lambda: ft.route(ds, *args.values(), None, ws))
    _passes_checks(lambda: ft.route_noalloc(ds, *args.values()))
    bad = [("x", bf(T, d + 256), "[T, 256]"), ("x", t(T, d), "bfloat16"), ("x", bf(T * d), "[T, 256]"),
           ("w_router", bf(E - 1, d), "w_router"), ("bias", t(E, dtype=torch.float64), "logit_bias"),
           ("ids", i32(T, k - 1), "topk_ids"), ("ids", t(T, k, dtype=torch.int64), "topk_ids"),
           ("w", t(T, k - 1), "topk_w")]
    for name, val, msg in bad:
        a = dict(args, **{name: val})
        _fails(lambda: ft.route(ds, *a.values(), None, ws), msg)
        _fails(lambda: ft.route_noalloc(ds, *a.values()), msg)
    _fails(lambda: ft.route(ds, *args.values(), t(T, E - 1), ws), "logits")
    _fails(lambda: ft.route(ds, *args.values(), None, None), "ws")


def test_permute():
    ds, ws = _dsc(), t(4096, dtype=torch.uint8)
    _passes_checks(lambda: ft.permute(ds, i32(T, k), i32(E + 1), i32(P), i32(P), ws))
    _fails(lambda: ft.permute(ds, i32(T, k + 1), i32(E + 1), i32(P), i32(P), ws), "topk_ids")
    _fails(lambda: ft.permute(ds, i32(P), i32(E + 1), i32(P), i32(P), ws), "topk_ids")
    _fails(lambda: ft.permute(ds, i32(T, k), i32(E), i32(P), i32(P), ws), "expert_offsets")
    _fails(lambda: ft.permute(ds, i32(T, k), i32(E + 1), i32(P - 1), i32(P), ws), "sorted_pair")
    _fails(lambda: ft.permute(ds, i32(T, k), i32(E + 1), i32(P), t(P), ws), "pair_pos")


def test_quantize_act():
    ds, d8 = _dsc(ft.NVFP4), _dsc(ft.FP8_B128)
    u8 = lambda n: t(n, dtype=torch.uint8)
    _passes_checks(lambda: ft.quantize_act(ds, bf(T, d), u8(T * d // 2), u8(T * d // 16)))
    _passes_checks(lambda: ft.quantize_act(d8, bf(T, d), u8(T * d), t(T, d // 128)))
    _passes_checks(lambda: ft.quantize_act(d8, bf(T, d), u8(T * d), t(T, d // 128).view(torch.uint8)))
    _fails(lambda: ft.quantize_act(ds, bf(T, d), u8(T * d // 2 - 1), u8(T * d // 16)), "codes")
    _fails(lambda: ft.quantize_act(d8, bf(T, d), u8(T * d // 2), t(T, d // 128)), "codes")
    _fails(lambda: ft.quantize_act(d8, bf(T, d), u8(T * d), u8(T * d // 128)), "scales")


def test_expert_ffn():
    ds, ws, st = _dsc(), t(4096, dtype=torch.uint8), ft.WeightsStruct()
    _passes_checks(lambda: ft.expert_ffn(ds, st, i32(E), bf(T, d), i32(E + 1), i32(P), None, t(P, d), ws))
    _passes_checks(lambda: ft.expert_ffn(ds, st, None, bf(T, d), i32(E + 1), i32(P), t(T, k), t(T, d), ws))
    _fails(lambda: ft.expert_ffn(ds, st, None, bf(T, d), i32(E + 1), i32(P), None, t(T, d), ws), "y_or_out")
    _fails(lambda: ft.expert_ffn(ds, st, i32(E - 1), bf(T, d), i32(E + 1), i32(P), None, t(P, d), ws), "slot_of")
    _fails(lambda: ft.expert_ffn(ds, st, None, bf(T, d), i32(E + 1), i32(P), t(T, k - 1), t(T, d), ws), "topk_w")
    _fails(lambda: ft.expert_ffn(ds, st, None, bf(T, d), i32(E + 1), i32(P), None, bf(P, d), ws), "y_or_out")


def test_combine():
    ds = _dsc()
    _passes_checks(lambda: ft.combine(ds, T, t(P, d), i32(P), t(T, k), i32(T, k), i32(E), None, t(T, d), bf(T, d)))
    _passes_checks(lambda: ft.combine(ds, T, None, None, None, None, None, t(T, d), t(T, d), None))
    _fails(lambda: ft.combine(ds, T, t(P, d - 1), i32(P), t(T, k), i32(T, k), None, None, t(T, d), None), "y")
    _fails(lambda: ft.combine(ds, T, t(P, d), None, t(T, k), i32(T, k), None, None, t(T, d), None), "pair_pos")
    _fails(lambda: ft.combine(ds, T, t(P, d), i32(P), t(T, k), None, i32(E), None, t(T, d), None), "topk_ids")
    _fails(lambda: ft.combine(ds, T, None, None, None, None, None, t(T, d - 1), t(T, d), None), "partial_b")
    _fails(lambda: ft.combine(ds, T, None, None, None, None, None, None, t(T, d), t(T, d)), "out_bf16")


def test_layer_forward():
    ds, ws, st = _dsc(), t(4096, dtype=torch.uint8), ft.WeightsStruct()
    ok = dict(slot_of=i32(E), x=bf(T, d), w_router=bf(E, d), bias=None, ids=i32(T, k), topk_w=t(T, k),
              out_f32=t(T, d), out_bf16=bf(T, d), ws=ws)
    _passes_checks(lambda: ft.layer_forward(ds, st, *ok.values()))
    _passes_checks(lambda: ft.layer_forward(ds, st, *dict(ok, ids=None, topk_w=None, out_bf16=None).values()))
    for name, val, msg in [("out_f32", None, "out_f32"), ("out_f32", t(T, d - 1), "out_f32"),
                           ("out_bf16", t(T, d), "out_bf16"), ("ids", i32(T, k - 1), "topk_ids"),
                           ("slot_of", t(E), "slot_of"), ("w_router", bf(E, d - 1), "w_router"),
                           ("x", bf(T, 2 * d), "[T, 256]")]:
        a = dict(ok, **{name: val})
        _fails(lambda: ft.layer_forward(ds, st, *a.values()), msg)


def test_lru_step_and_replay():
    lru = ft.LRU.__new__(ft.LRU)          # a handle without device state: only the checks run
    lru.L, lru.E, lru.C, lru._h = 2, 8, 4, None
    u8 = lambda n: t(n, dtype=torch.uint8)
    c = t(2, dtype=torch.int64)
    _passes_checks(lambda: lru.step(0, i32(3, 2), u8(6), i32(6), i32(6), c))
    _passes_checks(lambda: lru.step(0, i32(5, 2), u8(8), i32(8), i32(8), None))   # at most E accesses
    _fails(lambda: lru.step(0, i32(6), u8(6), i32(6), i32(6), c), "[B, k]")
    _fails(lambda: lru.step(0, i32(3, 2), u8(5), i32(6), i32(6), c), "hit")
    _fails(lambda: lru.step(0, i32(3, 2), u8(6), i32(6), i32(5), c), "evicted_key")
    _fails(lambda: lru.step(0, i32(3, 2), u8(6), i32(6), i32(6), t(2)), "counters")
    tr = i32(10, 2, 3, 2)
    _passes_checks(lambda: lru.replay(tr, u8(40), i32(40), i32(40), c))
    _fails(lambda: lru.replay(i32(10, 6), u8(40), i32(40), i32(40), c), "trace")
    _fails(lambda: lru.replay(tr, u8(40), i32(39), i32(40), c), "slot")


@pytest.mark.parametrize("fmt", [ft.BF16, ft.NVFP4, ft.MXFP4, ft.FP8_B128])
def test_weights_struct_checks_the_arena(fmt):
    import synth
    W = synth.make_experts(fmt, 3, 256, 256, 0)
    _passes_checks(lambda: ft.weights_struct(W))
    short = synth.make_experts(fmt, 3, 256, 256, 0)
    short.up = short.up[:2].contiguous()                  # two slots where the arena has three
    _fails(lambda: ft.weights_struct(short), "up")
    if fmt != ft.BF16:
        short = synth.make_experts(fmt, 3, 256, 256, 0)
        short.down_s = short.down_s[:2].contiguous()
        _fails(lambda: ft.weights_struct(short), "down_s")
    if fmt == ft.NVFP4:
        short = synth.make_experts(fmt, 3, 256, 256, 0)
        short.glob = short.glob[:2].contiguous()
        _fails(lambda: ft.weights_struct(short), "glob")


def test_host_buffer_call_wants_pinned_contiguous_host_tensors():
    """LayerHostCall (and the graph form built on it) copies x in and the bf16 output out by
    address, asynchronously: a pageable host tensor or a strided view of one is refused."""
    ds, ws = _dsc(), t(4096, dtype=torch.uint8)
    rest = dict(w_router=bf(E, d), bias=None, ids=i32(T, k), topk_w=t(T, k), out_f32=t(T, d))

    def call(xh, oh):
        return ft.LayerHostCall(ds, None, None, xh, rest["w_router"], None, rest["ids"], rest["topk_w"],
                                rest["out_f32"], oh, ws)
    _fails(lambda: call(bf(T, d), bf(T, d)), "pinned host memory")
    _fails(lambda: call(bf(d, T).t(), bf(T, d)), "contiguous")
    _fails(lambda: call(bf(T, d + 1), bf(T, d)), "host [T, 256]")
    _fails(lambda: call(t(T, d), bf(T, d)), "bfloat16")
