"""A bounded device wait that runs out returns an error status, and the library stays usable.

The decode FFN's two phases meet at a grid-wide sync whose arrival counter lives in the
workspace header (it only grows, and is a multiple of the grid between calls).  Setting that
counter to 1 before a call (the state a caller must clear after a timeout) means the last CTA
to arrive waits for a count that never comes.  With the wait limit shortened to 20 ms
(ftmoe_set_wait_limit) the call must end, the device error word must read a timeout code, and
after the header is zeroed the next call must match the oracle.  Nothing faults or hangs: the
wait is bounded, and the failure is made on the host (the counter's value).
"""
import numpy as np
import pytest
import torch

import synth
import sparse_moe_expert_sorted_b300 as ft
from oracle import ffn as OF

from gpu_helpers import ensure_built, permute, route
from helpers import bf16_bits, rel_l2, weights_to_numpy

pytestmark = pytest.mark.gpu
TIMEOUT_CODES = (6, 10)          # a bounded wait on a shared-memory barrier, on a grid sync


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def test_a_grid_sync_that_cannot_complete_times_out_and_the_next_call_is_correct():
    E, k, d, f, T = 16, 4, 256, 256, 16
    dsc = ft.desc(E, k, d, f, synth.NVFP4)
    assert ft.expert_ffn_path(dsc, T) == 0
    W = synth.make_experts(synth.NVFP4, E, d, f, 61, device="cuda")
    ft.prepare_weights(dsc, W)
    x = synth.make_x(T, d, 61).cuda()
    wr = synth.make_router(E, d, 61).cuda()
    ids, w, _ = route(dsc, x, wr)
    off, sp, pp = permute(dsc, ids)
    ws = ft.workspace(ft.expert_ffn_workspace_size(dsc, T))
    assert ft.get_device_error() == 0
    ws.view(torch.int64)[3] = 1            # bytes 24..31: the grid sync's arrival counter
    ft.set_wait_limit(20_000_000)
    try:
        y = torch.full((T * k, d), float("nan"), device="cuda")
        ft.expert_ffn(dsc, ft.weights_struct(W), None, x, off, sp, None, y, ws)
        torch.cuda.synchronize()           # ends: the wait gave up after 20 ms
        assert ft.get_device_error() in TIMEOUT_CODES
    finally:
        ft.set_wait_limit(0)
    ws[:ft.WS_ZERO_BYTES].zero_()          # what a caller does after a timeout
    y = torch.full((T * k, d), float("nan"), device="cuda")
    ft.expert_ffn(dsc, ft.weights_struct(W), None, x, off, sp, None, y, ws)
    torch.cuda.synchronize()
    assert ft.get_device_error() == 0
    ref = OF.expert_ffn(weights_to_numpy(W.to("cpu")), np.arange(E), bf16_bits(x.cpu()), k, off.cpu().numpy(),
                        sp.cpu().numpy())
    assert rel_l2(y.cpu().numpy(), ref) < 5e-3
