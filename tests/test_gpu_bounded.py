"""Failure detection on the device, without a GPU fault.

1. The layout's grid-wide hand-over is a bounded wait: with a 1 ms limit and
   the arrival counter set so that no block arrives last, every block gives
   up, the status word reports MOE_DEVERR_TIMEOUT, the launch returns, and a
   clear followed by a normal layout gives the oracle's layout again (the
   DeepSpeed AutoEP transport PR's review fix: run out, then fail; do not
   fault or hang).
2. Row indices and offsets read from the layout are range-checked: a
   corrupted entry is reported (MOE_DEVERR_BAD_LAYOUT) and skipped, every
   other entry is computed as the oracle computes it with that entry dropped.
   Each corrupted index points into slack rows that the test allocates past
   the end of the row tensors, so even an unchecked access would stay inside
   the allocation; the slack rows must come back untouched."""
import copy
import time

import numpy as np
import pytest
import torch

import combine_moe_route_05_gb300 as moe
import oracle
import synth
from tests.common import assert_ulp, gw_tolerance_ok, row_norms_for_gw
from tests.gpu_util import dev, layout_host, oracle_route, router, to_dev, to_host

pytestmark = pytest.mark.gpu

# the workspace plan: the status word in the first 256-byte slot, the
# layout's [arrival counter, epoch] at the start of the second
TICKET_OFFSET = 256


def test_layout_wait_runs_out_then_recovers():
    wl = synth.WORKLOADS[3].with_tokens(2600)
    inp = synth.make_inputs(wl, want=("logits", "bias"))
    idx, _ = oracle_route(wl, inp["logits"], inp["bias"])
    L = oracle.layout(idx, wl.E, wl.R)
    r = router(wl)
    assert moe.moe_dispatch_layout_launches(r.h, wl.T) == 1
    d_idx = to_dev(idx)
    ticket = r.h.workspace[TICKET_OFFSET:TICKET_OFFSET + 8].view(torch.int32)
    # where the counter and the epoch live: each single-launch layout leaves
    # the counter at 0 and advances the epoch by one
    r.layout(d_idx)
    torch.cuda.synchronize()
    e0 = int(ticket[1])
    r.layout(d_idx)
    torch.cuda.synchronize()
    assert int(ticket[0]) == 0 and int(ticket[1]) == e0 + 1

    moe.moe_set_wait_limit(r.h, 1_000_000)  # 1 ms
    ticket[0] = 1 << 30  # no block of the next layout is the last to arrive
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    r.layout(d_idx)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert moe.moe_read_device_status(r.h) & moe.MOE_DEVERR_TIMEOUT
    assert int(ticket[1]) == e0 + 1  # nobody published
    assert waited < 0.5, waited

    moe.moe_clear_device_status(r.h)
    moe.moe_set_wait_limit(r.h, 0)
    assert moe.moe_read_device_status(r.h) == 0
    assert int(ticket[0]) == 0
    r.layout(d_idx)
    got = layout_host(r)
    for f in oracle.Layout.FIELDS:
        assert np.array_equal(got[f].reshape(-1), getattr(L, f).reshape(-1)), f
    assert moe.moe_read_device_status(r.h) == 0


SLACK = 2048  # rows allocated past the end of every row tensor


def padded_rows(n, width, dtype, fill):
    full = torch.full((n + SLACK, width), fill, dtype=dtype, device=dev())
    return full, full[:n]


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def dropped(L, t, k):
    """The oracle layout with entry (t, k) dropped."""
    M = copy.deepcopy(L)
    M.pos[t, k] = -1
    M.send_row_of[t, k] = -1
    return M


@pytest.fixture()
def corrupt_case():
    wl = synth.WORKLOADS[1].with_tokens(600)
    inp = synth.make_inputs(wl, want=("logits", "x", "y", "g"))
    idx, w = oracle_route(wl, inp["logits"], None)
    L = oracle.layout(idx, wl.E, wl.R)
    r = router(wl)
    r.layout(to_dev(idx))
    torch.cuda.synchronize()
    return wl, inp, w, L, r


def test_out_of_range_receive_row_is_flagged_and_skipped(corrupt_case):
    wl, inp, w, L, r = corrupt_case
    T, K, H, RR = wl.T, wl.K, wl.H, r.h.recv_rows
    t, k = 5, 3
    good = int(L.pos[t, k])
    moe.layout_tensors(r.h)["pos"][t, k] = RR + 3
    M = dropped(L, t, k)
    x, wd, g = to_dev(inp["x"]), to_dev(w), to_dev(inp["g"])
    sentinel = -7.0

    # dispatch: the entry's receive row and the slack stay unwritten
    recv_full, recv = padded_rows(RR, H, torch.bfloat16, sentinel)
    rw_full = torch.full((RR + SLACK,), sentinel, device=dev())
    moe.moe_dispatch(r.h, x, wd, recv, rw_full[:RR])
    assert moe.moe_read_device_status(r.h) & moe.MOE_DEVERR_BAD_LAYOUT
    moe.moe_clear_device_status(r.h)
    orecv, orw, _ = oracle.dispatch(inp["x"], M, w)
    got = to_host(recv_full)
    keep = np.ones(RR, bool)
    keep[good] = False
    assert np.array_equal(got[:RR][keep], orecv[keep])
    assert (recv_full[good] == sentinel).all() and (recv_full[RR:] == sentinel).all()
    assert (rw_full[RR:] == sentinel).all() and float(rw_full[good]) == sentinel

    # combine (weighted and plain) and dispatch backward: the entry is left out
    y_full, y = padded_rows(RR, H, torch.bfloat16, 0.0)
    y.copy_(to_dev(inp["y"]))
    y_full[RR:] = 1e4  # would show in the sums if read
    for wt in (wd, None):
        out = to_host(r.combine(y, wt))
        assert moe.moe_read_device_status(r.h) & moe.MOE_DEVERR_BAD_LAYOUT
        moe.moe_clear_device_status(r.h)
        assert_ulp(out, oracle.combine(inp["y"], M, None if wt is None else w), 0, "combine")
    assert_ulp(to_host(r.dispatch_bwd(y)), oracle.dispatch_bwd(inp["y"], M), 0, "dispatch_bwd")
    moe.moe_clear_device_status(r.h)

    # combine backward: no gradient row for the entry, its score gradient 0
    gy_full, gy = padded_rows(RR, H, torch.bfloat16, sentinel)
    gw = torch.empty(T, K, device=dev())
    moe.moe_combine_bwd(r.h, g, y, wd, gy, gw)
    assert moe.moe_read_device_status(r.h) & moe.MOE_DEVERR_BAD_LAYOUT
    moe.moe_clear_device_status(r.h)
    ogy, ogw = oracle.combine_bwd(inp["g"], inp["y"], M, w)
    assert np.array_equal(to_host(gy)[keep], ogy[keep])
    assert (gy_full[good] == sentinel).all() and (gy_full[RR:] == sentinel).all()
    gn, yn = row_norms_for_gw(oracle.bf16_to_f32(inp["g"]), oracle.bf16_to_f32(inp["y"]), M.pos)
    assert gw_tolerance_ok(to_host(gw), ogw, gn, yn).all() and float(gw[t, k]) == 0.0


def test_out_of_range_send_row_is_flagged_and_skipped(corrupt_case):
    wl, inp, w, L, r = corrupt_case
    H = wl.H
    S_rows = wl.T * min(wl.K, wl.R)
    RR = r.h.recv_rows
    # the token's first entry carries its send row; give it a bad one
    t = 7
    k = 0
    moe.layout_tensors(r.h)["send_row_of"][t, k] = S_rows + 5
    x = to_dev(inp["x"])
    send_full, send = padded_rows(S_rows, H, torch.bfloat16, -7.0)
    recv = torch.empty(RR, H, dtype=torch.bfloat16, device=dev())
    moe.moe_dispatch(r.h, x, None, recv, None, send)
    assert moe.moe_read_device_status(r.h) & moe.MOE_DEVERR_BAD_LAYOUT
    moe.moe_clear_device_status(r.h)
    assert (send_full[S_rows:] == -7.0).all()
    # the receive rows do not depend on send rows: all of them are right
    orecv, _, _ = oracle.dispatch(inp["x"], L)
    assert np.array_equal(to_host(recv), orecv)
    # the staged calls read the same entry: flagged, and nothing past the end
    part_full, part = padded_rows(S_rows, H, torch.bfloat16, -7.0)
    moe.moe_combine_partial(r.h, recv, None, part)
    assert moe.moe_read_device_status(r.h) & moe.MOE_DEVERR_BAD_LAYOUT
    moe.moe_clear_device_status(r.h)
    assert (part_full[S_rows:] == -7.0).all()
    recv2_full, recv2 = padded_rows(RR, H, torch.bfloat16, -7.0)
    moe.moe_expand(r.h, send, recv2)
    assert moe.moe_read_device_status(r.h) & moe.MOE_DEVERR_BAD_LAYOUT
    moe.moe_clear_device_status(r.h)
    assert (recv2_full[RR:] == -7.0).all()


def test_out_of_range_offsets_stop_the_absorbed_kernels():
    """Offsets past the receive rows: scale_rows clamps to the rows it has,
    the fused W2 GEMM computes nothing; both report the bad layout."""
    wl = synth.WORKLOADS[4].with_tokens(300)
    inp = synth.make_inputs(wl, want=("logits",))
    idx, w = oracle_route(wl, inp["logits"], None)
    r = router(wl)
    r.layout(to_dev(idx))
    RR, I, Hout = r.h.recv_rows, 64, 256
    lay = moe.layout_tensors(r.h)
    lay["off_e"][wl.E] = RR + 1000
    lay["cnt_e"][wl.E - 1] += 1000
    h_full, h = padded_rows(RR, I, torch.bfloat16, 1.0)
    rw_full = torch.full((RR + SLACK,), 0.5, device=dev())
    hs_full, hs = padded_rows(RR, I, torch.bfloat16, -7.0)
    moe.moe_scale_rows(r.h, h, rw_full[:RR], hs)
    assert moe.moe_read_device_status(r.h) & moe.MOE_DEVERR_BAD_LAYOUT
    moe.moe_clear_device_status(r.h)
    assert (hs == 0.5).all() and (hs_full[RR:] == -7.0).all()
    w2 = torch.full((wl.E, Hout, I), 0.25, dtype=torch.bfloat16, device=dev())
    y_full, y = padded_rows(RR, Hout, torch.bfloat16, -7.0)
    moe.moe_w2_absorbed(r.h, h, rw_full[:RR], w2, y)
    assert moe.moe_read_device_status(r.h) & moe.MOE_DEVERR_BAD_LAYOUT
    assert (y_full == -7.0).all()
