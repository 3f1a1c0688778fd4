"""Padded (capacity-aligned) receive layout on the GPU against the oracle:
segments start at multiples of the alignment, pad rows carry -1 in the layout
and zeros in every receive-row tensor the kernels write, and the token-side
results are those of the packed layout."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from tests.common import assert_ulp, entry_row_norms, gw_tolerance_ok, row_norms_for_gw
from tests.gpu_util import layout_host, oracle_route, router, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("i,align", [(1, 128), (3, 128), (3, 48), (0, 4)])
def test_padded_chain(i, align):
    wl = dataclasses.replace(synth.WORKLOADS[i].with_tokens(min(2600, synth.WORKLOADS[i].T)),
                             pad_align=align)
    inp = synth.make_inputs(wl, want=("logits", "bias", "x", "g"))
    idx, w = oracle_route(wl, inp["logits"], inp["bias"])
    L = oracle.layout(idx, wl.E, wl.R, align)
    r = router(wl)
    r.layout(to_dev(idx))
    got = layout_host(r)
    for f in oracle.Layout.FIELDS:
        assert np.array_equal(got[f].reshape(-1), getattr(L, f).reshape(-1)), f
    rows = L.recv_rows
    # expert outputs: random rows at the entries, the oracle's zeros at the pads
    y = np.zeros((rows,) + inp["x"].shape[1:], inp["x"].dtype)
    y_entries = synth.rows(wl, wl.seed, "y", wl.T * wl.K, wl.H)
    y[L.pos.reshape(-1)] = y_entries
    y_d = to_dev(y)
    # rows past off_e[E] belong to no segment and are not written
    n = int(L.off_e[-1])
    recv, recv_w, send = r.dispatch(to_dev(inp["x"]), to_dev(w), with_send=True)
    orecv, orw, _ = oracle.dispatch(inp["x"], L, w)
    assert np.array_equal(to_host(recv)[:n], orecv[:n])  # includes the zero pad rows
    assert np.array_equal(to_host(recv_w)[:n], orw[:n])
    assert np.array_equal(to_host(r.expand(send))[:n], orecv[:n])
    assert_ulp(to_host(r.combine(y_d, to_dev(w))), oracle.combine(y, L, w), 0, "combine")
    gy, gw = r.combine_bwd(to_dev(inp["g"]), y_d, to_dev(w))
    ogy, ogw = oracle.combine_bwd(inp["g"], y, L, w)
    assert np.array_equal(to_host(gy)[:n], ogy[:n])       # zero pad rows
    f32 = (lambda a: a) if y.dtype == np.float32 else oracle.bf16_to_f32
    gn, yn = row_norms_for_gw(f32(inp["g"]), f32(y), L.pos)
    assert gw_tolerance_ok(to_host(gw), ogw, gn, yn).all()
    assert_ulp(to_host(r.dispatch_bwd(y_d)), oracle.dispatch_bwd(y, L), 0, "dispatch_bwd")
    # the token-side results equal those of the packed layout
    L0 = oracle.layout(idx, wl.E, wl.R)
    y0 = np.zeros((L0.recv_rows,) + y.shape[1:], y.dtype)
    y0[L0.pos.reshape(-1)] = y_entries
    assert np.array_equal(oracle.combine(y, L, w), oracle.combine(y0, L0, w))


def test_padded_absorption_rows():
    wl = dataclasses.replace(synth.WORKLOADS[4].with_tokens(1200), pad_align=64)
    inp = synth.make_inputs(wl, want=("logits",))
    idx, w = oracle_route(wl, inp["logits"], None)
    L = oracle.layout(idx, wl.E, wl.R, 64)
    r = router(wl)
    r.layout(to_dev(idx))
    rows = L.recv_rows
    h = np.zeros((rows, wl.I), np.uint16)
    ghs = np.zeros((rows, wl.I), np.uint16)
    h[L.pos.reshape(-1)] = synth.normal_bf16(0, "h", (wl.T * wl.K, wl.I))
    ghs[L.pos.reshape(-1)] = synth.normal_bf16(0, "ghs", (wl.T * wl.K, wl.I))
    _, recv_w, _ = oracle.dispatch(np.zeros((wl.T, 8), np.uint16), L, w)
    n = int(L.off_e[-1])
    hs = to_host(r.scale_rows(to_dev(h), to_dev(recv_w)))
    assert np.array_equal(hs[:n], oracle.scale_rows(h, recv_w, rows=n)[:n])
    gh, gw = r.scale_rows_bwd(to_dev(ghs), to_dev(h), to_dev(recv_w))
    ogh, ogw = oracle.scale_rows_bwd(ghs, h, recv_w, L, rows=n)
    assert np.array_equal(to_host(gh)[:n], ogh[:n])
    # the score gradient <ghs_row, h_row>, with the floor scaled by both rows' norms
    gn = entry_row_norms(oracle.bf16_to_f32(ghs), L.pos)
    hn = entry_row_norms(oracle.bf16_to_f32(h), L.pos)
    assert gw_tolerance_ok(to_host(gw), ogw, gn, hn).all()
