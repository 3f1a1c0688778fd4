"""Router backward to the logits on the GPU against the oracle's fp64
derivative of the routing weights (selection held fixed).

Acceptance: within 2 fp32 ulps of the oracle's value rounded to fp32, plus
1e-9 of the row's largest magnitude (both sides compute in fp64; device and
host exp may differ in the last fp64 bit, which matters only where the
difference gw_j - sum_k q_k gw_k cancels).

The dispatch backward with the router backward fused in is checked against
the oracle's dispatch backward (exact) and router backward (as above), and bit
for bit against the two separate GPU calls."""
import dataclasses

import numpy as np
import pytest
import torch

import combine_moe_route_05_gb300 as moe
import oracle
import synth
from tests.common import assert_ulp
from tests.gpu_util import oracle_route, router, to_dev, to_host

pytestmark = pytest.mark.gpu


def assert_close_rows(got, ref):
    ref32 = ref.astype(np.float32)
    ulp = np.abs(np.spacing(np.abs(ref32).astype(np.float32))).astype(np.float64)
    floor = 1e-9 * np.abs(ref).max(axis=1, keepdims=True)
    bad = np.abs(got.astype(np.float64) - ref) > 2 * ulp + floor
    assert not bad.any(), "%d entries out of tolerance" % int(bad.sum())


@pytest.mark.parametrize("i,renorm,scale", [(1, True, 1.0), (1, False, 1.0), (1, True, 2.5),
                                            (3, True, 1.0), (3, False, 1.0), (3, True, 2.5),
                                            (4, True, 1.0), (0, True, 1.0)])
def test_route_bwd(i, renorm, scale):
    wl = synth.WORKLOADS[i]
    wl = wl.with_tokens(min(wl.T, 2600))
    wl = dataclasses.replace(wl, renorm=renorm, route_scale=scale)
    inp = synth.make_inputs(wl, want=("logits", "bias"))
    idx, w = oracle_route(wl, inp["logits"], inp["bias"])
    gw = synth.normal_f32(wl.seed, "grecv", (wl.T, wl.K))
    ref = oracle.route_bwd(inp["logits"], idx, gw.astype(np.float64), wl.score_fn, renorm, scale)
    r = router(wl)
    got = to_host(r.route_bwd(to_dev(inp["logits"]), to_dev(idx), to_dev(gw)))
    assert_close_rows(got, ref)
    if not (wl.score_fn == "softmax" and not renorm):
        mask = np.zeros(ref.shape, bool)
        np.put_along_axis(mask, idx, True, 1)
        assert (got[~mask] == 0).all()


def test_route_bwd_full_size_deepseek_v3():
    wl = synth.WORKLOADS[3]
    inp = synth.make_inputs(wl, want=("logits", "bias"))
    idx, w = oracle_route(wl, inp["logits"], inp["bias"])
    gw = synth.normal_f32(wl.seed, "grecv", (wl.T, wl.K))
    ref = oracle.route_bwd(inp["logits"], idx, gw.astype(np.float64), "sigmoid", True, 1.0)
    got = to_host(router(wl).route_bwd(to_dev(inp["logits"]), to_dev(idx), to_dev(gw)))
    assert_close_rows(got, ref)


# ----------------------------------------------------------------------------
# dispatch backward with the router backward fused in


@pytest.mark.parametrize("i,renorm,scale", [(1, True, 1.0), (1, False, 1.0), (2, True, 1.0),
                                            (3, True, 1.0), (3, False, 2.5), (3, True, 2.5),
                                            (0, True, 1.0), (4, True, 1.0)])
def test_dispatch_bwd_route(i, renorm, scale):
    wl = synth.WORKLOADS[i]
    wl = dataclasses.replace(wl.with_tokens(min(wl.T, 2600)), renorm=renorm, route_scale=scale)
    inp = synth.make_inputs(wl, want=("logits", "bias", "grecv"))
    idx, w = oracle_route(wl, inp["logits"], inp["bias"])
    L = oracle.layout(idx, wl.E, wl.R)
    gw = synth.normal_f32(wl.seed, "grecv", (wl.T, wl.K))
    r = router(wl)
    r.layout(to_dev(idx))
    grecv, ld, idd, gwd = to_dev(inp["grecv"]), to_dev(inp["logits"]), to_dev(idx), to_dev(gw)
    gx, gl = r.dispatch_bwd_route(grecv, ld, idd, gwd)
    want_launches = 2 if (wl.score_fn == "softmax" and not renorm) else 1
    assert moe.moe_dispatch_bwd_route_launches(r.h) == want_launches
    assert moe.moe_read_device_status(r.h) == 0

    # against the oracle: gx exact, glogits within 2 fp32 ulps
    assert_ulp(to_host(gx), oracle.dispatch_bwd(inp["grecv"], L), 0, "gx")
    ref = oracle.route_bwd(inp["logits"], idx, gw.astype(np.float64), wl.score_fn, renorm, scale)
    assert_close_rows(to_host(gl), ref)
    if want_launches == 1:
        mask = np.zeros(ref.shape, bool)
        np.put_along_axis(mask, idx, True, 1)
        assert (to_host(gl)[~mask] == 0).all()

    # the same bits as the two separate calls
    gx2 = r.dispatch_bwd(grecv)
    gl2 = r.route_bwd(ld, idd, gwd)
    bits = (lambda t: t.view(torch.int16)) if gx.dtype == torch.bfloat16 else (lambda t: t)
    assert torch.equal(bits(gx), bits(gx2)) and torch.equal(gl, gl2)


def test_dispatch_bwd_route_full_size_deepseek_v3():
    wl = synth.WORKLOADS[3]
    inp = synth.make_inputs(wl, want=("logits", "bias"))
    idx, w = oracle_route(wl, inp["logits"], inp["bias"])
    gw = synth.normal_f32(wl.seed, "grecv", (wl.T, wl.K))
    r = router(wl)
    r.layout(to_dev(idx))
    rows = r.h.recv_rows
    grecv = torch.randn(rows, wl.H, device=to_dev(gw).device,
                        generator=torch.Generator(device="cuda").manual_seed(5)).to(torch.bfloat16)
    ld, idd, gwd = to_dev(inp["logits"]), to_dev(idx), to_dev(gw)
    gx, gl = r.dispatch_bwd_route(grecv, ld, idd, gwd)
    gx2 = r.dispatch_bwd(grecv)
    gl2 = r.route_bwd(ld, idd, gwd)
    assert torch.equal(gx.view(torch.int16), gx2.view(torch.int16)) and torch.equal(gl, gl2)
    ref = oracle.route_bwd(inp["logits"], idx, gw.astype(np.float64), "sigmoid", True, 1.0)
    assert_close_rows(to_host(gl), ref)
