"""Router backward to the logits on the GPU against the oracle's fp64
derivative of the routing weights (selection held fixed).

Acceptance: within 2 fp32 ulps of the oracle's value rounded to fp32, plus
1e-9 of the row's largest magnitude (both sides compute in fp64; device and
host exp may differ in the last fp64 bit, which matters only where the
difference gw_j - sum_k q_k gw_k cancels)."""
import numpy as np
import pytest

import oracle
import synth
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
    import dataclasses
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
