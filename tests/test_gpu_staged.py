"""Staged (wire-faithful) dispatch and combine on the GPU against the oracle:
send rows, expansion to expert rows, per-(token, rank) partial rows and their
reduction.  Integer and copy outputs bit-exact; the partial and reduced rows
follow the oracle's summation order, so they are bit-exact too (asserted
against the 1-ulp bound)."""
import numpy as np
import pytest

import oracle
import synth
from tests.common import assert_ulp
from tests.gpu_util import oracle_route, router, to_dev, to_host

pytestmark = pytest.mark.gpu

SIZES = {0: 256, 1: 2600, 2: 2600, 3: 2600}


@pytest.mark.parametrize("i", [0, 1, 2, 3])
def test_staged_path(i):
    wl = synth.WORKLOADS[i].with_tokens(SIZES[i])
    inp = synth.make_inputs(wl, want=("logits", "bias", "x", "y"))
    idx, w = oracle_route(wl, inp["logits"], inp["bias"])
    L = oracle.layout(idx, wl.E, wl.R)
    r = router(wl)
    r.layout(to_dev(idx))
    recv, _, send = r.dispatch(to_dev(inp["x"]), to_dev(w), with_send=True)
    orecv, _, osend = oracle.dispatch(inp["x"], L, w, with_send=True)
    n = int(L.off_e[-1])
    assert np.array_equal(to_host(send)[:L.S], osend[:L.S])
    expanded = to_host(r.expand(send))
    assert np.array_equal(expanded[:n], oracle.expand(osend, L)[:n])
    assert np.array_equal(expanded[:n], orecv[:n])
    for weighted in (True, False):
        ww = w if weighted else None
        part = r.combine_partial(to_dev(inp["y"]), to_dev(ww) if weighted else None)
        opart = oracle.combine_partial(inp["y"], L, ww)
        d = assert_ulp(to_host(part)[:L.S], opart[:L.S], 1, "partial")
        assert int(d.max()) == 0
        out = to_host(r.combine_reduce(part))
        d = assert_ulp(out, oracle.combine_reduce(opart, L), 1, "reduce")
        assert int(d.max()) == 0
    print("workload %d: dedup factor T*K/S = %.3f" % (i, wl.T * wl.K / L.S))


def test_staged_with_one_rank_equals_combine():
    wl = synth.WORKLOADS[1].with_tokens(1500)
    import dataclasses
    wl = dataclasses.replace(wl, R=1)
    inp = synth.make_inputs(wl, want=("logits", "y"))
    idx, w = oracle_route(wl, inp["logits"], None)
    r = router(wl)
    r.layout(to_dev(idx))
    y, wd = to_dev(inp["y"]), to_dev(w)
    staged = to_host(r.combine_reduce(r.combine_partial(y, wd)))
    assert np.array_equal(staged, to_host(r.combine(y, wd)))
