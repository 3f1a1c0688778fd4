"""Routing configurations of the eight-threads-per-token kernel (E of 64, 128
or 256, K <= 8) against the oracle: groups of one, two and four threads'
experts, all groups kept, a single-key group score, K not a power of two,
a route scale, sigmoid without renormalisation.  A quarter of the tokens
carry exact ties and one-ulp near-ties among their largest keys, so the
hand-over to the warp-per-token path runs in every configuration, and a few
tokens carry a non-finite logit."""
import numpy as np
import pytest

import combine_moe_route_05_gb300 as moe
import synth
from tests.common import assert_ulp
from tests.gpu_util import oracle_route, router, to_dev, to_host

pytestmark = pytest.mark.gpu

# (E, K, G, TG, GK, score_fn, renorm, route_scale)
CONFIGS = [
    (256, 8, 4, 2, 2, "sigmoid", True, 1.0),     # a group is two threads' experts
    (256, 8, 2, 1, 2, "sigmoid", True, 2.5),     # four threads per group
    (128, 6, 8, 8, 1, "sigmoid", True, 1.0),     # all groups kept, GK = 1
    (64, 4, 4, 2, 2, "sigmoid", True, 1.0),      # E = 64: eight experts per thread
    (128, 8, 1, 1, 1, "sigmoid", False, 2.5),    # no renormalisation
    (256, 7, 1, 1, 1, "softmax", True, 2.5),
    (64, 1, 1, 1, 1, "softmax", True, 1.0),
    (128, 5, 1, 1, 1, "softmax", True, 1.0),
]


def tied_logits(rng, T, E):
    logits = rng.standard_normal((T, E)).astype(np.float32)
    rows = rng.choice(T, size=T // 4, replace=False)
    for t in rows:
        order = np.argsort(-logits[t])
        a, b = order[rng.integers(0, 6)], order[rng.integers(0, 9)]
        if rng.random() < 0.5:
            logits[t, b] = logits[t, a]  # an exact tie
        else:
            logits[t, b] = np.nextafter(logits[t, a], np.float32(-np.inf))  # one ulp apart
    return logits


@pytest.mark.parametrize("cfg", CONFIGS, ids=lambda c: "E%d-K%d-G%d-TG%d-GK%d-%s-r%d-s%g" % c)
def test_team_routing_matches_oracle(cfg):
    E, K, G, TG, GK, score_fn, renorm, scale = cfg
    T = 2053  # a ragged last warp
    rng = np.random.default_rng(E * 131 + K * 7 + G)
    logits = tied_logits(rng, T, E)
    bias = None
    if score_fn == "sigmoid":
        bias = (rng.standard_normal(E) * 0.05).astype(np.float32)
        bias[rng.integers(0, E)] = bias[rng.integers(0, E)]  # two experts with equal bias
    wl = synth.Workload("team", T=T, H=16, E=E, K=K, R=E // 8, score_fn=score_fn, n_groups=G,
                        topk_groups=TG, group_score_topk=GK, renorm=renorm, route_scale=scale)
    r = router(wl)
    gi, gw_ = r.route(to_dev(logits), None if bias is None else to_dev(bias))
    idx, w = oracle_route(wl, logits, bias)
    gi = to_host(gi)
    assert np.array_equal(gi, idx), "%d tokens differ" % int((gi != idx).any(1).sum())
    assert_ulp(to_host(gw_), w, 1, "w")
    assert moe.moe_read_device_status(r.h) == 0


@pytest.mark.parametrize("score_fn", ["softmax", "sigmoid"])
def test_team_routing_with_nonfinite_logits(score_fn):
    """Tokens with a NaN or infinite logit are routed on the warp path, which
    raises the status bit; the other tokens of their warps are unaffected."""
    rng = np.random.default_rng(5)
    T, E, K = 300, 128, 8
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[7, 3] = np.nan
    logits[40, 100] = -np.inf
    logits[41, 5] = np.inf
    wl = synth.Workload("team", T=T, H=16, E=E, K=K, R=16, score_fn=score_fn)
    r = router(wl)
    gi, gw_ = r.route(to_dev(logits))
    assert moe.moe_read_device_status(r.h) & moe.MOE_DEVERR_NONFINITE
    clean = np.setdiff1d(np.arange(T), [7, 40, 41])
    idx, w = oracle_route(wl, logits[clean], None)
    assert np.array_equal(to_host(gi)[clean], idx)
    assert_ulp(to_host(gw_)[clean], w, 1, "w")
