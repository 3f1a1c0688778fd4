"""Edge cases of the CUDA path against the oracle: empty and single-token
batches, dropped (invalid or repeated) expert indices, capacity and call-order
errors, misaligned pointers, ties, and the extremes of E, K and R."""
import numpy as np
import pytest
import torch

import combine_moe_route_05_gb300 as moe
import oracle
import synth
from tests.common import assert_ulp, gw_tolerance_ok, row_norms_for_gw
from tests.gpu_util import dev, layout_host, router, to_dev, to_host

pytestmark = pytest.mark.gpu


def small(E, K, R, T, H=64, seed=0, **kw):
    wl = synth.Workload("edge", T=T, H=H, E=E, K=K, R=R, **kw)
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = synth.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    y = synth.to_bf16_bits(rng.standard_normal((T * K, H)).astype(np.float32))
    g = synth.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    return wl, logits, x, y, g


def rows_f32(a):
    return a if a.dtype == np.float32 else oracle.bf16_to_f32(a)


def check_chain(r, wl, idx, w, x, y, g):
    L = oracle.layout(idx, wl.E, wl.R)
    r.layout(to_dev(idx))
    got = layout_host(r)
    for f in oracle.Layout.FIELDS:
        assert np.array_equal(got[f].reshape(-1), getattr(L, f).reshape(-1)), f
    recv, recv_w, send = r.dispatch(to_dev(x), to_dev(w), with_send=True)
    orecv, orw, osend = oracle.dispatch(x, L, w, with_send=True)
    n = int(L.off_e[-1])
    assert np.array_equal(to_host(recv)[:n], orecv[:n])
    assert np.array_equal(to_host(send)[:L.S], osend[:L.S])
    assert_ulp(to_host(r.combine(to_dev(y), to_dev(w))), oracle.combine(y, L, w), 0, "combine")
    gy, gw_ = r.combine_bwd(to_dev(g), to_dev(y), to_dev(w))
    ogy, ogw = oracle.combine_bwd(g, y, L, w)
    assert_ulp(to_host(gy)[:n], ogy[:n], 0, "gy")
    gn, yn = row_norms_for_gw(rows_f32(g), rows_f32(y), L.pos)
    ok = gw_tolerance_ok(to_host(gw_), ogw, gn, yn)
    assert ok.all(), "router-score gradient out of tolerance at %d entries" % int((~ok).sum())
    assert_ulp(to_host(r.dispatch_bwd(to_dev(y))), oracle.dispatch_bwd(y, L), 0, "gx")
    return L


@pytest.mark.parametrize("E,K,R", [(512, 16, 512), (512, 16, 1), (8, 1, 1), (8, 8, 8), (64, 3, 4),
                                   (32, 5, 32), (128, 8, 128)])
@pytest.mark.parametrize("T", [1, 33, 1025, 3071])
def test_extremes_of_E_K_R(E, K, R, T):
    wl, logits, x, y, g = small(E, K, R, T)
    r = router(wl)
    gi, gw_ = r.route(to_dev(logits))
    idx, w = oracle.route_softmax(logits, K)
    assert np.array_equal(to_host(gi), idx)
    assert_ulp(to_host(gw_), w, 1, "w")
    L = check_chain(r, wl, idx, w, x, y, g)
    if R == 1:
        assert L.S == T
    if R == E:
        assert L.S == T * K


@pytest.mark.parametrize("E,K,R,T", [(64, 4, 8, 4096), (16, 2, 4, 160000)])
def test_layout_single_and_two_launch_paths(E, K, R, T):
    """The layout runs as one cooperative launch when all its tiles fit on the
    GPU at once and as two launches otherwise (here T = 160000: 313 tiles);
    both give the oracle's layout bit for bit, twice in a row (the arrival
    ticket and the epoch are reset / advanced correctly)."""
    wl = synth.Workload("edge", T=T, H=64, E=E, K=K, R=R)
    rng = np.random.default_rng(7)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int32)
    r = router(wl)
    n = moe.moe_dispatch_layout_launches(r.h, T)
    assert n == (1 if T <= 4096 else 2)
    L = oracle.layout(idx, E, R)
    for _ in range(2):
        r.layout(to_dev(idx))
        got = layout_host(r)
        for f in oracle.Layout.FIELDS:
            assert np.array_equal(got[f].reshape(-1), getattr(L, f).reshape(-1)), f
    assert moe.moe_read_device_status(r.h) == 0


def test_empty_batch():
    wl, logits, x, y, g = small(16, 4, 4, 8)
    r = router(wl)
    idx = torch.empty(0, 4, dtype=torch.int32, device=dev())
    lay = r.layout(idx)
    assert (to_host(lay["cnt_e"]) == 0).all() and (to_host(lay["off_e"]) == 0).all()
    assert int(to_host(lay["S"])[0]) == 0
    e = torch.empty(0, 64, dtype=torch.bfloat16, device=dev())
    recv, _, _ = r.dispatch(e, None)
    assert recv.shape == (0, 64)
    assert r.combine(torch.empty(0, 64, dtype=torch.bfloat16, device=dev())).shape == (0, 64)
    i2, w2 = r.route(torch.empty(0, 16, device=dev()))
    assert i2.shape == (0, 4)
    torch.cuda.synchronize()


def test_dropped_entries_set_flags_and_are_skipped():
    E, K, R, T, H = 16, 4, 4, 40, 32
    wl, logits, x, y, g = small(E, K, R, T, H)
    rng = np.random.default_rng(5)
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    idx[3, 1] = idx[3, 0]   # repeated expert
    idx[7, 2] = E           # out of range
    idx[8, 0] = -1          # out of range
    w = rng.random((T, K)).astype(np.float32)
    r = router(wl)
    L = check_chain(r, wl, idx, w, x, y, g)
    assert L.dropped == 3
    flags = moe.moe_read_device_status(r.h)
    assert flags & moe.MOE_DEVERR_BAD_EXPERT and flags & moe.MOE_DEVERR_DUP_EXPERT
    moe.moe_clear_device_status(r.h)
    assert moe.moe_read_device_status(r.h) == 0


def test_nonfinite_logits_are_flagged():
    wl, logits, x, y, g = small(16, 2, 2, 4)
    logits[2, 5] = np.nan
    r = router(wl)
    r.route(to_dev(logits))
    assert moe.moe_read_device_status(r.h) & moe.MOE_DEVERR_NONFINITE


def test_all_equal_logits_select_lowest_indices():
    for score in ("softmax", "sigmoid"):
        wl = synth.Workload("ties", T=64, H=16, E=64, K=8, R=8, score_fn=score)
        r = router(wl)
        gi, gw_ = r.route(torch.full((64, 64), 0.5, device=dev()))
        assert (to_host(gi) == np.arange(8)).all()
        assert (to_host(gw_) == np.float32(0.125)).all()


def test_tie_heavy_grouped_routing():
    rng = np.random.default_rng(3)
    wl = synth.Workload("ties", T=500, H=16, E=64, K=6, R=8, score_fn="sigmoid", n_groups=8,
                        topk_groups=3, group_score_topk=2)
    logits = (rng.integers(-2, 3, size=(500, 64)) * 0.5).astype(np.float32)
    bias = (rng.integers(-1, 2, size=64) * 0.125).astype(np.float32)
    r = router(wl)
    gi, gw_ = r.route(to_dev(logits), to_dev(bias))
    idx, w = oracle.route_sigmoid_grouped(logits, bias, 6, 8, 3, 2)
    assert np.array_equal(to_host(gi), idx)
    assert_ulp(to_host(gw_), w, 1, "w")


def test_capacity_and_call_order_errors():
    wl, logits, x, y, g = small(16, 4, 4, 8)
    r = router(wl, max_tokens=8)
    with pytest.raises(moe.MoeError) as e:
        r.combine(to_dev(y))
    assert e.value.status == moe.MOE_ERR_STATE
    too_many = torch.zeros(9, 4, dtype=torch.int32, device=dev())
    with pytest.raises(moe.MoeError) as e:
        r.layout(too_many)
    assert e.value.status == moe.MOE_ERR_CAPACITY
    with pytest.raises(moe.MoeError) as e:
        r.route(torch.zeros(9, 16, device=dev()))
    assert e.value.status == moe.MOE_ERR_CAPACITY


def test_misaligned_rows_are_rejected():
    wl, logits, x, y, g = small(16, 4, 4, 8, H=64)
    r = router(wl)
    idx, w = oracle.route_softmax(logits, 4)
    r.layout(to_dev(idx))
    xb = torch.empty(8 * 64 + 1, dtype=torch.bfloat16, device=dev())[1:].view(8, 64)
    recv = torch.empty(32, 64, dtype=torch.bfloat16, device=dev())
    st = moe.lib().moe_dispatch(r.h.ptr, xb.data_ptr(), 64, moe.MOE_BF16, None, recv.data_ptr(),
                                None, None, None)
    assert st == moe.MOE_ERR_INVALID
    st = moe.lib().moe_dispatch(r.h.ptr, recv.data_ptr(), 60, moe.MOE_BF16, None, recv.data_ptr(),
                                None, None, None)
    assert st == moe.MOE_ERR_INVALID  # 120-byte rows are not a multiple of 16


def test_fp32_rows_and_large_rows():
    """fp32 rows (the tiny workload's dtype) and rows longer than one bulk
    copy (16 KiB), which the dispatch splits into several chunks."""
    for H, dt in ((256, np.float32), (12288, np.uint16), (8200, np.float32)):
        rng = np.random.default_rng(H)
        T, E, K, R = 70, 16, 4, 4
        wl = synth.Workload("rows", T=T, H=H, E=E, K=K, R=R)
        logits = rng.standard_normal((T, E)).astype(np.float32)
        mk = (lambda a: a) if dt == np.float32 else synth.to_bf16_bits
        x = mk(rng.standard_normal((T, H)).astype(np.float32))
        y = mk(rng.standard_normal((T * K, H)).astype(np.float32))
        g = mk(rng.standard_normal((T, H)).astype(np.float32))
        idx, w = oracle.route_softmax(logits, K)
        check_chain(router(wl), wl, idx, w, x, y, g)


def near_tie_logits(rng, T, E):
    """Logits from a few values nudged by a few fp32 ulps, so that many keys
    are closer than the fp32 selection's error bound and the kernel must decide
    those tokens in fp64."""
    # no zero base: a bit-pattern nudge below +0 would make a NaN
    base = rng.choice(np.float32([-1.0, -0.125, 0.25, 0.5, 1.0, 2.0]), size=(T, E))
    ulps = rng.integers(-3, 4, size=(T, E)).astype(np.int32)
    out = (base.view(np.int32) + ulps).view(np.float32)
    assert np.isfinite(out).all()
    return out


@pytest.mark.parametrize("grouped", [False, True])
def test_near_tie_sigmoid_routing_matches_fp64_oracle(grouped):
    rng = np.random.default_rng(21 + grouped)
    T, E, K = 3000, 256, 8
    logits = near_tie_logits(rng, T, E)
    bias = (rng.integers(-2, 3, size=E) * np.float32(1e-7)).astype(np.float32)
    G, TG, GK = (8, 4, 2) if grouped else (1, 1, 1)
    wl = synth.Workload("neartie", T=T, H=16, E=E, K=K, R=64, score_fn="sigmoid", n_groups=G,
                        topk_groups=TG, group_score_topk=GK)
    r = router(wl)
    gi, gw_ = r.route(to_dev(logits), to_dev(bias))
    idx, w = oracle.route_sigmoid_grouped(logits, bias, K, G, TG, GK)
    assert np.array_equal(to_host(gi), idx)
    assert_ulp(to_host(gw_), w, 1, "w")


def test_near_tie_softmax_routing_is_exact():
    rng = np.random.default_rng(23)
    T, E, K = 3000, 128, 8
    logits = near_tie_logits(rng, T, E)
    wl = synth.Workload("neartie", T=T, H=16, E=E, K=K, R=8)
    gi, gw_ = router(wl).route(to_dev(logits))
    idx, w = oracle.route_softmax(logits, K)
    assert np.array_equal(to_host(gi), idx)
    assert_ulp(to_host(gw_), w, 1, "w")


@pytest.mark.parametrize("bias_std", [0.01, 0.3])
def test_large_random_grouped_routing_matches_fp64_oracle(bias_std):
    """131072 DeepSeek-V3-shaped tokens: any case where the fp32 selection's
    error bound were wrong would show up as an index mismatch."""
    T, E = 131072, 256
    rng = np.random.default_rng(int(bias_std * 1000))
    logits = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    bias = (rng.standard_normal(E) * bias_std).astype(np.float32)
    wl = synth.Workload("big", T=T, H=16, E=E, K=8, R=64, score_fn="sigmoid", n_groups=8,
                        topk_groups=4, group_score_topk=2)
    gi, gw_ = router(wl).route(to_dev(logits), to_dev(bias))
    idx, w = oracle.route_sigmoid_grouped(logits, bias, 8, 8, 4, 2)
    gi = to_host(gi)
    assert np.array_equal(gi, idx), "%d tokens differ" % int((gi != idx).any(1).sum())
    assert_ulp(to_host(gw_), w, 1, "w")


@pytest.mark.parametrize("score_fn,renorm", [("softmax", True), ("sigmoid", True), ("sigmoid", False)])
def test_weights_over_the_exponent_range(score_fn, renorm):
    """Logits of magnitude 1e-3 to 800 with either sign: softmax differences to
    the top pick run from 0 to beyond the fp64 range of exp, sigmoid scores
    saturate at both ends.  The weights' exponential and reciprocal are the
    kernel's own (not the library's), so they must stay within 1 fp32 ulp of
    the oracle's across that whole range."""
    rng = np.random.default_rng(31 + (score_fn == "sigmoid") + renorm)
    T, E, K = 4096, 64, 8
    mag = 10.0 ** rng.uniform(-3, np.log10(800.0), size=(T, E))
    logits = (mag * rng.choice([-1.0, 1.0], size=(T, E))).astype(np.float32)
    wl = synth.Workload("range", T=T, H=16, E=E, K=K, R=8, score_fn=score_fn, renorm=renorm)
    gi, gw_ = router(wl).route(to_dev(logits))
    if score_fn == "softmax":
        idx, w = oracle.route_softmax(logits, K, renorm)
    else:
        idx, w = oracle.route_sigmoid_grouped(logits, None, K, 1, 1, 1, renorm)
    assert np.array_equal(to_host(gi), idx)
    assert_ulp(to_host(gw_), w, 1, "w")
