"""Router-score absorption fused into the W2 grouped GEMM on the GPU (tensor
cores) against the oracle's definition: the scores scale the W2 input rows in
fp32, the scaled rows are rounded to bf16, and each expert's segment is
multiplied by that expert's W2; the oracle sums exactly (fp64) and rounds once.

Acceptance: the GPU accumulates in fp32 in its own order.  Each output must
lie within one bf16 spacing of the exact sum plus the fp32 summation bound
I * 2^-24 * sum_i |hs[r,i] * W2[e][n,i]| (the second term matters only where
the sum cancels to far below its terms; elsewhere the accumulation error is
~1e-3 of a bf16 spacing).  At most 1% of the outputs may differ from the
once-rounded exact sum at all (~0.01% seen): skipping the bf16 rounding of the
scaled rows would move ~20% of them, so the fraction pins that rounding.
Pad rows of a padded layout must be exactly 0; rows outside every expert
segment are left untouched."""
import dataclasses

import numpy as np
import pytest
import torch

import combine_moe_route_05_gb300 as moe
import oracle
import synth
from tests.common import ulp_dist
from tests.gpu_util import dev, oracle_route, router, to_dev, to_host

pytestmark = pytest.mark.gpu

MAX_OFF_BY_ONE = 0.01


def problem(wl, I, H, pad=1):
    """Routing, layouts (GPU and oracle), receive-row scores, h rows and W2."""
    wl = dataclasses.replace(wl, I=I, H=H, pad_align=pad)
    inp = synth.make_inputs(wl, want=("logits", "bias"))
    idx, w = oracle_route(wl, inp["logits"], inp["bias"])
    L = oracle.layout(idx, wl.E, wl.R, align=max(pad, 1))
    r = router(wl)
    r.layout(to_dev(idx))
    rows = r.h.recv_rows
    assert rows == L.recv_rows
    lay = moe.layout_tensors(r.h)
    assert np.array_equal(to_host(lay["off_e"]), L.off_e)
    assert np.array_equal(to_host(lay["cnt_e"]), L.cnt_e)
    _, recv_w, _ = r.dispatch(torch.zeros(wl.T, 8, dtype=torch.bfloat16, device=dev()), to_dev(w))
    h = synth.normal_bf16(wl.seed, "h", (rows, I))
    w2 = synth.w2_weights(wl.seed, wl.E, H, I)
    return wl, r, L, to_host(recv_w), h, w2


def abs_terms(h, recv_w, w2, seg_of_row):
    """sum_i |hs[r,i] * W2[e(r)][n,i]| for the given rows (fp64)."""
    hs = synth.bf16_bits_to_f32(synth.to_bf16_bits(synth.bf16_bits_to_f32(h) * recv_w[:, None]))
    hs = np.abs(hs.astype(np.float64))
    out = np.zeros((h.shape[0], w2.shape[1]))
    for e in np.unique(seg_of_row):
        m = seg_of_row == e
        out[m] = hs[m] @ np.abs(synth.bf16_bits_to_f32(w2[e]).astype(np.float64)).T
    return out


def check_rows(got, want64, want_bits, absum, I, label):
    g = synth.bf16_bits_to_f32(got).astype(np.float64)
    spacing = np.spacing(np.abs(synth.bf16_bits_to_f32(want_bits))) * 2.0 ** 16
    bound = spacing + I * 2.0 ** -24 * absum
    bad = np.abs(g - want64) > bound
    assert not bad.any(), "%s: %d outputs out of bound" % (label, int(bad.sum()))
    frac = float((ulp_dist(got, want_bits) > 0).mean())
    assert frac <= MAX_OFF_BY_ONE, "%s: %.4f of outputs differ" % (label, frac)
    return frac


def run_gpu(r, h, recv_w, w2, sentinel=None):
    y = torch.empty(h.shape[0], w2.shape[1], dtype=torch.bfloat16, device=dev())
    if sentinel is not None:
        y.view(torch.int16).fill_(sentinel)
    moe.moe_w2_absorbed(r.h, to_dev(h), to_dev(recv_w), to_dev(w2), y)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(r.h) == 0
    return to_host(y)


@pytest.mark.parametrize("case", ["qwen3_235b_small", "skewed", "ragged_I", "padded"])
def test_w2_absorbed_all_rows(case):
    if case == "qwen3_235b_small":
        wl, r, L, recv_w, h, w2 = problem(synth.WORKLOADS[4].with_tokens(700), I=256, H=512)
    elif case == "skewed":
        wl, r, L, recv_w, h, w2 = problem(synth.WORKLOADS[2].with_tokens(2048), I=128, H=256)
        assert (L.cnt_e == 0).any() and L.cnt_e.max() > 3 * 128
    elif case == "ragged_I":
        wl, r, L, recv_w, h, w2 = problem(synth.WORKLOADS[1].with_tokens(600), I=200, H=256)
    else:
        wl, r, L, recv_w, h, w2 = problem(synth.WORKLOADS[4].with_tokens(600), I=128, H=256, pad=128)
    sentinel = 0x7FC1  # a NaN pattern the kernel never writes
    y = run_gpu(r, h, recv_w, w2, sentinel=sentinel)
    n = int(L.off_e[-1])
    yb, y64 = oracle.w2_absorbed(h, recv_w, w2, L.off_e, L.cnt_e, rows=np.arange(n))
    real = np.zeros(n, bool)
    for e in range(wl.E):
        real[L.off_e[e]:L.off_e[e] + L.cnt_e[e]] = True
    seg_of = np.repeat(np.arange(wl.E), np.diff(L.off_e))[:n][real]
    absum = abs_terms(h[:n][real], recv_w[:n][real], w2, seg_of)
    frac = check_rows(y[:n][real], y64[real], yb[real], absum, h.shape[1], case)
    assert (y[:n][~real] == 0).all()  # pad rows
    assert (y[n:].view(np.int16) == sentinel).all()  # outside every segment
    # rounding the scaled rows is what keeps the fraction small
    hs_unrounded = synth.bf16_bits_to_f32(h[:n][real]).astype(np.float64) * recv_w[:n][real, None]
    print("%s: %.4f%% of outputs one ulp off" % (case, 100 * frac))
    sample = np.arange(0, hs_unrounded.shape[0], max(1, hs_unrounded.shape[0] // 64))
    alt = np.stack([hs_unrounded[i] @ synth.bf16_bits_to_f32(w2[seg_of[i]]).astype(np.float64).T
                    for i in sample])
    alt_frac = float((ulp_dist(oracle.f64_to_bf16(alt), yb[real][sample]) > 0).mean())
    assert alt_frac > 5 * max(frac, 0.002), (alt_frac, frac)


def test_w2_absorbed_repeated_runs_identical():
    """The pipeline hands shared-memory stages, tensor-memory stages and the
    accumulator between warps; a hand-over race shows up as run-to-run
    differences in whole rows.  Eight runs must be bitwise identical and each
    within the bound."""
    wl, r, L, recv_w, h, w2 = problem(synth.WORKLOADS[4].with_tokens(700), I=256, H=512)
    n = int(L.off_e[-1])
    first = run_gpu(r, h, recv_w, w2)
    for _ in range(7):
        assert np.array_equal(run_gpu(r, h, recv_w, w2)[:n], first[:n])
    yb, y64 = oracle.w2_absorbed(h, recv_w, w2, L.off_e, L.cnt_e, rows=np.arange(n))
    seg_of = np.repeat(np.arange(wl.E), np.diff(L.off_e))
    check_rows(first[:n], y64, yb, abs_terms(h[:n], recv_w[:n], w2, seg_of), h.shape[1], "repeat")


def test_w2_absorbed_full_size_sampled_rows():
    """The whole Qwen3-235B-shaped problem (T=32768, K=8, E=128, I=1536,
    H=4096), checked on sampled rows: the first, a middle and the last row of
    every 8th expert's segment and 64 random rows."""
    wl, r, L, recv_w, h, w2 = problem(synth.WORKLOADS[4], I=1536, H=4096)
    y = run_gpu(r, h, recv_w, w2)
    rng = np.random.default_rng(5)
    picks = []
    for e in range(0, wl.E, 8):
        lo, c = int(L.off_e[e]), int(L.cnt_e[e])
        if c:
            picks += [lo, lo + c // 2, lo + c - 1]
    picks += list(rng.integers(0, int(L.off_e[-1]), 64))
    rows = np.array(sorted(set(picks)), np.int64)
    yb, y64 = oracle.w2_absorbed(h, recv_w, w2, L.off_e, L.cnt_e, rows=rows)
    seg_of = np.searchsorted(L.off_e, rows, side="right") - 1
    absum = abs_terms(h[rows], recv_w[rows], w2, seg_of)
    frac = check_rows(y[rows], y64, yb, absum, h.shape[1], "full size")
    print("full size: %d rows, %.4f%% one ulp off" % (rows.size, 100 * frac))


@pytest.mark.parametrize("E,K,R,T,I,H", [(512, 8, 64, 300, 8, 256),   # E at its maximum, I at its minimum
                                         (8, 2, 2, 1, 64, 256),        # one token
                                         (16, 4, 4, 257, 72, 768)])    # ragged I past one slice, two n-tiles
def test_w2_absorbed_shapes(E, K, R, T, I, H):
    wl = dataclasses.replace(synth.WORKLOADS[1], E=E, K=K, R=R).with_tokens(T)
    wl, r, L, recv_w, h, w2 = problem(wl, I=I, H=H)
    y = run_gpu(r, h, recv_w, w2, sentinel=0x7FC1)
    n = int(L.off_e[-1])
    yb, y64 = oracle.w2_absorbed(h, recv_w, w2, L.off_e, L.cnt_e, rows=np.arange(n))
    seg_of = np.repeat(np.arange(wl.E), np.diff(L.off_e))
    check_rows(y[:n], y64, yb, abs_terms(h[:n], recv_w[:n], w2, seg_of), I, "shape")


def test_w2_absorbed_pad_rows_ignore_their_input():
    """Pad rows of a padded layout hold whatever the caller left there (NaN
    here): they come out 0 and no real row is touched by them."""
    wl, r, L, recv_w, h, w2 = problem(synth.WORKLOADS[4].with_tokens(300), I=64, H=256, pad=128)
    n = int(L.off_e[-1])
    real = np.zeros(h.shape[0], bool)
    for e in range(wl.E):
        real[L.off_e[e]:L.off_e[e] + L.cnt_e[e]] = True
    h = h.copy()
    h[~real] = 0x7FC0  # bf16 NaN in every pad row
    y = run_gpu(r, h, recv_w, w2)
    assert (y[:n][~real[:n]] == 0).all()
    yb, y64 = oracle.w2_absorbed(h, recv_w, w2, L.off_e, L.cnt_e, rows=np.nonzero(real)[0])
    seg_of = np.searchsorted(L.off_e, np.nonzero(real)[0], side="right") - 1
    check_rows(y[real], y64, yb, abs_terms(h[real], recv_w[real], w2, seg_of), 64, "pads")


def test_w2_absorbed_argument_checks():
    wl = dataclasses.replace(synth.WORKLOADS[4].with_tokens(64), I=64, H=256)
    r = router(wl)
    h = torch.zeros(wl.T * wl.K, 64, dtype=torch.bfloat16, device=dev())
    rw = torch.zeros(wl.T * wl.K, dtype=torch.float32, device=dev())
    w2 = torch.zeros(wl.E, 256, 64, dtype=torch.bfloat16, device=dev())
    y = torch.zeros(wl.T * wl.K, 256, dtype=torch.bfloat16, device=dev())
    with pytest.raises(moe.MoeError) as e:
        moe.moe_w2_absorbed(r.h, h, rw, w2, y)  # before any layout
    assert e.value.status == moe.MOE_ERR_STATE
    idx = torch.arange(wl.K, dtype=torch.int32, device=dev()).repeat(wl.T, 1)
    r.layout(idx)
    moe.moe_w2_absorbed(r.h, h, rw, w2, y)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(r.h) == 0
    for bad_I, bad_H in ((60, 256), (64, 200)):
        hb = torch.zeros(wl.T * wl.K, bad_I, dtype=torch.bfloat16, device=dev())
        w2b = torch.zeros(wl.E, bad_H, bad_I, dtype=torch.bfloat16, device=dev())
        yb = torch.zeros(wl.T * wl.K, bad_H, dtype=torch.bfloat16, device=dev())
        with pytest.raises(moe.MoeError) as e:
            moe.moe_w2_absorbed(r.h, hb, rw, w2b, yb)
        assert e.value.status == moe.MOE_ERR_INVALID
