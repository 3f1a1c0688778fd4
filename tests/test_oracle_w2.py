"""Pins of the oracle's absorbed W2 projection (router scores applied to the
W2 input rows in fp32, rounded to bf16, then the expert's W2 GEMM) and of its
single fp64 -> bf16 rounding, against things other than the oracle itself:
exact rational rounding, numpy's fp64 matmul, closed forms for diagonal
weights, and exact power-of-two scaling."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth


def _bf16(a):
    return synth.to_bf16_bits(np.asarray(a, np.float32))


def _f32(bits):
    return synth.bf16_bits_to_f32(bits)


def _segments(counts, pad=1):
    seg = [(c + pad - 1) // pad * pad for c in counts]
    off = np.concatenate([[0], np.cumsum(seg)]).astype(np.int32)
    return off, np.asarray(counts, np.int32)


def _problem(counts, I, H, pad=1, seed=3, unit=False):
    rng = np.random.default_rng(seed)
    off, cnt = _segments(counts, pad)
    rows = int(off[-1])
    E = len(counts)
    h = _bf16(rng.standard_normal((rows, I)))
    w2 = _bf16(rng.standard_normal((E, H, I)) / np.sqrt(I))
    w = np.ones(rows, np.float32) if unit else rng.uniform(0.05, 1.0, rows).astype(np.float32)
    return h, w, w2, off, cnt


def _bf16_exact_round(x):
    """Nearest bf16 to the fp64 value x in exact rational arithmetic, ties to
    an even significand (finite normal values only)."""
    f = np.float32(x)
    b = int(np.array([f]).view(np.uint32)[0] >> 16)
    cands = [c for c in (b - 1, b, b + 1, b + 2) if 0 <= c < 0x10000]
    best = None
    for c in cands:
        v = Fraction(float(_f32(np.array([c], np.uint16))[0]))
        d = abs(v - Fraction(float(x)))
        key = (d, c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_f64_to_bf16_rounds_once():
    rng = np.random.default_rng(7)
    base = _f32(_bf16(rng.standard_normal(400)))
    ulp = np.abs(base) * 2.0 ** -7
    # values on, just above and just below the bf16 midpoints, plus random ones
    mids = base.astype(np.float64) + ulp / 2
    xs = np.concatenate([mids, mids + ulp * 1e-9, mids - ulp * 1e-9,
                         rng.standard_normal(400) * 10.0])
    got = oracle.f64_to_bf16(xs)
    want = np.array([_bf16_exact_round(x) for x in xs], np.uint16)
    assert np.array_equal(got, want)
    # rounding through fp32 first would get the nudged midpoints wrong
    via32 = _bf16(xs.astype(np.float32))
    assert not np.array_equal(via32, want)


def test_w2_unit_scores_equal_matmul():
    h, w, w2, off, cnt = _problem([5, 0, 9, 3], I=40, H=24, unit=True)
    y, y64 = oracle.w2_absorbed(h, w, w2, off, cnt)
    for e in range(len(cnt)):
        lo, hi = off[e], off[e] + cnt[e]
        ref = _f32(h[lo:hi]).astype(np.float64) @ _f32(w2[e]).astype(np.float64).T
        np.testing.assert_allclose(y64[lo:hi], ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(y, oracle.f64_to_bf16(y64))


def test_w2_scores_scale_and_round_before_gemm():
    h, w, w2, off, cnt = _problem([7, 4, 11], I=64, H=16)
    _, y64 = oracle.w2_absorbed(h, w, w2, off, cnt)
    hs = _f32(_bf16(_f32(h) * w[:, None])).astype(np.float64)
    unrounded = (_f32(h) * w[:, None]).astype(np.float64)
    for e in range(len(cnt)):
        lo, hi = off[e], off[e] + cnt[e]
        wt = _f32(w2[e]).astype(np.float64).T
        np.testing.assert_allclose(y64[lo:hi], hs[lo:hi] @ wt, rtol=1e-12, atol=1e-12)
        # the test is sensitive to the rounding of the scaled rows
        assert np.abs(y64[lo:hi] - unrounded[lo:hi] @ wt).max() > 1e-6


def test_w2_diagonal_weights_closed_form():
    # W2[e] = (e + 1) * identity (H = I): y = round((e + 1) * hs) per segment
    counts = [3, 6, 0, 2]
    I = H = 32
    rng = np.random.default_rng(11)
    off, cnt = _segments(counts)
    rows = int(off[-1])
    h = _bf16(rng.standard_normal((rows, I)))
    w = rng.uniform(0.1, 1.0, rows).astype(np.float32)
    w2 = np.zeros((len(counts), H, I), np.uint16)
    for e in range(len(counts)):
        w2[e] = _bf16(np.eye(H, I) * (e + 1))
    y, y64 = oracle.w2_absorbed(h, w, w2, off, cnt)
    hs = _f32(_bf16(_f32(h) * w[:, None])).astype(np.float64)
    for e in range(len(counts)):
        lo, hi = off[e], off[e + 1]
        assert np.array_equal(y64[lo:hi], hs[lo:hi] * (e + 1))


def test_w2_power_of_two_scores_scale_exactly():
    h, w, w2, off, cnt = _problem([6, 5], I=48, H=8, unit=True)
    _, y1 = oracle.w2_absorbed(h, w, w2, off, cnt)
    _, y4 = oracle.w2_absorbed(h, w * 4.0, w2, off, cnt)
    assert np.array_equal(y4, 4.0 * y1)


def test_w2_pad_rows_and_row_subsets():
    h, w, w2, off, cnt = _problem([5, 1, 8], I=16, H=8, pad=4)
    y, y64 = oracle.w2_absorbed(h, w, w2, off, cnt)
    for e in range(len(cnt)):
        assert (y64[off[e] + cnt[e]:off[e + 1]] == 0).all()
        assert (y[off[e] + cnt[e]:off[e + 1]] == 0).all()
        assert (np.abs(y64[off[e]:off[e] + cnt[e]]).sum(axis=1) > 0).all()
    rows = np.array([off[2] + 3, 0, off[1]], np.int64)
    ys, ys64 = oracle.w2_absorbed(h, w, w2, off, cnt, rows=rows)
    assert np.array_equal(ys, y[rows]) and np.array_equal(ys64, y64[rows])


@pytest.mark.parametrize("planted", ["next_expert", "score_after_gemm"])
def test_w2_pins_catch_planted_mistakes(planted):
    """A wrong expert or a score applied after the GEMM (not to the bf16-rounded
    input) is caught by the matmul pin above."""
    h, w, w2, off, cnt = _problem([6, 7], I=64, H=16)
    _, y64 = oracle.w2_absorbed(h, w, w2, off, cnt)
    hs = _f32(_bf16(_f32(h) * w[:, None])).astype(np.float64)
    e = 0
    lo, hi = off[e], off[e] + cnt[e]
    if planted == "next_expert":
        wrong = hs[lo:hi] @ _f32(w2[e + 1]).astype(np.float64).T
    else:
        wrong = (_f32(h[lo:hi]).astype(np.float64) @ _f32(w2[e]).astype(np.float64).T) * w[lo:hi, None]
    assert not np.allclose(y64[lo:hi], wrong, rtol=1e-12, atol=1e-12)
