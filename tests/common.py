"""Comparison helpers shared by the tests (no method arithmetic here)."""
import numpy as np


def ordered_bf16(bits):
    """Map bf16 bit patterns to integers ordered like their values (+0 == -0)."""
    b = np.asarray(bits, np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ordered_f32(a):
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.int64)
    mag = u & 0x7FFFFFFF
    return np.where(u & 0x80000000, -mag, mag)


def ulp_dist(a, b):
    """Element-wise distance in units in the last place (bf16 bits or fp32)."""
    a = np.asarray(a)
    b = np.asarray(b)
    assert a.dtype == b.dtype and a.shape == b.shape, (a.dtype, b.dtype, a.shape, b.shape)
    if a.dtype == np.uint16:
        return np.abs(ordered_bf16(a) - ordered_bf16(b))
    if a.dtype == np.float32:
        return np.abs(ordered_f32(a) - ordered_f32(b))
    raise TypeError(a.dtype)


def assert_ulp(a, b, max_ulp=1, what=""):
    d = ulp_dist(a, b)
    worst = int(d.max()) if d.size else 0
    assert worst <= max_ulp, "%s: max ulp distance %d > %d (%d elements differ)" % (
        what, worst, max_ulp, int((d > 0).sum()))
    return d


def gw_tolerance_ok(gw, gw_ref, g_norm, y_norm, rel=1e-3, floor=1e-6):
    """Router-score gradient acceptance: |gw - ref| <= rel*|ref| + floor*|g_t|*|y_row|.
    The second term covers near-zero dot products, where a relative bound alone
    is undefined."""
    gw = np.asarray(gw, np.float64)
    gw_ref = np.asarray(gw_ref, np.float64)
    bound = rel * np.abs(gw_ref) + floor * np.asarray(g_norm) * np.asarray(y_norm)
    return np.abs(gw - gw_ref) <= bound


def entry_row_norms(rows_f32, pos):
    """|rows[pos[t,k]]| per entry (0 for a dropped entry)."""
    n = np.linalg.norm(rows_f32.astype(np.float64), axis=1)
    return np.where(pos >= 0, n[np.clip(pos, 0, None)], 0.0)


def row_norms_for_gw(g_f32, y_f32, pos):
    """|g_t| broadcast over k and |y[pos[t,k]]|, for the gw tolerance floor."""
    gn = np.linalg.norm(g_f32.astype(np.float64), axis=1)[:, None] * np.ones(pos.shape)
    return gn, entry_row_norms(y_f32, pos)
