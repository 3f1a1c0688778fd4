"""CPU oracle for the MoE token dispatch / combine path -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product library never loads it, and it never loads
the product library: the two share no code.

Each wrapper below marshals numpy arrays into the plain C++ definitions in
``oracle.cpp`` (which cite the passages they follow) and returns numpy arrays.
bf16 tensors travel as ``np.uint16`` bit patterns.
"""
import ctypes
import numpy as np

from . import build as _build

BF16 = 0
F32 = 1

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        i32 = ctypes.c_int
        d = ctypes.c_double
        L.orc_route_softmax.argtypes = [P, i64, i32, i32, i32, d, P, P]
        L.orc_route_softmax.restype = i32
        L.orc_route_sigmoid_grouped.argtypes = [P, P, i64, i32, i32, i32, i32, i32, i32, d, P, P]
        L.orc_route_sigmoid_grouped.restype = i32
        L.orc_layout.argtypes = [P, i64, i32, i32, i32, i32] + [P] * 12 + [P]
        L.orc_layout.restype = i64
        L.orc_dispatch.argtypes = [P, i64, i64, i32, P, P, P, P, P, P]
        L.orc_dispatch.restype = None
        L.orc_combine.argtypes = [P, i32, i64, i64, i32, P, P, P]
        L.orc_combine.restype = None
        L.orc_combine_bwd.argtypes = [P, P, i32, i64, i64, i32, P, P, P, P]
        L.orc_combine_bwd.restype = None
        L.orc_dispatch_bwd.argtypes = [P, i32, i64, i64, i32, P, P]
        L.orc_dispatch_bwd.restype = None
        L.orc_scale_rows.argtypes = [P, i32, i64, i64, P, P]
        L.orc_scale_rows.restype = None
        L.orc_scale_rows_bwd.argtypes = [P, P, i32, i64, i64, i64, i32, P, P, P, P]
        L.orc_scale_rows_bwd.restype = None
        L.orc_combine_f64.argtypes = [P, i64, i64, i32, P, P, P]
        L.orc_combine_f64.restype = None
        L.orc_dispatch_f64.argtypes = [P, i64, i64, i32, P, P]
        L.orc_dispatch_f64.restype = None
        L.orc_route_bwd.argtypes = [P, i64, i32, i32, i32, i32, d, P, P, P]
        L.orc_route_bwd.restype = i32
        L.orc_expand.argtypes = [P, i64, i64, i32, P, P, P]
        L.orc_expand.restype = None
        L.orc_combine_partial.argtypes = [P, i32, i64, i64, i32, P, P, P, P]
        L.orc_combine_partial.restype = None
        L.orc_combine_reduce.argtypes = [P, i32, i64, i64, i32, P, P]
        L.orc_combine_reduce.restype = None
        L.orc_f32_to_bf16.argtypes = [P, i64, P]
        L.orc_f32_to_bf16.restype = None
        L.orc_w2_absorbed.argtypes = [P, i64, P, P, i64, i32, P, P, P, i64, P, P]
        L.orc_w2_absorbed.restype = None
        L.orc_f64_to_bf16.argtypes = [P, i64, P]
        L.orc_f64_to_bf16.restype = None
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _dtype_of(a):
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    raise TypeError("rows must be np.uint16 (bf16 bits) or np.float32, got %s" % a.dtype)


def route_softmax(logits, K, renorm=True, route_scale=1.0):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    rc = lib().orc_route_softmax(_p(logits), T, E, K, int(renorm), float(route_scale), _p(idx), _p(w))
    if rc != 0:
        raise ValueError("orc_route_softmax: invalid sizes")
    return idx, w


def route_sigmoid_grouped(logits, bias, K, n_groups, topk_groups, group_score_topk=2,
                          renorm=True, route_scale=1.0):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    bias = None if bias is None else _c(bias, np.float32)
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    rc = lib().orc_route_sigmoid_grouped(_p(logits), _p(bias), T, E, K, n_groups, topk_groups,
                                         group_score_topk, int(renorm), float(route_scale),
                                         _p(idx), _p(w))
    if rc != 0:
        raise ValueError("orc_route_sigmoid_grouped: invalid sizes")
    return idx, w


def route_bwd(logits, idx, gw, score_fn="softmax", renorm=True, route_scale=1.0):
    """dL/dlogits [T,E] fp64 of the routing weights, selection held fixed."""
    logits = _c(logits, np.float32)
    idx = _c(idx, np.int32)
    gw = _c(gw, np.float64)
    T, E = logits.shape
    K = idx.shape[1]
    out = np.empty((T, E), np.float64)
    fn = {"softmax": 0, "sigmoid": 1}[score_fn]
    rc = lib().orc_route_bwd(_p(logits), T, E, K, fn, int(renorm), float(route_scale), _p(idx),
                             _p(gw), _p(out))
    if rc != 0:
        raise ValueError("orc_route_bwd: invalid sizes")
    return out


class Layout:
    """Outputs of the dispatch layout, as numpy int32 arrays."""

    def __init__(self, T, K, E, R, align=1):
        self.T, self.K, self.E, self.R, self.align = T, K, E, R, align
        self.recv_rows = T * K + E * (align - 1)
        self.cnt_e = np.empty(E, np.int32)
        self.off_e = np.empty(E + 1, np.int32)
        self.cnt_send_r = np.empty(R, np.int32)
        self.off_send_r = np.empty(R + 1, np.int32)
        self.cnt_recv_r = np.empty(R, np.int32)
        self.off_recv_r = np.empty(R + 1, np.int32)
        self.pos = np.empty((T, K), np.int32)
        self.recv_token = np.empty(self.recv_rows, np.int32)
        self.recv_k = np.empty(self.recv_rows, np.int32)
        self.send_token = np.empty(T * min(K, R), np.int32)
        self.send_row_of = np.empty((T, K), np.int32)
        self.recv_send_row = np.empty(self.recv_rows, np.int32)
        self.S = 0
        self.dropped = 0

    FIELDS = ("cnt_e", "off_e", "cnt_send_r", "off_send_r", "cnt_recv_r", "off_recv_r", "pos",
              "recv_token", "recv_k", "send_token", "send_row_of", "recv_send_row")


def layout(idx, E, R, align=1):
    idx = _c(idx, np.int32)
    T, K = idx.shape
    L = Layout(T, K, E, R, align)
    S = ctypes.c_int64(0)
    dropped = lib().orc_layout(_p(idx), T, K, E, R, align,
                               *[_p(getattr(L, f)) for f in Layout.FIELDS], ctypes.addressof(S))
    if dropped < 0:
        raise ValueError("orc_layout: invalid sizes")
    L.S = int(S.value)
    L.dropped = int(dropped)
    return L


def dispatch(x, lay, w=None, with_send=False):
    x = np.ascontiguousarray(x)
    T, H = x.shape
    K = lay.K
    recv = np.zeros((lay.recv_rows, H), x.dtype)
    recv_w = np.zeros(lay.recv_rows, np.float32) if w is not None else None
    send = np.zeros((T * min(K, lay.R), H), x.dtype) if with_send else None
    wc = None if w is None else _c(w, np.float32)
    lib().orc_dispatch(_p(x), H * x.itemsize, T, K, _p(lay.pos), _p(wc), _p(lay.send_row_of),
                       _p(recv), _p(recv_w), _p(send))
    return recv, recv_w, send


def combine(y, lay, w=None):
    y = np.ascontiguousarray(y)
    H = y.shape[1]
    out = np.empty((lay.T, H), y.dtype)
    wc = None if w is None else _c(w, np.float32)
    lib().orc_combine(_p(y), _dtype_of(y), H, lay.T, lay.K, _p(lay.pos), _p(wc), _p(out))
    return out


def combine_bwd(g, y, lay, w=None):
    g = np.ascontiguousarray(g)
    y = np.ascontiguousarray(y)
    assert g.dtype == y.dtype
    H = g.shape[1]
    gy = np.zeros((getattr(lay, "recv_rows", lay.T * lay.K), H), g.dtype)
    wc = None if w is None else _c(w, np.float32)
    gw = np.zeros((lay.T, lay.K), np.float64) if w is not None else None
    lib().orc_combine_bwd(_p(g), _p(y), _dtype_of(g), H, lay.T, lay.K, _p(lay.pos), _p(wc), _p(gy),
                          _p(gw))
    return gy, gw


def dispatch_bwd(grecv, lay):
    grecv = np.ascontiguousarray(grecv)
    H = grecv.shape[1]
    gx = np.empty((lay.T, H), grecv.dtype)
    lib().orc_dispatch_bwd(_p(grecv), _dtype_of(grecv), H, lay.T, lay.K, _p(lay.pos), _p(gx))
    return gx


def expand(send, lay):
    """recv[pos[t,k]] = send[send_row_of[t,k]] (rows of dropped entries stay 0)."""
    send = np.ascontiguousarray(send)
    H = send.shape[1]
    recv = np.zeros((getattr(lay, "recv_rows", lay.T * lay.K), H), send.dtype)
    lib().orc_expand(_p(send), H * send.itemsize, lay.T, lay.K, _p(lay.pos), _p(lay.send_row_of),
                     _p(recv))
    return recv


def combine_partial(y, lay, w=None):
    """Stage-1 partial rows [T*min(K,R), H] (rows past S stay 0)."""
    y = np.ascontiguousarray(y)
    H = y.shape[1]
    partial = np.zeros((lay.T * min(lay.K, lay.R), H), y.dtype)
    wc = None if w is None else _c(w, np.float32)
    lib().orc_combine_partial(_p(y), _dtype_of(y), H, lay.T, lay.K, _p(lay.pos),
                              _p(lay.send_row_of), _p(wc), _p(partial))
    return partial


def combine_reduce(partial, lay):
    partial = np.ascontiguousarray(partial)
    H = partial.shape[1]
    out = np.empty((lay.T, H), partial.dtype)
    lib().orc_combine_reduce(_p(partial), _dtype_of(partial), H, lay.T, lay.K,
                             _p(lay.send_row_of), _p(out))
    return out


def scale_rows(h, recv_w, rows=None):
    h = np.ascontiguousarray(h)
    R_, I = h.shape
    rows = R_ if rows is None else rows
    hs = np.zeros_like(h)
    rw = _c(recv_w, np.float32)
    lib().orc_scale_rows(_p(h), _dtype_of(h), I, rows, _p(rw), _p(hs))
    return hs


def w2_absorbed(h, recv_w, w2, off_e, cnt_e, rows=None):
    """Absorbed W2 projection of the listed receive rows (all rows if None):
    returns (y as bf16 bits [n, H], its fp64 value before rounding [n, H]).
    h is bf16 bits [rows, I]; w2 is bf16 bits [E, H, I]."""
    h = _c(h, np.uint16)
    w2 = _c(w2, np.uint16)
    E, H, I = w2.shape
    assert h.shape[1] == I
    off_e = _c(off_e, np.int32)
    cnt_e = _c(cnt_e, np.int32)
    assert off_e.shape == (E + 1,) and cnt_e.shape == (E,)
    rows = np.arange(h.shape[0], dtype=np.int64) if rows is None else _c(rows, np.int64)
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < h.shape[0])
    rw = _c(recv_w, np.float32)
    y = np.zeros((rows.size, H), np.uint16)
    y64 = np.zeros((rows.size, H), np.float64)
    lib().orc_w2_absorbed(_p(h), I, _p(rw), _p(w2), H, E, _p(off_e), _p(cnt_e), _p(rows),
                          rows.size, _p(y), _p(y64))
    return y, y64


def f64_to_bf16(a):
    """Round-to-nearest-even of fp64 values to bf16 bits, rounding once."""
    a = _c(a, np.float64)
    out = np.zeros(a.shape, np.uint16)
    lib().orc_f64_to_bf16(_p(a), a.size, _p(out))
    return out


def scale_rows_bwd(ghs, h, recv_w, lay, rows=None):
    ghs = np.ascontiguousarray(ghs)
    h = np.ascontiguousarray(h)
    R_, I = h.shape
    rows = R_ if rows is None else rows
    gh = np.zeros_like(h)
    gw = np.zeros((lay.T, lay.K), np.float64)
    rw = _c(recv_w, np.float32)
    lib().orc_scale_rows_bwd(_p(ghs), _p(h), _dtype_of(h), I, rows, lay.T, lay.K, _p(lay.pos),
                             _p(rw), _p(gh), _p(gw))
    return gh, gw


def combine_f64(y, lay, w=None):
    y = _c(y, np.float64)
    H = y.shape[1]
    out = np.empty((lay.T, H), np.float64)
    wc = None if w is None else _c(w, np.float64)
    lib().orc_combine_f64(_p(y), H, lay.T, lay.K, _p(lay.pos), _p(wc), _p(out))
    return out


def dispatch_f64(x, lay):
    x = _c(x, np.float64)
    H = x.shape[1]
    recv = np.zeros((getattr(lay, "recv_rows", lay.T * lay.K), H), np.float64)
    lib().orc_dispatch_f64(_p(x), H, lay.T, lay.K, _p(lay.pos), _p(recv))
    return recv


def f32_to_bf16(a):
    a = _c(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    lib().orc_f32_to_bf16(_p(a), a.size, _p(out))
    return out


def bf16_to_f32(a):
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32)
