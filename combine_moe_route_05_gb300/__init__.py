"""Python binding of libmoeroute.so, the C-ABI MoE routing / dispatch / combine
library for one GB300 (sm_103a).

The functions named ``moe_*`` mirror the C entry points of
``include/moe_route.h`` one to one: they take torch CUDA tensors (PyTorch only
provides device memory and streams), check shapes and dtypes, and pass raw
pointers; every step of the computation runs in the library's CUDA kernels.
There is no fallback: if the library is missing or fails to load, the import
of :func:`lib` raises.

``MoeRouter`` is a convenience owner of a handle and its workspace with
methods that allocate their outputs.
"""
import ctypes
import os

import torch

from . import build as _build

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = _build.LIB

MOE_OK, MOE_ERR_INVALID, MOE_ERR_CAPACITY, MOE_ERR_CUDA, MOE_ERR_STATE = range(5)
MOE_BF16, MOE_F32 = 0, 1
MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID = 0, 1
MOE_DEVERR_BAD_EXPERT, MOE_DEVERR_DUP_EXPERT, MOE_DEVERR_NONFINITE, MOE_DEVERR_TIMEOUT = 1, 2, 4, 8
MOE_DEVERR_INTERNAL, MOE_DEVERR_BAD_LAYOUT = 16, 32
MOE_MAX_EXPERTS, MOE_MAX_TOPK = 512, 16

EXPORTS = ("moe_status_string", "moe_workspace_bytes", "moe_handle_create", "moe_handle_destroy",
           "moe_route_topk", "moe_dispatch_layout", "moe_layout_view", "moe_dispatch",
           "moe_combine", "moe_combine_bwd", "moe_dispatch_bwd", "moe_scale_rows",
           "moe_scale_rows_bwd", "moe_read_device_status", "moe_clear_device_status",
           "moe_dispatch_layout_static", "moe_route_bwd", "moe_expand", "moe_combine_partial",
           "moe_combine_reduce", "moe_w2_absorbed", "moe_dispatch_layout_launches",
           "moe_dispatch_bwd_route", "moe_dispatch_bwd_route_launches", "moe_set_wait_limit")
MOE_LAYOUT_STATIC_COUNTERS = 65536
MOE_LAYOUT_TILE_TOKENS = 512


class MoeConfig(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("num_ranks", ctypes.c_int32), ("score_fn", ctypes.c_int32),
                ("num_groups", ctypes.c_int32), ("topk_groups", ctypes.c_int32),
                ("group_score_topk", ctypes.c_int32), ("renorm", ctypes.c_int32),
                ("route_scale", ctypes.c_double), ("max_tokens", ctypes.c_int32),
                ("pad_align", ctypes.c_int32)]


class MoeLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "cnt_e", "off_e", "cnt_send_r", "off_send_r", "cnt_recv_r", "off_recv_r", "pos",
        "recv_token", "recv_k", "send_token", "send_row_of", "recv_send_row", "S")] + [
        ("num_tokens", ctypes.c_int32), ("pad_align", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s" % (fn, status_string(status)))


_lib = None


def lib():
    """The loaded CUDA library (raises if it is not built or cannot load)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmoeroute.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        st = ctypes.c_int
        sigs = {
            "moe_status_string": ([st], ctypes.c_char_p),
            "moe_workspace_bytes": ([P], sz),
            "moe_handle_create": ([P, P, sz, P], st),
            "moe_handle_destroy": ([P], st),
            "moe_route_topk": ([P, P, P, i32, P, P, P], st),
            "moe_dispatch_layout": ([P, P, i32, P], st),
            "moe_layout_view": ([P, P], st),
            "moe_dispatch": ([P, P, i32, i32, P, P, P, P, P], st),
            "moe_combine": ([P, P, i32, i32, P, P, P], st),
            "moe_combine_bwd": ([P, P, P, i32, i32, P, P, P, P], st),
            "moe_dispatch_bwd": ([P, P, i32, i32, P, P], st),
            "moe_scale_rows": ([P, P, i32, i32, P, P, P], st),
            "moe_scale_rows_bwd": ([P, P, P, i32, i32, P, P, P, P], st),
            "moe_read_device_status": ([P, P], st),
            "moe_clear_device_status": ([P, P], st),
            "moe_dispatch_layout_static": ([P, P, i32, P, P, P], st),
            "moe_route_bwd": ([P, P, P, P, i32, P, P], st),
            "moe_expand": ([P, P, i32, i32, P, P], st),
            "moe_combine_partial": ([P, P, i32, i32, P, P, P], st),
            "moe_combine_reduce": ([P, P, i32, i32, P, P], st),
            "moe_w2_absorbed": ([P, P, i32, P, P, i32, P, P], st),
            "moe_dispatch_layout_launches": ([P, i32, P], st),
            "moe_dispatch_bwd_route": ([P, P, i32, i32, P, P, P, P, P, P], st),
            "moe_dispatch_bwd_route_launches": ([P, P], st),
            "moe_set_wait_limit": ([P, ctypes.c_uint64], st),
        }
        for name, (args, res) in sigs.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def status_string(s):
    return lib().moe_status_string(s).decode()


def _check(fn, s):
    if s != MOE_OK:
        raise MoeError(fn, s)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream, device=None):
    """The raw handle of `stream`, else of the current stream of `device` (the
    handle's device; the current device when None)."""
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if device is not None and stream.device != device:
        raise ValueError("stream is on %s, the handle on %s" % (stream.device, device))
    return stream.cuda_stream


def _call(h, fn, *args):
    """Library function `fn` called with the handle's device current (the
    library refuses a call made while another device is current)."""
    f = getattr(lib(), fn)
    if torch.cuda.current_device() != h.device.index:
        with torch.cuda.device(h.device):
            _check(fn, f(*args))
    else:
        _check(fn, f(*args))


def _row_dtype(t):
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    if t.dtype == torch.float32:
        return MOE_F32
    raise TypeError("row tensors must be bfloat16 or float32, got %s" % t.dtype)


def _req(t, dtype=None, shape=None, name="tensor", device=None):
    if t is None:
        return
    if shape is not None and any(d < 0 for d in shape):
        shape = None  # no layout yet: the library itself reports MOE_ERR_STATE
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, the handle on %s" % (name, t.device, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def make_config(num_experts, top_k, num_ranks, max_tokens, score_fn="softmax", num_groups=1,
                topk_groups=1, group_score_topk=1, renorm=True, route_scale=1.0, pad_align=0):
    fn = {"softmax": MOE_SCORE_SOFTMAX, "sigmoid": MOE_SCORE_SIGMOID}[score_fn] \
        if isinstance(score_fn, str) else int(score_fn)
    return MoeConfig(num_experts, top_k, num_ranks, fn, num_groups, topk_groups, group_score_topk,
                     int(bool(renorm)), float(route_scale), max_tokens, int(pad_align))


def moe_workspace_bytes(cfg):
    return lib().moe_workspace_bytes(ctypes.byref(cfg))


class Handle:
    """A moe_handle plus the device workspace it lives in (owned here)."""

    def __init__(self, cfg, device=None):
        self.cfg = cfg
        nbytes = moe_workspace_bytes(cfg)
        if nbytes == 0:
            raise MoeError("moe_workspace_bytes", MOE_ERR_INVALID)
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        with torch.cuda.device(dev):
            # 256-byte aligned: the caching allocator returns 512-byte aligned blocks
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            torch.cuda.current_stream().synchronize()
            h = ctypes.c_void_p()
            _check("moe_handle_create",
                   lib().moe_handle_create(ctypes.byref(cfg), self.workspace.data_ptr(), nbytes,
                                           ctypes.byref(h)))
        self.ptr = h
        self.device = dev
        self.T = -1

    def close(self):
        if getattr(self, "ptr", None):
            lib().moe_handle_destroy(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def E(self):
        return self.cfg.num_experts

    @property
    def K(self):
        return self.cfg.top_k

    @property
    def R(self):
        return self.cfg.num_ranks

    @property
    def pad(self):
        return max(1, self.cfg.pad_align)

    @property
    def recv_rows(self):
        """Rows of a receive-row tensor for the current layout (-1 before the
        first layout, so that the library itself reports MOE_ERR_STATE)."""
        if self.T < 0:
            return -1
        return self.T * self.K + self.E * (self.pad - 1)


def moe_route_topk(h, logits, bias, idx, w, stream=None):
    T = logits.shape[0]
    d = h.device
    _req(logits, torch.float32, (T, h.E), "logits", d)
    _req(bias, torch.float32, (h.E,), "bias", d)
    _req(idx, torch.int32, (T, h.K), "idx", d)
    _req(w, torch.float32, (T, h.K), "w", d)
    _call(h, "moe_route_topk", h.ptr, _ptr(logits), _ptr(bias), T, _ptr(idx), _ptr(w),
          _stream(stream, d))


def moe_route_bwd(h, logits, idx, gw, glogits, stream=None):
    T = logits.shape[0]
    d = h.device
    _req(logits, torch.float32, (T, h.E), "logits", d)
    _req(idx, torch.int32, (T, h.K), "idx", d)
    _req(gw, torch.float32, (T, h.K), "gw", d)
    _req(glogits, torch.float32, (T, h.E), "glogits", d)
    _call(h, "moe_route_bwd", h.ptr, _ptr(logits), _ptr(idx), _ptr(gw), T, _ptr(glogits),
          _stream(stream, d))


def moe_dispatch_layout(h, idx, stream=None):
    T = idx.shape[0]
    _req(idx, torch.int32, (T, h.K), "idx", h.device)
    _call(h, "moe_dispatch_layout", h.ptr, _ptr(idx), T, _stream(stream, h.device))
    h.T = T


def moe_layout_view(h):
    v = MoeLayout()
    _check("moe_layout_view", lib().moe_layout_view(h.ptr, ctypes.byref(v)))
    return v


def moe_dispatch(h, x, w, recv, recv_w, send=None, stream=None):
    T, H = x.shape
    d = h.device
    _req(x, None, (h.T, H), "x", d)
    _req(recv, x.dtype, (h.recv_rows, H), "recv", d)
    _req(w, torch.float32, (h.T, h.K), "w", d)
    _req(recv_w, torch.float32, (h.recv_rows,), "recv_w", d)
    _req(send, x.dtype, (h.T * min(h.K, h.R), H), "send", d)
    _call(h, "moe_dispatch", h.ptr, _ptr(x), H, _row_dtype(x), _ptr(w), _ptr(recv),
          _ptr(recv_w), _ptr(send), _stream(stream, d))


def moe_combine(h, y, w, out, stream=None):
    H = y.shape[1]
    d = h.device
    _req(y, None, (h.recv_rows, H), "y", d)
    _req(w, torch.float32, (h.T, h.K), "w", d)
    _req(out, y.dtype, (h.T, H), "out", d)
    _call(h, "moe_combine", h.ptr, _ptr(y), H, _row_dtype(y), _ptr(w), _ptr(out),
          _stream(stream, d))


def moe_combine_bwd(h, g, y, w, gy, gw, stream=None):
    H = g.shape[1]
    d = h.device
    _req(g, None, (h.T, H), "g", d)
    _req(y, g.dtype, (h.recv_rows, H), "y", d)
    _req(w, torch.float32, (h.T, h.K), "w", d)
    _req(gy, g.dtype, (h.recv_rows, H), "gy", d)
    _req(gw, torch.float32, (h.T, h.K), "gw", d)
    _call(h, "moe_combine_bwd", h.ptr, _ptr(g), _ptr(y), H, _row_dtype(g), _ptr(w), _ptr(gy),
          _ptr(gw), _stream(stream, d))


def moe_dispatch_bwd(h, grecv, gx, stream=None):
    H = grecv.shape[1]
    d = h.device
    _req(grecv, None, (h.recv_rows, H), "grecv", d)
    _req(gx, grecv.dtype, (h.T, H), "gx", d)
    _call(h, "moe_dispatch_bwd", h.ptr, _ptr(grecv), H, _row_dtype(grecv), _ptr(gx),
          _stream(stream, d))


def moe_dispatch_bwd_route(h, grecv, logits, idx, gw, gx, glogits, stream=None):
    H = grecv.shape[1]
    d = h.device
    _req(grecv, None, (h.recv_rows, H), "grecv", d)
    _req(logits, torch.float32, (h.T, h.E), "logits", d)
    _req(idx, torch.int32, (h.T, h.K), "idx", d)
    _req(gw, torch.float32, (h.T, h.K), "gw", d)
    _req(gx, grecv.dtype, (h.T, H), "gx", d)
    _req(glogits, torch.float32, (h.T, h.E), "glogits", d)
    _call(h, "moe_dispatch_bwd_route", h.ptr, _ptr(grecv), H, _row_dtype(grecv), _ptr(logits),
          _ptr(idx), _ptr(gw), _ptr(gx), _ptr(glogits), _stream(stream, d))


def moe_dispatch_bwd_route_launches(h):
    """Kernel launches moe_dispatch_bwd_route makes for the handle's routing."""
    n = ctypes.c_int32(0)
    _check("moe_dispatch_bwd_route_launches",
           lib().moe_dispatch_bwd_route_launches(h.ptr, ctypes.byref(n)))
    return n.value


def moe_expand(h, send, recv, stream=None):
    H = send.shape[1]
    d = h.device
    _req(send, None, (h.T * min(h.K, h.R), H), "send", d)
    _req(recv, send.dtype, (h.recv_rows, H), "recv", d)
    _call(h, "moe_expand", h.ptr, _ptr(send), H, _row_dtype(send), _ptr(recv), _stream(stream, d))


def moe_combine_partial(h, y, w, partial, stream=None):
    H = y.shape[1]
    d = h.device
    _req(y, None, (h.recv_rows, H), "y", d)
    _req(w, torch.float32, (h.T, h.K), "w", d)
    _req(partial, y.dtype, (h.T * min(h.K, h.R), H), "partial", d)
    _call(h, "moe_combine_partial", h.ptr, _ptr(y), H, _row_dtype(y), _ptr(w), _ptr(partial),
          _stream(stream, d))


def moe_combine_reduce(h, partial, out, stream=None):
    H = partial.shape[1]
    d = h.device
    _req(partial, None, (h.T * min(h.K, h.R), H), "partial", d)
    _req(out, partial.dtype, (h.T, H), "out", d)
    _call(h, "moe_combine_reduce", h.ptr, _ptr(partial), H, _row_dtype(partial), _ptr(out),
          _stream(stream, d))


def moe_scale_rows(h, hrows, recv_w, hs, stream=None):
    I = hrows.shape[1]
    d = h.device
    _req(hrows, None, (h.recv_rows, I), "h", d)
    _req(recv_w, torch.float32, (h.recv_rows,), "recv_w", d)
    _req(hs, hrows.dtype, (h.recv_rows, I), "hs", d)
    _call(h, "moe_scale_rows", h.ptr, _ptr(hrows), I, _row_dtype(hrows), _ptr(recv_w), _ptr(hs),
          _stream(stream, d))


def moe_scale_rows_bwd(h, ghs, hrows, recv_w, gh, gw, stream=None):
    I = hrows.shape[1]
    d = h.device
    _req(ghs, None, (h.recv_rows, I), "ghs", d)
    _req(hrows, ghs.dtype, (h.recv_rows, I), "h", d)
    _req(recv_w, torch.float32, (h.recv_rows,), "recv_w", d)
    _req(gh, ghs.dtype, (h.recv_rows, I), "gh", d)
    _req(gw, torch.float32, (h.T, h.K), "gw", d)
    _call(h, "moe_scale_rows_bwd", h.ptr, _ptr(ghs), _ptr(hrows), I, _row_dtype(ghs),
          _ptr(recv_w), _ptr(gh), _ptr(gw), _stream(stream, d))


def moe_w2_absorbed(h, hrows, recv_w, w2, y, stream=None):
    """y = bf16(bf16(h * recv_w) @ W2[e].T) per expert segment (W2 [E, H, I])."""
    I = hrows.shape[1]
    H = w2.shape[1]
    d = h.device
    _req(hrows, torch.bfloat16, (h.recv_rows, I), "h", d)
    _req(recv_w, torch.float32, (h.recv_rows,), "recv_w", d)
    _req(w2, torch.bfloat16, (h.E, H, I), "w2", d)
    _req(y, torch.bfloat16, (h.recv_rows, H), "y", d)
    _call(h, "moe_w2_absorbed", h.ptr, _ptr(hrows), I, _ptr(recv_w), _ptr(w2), H, _ptr(y),
          _stream(stream, d))


def moe_dispatch_layout_launches(h, T):
    """Kernel launches moe_dispatch_layout makes for T tokens (1 or 2)."""
    n = ctypes.c_int32(0)
    _check("moe_dispatch_layout_launches",
           lib().moe_dispatch_layout_launches(h.ptr, T, ctypes.byref(n)))
    return n.value


def moe_read_device_status(h):
    flags = ctypes.c_uint32(0)
    _check("moe_read_device_status", lib().moe_read_device_status(h.ptr, ctypes.byref(flags)))
    return flags.value


def moe_clear_device_status(h, stream=None):
    _call(h, "moe_clear_device_status", h.ptr, _stream(stream, h.device))


def moe_set_wait_limit(h, limit_ns):
    """Limit of the kernels' bounded waits on this handle (0: the 1 s default)."""
    _check("moe_set_wait_limit", lib().moe_set_wait_limit(h.ptr, int(limit_ns)))


LAYOUT_FIELDS = ("cnt_e", "off_e", "cnt_send_r", "off_send_r", "cnt_recv_r", "off_recv_r", "pos",
                 "recv_token", "recv_k", "send_token", "send_row_of", "recv_send_row", "S")


def layout_sizes(T, K, E, R, pad=1):
    """Element counts (int32) of the layout arrays for T tokens."""
    RR = T * K + E * (max(1, pad) - 1)
    return {"cnt_e": E, "off_e": E + 1, "cnt_send_r": R, "off_send_r": R + 1, "cnt_recv_r": R,
            "off_recv_r": R + 1, "pos": T * K, "recv_token": RR, "recv_k": RR,
            "send_token": T * min(K, R), "send_row_of": T * K, "recv_send_row": RR, "S": 1}


def moe_dispatch_layout_static(cfg, idx, out, status=None, stream=None):
    """Allocation-free layout into caller-owned int32 tensors `out` (a dict
    keyed like LAYOUT_FIELDS, sized by layout_sizes); `status` an optional
    one-element int32 CUDA tensor that collects MOE_DEVERR_* bits.  Every
    tensor and the stream are on idx's device; the call runs there."""
    T = idx.shape[0]
    _req(idx, torch.int32, (T, cfg.top_k), "idx")
    d = idx.device
    sizes = layout_sizes(T, cfg.top_k, cfg.num_experts, cfg.num_ranks, cfg.pad_align)
    v = MoeLayout()
    for name in LAYOUT_FIELDS:
        t = out[name]
        _req(t, torch.int32, None, name, d)
        if t.numel() != sizes[name]:
            raise ValueError("%s must have %d elements, got %d" % (name, sizes[name], t.numel()))
        setattr(v, name, t.data_ptr() if t.numel() else None)
    v.num_tokens = T
    _req(status, torch.int32, (1,), "status", d)
    with torch.cuda.device(d):
        _check("moe_dispatch_layout_static",
               lib().moe_dispatch_layout_static(ctypes.byref(cfg), _ptr(idx), T, ctypes.byref(v),
                                                _ptr(status), _stream(stream, d)))


def layout_tensors(h):
    """Torch views (int32, on the handle's device) of the current layout arrays."""
    v = moe_layout_view(h)
    T, K, E, R = h.T, h.K, h.E, h.R
    sizes = layout_sizes(T, K, E, R, h.pad)
    out = {}
    ws = h.workspace
    base = ws.data_ptr()
    for name, n in sizes.items():
        off = getattr(v, name) - base
        out[name] = ws[off:off + 4 * n].view(torch.int32)
    out["pos"] = out["pos"].view(T, K)
    out["send_row_of"] = out["send_row_of"].view(T, K)
    return out


class MoeRouter:
    """Owns a handle; methods allocate their outputs and call the moe_* bindings."""

    def __init__(self, num_experts, top_k, num_ranks, max_tokens, **kw):
        self.cfg = make_config(num_experts, top_k, num_ranks, max_tokens, **kw)
        self.h = Handle(self.cfg)

    def route(self, logits, bias=None, stream=None):
        T = logits.shape[0]
        idx = torch.empty(T, self.h.K, dtype=torch.int32, device=logits.device)
        w = torch.empty(T, self.h.K, dtype=torch.float32, device=logits.device)
        moe_route_topk(self.h, logits, bias, idx, w, stream)
        return idx, w

    def route_bwd(self, logits, idx, gw, stream=None):
        glogits = torch.empty_like(logits)
        moe_route_bwd(self.h, logits, idx, gw, glogits, stream)
        return glogits

    def layout(self, idx, stream=None):
        moe_dispatch_layout(self.h, idx, stream)
        return layout_tensors(self.h)

    def dispatch(self, x, w=None, with_send=False, stream=None):
        T, H = x.shape
        rr = max(self.h.recv_rows, 0)
        recv = torch.empty(rr, H, dtype=x.dtype, device=x.device)
        recv_w = torch.empty(rr, dtype=torch.float32, device=x.device) if w is not None else None
        send = torch.empty(T * min(self.h.K, self.h.R), H, dtype=x.dtype, device=x.device) if with_send else None
        moe_dispatch(self.h, x, w, recv, recv_w, send, stream)
        return recv, recv_w, send

    def combine(self, y, w=None, stream=None):
        out = torch.empty(max(self.h.T, 0), y.shape[1], dtype=y.dtype, device=y.device)
        moe_combine(self.h, y, w, out, stream)
        return out

    def combine_bwd(self, g, y=None, w=None, stream=None):
        gy = torch.empty(max(self.h.recv_rows, 0), g.shape[1], dtype=g.dtype, device=g.device)
        gw = torch.empty(max(self.h.T, 0), self.h.K, dtype=torch.float32, device=g.device) if w is not None else None
        moe_combine_bwd(self.h, g, y, w, gy, gw, stream)
        return gy, gw

    def dispatch_bwd(self, grecv, stream=None):
        gx = torch.empty(max(self.h.T, 0), grecv.shape[1], dtype=grecv.dtype, device=grecv.device)
        moe_dispatch_bwd(self.h, grecv, gx, stream)
        return gx

    def dispatch_bwd_route(self, grecv, logits, idx, gw, stream=None):
        """Dispatch backward and router backward to the logits in one call:
        (gx, glogits)."""
        gx = torch.empty(max(self.h.T, 0), grecv.shape[1], dtype=grecv.dtype, device=grecv.device)
        glogits = torch.empty(max(self.h.T, 0), self.h.E, dtype=torch.float32, device=grecv.device)
        moe_dispatch_bwd_route(self.h, grecv, logits, idx, gw, gx, glogits, stream)
        return gx, glogits

    def expand(self, send, stream=None):
        recv = torch.empty(max(self.h.recv_rows, 0), send.shape[1], dtype=send.dtype,
                           device=send.device)
        moe_expand(self.h, send, recv, stream)
        return recv

    def combine_partial(self, y, w=None, stream=None):
        partial = torch.empty(max(self.h.T, 0) * min(self.h.K, self.h.R), y.shape[1],
                              dtype=y.dtype, device=y.device)
        moe_combine_partial(self.h, y, w, partial, stream)
        return partial

    def combine_reduce(self, partial, stream=None):
        out = torch.empty(max(self.h.T, 0), partial.shape[1], dtype=partial.dtype,
                          device=partial.device)
        moe_combine_reduce(self.h, partial, out, stream)
        return out

    def scale_rows(self, hrows, recv_w, stream=None):
        hs = torch.empty_like(hrows)
        moe_scale_rows(self.h, hrows, recv_w, hs, stream)
        return hs

    def w2_absorbed(self, hrows, recv_w, w2, stream=None):
        y = torch.empty(hrows.shape[0], w2.shape[1], dtype=torch.bfloat16, device=hrows.device)
        moe_w2_absorbed(self.h, hrows, recv_w, w2, y, stream)
        return y

    def scale_rows_bwd(self, ghs, hrows, recv_w, stream=None):
        gh = torch.empty_like(hrows)
        gw = torch.empty(max(self.h.T, 0), self.h.K, dtype=torch.float32, device=hrows.device)
        moe_scale_rows_bwd(self.h, ghs, hrows, recv_w, gh, gw, stream)
        return gh, gw
