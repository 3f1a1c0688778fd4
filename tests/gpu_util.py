"""Helpers shared by the GPU parity tests: host <-> device marshalling, the
oracle's routing for a workload, and token-sampled oracle sub-problems."""
import numpy as np
import torch

import combine_moe_route_05_gb300 as moe
import oracle


def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda", 0)


def to_dev(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev()).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev())


def to_host(t):
    if t is None:
        return None
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def router(wl, max_tokens=None):
    return moe.MoeRouter(wl.E, wl.K, wl.R, wl.T if max_tokens is None else max_tokens,
                         score_fn=wl.score_fn, num_groups=wl.n_groups, topk_groups=wl.topk_groups,
                         group_score_topk=wl.group_score_topk, renorm=wl.renorm,
                         route_scale=wl.route_scale, pad_align=wl.pad_align)


def oracle_route(wl, logits, bias):
    if wl.score_fn == "softmax":
        return oracle.route_softmax(logits, wl.K, wl.renorm, wl.route_scale)
    return oracle.route_sigmoid_grouped(logits, bias, wl.K, wl.n_groups, wl.topk_groups,
                                        wl.group_score_topk, wl.renorm, wl.route_scale)


class SubLayout:
    """An oracle layout restricted to some tokens: their entries are renumbered
    0..n*K-1 in token-then-k order, and `rows` holds the global receive row of
    each renumbered entry (-1 for a dropped entry), so oracle row operations
    run on gathered copies of just those rows."""

    def __init__(self, L, tokens):
        self.T = len(tokens)
        self.K = L.K
        self.R = L.R
        self.recv_rows = self.T * self.K
        self.rows = L.pos[tokens].reshape(-1)
        local = np.arange(self.T * self.K, dtype=np.int32)
        self.pos = np.where(self.rows >= 0, local, -1).astype(np.int32).reshape(self.T, self.K)
        self.send_row_of = np.full((self.T, self.K), -1, np.int32)

    def gather(self, rows_array):
        out = np.zeros((self.T * self.K,) + rows_array.shape[1:], rows_array.dtype)
        ok = self.rows >= 0
        out[ok] = rows_array[self.rows[ok]]
        return out


def layout_host(r):
    return {k: to_host(v) for k, v in moe.layout_tensors(r.h).items()}
