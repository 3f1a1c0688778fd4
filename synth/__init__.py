"""Seeded synthetic inputs for the MoE dispatch / combine workloads.

This module only draws random numbers and shapes them; it holds none of the
routing, layout or combine arithmetic.  Both the CUDA path's tests and the CPU
oracle receive the arrays it produces.

Recipe: numpy ``Generator(PCG64)`` streams spawned from ``SeedSequence(seed)``,
one child stream per tensor in the fixed order of ``STREAMS``; large tensors
are drawn in fixed chunks of ``CHUNK`` elements, each from its own grandchild
stream, so that a tensor is the same whatever the thread count.  Normals are
drawn in fp32; bf16 tensors are the round-to-nearest-even bf16 of those fp32
draws, returned as ``np.uint16`` bit patterns.

Workloads (one per MoE layer shape the pages discuss):
  0 tiny            T=256,   H=256,  E=8,   K=2, R=2,  fp32 rows, softmax
  1 qwen3_30b_a3b   T=8192,  H=2048, E=128, K=8, R=8,  bf16, softmax
  2 skewed          as 1, plus a per-expert logit bias 3.0*(e+1)^-1.2 and a
                    bias of -1e4 on the last expert (it receives no token)
  3 deepseek_v3     T=16384, H=7168, E=256, K=8, R=64, bf16, sigmoid scores in
                    8 groups, top-4 groups then top-8, correction bias N(0,0.01)
  4 qwen3_235b_abs  T=32768, H=4096, E=128, K=8, R=32, bf16, softmax, router
                    scores absorbed into the W2 input (I=1536): plain-sum combine
"""
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace
import os

import numpy as np

STREAMS = ("x", "logits", "bias", "y", "g", "h", "w2", "grecv", "ghs")
CHUNK = 1 << 22


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    K: int
    R: int
    dtype: str = "bf16"          # row dtype: "bf16" or "f32"
    score_fn: str = "softmax"    # "softmax" or "sigmoid"
    n_groups: int = 1
    topk_groups: int = 1
    group_score_topk: int = 1
    renorm: bool = True
    route_scale: float = 1.0
    bias: str = "none"           # "none" | "normal" (selection bias) | "zipf" (added to logits)
    bias_std: float = 0.0
    zipf_s: float = 1.2
    zipf_max: float = 3.0
    absorb: bool = False
    I: int = 0                   # W2 input width when scores are absorbed
    identity_experts: bool = False
    pad_align: int = 0           # receive segments rounded up to this many rows (0: packed)
    seed: int = 0
    extra: dict = field(default_factory=dict)

    def with_tokens(self, T):
        return replace(self, T=T)


WORKLOADS = {
    0: Workload("tiny", T=256, H=256, E=8, K=2, R=2, dtype="f32", identity_experts=True),
    1: Workload("qwen3_30b_a3b", T=8192, H=2048, E=128, K=8, R=8),
    2: Workload("qwen3_30b_a3b_skewed", T=8192, H=2048, E=128, K=8, R=8, bias="zipf"),
    3: Workload("deepseek_v3", T=16384, H=7168, E=256, K=8, R=64, score_fn="sigmoid", n_groups=8,
                topk_groups=4, group_score_topk=2, bias="normal", bias_std=0.01),
    4: Workload("qwen3_235b_absorbed", T=32768, H=4096, E=128, K=8, R=32, absorb=True, I=1536),
}


def _child(seed, name):
    """The SeedSequence of tensor stream `name` for base seed `seed`."""
    return np.random.SeedSequence(seed).spawn(len(STREAMS))[STREAMS.index(name)]


def _fill_chunks(seed, name, n, out, convert, threads):
    nchunks = (n + CHUNK - 1) // CHUNK
    seqs = _child(seed, name).spawn(nchunks)

    def fill(c):
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        a = np.random.Generator(np.random.PCG64(seqs[c])).standard_normal(hi - lo, dtype=np.float32)
        out[lo:hi] = convert(a)

    threads = threads or min(16, os.cpu_count() or 1)
    if nchunks <= 1 or threads == 1:
        for c in range(nchunks):
            fill(c)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(nchunks)))


def normal_f32(seed, name, shape, threads=None):
    """fp32 N(0,1) array of `shape` from stream `name`, drawn chunk by chunk."""
    n = int(np.prod(shape))
    out = np.empty(n, np.float32)
    _fill_chunks(seed, name, n, out, lambda a: a, threads)
    return out.reshape(shape)


def normal_bf16(seed, name, shape, threads=None):
    """bf16 bits of the same fp32 draws as normal_f32(seed, name, shape)."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    _fill_chunks(seed, name, n, out, to_bf16_bits, threads)
    return out.reshape(shape)


def to_bf16_bits(a):
    """Round fp32 -> bf16 to nearest even; returns np.uint16 bit patterns."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32)
    out = np.empty(u.shape, np.uint16)
    flat_u = u.reshape(-1)
    flat_o = out.reshape(-1)
    for lo in range(0, flat_u.size, CHUNK):
        v = flat_u[lo:lo + CHUNK]
        r = (v + np.uint32(0x7FFF) + ((v >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        nan = (v & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
        r = np.where(nan, (v >> np.uint32(16)) | np.uint32(0x40), r)
        flat_o[lo:lo + CHUNK] = r.astype(np.uint16)
    return out


def bf16_bits_to_f32(a):
    return (np.asarray(a, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def rows(wl, seed, name, nrows, width):
    """A [nrows, width] row tensor in the workload's row dtype (bf16 bits or fp32)."""
    if wl.dtype == "bf16":
        return normal_bf16(seed, name, (nrows, width))
    return normal_f32(seed, name, (nrows, width))


def router_logits(wl, seed=None):
    """Router logits [T,E] fp32 ~ N(0,1); workload 2 adds its Zipf profile."""
    seed = wl.seed if seed is None else seed
    logits = normal_f32(seed, "logits", (wl.T, wl.E))
    if wl.bias == "zipf":
        logits = logits + zipf_logit_bias(wl)[None, :]
    return np.ascontiguousarray(logits, np.float32)


def zipf_logit_bias(wl):
    """Per-expert logit bias zipf_max * (e+1)^-s (expert 0 heaviest), and -1e4 on
    the last expert so that it receives no token."""
    e = np.arange(wl.E, dtype=np.float64)
    b = (wl.zipf_max * (e + 1.0) ** (-wl.zipf_s)).astype(np.float32)
    b[wl.E - 1] = np.float32(-1.0e4)
    return b


def selection_bias(wl, seed=None):
    """Score-correction bias [E] fp32 ~ N(0, bias_std) (None if the workload has none)."""
    seed = wl.seed if seed is None else seed
    if wl.bias != "normal":
        return None
    return (normal_f32(seed, "bias", (wl.E,)) * np.float32(wl.bias_std)).astype(np.float32)


def make_inputs(wl, seed=None, want=("logits", "bias", "x", "y", "g")):
    """Dict of the requested host arrays for workload `wl`."""
    seed = wl.seed if seed is None else seed
    out = {}
    for k in want:
        if k == "logits":
            out[k] = router_logits(wl, seed)
        elif k == "bias":
            out[k] = selection_bias(wl, seed)
        elif k == "x":
            out[k] = rows(wl, seed, "x", wl.T, wl.H)
        elif k == "y":
            out[k] = rows(wl, seed, "y", wl.T * wl.K, wl.H)
        elif k == "g":
            out[k] = rows(wl, seed, "g", wl.T, wl.H)
        elif k == "grecv":
            out[k] = rows(wl, seed, "grecv", wl.T * wl.K, wl.H)
        elif k == "h":
            out[k] = normal_bf16(seed, "h", (wl.T * wl.K, wl.I))
        elif k == "ghs":
            out[k] = normal_bf16(seed, "ghs", (wl.T * wl.K, wl.I))
        elif k == "w2":
            out[k] = w2_weights(seed, wl.E, wl.H, wl.I)
        else:
            raise KeyError(k)
    return out


def w2_weights(seed, E, H, I):
    """Random W2 weights, bf16 bits [E, H, I] ~ N(0, 1/I): row n of expert e
    holds the I input weights of output n."""
    return to_bf16_bits(normal_f32(seed, "w2", (E, H, I)) * np.float32(1.0 / np.sqrt(I)))


def shard_seed(seed, rank):
    """Base seed of data-parallel replica `rank`: each replica draws its own batch."""
    return int(np.random.SeedSequence([seed, rank]).generate_state(1)[0])
