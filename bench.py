"""Benchmark of the MoE routing / dispatch / combine path on GB300.

One step = one pass of the whole path over one batch of synthetic input on one
GPU: route_topk -> dispatch_layout -> dispatch -> combine -> combine_bwd ->
dispatch_bwd (the expert GEMMs between them are out of scope: the expert output
y is a synthetic input and the expert backward is the identity, grecv = gy).

Workload (default): DeepSeek-V3-shaped layer, T=16384, H=7168, E=256 sigmoid
experts in 8 groups (top-4 groups, top-8 experts, correction bias), 64 virtual
ranks, bf16 rows.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

The timed region replays the step captured as one CUDA graph (the same
kernels and work, without per-launch host overhead; --eager times eager
calls); per-stage times come from a second, eager pass with CUDA events
between the calls.  Under torchrun (N > 1) every rank runs an independent
data-parallel replica on its own batch (the path shards by token; there is
no exchange), and the step time is the max over ranks.  Prints one JSON line
on rank 0.
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "dispatch+combine fwd+bwd tokens/s and achieved HBM GB/s (% of GB300 peak)"
UNIT = "tokens/s"
DOMINANT = "combine_bwd"
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e data-sheet bandwidth, for context beside the measured peak
KERNEL_SOURCES = ("combine_moe_route_05_gb300/csrc/rows.cu", "combine_moe_route_05_gb300/csrc/common.cuh",
                  "combine_moe_route_05_gb300/csrc/router_grad.cuh")
W2_SOURCES = ("combine_moe_route_05_gb300/csrc/w2_gemm.cu", "combine_moe_route_05_gb300/csrc/common.cuh")
# per-launch DRAM traffic of the roofline kernels, from one ncu pass each
TRAFFIC_RECORDS = os.path.join(ROOT, "profiles", "traffic.json")
L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2


# ----------------------------------------------------------------------------
# byte accounting (algorithmic: every tensor read once and written once)


def step_bytes(wl):
    """Algorithmic HBM bytes of each stage of one step.  With absorbed scores
    the combine is a plain sum, its backward copies g (no score gradient
    there), and scale_rows / scale_rows_bwd apply the scores to the W2 input
    rows (I wide) and produce the score gradient."""
    T, H, E, K, R = wl.T, wl.H, wl.E, wl.K, wl.R
    eb = 2 if wl.dtype == "bf16" else 4
    row, tk = H * eb, T * K
    b = {
        "route_topk": T * E * 4 + (E * 4 if wl.bias == "normal" else 0) + tk * 8,
        "dispatch_layout": tk * 4 + 6 * tk * 4 + T * min(K, R) * 4,
        "dispatch": T * row + tk * row + tk * 4 * 3,
    }
    if wl.absorb:
        irow = wl.I * eb
        b["scale_rows"] = 2 * tk * irow + tk * 4
        b["combine"] = tk * row + T * row + tk * 4
        b["combine_bwd"] = T * row + tk * row + tk * 4
        b["scale_rows_bwd"] = 3 * tk * irow + tk * 4 + tk * 8
    else:
        b["combine"] = tk * row + T * row + tk * 8
        b["combine_bwd"] = T * row + 2 * tk * row + tk * 12
    b["dispatch_bwd"] = tk * row + T * row + tk * 4
    return b


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def read_bf16_peak():
    """Dense bf16 tensor peak in TFLOP/s: the burst figure (the W2 GEMM is
    timed on its own, not inside a long step)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured (burst)"
    return 1900.0, "fallback"


def w2_absorbed_extra(device, stream, reps, tokens=None):
    """Router scores absorbed into the W2 input, fused into the W2 grouped GEMM
    (tensor cores), on the Qwen3-235B-shaped layer (T=32768, K=8, E=128,
    I=1536, H=4096), against the unfused path: scale_rows, then cuBLAS per
    expert.  Inputs: N(0,1) logits and h, W2 ~ N(0, 1/I), seeded on device."""
    import torch
    import combine_moe_route_05_gb300 as moe
    wl = synth.WORKLOADS[4]
    T = tokens or wl.T
    E, K, R, I, H = wl.E, wl.K, wl.R, wl.I, 4096
    g = torch.Generator(device=device).manual_seed(wl.seed)
    r = moe.MoeRouter(E, K, R, T)
    idx, w = r.route(torch.randn(T, E, device=device, generator=g))
    r.layout(idx)
    rows = r.h.recv_rows
    hrows = torch.randn(rows, I, device=device, generator=g).to(torch.bfloat16)
    w2 = (torch.randn(E, H, I, device=device, generator=g) * (1.0 / I ** 0.5)).to(torch.bfloat16)
    _, recv_w, _ = r.dispatch(torch.zeros(T, 8, dtype=torch.bfloat16, device=device), w)
    y = torch.empty(rows, H, dtype=torch.bfloat16, device=device)
    hs = torch.empty_like(hrows)
    y_ref = torch.empty_like(y)
    cnt = moe.layout_tensors(r.h)["cnt_e"].tolist()

    def unfused():
        moe.moe_scale_rows(r.h, hrows, recv_w, hs)
        o = 0
        for e in range(E):
            if cnt[e]:
                torch.matmul(hs[o:o + cnt[e]], w2[e].t(), out=y_ref[o:o + cnt[e]])
            o += cnt[e]

    def timed(fn):
        for _ in range(3):
            fn()
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        for _ in range(reps):
            fn()
        b_.record(stream)
        torch.cuda.synchronize()
        return a_.elapsed_time(b_) / reps

    t_fused = timed(lambda: moe.moe_w2_absorbed(r.h, hrows, recv_w, w2, y))
    t_unfused = timed(unfused)
    # the absorption row on its own: scale_rows forward and backward
    ghs = torch.randn(rows, I, device=device, generator=g).to(torch.bfloat16)
    gh = torch.empty_like(hrows)
    gws = torch.empty(T, K, dtype=torch.float32, device=device)
    t_sr = timed(lambda: moe.moe_scale_rows(r.h, hrows, recv_w, hs))
    t_srb = timed(lambda: moe.moe_scale_rows_bwd(r.h, ghs, hrows, recv_w, gh, gws))
    assert moe.moe_read_device_status(r.h) == 0
    hbm_peak, hbm_src = read_peaks()
    sr_bytes = rows * I * 2 * 2 + rows * 4
    srb_bytes = rows * I * 2 * 3 + rows * 4 + T * K * 8
    same = bool(torch.equal(y, y_ref))
    flop = 2.0 * T * K * H * I
    peak, src = read_bf16_peak()
    achieved = flop / (t_fused / 1e3) / 1e12
    return {
        "workload": "qwen3_235b_absorbed T=%d K=%d E=%d I=%d H=%d (W2 [E,H,I] bf16)" % (T, K, E, I, H),
        "fused_ms": t_fused, "unfused_ms": t_unfused, "scale_rows_plus_cublas_per_expert_ms": t_unfused,
        "bitwise_equal_to_unfused": same,
        "roofline": {"kernel": "w2_absorbed", "bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak,
                     "traffic": (measured_traffic_per_launch("w2_absorbed", wl.name, W2_SOURCES)
                                 if T == wl.T else None),
                     "algorithmic_flops": flop,
                     "algorithmic_bytes": rows * I * 2 + E * H * I * 2 + rows * H * 2 + rows * 4,
                     "peak_source": src},
        "kernel_source": kernel_source_hash(W2_SOURCES),
        "scale_rows": {"rows": rows, "I": I, "ms": t_sr, "gbs": sr_bytes / (t_sr / 1e3) / 1e9,
                       "frac_of_hbm_peak": sr_bytes / (t_sr / 1e3) / 1e9 / hbm_peak},
        "scale_rows_bwd": {"ms": t_srb, "gbs": srb_bytes / (t_srb / 1e3) / 1e9,
                           "frac_of_hbm_peak": srb_bytes / (t_srb / 1e3) / 1e9 / hbm_peak},
    }


def kernel_source_hash(sources=KERNEL_SOURCES):
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic_per_launch(kernel, workload_name, sources=KERNEL_SOURCES):
    """DRAM bytes (read + write) per launch of `kernel` on the named workload,
    from its ncu record, if that was taken on the current kernel source."""
    if not os.path.exists(TRAFFIC_RECORDS):
        return None
    with open(TRAFFIC_RECORDS) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("workload") != workload_name or rec.get("source") != kernel_source_hash(sources):
        return None
    return float(rec["traffic_bytes_per_launch"])


# ----------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only: a barrier and a max of the step time)


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def replica_seed(base_seed, rank, world):
    return base_seed if world == 1 else synth.shard_seed(base_seed, rank)


def reduce_max(value, world, device=None):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def relaunch_under_torchrun(nproc):
    """`--gpus N` (N > 1) started as a plain process: run this same command as
    N ranks, one process per GPU, under torch.distributed.run on this node,
    and return its exit code."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           "--nproc-per-node", str(nproc), "--master-addr", "127.0.0.1",
           "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------
# CPU oracle leg (rank 0 only)


def oracle_chain(wl, inp):
    import oracle
    if wl.score_fn == "softmax":
        idx, w = oracle.route_softmax(inp["logits"], wl.K, wl.renorm, wl.route_scale)
    else:
        idx, w = oracle.route_sigmoid_grouped(inp["logits"], inp["bias"], wl.K, wl.n_groups,
                                              wl.topk_groups, wl.group_score_topk, wl.renorm,
                                              wl.route_scale)
    L = oracle.layout(idx, wl.E, wl.R)
    _, recv_w, _ = oracle.dispatch(inp["x"], L, w)
    if wl.absorb:
        oracle.scale_rows(inp["h"], recv_w)
        oracle.combine(inp["y"], L)
        gy, _ = oracle.combine_bwd(inp["g"], inp["y"], L)
        oracle.scale_rows_bwd(inp["ghs"], inp["h"], recv_w, L)
    else:
        oracle.combine(inp["y"], L, w)
        gy, _ = oracle.combine_bwd(inp["g"], inp["y"], L, w)
    oracle.dispatch_bwd(gy, L)


def oracle_inputs(wl, seed):
    want = ("logits", "bias", "x", "y", "g") + (("h", "ghs") if wl.absorb else ())
    return synth.make_inputs(wl, seed=seed, want=want)


def time_oracle(wl, tokens, reps=1):
    sub = wl.with_tokens(tokens)
    inp = oracle_inputs(sub, wl.seed)
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle_chain(sub, inp)
        times.append(time.perf_counter() - t0)
    return times


def cpu_baseline(wl, tokens):
    tokens = min(tokens, wl.T) if tokens > 0 else wl.T
    t = time_oracle(wl, tokens)[0]
    return {"value": tokens / t, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "first %d of %d tokens of the same workload, whole path (route, layout, "
                      "dispatch, combine, combine_bwd, dispatch_bwd), single-threaded C++ oracle, "
                      "%.1f s" % (tokens, wl.T, t)}


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from oracle import build as ob
    ob.build()
    tokens = args.ref_tokens
    sub = wl.with_tokens(tokens)
    inp = oracle_inputs(sub, wl.seed)
    for _ in range(args.warmup):
        oracle_chain(sub, inp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_chain(sub, inp)
    el = time.perf_counter() - t0
    value = tokens * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic", "config": workload_config(wl, extra={"sample_tokens_per_step": tokens}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "first %d of %d tokens per step, whole path, single-threaded "
                                   "C++ oracle" % (tokens, wl.T)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# GPU leg


L2_BYTES = 129e6


def workload_config(wl, extra=None, cold=False):
    eb = 2 if wl.dtype == "bf16" else 4
    xb, yb = wl.T * wl.H * eb, wl.T * wl.K * wl.H * eb
    if cold:
        l2 = "cold: L2 flushed by a 256 MB device write before every timed step"
    elif xb > L2_BYTES:
        l2 = "inputs larger than L2 (x %.0f MB, y %.0f MB per step; L2 129 MB)" % (xb / 1e6, yb / 1e6)
    else:
        l2 = ("warm: steps back to back; y (%.0f MB) is larger than L2 (129 MB), x (%.0f MB) "
              "is not and may stay in L2 across steps" % (yb / 1e6, xb / 1e6))
    c = {"workload": "%s T=%d H=%d E=%d K=%d R=%d %s%s" % (
        wl.name, wl.T, wl.H, wl.E, wl.K, wl.R, wl.score_fn,
        (" groups=%d/%d" % (wl.topk_groups, wl.n_groups)) if wl.n_groups > 1 else ""),
        "tokens_per_gpu": wl.T, "hidden": wl.H, "experts": wl.E, "top_k": wl.K,
        "virtual_ranks": wl.R, "row_dtype": wl.dtype, "parallelism": "replicas",
        "l2": l2}
    if extra:
        c.update(extra)
    return c


def run_gpu(args, wl):
    import torch
    import combine_moe_route_05_gb300 as moe

    rank, world, local = dist_env()
    if torch.cuda.device_count() <= local:
        raise SystemExit("rank %d needs GPU %d, but %d are visible" % (rank, local,
                                                                      torch.cuda.device_count()))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    seed = replica_seed(wl.seed, rank, world)
    want = ("logits", "bias", "x", "y", "g") + (("h", "ghs") if wl.absorb else ())
    inp = synth.make_inputs(wl, seed=seed, want=want)

    def dev_tensor(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
        return torch.from_numpy(a).to(device)

    T, H, E, K = wl.T, wl.H, wl.E, wl.K
    r = moe.MoeRouter(E, K, wl.R, T, score_fn=wl.score_fn, num_groups=wl.n_groups,
                      topk_groups=wl.topk_groups, group_score_topk=wl.group_score_topk,
                      renorm=wl.renorm, route_scale=wl.route_scale)
    h = r.h
    logits, bias, x, y, g = (dev_tensor(inp[k]) for k in ("logits", "bias", "x", "y", "g"))
    hrows = dev_tensor(inp["h"]) if wl.absorb else None
    ghs = dev_tensor(inp["ghs"]) if wl.absorb else None
    bf = torch.bfloat16
    rd = bf if wl.dtype == "bf16" else torch.float32  # row dtype of the workload
    bits = (lambda t: t.view(torch.int16)) if rd == bf else (lambda t: t)
    idx = torch.empty(T, K, dtype=torch.int32, device=device)
    w = torch.empty(T, K, dtype=torch.float32, device=device)
    recv = torch.empty(T * K, H, dtype=rd, device=device)
    recv_w = torch.empty(T * K, dtype=torch.float32, device=device)
    out = torch.empty(T, H, dtype=rd, device=device)
    gy = torch.empty(T * K, H, dtype=rd, device=device)
    gw = torch.empty(T, K, dtype=torch.float32, device=device)
    gx = torch.empty(T, H, dtype=rd, device=device)
    stream = torch.cuda.current_stream()
    if wl.absorb:
        hs = torch.empty_like(hrows)
        gh = torch.empty_like(hrows)

    def stages(logits, bias, x, y, g, h_in=None, ghs_in=None):
        """The step's calls in order, as (name, call)."""
        st = [("route_topk", lambda: moe.moe_route_topk(h, logits, bias, idx, w)),
              ("dispatch_layout", lambda: moe.moe_dispatch_layout(h, idx)),
              ("dispatch", lambda: moe.moe_dispatch(h, x, w, recv, recv_w))]
        if wl.absorb:
            # scores go into the W2 input; the W2 GEMM itself (y from hs) and
            # its backward (ghs from g) sit between these calls and are not
            # part of the path: y and ghs are synthetic inputs
            st += [("scale_rows", lambda: moe.moe_scale_rows(h, h_in, recv_w, hs)),
                   ("combine", lambda: moe.moe_combine(h, y, None, out)),
                   ("combine_bwd", lambda: moe.moe_combine_bwd(h, g, y, None, gy, None)),
                   ("scale_rows_bwd", lambda: moe.moe_scale_rows_bwd(h, ghs_in, h_in, recv_w, gh, gw))]
        else:
            st += [("combine", lambda: moe.moe_combine(h, y, w, out)),
                   ("combine_bwd", lambda: moe.moe_combine_bwd(h, g, y, w, gy, gw))]
        st.append(("dispatch_bwd", lambda: moe.moe_dispatch_bwd(h, gy, gx)))
        return st

    main_stages = stages(logits, bias, x, y, g, hrows, ghs)
    names = tuple(n for n, _ in main_stages)
    launches_per_step = len(main_stages) - 1 + moe.moe_dispatch_layout_launches(h, T)

    def step(ev=None, st=main_stages):
        for j, (_, call) in enumerate(st):
            if ev is not None:
                ev[j].record(stream)
            call()
        if ev is not None:
            ev[len(st)].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(h) == 0
    # expert load of the routed batch (read outside the timed region); the
    # skewed workload must put more than 5x the mean load on its heaviest
    # expert and no token at all on exactly one expert
    cnt = moe.layout_tensors(h)["cnt_e"].cpu().numpy()
    load = {"max_over_mean": float(cnt.max() / cnt.mean()), "zero_load_experts": int((cnt == 0).sum()),
            "histogram_top8": [int(c) for c in np.sort(cnt)[::-1][:8]]}
    if wl.bias == "zipf" and not args.tokens:
        assert load["max_over_mean"] > 5 and load["zero_load_experts"] == 1, load

    # the step as one CUDA graph (captured once, replayed every step): the same
    # kernels and work, without the per-launch host and driver overhead
    graph = None
    if not args.eager:
        side = torch.cuda.Stream(device)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        assert moe.moe_read_device_status(h) == 0

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            step()

    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device) if args.cold else None
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if flush is None:
        # inputs larger than L2 (or warm L2, see the line's config): back to back
        start.record(stream)
        for i in range(args.steps):
            run_step()
        end.record(stream)
        torch.cuda.synchronize()
        el_ms = start.elapsed_time(end)
    else:
        # cold L2: every step runs after a write of twice the L2 size, which
        # sits between the step's own events
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(i)
            ev[i][0].record(stream)
            run_step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        el_ms = sum(a_.elapsed_time(b_) for a_, b_ in ev)
    clk = clocks.stop()
    barrier(world)
    ms_step = reduce_max(el_ms / args.steps, world, device)

    # stage times: a second pass of K eager steps with CUDA events between the
    # calls (the events themselves cost about 2 us each, so this pass runs a
    # little slower than the timed one)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize()
    stage_ms = {n: float(np.mean([e[j].elapsed_time(e[j + 1]) for e in evs])) for j, n in enumerate(names)}
    step_median_ms = float(np.median([e[0].elapsed_time(e[-1]) for e in evs]))
    stage_pass_ms = float(np.mean([e[0].elapsed_time(e[-1]) for e in evs]))

    # end to end through the same public calls, inputs from pinned host memory
    # and outputs read back every step
    e2e = None
    if not args.no_e2e:
        host_in = {k: torch.from_numpy(inp[k].view(np.int16) if inp[k].dtype == np.uint16 else inp[k])
                   .pin_memory() for k in want if inp[k] is not None}
        dev_in = {"logits": logits, "bias": bias, "x": x, "y": y, "g": g}
        if wl.absorb:
            dev_in.update({"h": hrows, "ghs": ghs})
        host_out = {"idx": torch.empty(T, K, dtype=torch.int32).pin_memory(),
                    "w": torch.empty(T, K, dtype=torch.float32).pin_memory(),
                    "out": bits(torch.empty(T, H, dtype=rd)).pin_memory(),
                    "gw": torch.empty(T, K, dtype=torch.float32).pin_memory(),
                    "gx": bits(torch.empty(T, H, dtype=rd)).pin_memory()}
        dev_out = {"idx": idx, "w": w, "out": bits(out), "gw": gw, "gx": bits(gx)}
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())

        # copies overlap compute: step i+1's inputs go up on their own stream
        # into the second of two device input sets while step i computes, and
        # step i's outputs come back on a third stream
        dev_sets = [dev_in, {k: (torch.empty_like(v) if v is not None else None)
                             for k, v in dev_in.items()}]
        set_stages = [stages(d["logits"], d["bias"], d["x"], d["y"], d["g"], d.get("h"), d.get("ghs"))
                      for d in dev_sets]
        s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_comp = [torch.cuda.Event(), torch.cuda.Event()]
        ev_out = torch.cuda.Event()

        def e2e_run(n):
            s_in.wait_stream(stream)
            for i in range(n):
                b = i % 2
                din = dev_sets[b]
                if i >= 2:
                    s_in.wait_event(ev_comp[b])  # input set b no longer read
                with torch.cuda.stream(s_in):
                    for k, t in host_in.items():
                        d = din[k]
                        (d.view(torch.int16) if d.dtype == bf else d).copy_(t, non_blocking=True)
                    ev_in[b].record(s_in)
                stream.wait_event(ev_in[b])
                if i >= 1:
                    stream.wait_event(ev_out)  # the previous outputs are read back
                step(st=set_stages[b])
                ev_comp[b].record(stream)
                s_out.wait_event(ev_comp[b])
                with torch.cuda.stream(s_out):
                    for k, t in host_out.items():
                        t.copy_(dev_out[k], non_blocking=True)
                    ev_out.record(s_out)
            stream.wait_stream(s_out)

        e2e_run(max(1, args.warmup))
        torch.cuda.synchronize()
        barrier(world)
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        e2e_run(args.steps)
        e2.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max(s2.elapsed_time(e2) / args.steps, world, device)
        e2e = {"value": world * T / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "copies": "pinned host buffers; host-to-device, compute and device-to-host "
                         "of consecutive steps overlap on three streams"}
    assert moe.moe_read_device_status(h) == 0

    # widened rows, timed apart from the step: router backward to the logits,
    # and the staged (token once per destination rank) dispatch and combine
    extras = None
    if not args.no_extras:
        def time_op(fn, reps=max(3, args.steps)):
            for _ in range(2):
                fn()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            for _ in range(reps):
                fn()
            b_.record(stream)
            torch.cuda.synchronize()
            return a_.elapsed_time(b_) / reps
        R = wl.R
        step()
        glogits = torch.empty(T, E, dtype=torch.float32, device=device)
        t_rb = time_op(lambda: moe.moe_route_bwd(h, logits, idx, gw, glogits))
        # the same router backward fused into the dispatch backward
        t_db = time_op(lambda: moe.moe_dispatch_bwd(h, gy, gx))
        t_dbr = time_op(lambda: moe.moe_dispatch_bwd_route(h, gy, logits, idx, gw, gx, glogits))
        send = torch.empty(T * min(K, R), H, dtype=rd, device=device)
        partial = torch.empty_like(send)
        t_ds = time_op(lambda: moe.moe_dispatch(h, x, w, recv, recv_w, send))
        t_ex = time_op(lambda: moe.moe_expand(h, send, recv))
        t_cp = time_op(lambda: moe.moe_combine_partial(h, y, w, partial))
        t_cr = time_op(lambda: moe.moe_combine_reduce(h, partial, out))
        S = int(moe.layout_tensors(h)["S"].item())
        row = H * (2 if wl.dtype == "bf16" else 4)
        extras = {
            "route_bwd": {"ms": t_rb, "gbs": (T * E * 4 + T * K * 12) / (t_rb / 1e3) / 1e9},
            "dispatch_bwd_route": {
                "fused_ms": t_dbr, "dispatch_bwd_ms": t_db, "separate_ms": t_db + t_rb,
                "launches": moe.moe_dispatch_bwd_route_launches(h)},
            "staged": {
                "dedup_factor": T * K / S, "send_rows": S,
                "dispatch_with_send_ms": t_ds, "expand_ms": t_ex, "combine_partial_ms": t_cp,
                "combine_reduce_ms": t_cr,
                "dispatch_with_send_gbs": (T + T * K + S) * row / (t_ds / 1e3) / 1e9,
                "expand_gbs": (S + T * K) * row / (t_ex / 1e3) / 1e9,
                "combine_partial_gbs": (T * K + S) * row / (t_cp / 1e3) / 1e9,
                "combine_reduce_gbs": (S + T) * row / (t_cr / 1e3) / 1e9},
        }
        assert moe.moe_read_device_status(h) == 0
        # the padded, capacity-aligned layout (segments rounded up to 128 rows)
        rp = moe.MoeRouter(E, K, R, T, score_fn=wl.score_fn, num_groups=wl.n_groups,
                           topk_groups=wl.topk_groups, group_score_topk=wl.group_score_topk,
                           renorm=wl.renorm, route_scale=wl.route_scale, pad_align=128)
        moe.moe_dispatch_layout(rp.h, idx)
        recv_p = torch.empty(rp.h.recv_rows, H, dtype=rd, device=device)
        recv_wp = torch.empty(rp.h.recv_rows, dtype=torch.float32, device=device)
        t_lp = time_op(lambda: moe.moe_dispatch_layout(rp.h, idx))
        t_dp = time_op(lambda: moe.moe_dispatch(rp.h, x, w, recv_p, recv_wp))
        assert moe.moe_read_device_status(rp.h) == 0
        extras["padded_layout"] = {
            "pad_align": 128, "receive_rows": rp.h.recv_rows, "layout_ms": t_lp,
            "dispatch_ms": t_dp,
            "dispatch_gbs": (T * row + rp.h.recv_rows * row) / (t_dp / 1e3) / 1e9}
        del recv_p, recv_wp
        extras["w2_absorbed"] = w2_absorbed_extra(device, stream, max(5, args.steps // 5),
                                                  tokens=args.tokens or None)

    if rank != 0:
        return
    peak, peak_src = read_peaks()
    sb = step_bytes(wl)
    total_bytes = sum(sb.values())
    dom_ms = stage_ms[DOMINANT]
    achieved = sb[DOMINANT] / (dom_ms / 1e3) / 1e9
    # the committed summary is for the full-size workload
    traffic = measured_traffic_per_launch(DOMINANT, wl.name) if not args.tokens else None
    cpu = None
    if world == 1 and not args.no_cpu:
        cpu = cpu_baseline(wl, args.cpu_tokens)
    line = {
        "metric": METRIC, "value": world * T / (ms_step / 1e3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic", "config": workload_config(wl, cold=args.cold),
        "hbm_gbs": total_bytes / (ms_step / 1e3) / 1e9,
        "hbm_frac_of_peak": total_bytes / (ms_step / 1e3) / 1e9 / peak,
        "hbm_frac_of_nominal": total_bytes / (ms_step / 1e3) / 1e9 / NOMINAL_HBM_GBS,
        "launch": "eager" if args.eager else "cuda_graph",
        "bytes_per_step": total_bytes,
        "stage_pass": {"launch": "eager, CUDA events between the calls", "steps": args.steps,
                       "ms_per_step": stage_pass_ms, "ms_per_step_median": step_median_ms},
        "stage_ms": stage_ms,
        "stage_gbs": {n: sb[n] / (stage_ms[n] / 1e3) / 1e9 for n in names},
        "roofline": {"kernel": DOMINANT, "bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes": sb[DOMINANT], "peak_source": peak_src},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "kernel_source": kernel_source_hash(),
        "expert_load": load,
        "extras": extras,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", type=int, default=3)
    ap.add_argument("--tokens", type=int, default=0, help="override T (small profiling cases)")
    ap.add_argument("--cpu-tokens", type=int, default=0,
                    help="oracle baseline sample in tokens (0 = the whole batch)")
    ap.add_argument("--ref-tokens", type=int, default=256)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="time eager launches instead of the step replayed as a CUDA graph")
    ap.add_argument("--cold", action="store_true",
                    help="flush L2 (a 256 MB device write) before every timed step, outside "
                         "the step's own events")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(relaunch_under_torchrun(args.gpus))
    world = dist_env()[1]
    if world != args.gpus:
        ap.error("--gpus %d but %d ranks were started" % (args.gpus, world))
    wl = synth.WORKLOADS[args.workload]
    if args.tokens:
        wl = wl.with_tokens(args.tokens)
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_gpu(args, wl)


if __name__ == "__main__":
    main()
