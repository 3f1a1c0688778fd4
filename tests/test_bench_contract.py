"""The benchmark's contract, on the CPU: the algorithmic bytes it divides by
(the numerator of every bandwidth and roofline figure) against the closed
forms of the step, and the JSON line of its reference arm."""
import json
import os
import subprocess
import sys

import pytest

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ROW_STAGES = ("dispatch", "combine", "combine_bwd", "dispatch_bwd", "scale_rows", "scale_rows_bwd")


@pytest.mark.parametrize("i", [0, 1, 2, 3, 4])
def test_step_bytes_match_the_closed_forms(i):
    """Each row tensor crosses HBM once per stage: dispatch reads x and writes
    K rows, combine reads K rows and writes one, the weighted combine backward
    reads g and y and writes gy (1 + 2K rows), the dispatch backward reads K
    and writes one: 2H (5K + 4) bytes per bf16 token.  Under absorption the
    combine backward is a copy (1 + K rows) and scale_rows moves 2 + 3 rows
    of I per entry: 2H (4K + 4) + 2I 5K.  Index and score arrays are 4 bytes
    per entry and array."""
    wl = synth.WORKLOADS[i]
    b = bench.step_bytes(wl)
    T, H, K = wl.T, wl.H, wl.K
    eb = 2 if wl.dtype == "bf16" else 4
    rows = sum(v for k, v in b.items() if k in ROW_STAGES)
    if wl.absorb:
        # pos + score + send row (dispatch), score (scale_rows), pos (combine,
        # its backward, dispatch_bwd), score + pos + gw (scale_rows_bwd)
        index = T * K * 4 * (3 + 1 + 1 + 1 + 3 + 1)
        want = T * (eb * H * (4 * K + 4) + eb * wl.I * 5 * K)
    else:
        # pos + score + send row (dispatch), pos + score (combine),
        # pos + score + gw (combine_bwd), pos (dispatch_bwd)
        index = T * K * 4 * (3 + 2 + 3 + 1)
        want = T * eb * H * (5 * K + 4)
    assert rows - index == want
    if i == 3:
        assert want // T == 630784  # the DeepSeek-V3 figure per token
    if i == 1:
        assert want // T == 180224
    if i == 4:
        assert want // T == 417792
    # routing reads the logits (and the bias) and writes idx and w
    assert b["route_topk"] == T * wl.E * 4 + (wl.E * 4 if wl.bias == "normal" else 0) + T * K * 8


def test_reference_arm_line():
    """`--impl reference` times the oracle on the host and prints one JSON
    line with the base contract's keys, its own cpu_baseline and an e2e that
    moves no bytes."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3", "--ref-tokens", "32", "--workload", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["warmup"] == 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["unit"] == line["unit"]
    assert line["config"]["workload"].startswith("qwen3_30b")


def test_traffic_records_are_consistent():
    """The per-launch DRAM traffic the benchmark reports beside its roofline
    (profiles/traffic.json) is one ncu pass per record: each names a workload,
    the hash of the kernel sources it was taken on and the summary that cites
    it; the figure lies at or a little below the kernel's algorithmic bytes
    (the write-back L2 still holds the last writes when a launch ends) and
    never well above them, which would mean re-reads."""
    import re
    with open(bench.TRAFFIC_RECORDS) as f:
        recs = json.load(f)
    by_name = {w.name: w for w in synth.WORKLOADS.values()}
    algo = {}
    wl = by_name[recs["combine_bwd"]["workload"]]
    algo["combine_bwd"] = bench.step_bytes(wl)["combine_bwd"]
    wl = by_name[recs["w2_absorbed"]["workload"]]
    rows, H = wl.T * wl.K, 4096
    algo["w2_absorbed"] = rows * wl.I * 2 + wl.E * H * wl.I * 2 + rows * H * 2 + rows * 4
    for key, a in algo.items():
        rec = recs[key]
        traffic = rec["traffic_bytes_per_launch"]
        assert 0.95 * a <= traffic <= 1.01 * a, (key, traffic, a)
        assert re.fullmatch(r"[0-9a-f]{16}", rec["source"])
        with open(os.path.join(ROOT, rec["summary"])) as f:
            text = f.read()
        cite = "(key `%s`): %.3fe9 bytes, workload %s, kernel source %s" % (
            key, traffic / 1e9, rec["workload"], rec["source"])
        assert cite in text, cite
