"""moe_dispatch_layout_static, the allocation-free layout, against the
handle-based moe_dispatch_layout.

The allocation-free entry point serves callers that may not allocate device
memory (for instance a plugin that receives only its input and output buffers
from a host framework which forbids cudaMalloc while it runs or captures the
stream).  Its scratch is a static device array shared by all calls, so this
test calls it twice in a row, on two different batches, and requires each
result to equal, bit for bit, the handle-based layout of the same batch.  The
file is collected last so that a failure here leaves every other test run."""
import numpy as np
import pytest
import torch

import combine_moe_route_05_gb300 as moe
import oracle
import synth
from tests.gpu_util import dev, oracle_route, router, to_dev

pytestmark = pytest.mark.gpu


def batches():
    wl = synth.WORKLOADS[3].with_tokens(2600)
    inp = synth.make_inputs(wl, want=("logits", "bias"))
    idx_a, _ = oracle_route(wl, inp["logits"], inp["bias"])
    # a second, smaller batch with dropped entries (a repeat and an out-of-range index)
    rng = np.random.default_rng(7)
    idx_b = np.stack([rng.choice(wl.E, wl.K, replace=False) for _ in range(1500)]).astype(np.int32)
    idx_b[10, 3] = idx_b[10, 0]
    idx_b[99, 7] = wl.E + 5
    return wl, [idx_a, idx_b]


def empty_outputs(wl, T):
    sizes = moe.layout_sizes(T, wl.K, wl.E, wl.R)
    # filled with a sentinel so that an unwritten entry cannot pass as written
    return {n: torch.full((sizes[n],), -7, dtype=torch.int32, device=dev()) for n in moe.LAYOUT_FIELDS}


def test_static_layout_equals_handle_layout_on_two_calls_in_a_row():
    wl, idxs = batches()
    cfg = moe.make_config(wl.E, wl.K, wl.R, max(i.shape[0] for i in idxs), score_fn=wl.score_fn,
                          num_groups=wl.n_groups, topk_groups=wl.topk_groups,
                          group_score_topk=wl.group_score_topk)
    for idx in idxs:
        T = idx.shape[0]
        d_idx = to_dev(idx)
        r = router(wl, max_tokens=T)
        ref = {k: v.clone() for k, v in r.layout(d_idx).items()}
        ref_flags = moe.moe_read_device_status(r.h)
        out = empty_outputs(wl, T)
        status = torch.zeros(1, dtype=torch.int32, device=dev())
        moe.moe_dispatch_layout_static(cfg, d_idx, out, status)
        torch.cuda.synchronize()
        for name in moe.LAYOUT_FIELDS:
            assert torch.equal(out[name], ref[name].reshape(-1)), name
        assert int(status.item()) == ref_flags
        # and the handle-based layout itself matches the oracle
        L = oracle.layout(idx, wl.E, wl.R)
        assert np.array_equal(out["pos"].cpu().numpy().reshape(T, wl.K), L.pos)


def test_static_layout_rejects_sizes_beyond_its_scratch():
    wl = synth.WORKLOADS[3]
    cfg = moe.make_config(wl.E, wl.K, wl.R, 16, score_fn="sigmoid", num_groups=8, topk_groups=4,
                          group_score_topk=2)
    tiles_max = moe.MOE_LAYOUT_STATIC_COUNTERS // (wl.E + wl.R)
    T = tiles_max * moe.MOE_LAYOUT_TILE_TOKENS + 1
    v = moe.MoeLayout()
    st = moe.lib().moe_dispatch_layout_static(
        __import__("ctypes").byref(cfg), None, T, __import__("ctypes").byref(v), None, None)
    assert st == moe.MOE_ERR_CAPACITY


def test_static_layout_two_launch_path_on_two_calls_in_a_row():
    """A batch whose tiles do not all fit on the GPU at once (160000 tokens:
    313 tiles of 512) takes the two-launch path, in which the count kernel's
    last block uses and re-arms the arrival counter in the static array.  Two
    calls in a row must each equal the handle-based layout and the oracle, and
    a single-launch call after them must still be right."""
    E, K, R, T = 16, 2, 4, 160000
    wl = synth.Workload("two_launch", T=T, H=64, E=E, K=K, R=R)
    assert moe.layout_sizes(T, K, E, R)["pos"] == T * K
    assert (T + moe.MOE_LAYOUT_TILE_TOKENS - 1) // moe.MOE_LAYOUT_TILE_TOKENS * (E + R) \
        <= moe.MOE_LAYOUT_STATIC_COUNTERS
    rng = np.random.default_rng(11)
    cfg = moe.make_config(E, K, R, T)
    r = router(wl)
    assert moe.moe_dispatch_layout_launches(r.h, T) == 2
    for call in range(2):
        idx = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int32)
        d_idx = to_dev(idx)
        ref = {k: v.clone() for k, v in r.layout(d_idx).items()}
        out = empty_outputs(wl, T)
        status = torch.zeros(1, dtype=torch.int32, device=dev())
        moe.moe_dispatch_layout_static(cfg, d_idx, out, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for name in moe.LAYOUT_FIELDS:
            assert torch.equal(out[name], ref[name].reshape(-1)), (call, name)
        L = oracle.layout(idx, E, R)
        for f in oracle.Layout.FIELDS:
            assert np.array_equal(out[f].cpu().numpy(), getattr(L, f).reshape(-1)), (call, f)
        assert int(out["S"].item()) == L.S
    # back to the single launch on the same static array
    test_static_layout_equals_handle_layout_on_two_calls_in_a_row()
