"""The C-ABI library builds, loads and exports every entry point that
include/moe_route.h declares; host-side argument validation (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_route.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(moe_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from combine_moe_route_05_gb300 import build
    build.build()
    import combine_moe_route_05_gb300 as m
    return m


def test_header_declares_the_six_path_calls():
    names = declared_functions()
    for n in ("moe_route_topk", "moe_dispatch_layout", "moe_dispatch", "moe_combine",
              "moe_dispatch_bwd", "moe_combine_bwd"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 15
    L = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (moe_\w+)$", out, flags=re.M))
    assert set(names) <= exported
    assert set(lib.EXPORTS) == set(names)


def test_binding_covers_every_declared_function(lib):
    """The Python binding names exactly the header's functions, and sets a
    signature for each (no call goes through ctypes' default int marshalling)."""
    assert set(declared_functions()) == set(lib.EXPORTS)
    L = lib.lib()
    for n in lib.EXPORTS:
        assert getattr(L, n).argtypes is not None, n


def test_library_is_built_for_sm_103a_only():
    """The build compiles every translation unit and links for sm_103a, one
    -gencode and no other architecture flag."""
    from combine_moe_route_05_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert not any("arch" in f or "gencode" in f for f in build.FLAGS)


def test_status_strings(lib):
    for s in range(5):
        assert lib.status_string(s).startswith("MOE_")


@pytest.mark.parametrize("kw,ok", [
    (dict(num_experts=256, top_k=8, num_ranks=64, max_tokens=16384, score_fn="sigmoid",
          num_groups=8, topk_groups=4, group_score_topk=2), True),
    (dict(num_experts=128, top_k=8, num_ranks=8, max_tokens=8192), True),
    (dict(num_experts=8, top_k=2, num_ranks=2, max_tokens=0), True),
    (dict(num_experts=512, top_k=16, num_ranks=512, max_tokens=4096), True),
    (dict(num_experts=256, top_k=8, num_ranks=64, max_tokens=16, num_groups=8, topk_groups=4,
          group_score_topk=2), False),  # groups need sigmoid scores
    (dict(num_experts=128, top_k=8, num_ranks=7, max_tokens=16), False),    # E % R
    (dict(num_experts=8, top_k=9, num_ranks=1, max_tokens=16), False),      # K > E
    (dict(num_experts=1024, top_k=8, num_ranks=1, max_tokens=16), False),   # E > 512
    (dict(num_experts=64, top_k=17, num_ranks=1, max_tokens=16), False),    # K > 16
    (dict(num_experts=8, top_k=2, num_ranks=2, max_tokens=-1), False),
    (dict(num_experts=64, top_k=9, num_ranks=1, max_tokens=16, score_fn="sigmoid",
          num_groups=8, topk_groups=1, group_score_topk=2), False),         # K > kept experts
])
def test_workspace_bytes_validates_config(lib, kw, ok):
    cfg = lib.make_config(**kw)
    n = lib.moe_workspace_bytes(cfg)
    assert (n > 0) == ok
    if ok:
        T, K, R = kw["max_tokens"], kw["top_k"], kw["num_ranks"]
        assert n >= 4 * T * K * 5 + 4 * T * min(K, R)


def test_host_validation_rejects_bad_arguments_without_a_gpu(lib):
    L = lib.lib()
    cfg = lib.make_config(8, 2, 2, 64)
    h = ctypes.c_void_p()
    # null workspace, misaligned workspace, too small workspace, null out
    assert L.moe_handle_create(ctypes.byref(cfg), None, 1 << 20, ctypes.byref(h)) == lib.MOE_ERR_INVALID
    assert L.moe_handle_create(ctypes.byref(cfg), 0x1008, 1 << 20, ctypes.byref(h)) == lib.MOE_ERR_INVALID
    assert L.moe_handle_create(ctypes.byref(cfg), 0x10000, 16, ctypes.byref(h)) == lib.MOE_ERR_INVALID
    assert L.moe_handle_create(ctypes.byref(cfg), 0x10000, 1 << 20, None) == lib.MOE_ERR_INVALID
    # every compute call rejects a null handle before touching the device
    assert L.moe_route_topk(None, 0x1000, None, 4, 0x1000, 0x1000, None) == lib.MOE_ERR_INVALID
    assert L.moe_dispatch_layout(None, 0x1000, 4, None) == lib.MOE_ERR_INVALID
    assert L.moe_dispatch(None, 0x1000, 8, 0, None, 0x1000, None, None, None) == lib.MOE_ERR_INVALID
    assert L.moe_combine(None, 0x1000, 8, 0, None, 0x1000, None) == lib.MOE_ERR_INVALID
    assert L.moe_combine_bwd(None, 0x1000, 0x1000, 8, 0, None, 0x1000, None, None) == lib.MOE_ERR_INVALID
    assert L.moe_dispatch_bwd(None, 0x1000, 8, 0, 0x1000, None) == lib.MOE_ERR_INVALID
    assert L.moe_read_device_status(None, None) == lib.MOE_ERR_INVALID
    assert L.moe_handle_destroy(None) == lib.MOE_ERR_INVALID


class _FakeCudaTensor:
    """Stands in for a CUDA tensor on a given device (no GPU needed)."""
    is_cuda = True

    def __init__(self, device, shape, dtype):
        self.device, self.shape, self.dtype = device, shape, dtype

    def is_contiguous(self):
        return True


class _FakeStream:
    def __init__(self, device):
        self.device, self.cuda_stream = device, 0


def test_binding_rejects_tensors_and_streams_of_another_device(lib):
    import torch
    d0, d1 = torch.device("cuda", 0), torch.device("cuda", 1)
    lib._req(_FakeCudaTensor(d0, (4, 8), torch.float32), torch.float32, (4, 8), "x", d0)
    with pytest.raises(ValueError, match="x is on cuda:1, the handle on cuda:0"):
        lib._req(_FakeCudaTensor(d1, (4, 8), torch.float32), torch.float32, (4, 8), "x", d0)
    assert lib._stream(_FakeStream(d0), d0) == 0
    with pytest.raises(ValueError, match="stream is on cuda:1"):
        lib._stream(_FakeStream(d1), d0)
