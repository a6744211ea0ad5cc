"""The allocation-free entry point, mxfp4_expert_linear_static_scratch.

It serves callers that cannot allocate device memory: its scratch is a fixed
array compiled into the library. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

from gpu_util import TOL, oracle_rows, worst_ratio
from mxfp4_routed_expert_route_gb300 import _native, mxfp4_expert_linear, workloads


@pytest.fixture(scope="module")
def lib():
    from mxfp4_routed_expert_route_gb300 import build
    build.build()
    return _native.load()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else None


def _call_static(lib, d, wl, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dtype = _native.DTYPE_BF16 if wl.dtype == torch.bfloat16 else _native.DTYPE_F32
    return lib.mxfp4_expert_linear_static_scratch(
        _ptr(d["x"]), _ptr(d["packed"]), _ptr(d["scales"]), _ptr(d["sel"]),
        _ptr(d["p"]), _ptr(d["y_shared"]), _ptr(out), wl.T, wl.E, wl.I, wl.O, wl.K,
        dtype, _native.INDEX_I32, stream)


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point_twice(lib):
    # Two different calls in a row: the second must not see the first's scratch.
    cases = [workloads.make(8, 32, 4, 512, 640, dtype=torch.bfloat16, seed=71,
                            name="first"),
             workloads.make(13, 20, 3, 256, 300, dtype=torch.float32, seed=72,
                            name="second")]
    for wl in cases:
        d = wl.device_tensors("cuda")
        ref = mxfp4_expert_linear(d["x"], d["packed"], d["scales"], d["sel"], d["p"],
                                  d["y_shared"])
        out = torch.full_like(ref, float("nan"))
        assert _call_static(lib, d, wl, out) == _native.OK
        torch.cuda.synchronize()
        _, abs_terms, _ = oracle_rows(wl)
        assert worst_ratio(out, ref.cpu().double().numpy(), abs_terms) <= TOL[wl.dtype], wl.name


@pytest.mark.gpu
def test_static_scratch_rejects_oversized_calls(lib):
    limit = lib.mxfp4_expert_linear_static_scratch_bytes()
    assert limit == 8 << 20
    # 64 tokens x 8 slots x 8192 rows of float32 partials is 16 MiB: refused
    # before any GPU work (the pointers are never touched).
    fake = ctypes.c_void_p(1 << 24)
    out = ctypes.c_void_p(1 << 40)
    rc = lib.mxfp4_expert_linear_static_scratch(fake, fake, fake, fake, fake, fake,
                                                out, 64, 16, 256, 8192, 8,
                                                _native.DTYPE_BF16, _native.INDEX_I32,
                                                None)
    assert rc == _native.ERR_TOO_LARGE
