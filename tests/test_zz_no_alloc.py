"""The allocation-free entry point, mxfp4_expert_linear_static_scratch.

It is for callers that cannot allocate device memory while they run (a
serving process whose memory budget is fixed at start-up, a plugin inside a
host framework that owns every device allocation): its scratch is a fixed
array compiled into the library. The tests check that, on each kernel path
the library picks (the GEMV routing for itself, the GEMV after the separate
bucketer, the tensor-core GEMM), the call gives exactly the bits of the
caller-workspace entry point and matches the float64 oracle within the
tolerance of the other parity tests; that two calls in a row (the array
keeping the previous call's contents) stay correct; and that the calls leave
the device's free memory unchanged.

This file is collected last on purpose, so that a run stopping at its first
failure has run every other test.
"""
import ctypes

import pytest
import torch

from gpu_util import assert_parity, oracle_rows
from mxfp4_routed_expert_route_gb300 import (_native, mxfp4_expert_linear, workloads,
                                             workspace_size)


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


# (workload, environment): the three kernel paths, each within the 8 MiB array.
CASES = [
    # 32 pairs: the GEMV routes for itself (bf16 tokens scaled on load).
    (dict(T=8, E=32, K=4, I=512, O=640, dtype=torch.bfloat16, seed=71), {}),
    # fp32 tokens, ragged sizes.
    (dict(T=13, E=20, K=3, I=256, O=300, dtype=torch.float32, seed=72), {}),
    # The separate bucketer launch before the GEMV, with its own scratch.
    (dict(T=40, E=24, K=4, I=320, O=200, dtype=torch.bfloat16, seed=73),
     {"MXFP4EL_ROUTE": "bucketer"}),
    # The tensor-core GEMM: 256 pairs over 4 experts (64 tokens per expert),
    # the f16 token copy and partial results in the array.
    (dict(T=128, E=4, K=2, I=256, O=192, dtype=torch.bfloat16, seed=74),
     {"MXFP4EL_PATH": "gemm"}),
]


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point_twice(lib, monkeypatch):
    limit = lib.mxfp4_expert_linear_static_scratch_bytes()
    runs = []
    for cfg, env in CASES:
        wl = workloads.make(name=f"static_{cfg['seed']}", **cfg)
        need = workspace_size(wl.T, wl.E, wl.I, wl.O, wl.K, wl.dtype)
        assert 0 < need <= limit, (cfg, need)
        d = wl.device_tensors("cuda")
        for k in ("MXFP4EL_ROUTE", "MXFP4EL_PATH"):
            monkeypatch.delenv(k, raising=False)
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        # The reference: the caller-workspace entry point on a torch buffer.
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        ref = mxfp4_expert_linear(d["x"], d["packed"], d["scales"], d["sel"], d["p"],
                                  d["y_shared"], workspace=ws)
        outs = [torch.full_like(ref, float("nan")) for _ in range(2)]
        runs.append((wl, env, d, ref, outs))
    torch.cuda.synchronize()

    # First call on this device: it looks up the array's address (and may load
    # the library's device code); not part of the measured calls below.
    wl0, env0, d0, _, outs0 = runs[0]
    for k, v in env0.items():
        monkeypatch.setenv(k, v)
    assert _call_static(lib, d0, wl0, outs0[0]) == _native.OK
    torch.cuda.synchronize()

    free_before = torch.cuda.mem_get_info()[0]
    # Every case twice in a row; the array keeps whatever the previous call
    # (another case, or the same one) left in it.
    for rep in range(2):
        for wl, env, d, ref, outs in runs:
            for k in ("MXFP4EL_ROUTE", "MXFP4EL_PATH"):
                monkeypatch.delenv(k, raising=False)
            for k, v in env.items():
                monkeypatch.setenv(k, v)
            assert _call_static(lib, d, wl, outs[rep]) == _native.OK, (wl.name, rep)
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before, "the allocation-free calls changed free device memory"

    for wl, env, d, ref, outs in runs:
        want, abs_terms, bad = oracle_rows(wl)
        assert bad == 0
        for rep in range(2):
            assert torch.equal(outs[rep], ref), (wl.name, env, rep)
            assert_parity(outs[rep], want, abs_terms, wl.dtype, f"static {wl.name} call {rep}")
