"""GPU checks of the prepared weight layout and of the calls that read it.

The prepared copy is a load-time re-layout of the same bytes ("MoE Expert
Kernels: Grouped Prefill and Mixed-Quant Compact Experts", section 2, the
weight preparation built once at load time), so:
  * its bytes must equal a re-layout written here from the header's
    definition (blocks of 128 rows x one 64-wide K chunk, 16-byte halves
    swapped on rows with bit 2 set, scale bytes after each block's codes);
  * every call on it must give the same bits as the same call on the plain
    layout, through both kernels (GEMV and tensor-core GEMM), whatever the
    tile modes, and agree with the oracle.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_parity, oracle_rows, parity_rows
from mxfp4_routed_expert_route_gb300 import (mxfp4_expert_linear, mxfp4_expert_linear_prepared,
                                             prepare_weights, prepared_bytes, wait_timeouts,
                                             workloads)

pytestmark = pytest.mark.gpu


def _align256(n):
    return (n + 255) // 256 * 256


def _expected_blocks(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """The block region of the prepared copy, from the header's definition."""
    E, O, G, _ = packed.shape
    nk, mt = (G + 1) // 2, (O + 127) // 128
    out = np.zeros((E, mt, nk, 4352), dtype=np.uint8)
    for e in range(E):
        for t in range(mt):
            for kc in range(nk):
                blk = out[e, t, kc]
                for m in range(128):
                    o = 128 * t + m
                    row = min(o, O - 1)
                    g0, g1 = 2 * kc, 2 * kc + 1
                    c0 = packed[e, o, g0] if o < O else np.zeros(16, np.uint8)
                    c1 = packed[e, o, g1] if o < O and g1 < G else np.zeros(16, np.uint8)
                    sw = (m >> 2) & 1
                    blk[32 * m + 16 * sw: 32 * m + 16 * sw + 16] = c0
                    blk[32 * m + 16 * (1 - sw): 32 * m + 16 * (1 - sw) + 16] = c1
                    blk[4096 + 2 * m] = scales[e, row, g0]
                    blk[4097 + 2 * m] = scales[e, row, g1] if g1 < G else scales[e, row, g0]
    return out.reshape(-1)


@pytest.mark.parametrize("E,O,I", [(2, 128, 64), (3, 200, 96), (1, 77, 160), (2, 300, 2880)])
def test_prepared_bytes_match_the_documented_layout(E, O, I):
    wl = workloads.make(4, E, 1, I, O, seed=E * 1000 + O + I)
    G = I // 32
    nk, mt = (G + 1) // 2, (O + 127) // 128
    n = prepared_bytes(E, I, O)
    assert n == (_align256(E * mt * nk * 4352) + _align256(E * O * 2) + _align256(E * mt))
    pw = prepare_weights(wl.packed.cuda(), wl.scales.cuda())
    torch.cuda.synchronize()
    got = pw.buffer.cpu().numpy()
    want = _expected_blocks(wl.packed.numpy(), wl.scales.numpy())
    np.testing.assert_array_equal(got[:want.size], want)
    # The tensor-core kernel's f16 mode data: offset = the row's largest
    # scale byte - 140; a tile takes the mode when every row's bytes span at
    # most 26 binades.
    off = _align256(E * mt * nk * 4352)
    row_off = got[off:off + E * O * 2].view(np.int16).reshape(E, O)
    sc = wl.scales.numpy().astype(np.int32)
    np.testing.assert_array_equal(row_off, sc.max(axis=2) - 140)
    off += _align256(E * O * 2)
    modes = got[off:off + E * mt].reshape(E, mt)
    span = sc.max(axis=2) - sc.min(axis=2)
    for e in range(E):
        for t in range(mt):
            assert modes[e, t] == int((span[e, 128 * t:128 * t + 128] <= 26).all())


def _both(wl, sel=None):
    d = wl.device_tensors("cuda")
    if sel is not None:
        d["sel"] = sel.cuda()
    plain = mxfp4_expert_linear(d["x"], d["packed"], d["scales"], d["sel"], d["p"],
                                d["y_shared"])
    pw = prepare_weights(d["packed"], d["scales"])
    prep = mxfp4_expert_linear_prepared(d["x"], pw, d["sel"], d["p"], d["y_shared"])
    torch.cuda.synchronize()
    assert wait_timeouts() == 0
    return plain, prep


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,E,K,I,O", [
    (1, 4, 2, 64, 130),         # one token: self-routed GEMV
    (16, 8, 4, 96, 257),        # odd group count, ragged rows
    (200, 6, 2, 2880, 384),     # tensor-core GEMM for bf16
    (1500, 16, 4, 256, 520),    # many pairs: the bucketer's multi-CTA sort
])
def test_prepared_matches_plain_bitwise(dtype, T, E, K, I, O):
    wl = workloads.make(T, E, K, I, O, dtype=dtype, seed=T + E + I + O)
    plain, prep = _both(wl)
    assert torch.equal(plain, prep)
    want, absm, _ = oracle_rows(wl)
    assert_parity(prep, want, absm, wl.dtype, f"prepared {T},{E},{K},{I},{O}")


@pytest.mark.parametrize("path", ["gemm", "gemv"])
def test_prepared_matches_plain_on_each_kernel(monkeypatch, path):
    monkeypatch.setenv("MXFP4EL_PATH", path)
    wl = workloads.make(300, 5, 2, 512, 390, dtype=torch.bfloat16, seed=11)
    plain, prep = _both(wl)
    assert torch.equal(plain, prep)


def test_prepared_mixed_operand_modes_bitwise(monkeypatch):
    # Expert 0's tiles take the f16 operands, expert 1's (one row spanning
    # 34 binades) the bf16 operands, in one tensor-core launch.
    monkeypatch.setenv("MXFP4EL_PATH", "gemm")
    T, E, K, I, O = 160, 2, 1, 512, 256
    wl = workloads.make(T, E, K, I, O, dtype=torch.bfloat16, scale_lo=116, scale_hi=124,
                        seed=5)
    wl.scales[1, :, 0] = 90
    sel = torch.from_numpy((np.arange(T) % 2).reshape(T, 1).astype(np.int32))
    plain, prep = _both(wl, sel=sel)
    assert torch.equal(plain, prep)
    want, absm, _ = oracle_rows(wl, sel=sel)
    assert_parity(prep, want, absm, wl.dtype, "prepared mixed tiles")


@pytest.mark.parametrize("name", ["decode", "wide_decode", "prefill", "skewed_prefill"])
def test_prepared_named_workloads_bitwise(name):
    wl = workloads.named(name)
    plain, prep = _both(wl)
    assert torch.equal(plain, prep), name
    rows = parity_rows(wl, n_random=64)
    want, absm, _ = oracle_rows(wl, rows=rows)
    assert_parity(prep[torch.from_numpy(rows).cuda()], want, absm, wl.dtype,
                  f"prepared {name} ({len(rows)} rows)")
