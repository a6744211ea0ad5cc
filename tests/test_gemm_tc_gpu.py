"""GPU parity of the tensor-core (tcgen05) grouped GEMM path.

The library picks the tensor-core kernel for bf16 tokens when experts
average at least 16 tokens; MXFP4EL_PATH=gemm forces it for these cases so
that small shapes exercise every edge: output widths that are not a multiple
of the 128-row tile, token counts around the 16-token MMA granule and the
192-token block, a single 64-wide K chunk, and many experts.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_parity, oracle_rows, run_gpu
from mxfp4_routed_expert_route_gb300 import wait_timeouts, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _force_gemm(monkeypatch):
    monkeypatch.setenv("MXFP4EL_PATH", "gemm")


def _one_expert_sel(T, K, E, hot, rng):
    """Slot 0 of every token on expert `hot`, the other slots elsewhere."""
    sel = np.zeros((T, K), dtype=np.int32)
    for t in range(T):
        others = rng.permutation([e for e in range(E) if e != hot])[:K - 1]
        sel[t] = np.concatenate([[hot], others])
    return torch.from_numpy(sel)


@pytest.mark.parametrize("T,E,K,I,O", [
    (8, 2, 1, 64, 128),        # one K chunk, one row tile
    (40, 3, 2, 128, 200),      # row tile with 72 rows
    (64, 4, 2, 320, 257),
    (300, 12, 3, 256, 130),
    (97, 5, 4, 2880, 384),     # the decode/prefill width
])
def test_gemm_path_matches_oracle(T, E, K, I, O):
    wl = workloads.make(T, E, K, I, O, dtype=torch.bfloat16, seed=T + O)
    out = run_gpu(wl)
    torch.cuda.synchronize()
    assert wait_timeouts() == 0
    want, absm, _ = oracle_rows(wl)
    assert_parity(out, want, absm, wl.dtype, f"gemm {T},{E},{K},{I},{O}")


@pytest.mark.parametrize("ntok", [1, 15, 16, 17, 191, 192, 193, 400])
def test_gemm_token_block_edges(ntok):
    # Expert 1 receives exactly ntok tokens (slot 0 of each); the other
    # slot spreads over the remaining experts.
    rng = np.random.default_rng(ntok)
    T, E, K, I, O = ntok, 6, 2, 128, 136
    wl = workloads.make(T, E, K, I, O, dtype=torch.bfloat16, seed=ntok)
    sel = _one_expert_sel(T, K, E, 1, rng)
    out = run_gpu(wl, sel=sel)
    torch.cuda.synchronize()
    assert wait_timeouts() == 0
    want, absm, _ = oracle_rows(wl, sel=sel)
    assert_parity(out, want, absm, wl.dtype, f"ntok={ntok}")


def test_gemm_integer_inputs_exact():
    # Integer tokens, unit scales, one slot with weight 1, zero shared output:
    # every product and sum is exact in float32, so the bf16 result must be
    # the oracle's value rounded to bf16.
    rng = np.random.default_rng(31)
    T, E, K, I, O = 48, 3, 1, 256, 160
    wl = workloads.make(T, E, K, I, O, dtype=torch.bfloat16, scale_lo=127,
                        scale_hi=127, seed=31)
    wl.x = torch.from_numpy(rng.integers(-8, 9, (T, I)).astype(np.float32)).to(torch.bfloat16)
    wl.y_shared = torch.zeros((T, O), dtype=torch.bfloat16)
    wl.p = torch.ones((T, K), dtype=torch.float32)
    out = run_gpu(wl)
    want, _, _ = oracle_rows(wl)
    assert torch.equal(out.cpu(), torch.from_numpy(want).to(torch.bfloat16))


def test_gemm_and_gemv_agree(monkeypatch):
    wl = workloads.make(160, 8, 4, 512, 264, dtype=torch.bfloat16, seed=33)
    a = run_gpu(wl)
    monkeypatch.setenv("MXFP4EL_PATH", "gemv")
    b = run_gpu(wl)
    want, absm, _ = oracle_rows(wl)
    assert_parity(a, want, absm, wl.dtype, "gemm")
    assert_parity(b, want, absm, wl.dtype, "gemv")


def test_more_experts_than_the_tensor_core_lists_take_the_gemv(monkeypatch):
    # The tensor-core kernel keeps per-expert lists for up to 512 experts in
    # shared memory; beyond that a call runs on the GEMV, even when experts
    # average many tokens, and still matches the oracle.
    from mxfp4_routed_expert_route_gb300 import _native
    monkeypatch.delenv("MXFP4EL_PATH", raising=False)
    T, E, K, I, O = 640, 600, 16, 64, 48
    lib = _native.load()
    assert lib.mxfp4el_linear_path(T, E, I, O, K, _native.DTYPE_BF16) == _native.PATH_GEMV
    assert lib.mxfp4el_linear_path(T, 512, I, O, K, _native.DTYPE_BF16) == _native.PATH_GEMM
    wl = workloads.make(T, E, K, I, O, dtype=torch.bfloat16, seed=44)
    out = run_gpu(wl)
    rows = np.arange(0, T, 37)
    want, absm, _ = oracle_rows(wl, rows=rows)
    assert_parity(out[torch.from_numpy(rows).cuda()], want, absm, wl.dtype, "E=600")


def test_gemm_operand_modes_agree(monkeypatch):
    # Scale bytes 118..124 let every tile take the f16 operands; the knob
    # keeps the bf16 operands. Products are exact in both and accumulate in
    # float32: the results agree with the oracle and with each other.
    T, E, K, I, O = 256, 4, 2, 2880, 384
    wl = workloads.make(T, E, K, I, O, dtype=torch.bfloat16, seed=77)
    want, absm, _ = oracle_rows(wl)
    out_f16 = run_gpu(wl)
    monkeypatch.setenv("MXFP4EL_TC_MODE", "bf16")
    out_bf16 = run_gpu(wl)
    torch.cuda.synchronize()
    assert wait_timeouts() == 0
    assert_parity(out_f16, want, absm, wl.dtype, "f16 operands")
    assert_parity(out_bf16, want, absm, wl.dtype, "bf16 operands")
    same = float((out_f16 == out_bf16).float().mean())
    print(f"[gemm modes] identical outputs: {same:.6f}")
    assert same > 0.999


@pytest.mark.parametrize("lo,hi", [(0, 255), (100, 140)])
def test_gemm_wide_scale_spans_take_bf16_tiles(lo, hi):
    # Rows whose scale bytes span more than 26 binades cannot be held exactly
    # by f16 operands: their tiles take the bf16 mode. (0, 255): every tile;
    # (100, 140): some rows span up to 40, most tiles mix both kinds of rows.
    T, E, K, I, O = 96, 3, 2, 256, 260
    wl = workloads.make(T, E, K, I, O, dtype=torch.bfloat16, scale_lo=lo, scale_hi=hi,
                        seed=lo + hi)
    # Keep every result inside the bf16 range (scale bytes up to 170: weights
    # up to 6 * 2^43); the exhaustive scale tests cover the bytes beyond.
    wl.scales.clamp_(2, 170)
    out = run_gpu(wl)
    torch.cuda.synchronize()
    assert wait_timeouts() == 0
    want, absm, _ = oracle_rows(wl)
    assert_parity(out, want, absm, wl.dtype, f"scales {lo}..{hi}")


def test_gemm_mixed_tiles_in_one_call():
    # Expert 0's rows span 116..124 (f16 tiles), expert 1's rows one byte
    # 90 and the rest 124 (bf16 tiles): one launch holds both modes.
    T, E, K, I, O = 160, 2, 1, 512, 256
    wl = workloads.make(T, E, K, I, O, dtype=torch.bfloat16, scale_lo=116, scale_hi=124,
                        seed=5)
    wl.scales[1, :, 0] = 90
    sel = torch.from_numpy((np.arange(T) % 2).reshape(T, 1).astype(np.int32))
    out = run_gpu(wl, sel=sel)
    torch.cuda.synchronize()
    assert wait_timeouts() == 0
    want, absm, _ = oracle_rows(wl, sel=sel)
    assert_parity(out, want, absm, wl.dtype, "mixed tiles")
