"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Tolerance (elementwise): |gpu - oracle| <= tol * abs_terms with
abs_terms = |y_shared| + sum_k sum_i |p w x|; tol = 1e-5 for fp32 tokens and
8e-3 for bf16 tokens and outputs. Integer-valued inputs that keep every
partial sum exact are compared bit for bit.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (TOL, assert_parity, digest, oracle_rows, parity_rows, run_gpu,
                      sample_rows)
from mxfp4_routed_expert_route_gb300 import (_native, device_errors, wait_timeouts,
                                             mxfp4_expert_linear, workloads)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mxfp4_routed_expert_route_gb300 import build
    build.build()
    _native.load()


# ------------------------------------------------------------ named workloads
@pytest.mark.parametrize("name", ["tiny_fp32", "decode", "wide_decode"])
def test_named_workload_full(name):
    wl = workloads.named(name)
    out = run_gpu(wl)
    assert out.shape == (wl.T, wl.O) and out.dtype == wl.dtype and out.is_cuda
    want, absm, bad = oracle_rows(wl)
    assert bad == 0
    assert_parity(out, want, absm, wl.dtype, name)


@pytest.mark.parametrize("name", ["prefill", "skewed_prefill"])
def test_named_workload_sampled(name):
    wl = workloads.named(name)
    out = run_gpu(wl)
    assert torch.isfinite(out.float()).all()
    # At least 256 token rows element by element, including every token of
    # the least-loaded expert and whole token blocks of the most-loaded one.
    rows = parity_rows(wl)
    assert len(rows) >= 256
    want, absm, _ = oracle_rows(wl, rows=rows)
    assert_parity(out[torch.from_numpy(rows).cuda()], want, absm, wl.dtype,
                  f"{name} ({len(rows)} rows)")
    # Token permutation permutes the output rows, bit for bit, at full size.
    perm = torch.from_numpy(np.random.default_rng(1).permutation(wl.T))
    d = wl.device_tensors("cuda")
    pc = perm.cuda()
    out2 = mxfp4_expert_linear(d["x"][pc], d["packed"], d["scales"], d["sel"][pc],
                               d["p"][pc], d["y_shared"][pc])
    assert torch.equal(out2, out[pc])


# ------------------------------------------------ ragged sizes and edge cases
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,E,K,I,O", [(37, 9, 3, 320, 100), (5, 3, 1, 32, 1),
                                       (64, 40, 6, 96, 257), (3, 200, 2, 1024, 33)])
def test_ragged_sizes(dtype, T, E, K, I, O):
    wl = workloads.make(T, E, K, I, O, dtype=dtype, scale_lo=112, scale_hi=140,
                        seed=T * 1000 + O)
    out = run_gpu(wl)
    want, absm, _ = oracle_rows(wl)
    assert_parity(out, want, absm, dtype, f"{T},{E},{K},{I},{O}")


def test_one_expert_takes_every_token():
    # 70 tokens, every slot 0 on expert 2: the expert's token list spans
    # several passes of the kernel.
    wl = workloads.make(70, 5, 2, 192, 48, dtype=torch.bfloat16, seed=5)
    sel = wl.sel.clone()
    sel[:, 0] = 2
    sel[:, 1] = torch.where(sel[:, 1] == 2, torch.full_like(sel[:, 1], 3), sel[:, 1])
    out = run_gpu(wl, sel=sel)
    want, absm, _ = oracle_rows(wl, sel=sel)
    assert_parity(out, want, absm, wl.dtype)


def test_duplicate_picks_are_summed_per_slot():
    wl = workloads.make(6, 4, 3, 64, 20, dtype=torch.float32, seed=6)
    sel = torch.tensor([[1, 1, 2]] * 6, dtype=torch.int32)
    out = run_gpu(wl, sel=sel)
    want, absm, _ = oracle_rows(wl, sel=sel)
    assert_parity(out, want, absm, wl.dtype)


def test_k_zero_returns_shared_output():
    wl = workloads.make(4, 3, 0, 64, 10, dtype=torch.bfloat16, seed=7)
    out = run_gpu(wl)
    assert torch.equal(out.cpu(), wl.y_shared)


def test_zero_weights_return_shared_output_bits():
    wl = workloads.make(9, 6, 2, 128, 40, dtype=torch.bfloat16, seed=8)
    wl.p.zero_()
    out = run_gpu(wl)
    assert torch.equal(out.cpu(), wl.y_shared)


def test_t_zero_is_a_no_op():
    wl = workloads.make(0, 3, 2, 64, 10, dtype=torch.bfloat16, seed=9)
    out = run_gpu(wl)
    assert out.shape == (0, 10)


def test_invalid_ids_are_skipped_and_counted():
    wl = workloads.make(8, 5, 2, 64, 16, dtype=torch.float32, seed=10)
    device_errors()                                    # reset the counter
    sel = wl.sel.clone()
    sel[1, 0] = 5
    sel[6, 1] = -3
    out = run_gpu(wl, sel=sel)
    assert device_errors() == 2
    want, absm, bad = oracle_rows(wl, sel=sel)
    assert bad == 2
    assert_parity(out, want, absm, wl.dtype)


def test_no_experts_at_all():
    wl = workloads.make(3, 1, 2, 32, 4, dtype=torch.float32, seed=11)
    device_errors()
    sel = torch.full((3, 2), 7, dtype=torch.int32)
    out = run_gpu(wl, sel=sel)
    assert device_errors() == 6
    assert torch.equal(out.cpu(), wl.y_shared)


@pytest.mark.parametrize("T,K,dtype", [(64, 2, torch.bfloat16), (4200, 2, torch.bfloat16),
                                       (5, 3, torch.float32)])
def test_zero_experts_counts_every_id(T, K, dtype):
    # E == 0: every id is out of range; the call returns the shared output
    # and counts every pair, on every path the sizes would otherwise pick.
    wl = workloads.make(T, 1, K, 64, 24, dtype=dtype, seed=13)
    d = wl.device_tensors("cuda")
    device_errors()
    sel = torch.randint(-3, 5, (T, K), dtype=torch.int64, device="cuda")
    out = mxfp4_expert_linear(d["x"], d["packed"][:0], d["scales"][:0], sel, d["p"],
                              d["y_shared"])
    assert torch.equal(out.cpu(), wl.y_shared)
    assert device_errors() == T * K


def test_int64_ids_match_int32():
    wl = workloads.make(11, 7, 3, 96, 30, dtype=torch.bfloat16, seed=12)
    a = run_gpu(wl)
    b = run_gpu(wl, sel=wl.sel.to(torch.int64))
    assert torch.equal(a, b)


# ------------------------------------------------------------- exactness ----
def test_every_code_and_scale_exact_fp32():
    # Rows o = 0..253 use scale byte s = o + 1; the group's 32 positions hold
    # the 16 codes twice, once from low nibbles and once from high nibbles.
    O, I = 254, 32
    codes = np.arange(32) % 16
    codes = np.concatenate([codes[:16], codes[:16][::-1]])          # 32 codes
    bytes_ = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)      # 16 bytes
    packed = np.broadcast_to(bytes_, (1, O, 1, 16)).copy()
    scales = (np.arange(O) + 1).astype(np.uint8).reshape(1, O, 1)
    T = 32
    x = torch.eye(T, I, dtype=torch.float32)                          # token t = e_t
    sel = torch.zeros((T, 1), dtype=torch.int32)
    p = torch.ones((T, 1), dtype=torch.float32)
    ys = torch.zeros((T, O), dtype=torch.float32)
    out = mxfp4_expert_linear(x.cuda(), torch.from_numpy(packed).cuda(),
                              torch.from_numpy(scales).cuda(), sel.cuda(), p.cuda(),
                              ys.cuda())
    want, _, _ = oracle.expert_linear(x, packed, scales, sel, p, ys)
    got = out.cpu().double().numpy()
    finite = np.abs(want) <= np.finfo(np.float32).max
    assert np.array_equal(got[finite], want[finite])


def test_scale_byte_zero_and_255_fp32():
    # s = 0 is 2^-127 (subnormal factor); s = 255 is 2^128, exact for code 1.
    packed = np.zeros((1, 2, 1, 16), dtype=np.uint8)
    packed[0, :, 0, 0] = 0x71          # codes 1 (0.5) and 7 (6.0)
    scales = np.array([[[0], [255]]], dtype=np.uint8)
    x = torch.zeros((1, 32), dtype=torch.float32)
    x[0, 0] = 1.0                       # picks the low-nibble code 1 -> 0.5
    out = mxfp4_expert_linear(x.cuda(), torch.from_numpy(packed).cuda(),
                              torch.from_numpy(scales).cuda(),
                              torch.zeros((1, 1), dtype=torch.int32).cuda(),
                              torch.ones((1, 1)).cuda(), torch.zeros((1, 2)).cuda())
    got = out.cpu().double().numpy()[0]
    assert got[0] == 2.0 ** -128 and got[1] == 2.0 ** 127


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_every_scale_byte_exact(dtype):
    # Output row r uses scale byte r for its one group of codes 1.0, and the
    # token is all ones: the row is 32 * 2^(r - 127) = 2^(r - 122), exact in
    # float32 (bf16 holds every power of two in range too) and +inf past the
    # largest finite value.
    O = 256
    packed = np.full((1, O, 1, 16), 0x22, dtype=np.uint8)
    scales = np.arange(O, dtype=np.uint8).reshape(1, O, 1)
    x = torch.ones((1, 32), dtype=dtype)
    out = mxfp4_expert_linear(x.cuda(), torch.from_numpy(packed).cuda(),
                              torch.from_numpy(scales).cuda(),
                              torch.zeros((1, 1), dtype=torch.int32).cuda(),
                              torch.ones((1, 1)).cuda(), torch.zeros((1, O), dtype=dtype).cuda())
    got = out.float().cpu().double().numpy()[0]
    want, _, _ = oracle.expert_linear(x.double().numpy(), packed, scales,
                                      np.zeros((1, 1), dtype=np.int64), np.ones((1, 1)),
                                      np.zeros((1, O)))
    want = want[0]
    fmax = float(torch.finfo(dtype).max)
    finite = np.abs(want) <= fmax
    assert np.array_equal(got[finite], want[finite])
    assert np.all(np.isinf(got[~finite]) & (got[~finite] > 0))
    assert finite[:250].all() and not finite[250:].any()


def test_extreme_token_magnitudes_bf16():
    # bf16 tokens of magnitude 2^m (m from -120 to 100) against every scale
    # byte: the GEMV pre-scales each token by its own power of two into f16,
    # so weight scale and token scale meet in one factor 2^(s-127-sigma)
    # that spans 2^-253 .. 2^247. Elements whose terms stay within float32
    # range match the oracle to the bf16 tolerance; those past it are not
    # finite (inf, or NaN where terms of both signs overflow).
    rng = np.random.default_rng(21)
    T, E, K, I, O = 8, 3, 2, 64, 96
    wl = workloads.make(T, E, K, I, O, dtype=torch.bfloat16, scale_lo=0, scale_hi=255, seed=21)
    mags = torch.tensor([-120, -100, -30, 0, 30, 60, 90, 100], dtype=torch.float32)
    wl.x = (wl.x.float() * torch.exp2(mags)[:, None]).to(torch.bfloat16)
    wl.y_shared = torch.zeros((T, O), dtype=torch.bfloat16)
    out = run_gpu(wl).float().cpu().double().numpy()
    want, absm, _ = oracle_rows(wl)
    fmax = float(torch.finfo(torch.float32).max)
    inside = (absm >= 2.0 ** -100) & (absm <= fmax / 4)
    assert inside.sum() > T * O // 4
    err = np.abs(out[inside] - want[inside])
    assert np.all(err <= TOL[torch.bfloat16] * absm[inside])
    over = np.abs(want) >= 2 * fmax
    assert over.any()
    assert not np.isfinite(out[over]).any()
    assert not np.isnan(out[absm <= fmax / 4]).any()


def test_integer_inputs_exact_bf16():
    rng = np.random.default_rng(13)
    T, E, K, I, O = 16, 3, 1, 256, 64
    wl = workloads.make(T, E, K, I, O, dtype=torch.bfloat16, scale_lo=127,
                        scale_hi=127, seed=13)
    wl.x = torch.from_numpy(rng.integers(-8, 9, (T, I)).astype(np.float32)).to(torch.bfloat16)
    wl.y_shared = torch.zeros((T, O), dtype=torch.bfloat16)
    wl.p = torch.ones((T, K), dtype=torch.float32)
    out = run_gpu(wl)
    want, _, _ = oracle_rows(wl)
    want_bf16 = torch.from_numpy(want).to(torch.bfloat16)
    assert torch.equal(out.cpu(), want_bf16)


# ------------------------------------------------------------- properties ---
def test_inputs_not_mutated_and_deterministic():
    wl = workloads.make(33, 12, 4, 160, 70, dtype=torch.bfloat16, seed=14)
    d = wl.device_tensors("cuda")
    before = digest(*d.values())
    a = mxfp4_expert_linear(d["x"], d["packed"], d["scales"], d["sel"], d["p"], d["y_shared"])
    b = mxfp4_expert_linear(d["x"], d["packed"], d["scales"], d["sel"], d["p"], d["y_shared"])
    torch.cuda.synchronize()
    assert digest(*d.values()) == before
    assert torch.equal(a, b)


def test_unselected_experts_are_never_read():
    wl = workloads.make(10, 8, 2, 128, 24, dtype=torch.bfloat16, seed=15)
    sel = torch.tensor([[0, 3]] * 10, dtype=torch.int32)
    a = run_gpu(wl, sel=sel)
    rng = np.random.default_rng(16)
    for e in (1, 2, 4, 5, 6, 7):
        wl.packed[e] = torch.from_numpy(rng.integers(0, 256, wl.packed[e].shape, dtype=np.uint8))
        wl.scales[e] = torch.from_numpy(rng.integers(0, 256, wl.scales[e].shape, dtype=np.uint8))
    b = run_gpu(wl, sel=sel)
    assert torch.equal(a, b)


def test_library_owned_workspace_entry_point():
    wl = workloads.make(21, 9, 3, 224, 90, dtype=torch.bfloat16, seed=17)
    d = wl.device_tensors("cuda")
    ref = mxfp4_expert_linear(d["x"], d["packed"], d["scales"], d["sel"], d["p"], d["y_shared"])
    out = torch.empty_like(ref)
    lib = _native.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    for _ in range(2):
        rc = lib.mxfp4_expert_linear(ptr(d["x"]), ptr(d["packed"]), ptr(d["scales"]),
                                     ptr(d["sel"]), ptr(d["p"]), ptr(d["y_shared"]),
                                     ptr(out), wl.T, wl.E, wl.I, wl.O, wl.K,
                                     _native.DTYPE_BF16, _native.INDEX_I32, stream)
        assert rc == _native.OK
        torch.cuda.synchronize()
        assert torch.equal(out, ref)


def test_alias_is_refused():
    wl = workloads.make(4, 3, 2, 64, 8, dtype=torch.float32, seed=18)
    d = wl.device_tensors("cuda")
    with pytest.raises(_native.MXFP4Error):
        mxfp4_expert_linear(d["x"], d["packed"], d["scales"], d["sel"], d["p"],
                            d["y_shared"], out=d["y_shared"])


# ------------------------------------------------ kernel variants, numerics --
def test_rows_too_wide_for_a_stage_use_the_direct_kernel():
    # I = 16384 (512 groups): one row per warp no longer fits a shared-memory
    # stage, so the unstaged GEMV runs.
    for dtype in (torch.bfloat16, torch.float32):
        wl = workloads.make(3, 4, 2, 16384, 40, dtype=dtype, seed=19)
        out = run_gpu(wl)
        want, absm, _ = oracle_rows(wl)
        assert_parity(out, want, absm, dtype, str(dtype))


@pytest.mark.parametrize("seed", [20, 21])
def test_bf16_tokens_with_extreme_dynamic_range(seed):
    # Per-token magnitudes from 2^-60 to 2^60 and per-element spread of 2^+-12
    # stress the per-token power-of-two scaling and the f16 product chains.
    rng = np.random.default_rng(seed)
    T, E, K, I, O = 12, 6, 3, 640, 96
    wl = workloads.make(T, E, K, I, O, dtype=torch.bfloat16, scale_lo=100,
                        scale_hi=150, seed=seed)
    tok_scale = np.ldexp(1.0, rng.integers(-60, 61, size=(T, 1)))
    elem = np.ldexp(rng.standard_normal((T, I)), rng.integers(-12, 13, size=(T, I)))
    wl.x = torch.from_numpy((elem * tok_scale).astype(np.float32)).to(torch.bfloat16)
    out = run_gpu(wl)
    want, absm, _ = oracle_rows(wl)
    assert_parity(out, want, absm, wl.dtype)


def test_no_kernel_wait_timed_out():
    from mxfp4_routed_expert_route_gb300 import wait_timeouts
    wl = workloads.make(9, 10, 3, 288, 130, dtype=torch.bfloat16, seed=22)
    run_gpu(wl)
    assert wait_timeouts() == 0


@pytest.mark.parametrize("T,E,K,I,O", [
    (24, 6, 3, 256, 64),      # GEMV partials, several columns
    (4096, 8, 4, 256, 512),   # tensor-core partials, many segments per warp
])
def test_combine_vector_and_scalar_paths_agree_bitwise(T, E, K, I, O):
    # The combine has 16-byte vector paths (width a multiple of 4, aligned
    # buffers) and an elementwise path. A shared-output view that starts one
    # element into its storage is misaligned and takes the elementwise path;
    # all evaluate the same expression in the same order.
    wl = workloads.make(T, E, K, I, O, dtype=torch.bfloat16, seed=41)
    d = wl.device_tensors("cuda")
    a = mxfp4_expert_linear(d["x"], d["packed"], d["scales"], d["sel"], d["p"], d["y_shared"])
    store = torch.empty(wl.T * wl.O + 1, dtype=torch.bfloat16, device="cuda")
    ys_off = store[1:].view(wl.T, wl.O)
    ys_off.copy_(d["y_shared"])
    assert ys_off.data_ptr() % 16 != 0
    b = mxfp4_expert_linear(d["x"], d["packed"], d["scales"], d["sel"], d["p"], ys_off)
    assert torch.equal(a, b)


def test_many_pairs_gemv_path_with_invalid_ids():
    # 9600 (token, slot) pairs: the bucketer runs as several CTAs (count,
    # scan, scatter) and writes the GEMV's cost-balanced CTA ranges; fp32
    # tokens keep the GEMV path. Two out-of-range ids are skipped and counted.
    wl = workloads.make(2400, 48, 4, 96, 72, dtype=torch.float32, seed=42)
    sel = wl.sel.clone()
    sel[17, 2] = 48
    sel[2399, 0] = -1
    device_errors()                                    # reset the counter
    out = run_gpu(wl, sel=sel)
    assert device_errors() == 2
    assert wait_timeouts() == 0
    rows = sample_rows(wl, 64, seed=3)
    rows = np.union1d(rows, [17, 2399])
    want, absm, bad = oracle_rows(wl, rows=rows, sel=sel)
    assert_parity(out[torch.from_numpy(rows).cuda()], want, absm, wl.dtype, "9600 pairs")


@pytest.mark.parametrize("dtype,idx", [(torch.bfloat16, torch.int32), (torch.float32, torch.int64)])
def test_self_routed_gemv_matches_bucketer_bitwise(monkeypatch, dtype, idx):
    # Small batches on the GEMV route inside the GEMV's own CTAs; the
    # bucketer path computes the same lists, split and token scales, so the
    # two give the same bits. Some ids are out of range.
    wl = workloads.make(24, 40, 5, 320, 150, dtype=dtype, seed=43)
    sel = wl.sel.clone().to(idx)
    sel[3, 1] = 40
    sel[20, 4] = -2
    device_errors()
    a = run_gpu(wl, sel=sel)
    assert device_errors() == 2
    monkeypatch.setenv("MXFP4EL_ROUTE", "bucketer")
    b = run_gpu(wl, sel=sel)
    assert device_errors() == 2
    assert torch.equal(a, b)
    want, absm, _ = oracle_rows(wl, sel=sel)
    assert_parity(a, want, absm, dtype, "self-routed")


@pytest.mark.parametrize("name", ["decode", "wide_decode", "prefill"])
def test_poisoned_workspace(name):
    # A caller workspace full of 0xFF bytes: the GEMV's pool counter reads -1
    # and every partial result NaN until written. The results must not
    # depend on it: every unit is claimed and every partial written, on
    # repeated calls.
    from mxfp4_routed_expert_route_gb300 import workspace_size
    wl = workloads.named(name)
    d = wl.device_tensors("cuda")
    n = workspace_size(wl.T, wl.E, wl.I, wl.O, wl.K, wl.dtype)
    rows = np.array([0, wl.T // 3, wl.T - 1])
    want, absm, _ = oracle_rows(wl, rows=rows)
    r = torch.from_numpy(rows).cuda()
    for _ in range(3):
        ws = torch.full((max(n, 1),), 0xFF, dtype=torch.uint8, device="cuda")
        out = mxfp4_expert_linear(d["x"], d["packed"], d["scales"], d["sel"], d["p"],
                                  d["y_shared"], workspace=ws)
        torch.cuda.synchronize()
        assert wait_timeouts() == 0
        assert torch.isfinite(out.float()).all()
        assert_parity(out[r], want, absm, wl.dtype, f"{name}, poisoned workspace")
