"""GPU parity of the routed MXFP4 SwiGLU expert against the float64 oracle.

Tolerance (elementwise, derived from the arithmetic in oracle/swiglu.py):
|gpu - oracle| <= tolerance(terms, tau, tau1, rho), each projection's bound
relative to its sum of |terms| and taken from the kernel that runs it:
  * fp32 tokens (GEMV, exact products, float32 sums): 1e-5;
  * bf16 tokens on the GEMV: 8 * 2^-11 per group (two f16x2 chains of 8
    products added in f16) plus G * 2^-24 for the float32 sum of the groups;
  * bf16 tokens on the tensor cores: exact products summed in float32,
    width * 2^-24;
tau (the down projection) also carries the combine's (K + 1) * 2^-24, rho is
the relative error of h = silu(g) u evaluated in float32 and rounded to the
token dtype (2^-20 fp32; 2^-9 + 2^-20 bf16), and the output's own rounding
to the token dtype adds OUT_ROUND |out| (half an ulp: 2^-8 bf16, 2^-24 fp32).

Such a bound holds for every element. Where the tensor cores run both
projections the roundings of h and of the output dominate it, and it came
within 1.2 to 3 times the error at the worst element (max err/bound 0.34 to
0.84 over the gate/up-tile cases). Where the GEMV runs, its f16 chains' bound
sums |terms|, which for F terms of mixed sign lies about sqrt(F) above the
error random-signed roundings produce, whatever the constant in front: there
it came out 25 to 750 times the error. The ratio is printed for every case.
The bf16 cases are also checked by
  * an exact case: integer-valued tokens and weights that keep every gate/up
    partial sum exact, and a down matrix that copies h to the output, so the
    output is h rounded to bf16: equal to the oracle's h rounded to bf16 but
    for values within a few float32 ulps of a rounding midpoint;
  * the relative RMS error over all outputs, at most 1e-2 (the expected
    value from bf16 rounding of h and of the output is near 1e-3).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle.swiglu as osw
from mxfp4_routed_expert_route_gb300 import (_native, device_errors, mxfp4_swiglu_expert,
                                             swiglu_workspace_size, workloads)

pytestmark = pytest.mark.gpu

RHO = {torch.float32: 2.0 ** -20, torch.bfloat16: 2.0 ** -9 + 2.0 ** -20}
OUT_ROUND = {torch.float32: 2.0 ** -24, torch.bfloat16: 2.0 ** -8}
RMS_BF16 = 1e-2


def linear_tau(T, E, I, O, K, dtype):
    """Error bound of one routed projection, relative to its sum of |terms|,
    for the kernel the library runs at these sizes."""
    if dtype == torch.float32:
        return 1e-5
    lib = _native.load()
    gemm = lib.mxfp4el_linear_path(T, E, I, O, K, _native.DTYPE_BF16) == _native.PATH_GEMM
    return I * 2.0 ** -24 if gemm else 8 * 2.0 ** -11 + (I // 32) * 2.0 ** -24


def taus(wl):
    """(tau for the down projection and combine, tau1 for gate/up)."""
    P = wl.T * wl.K
    tau1 = linear_tau(wl.T, wl.E, wl.I, 2 * wl.F, wl.K, wl.dtype)
    tau = linear_tau(P, wl.E, wl.F, wl.O, 1, wl.dtype) + (wl.K + 1) * 2.0 ** -24
    return tau, tau1


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mxfp4_routed_expert_route_gb300 import build
    build.build()
    _native.load()


def run(wl, **kw):
    d = wl.device_tensors("cuda")
    return mxfp4_swiglu_expert(d["x"], d["gate_up_packed"], d["gate_up_scales"],
                               d["down_packed"], d["down_scales"], d["sel"], d["p"],
                               d["y_shared"], **kw)


def check(out_rows, wl, rows=None, what=""):
    r = osw.swiglu_expert(*wl.args(), rows=rows)
    got = out_rows.detach().cpu().double().numpy()
    assert np.all(np.isfinite(got)), what
    tau, tau1 = taus(wl)
    bound = osw.tolerance(r, tau, tau1, RHO[wl.dtype])
    bound = bound + OUT_ROUND[wl.dtype] * (np.abs(r["out"]) + bound)
    err = np.abs(got - r["out"])
    ratio = float(np.max(err / np.maximum(bound, np.finfo(np.float64).tiny)))
    rms = float(np.sqrt(np.mean(err ** 2)) / max(np.sqrt(np.mean(r["out"] ** 2)), 1e-300))
    print(f"[swiglu parity] {what}: tau1 {tau1:.2e}, tau {tau:.2e}: max err/bound = "
          f"{ratio:.3e} (the bound {1.0 / max(ratio, 1e-300):.0f}x the error there), "
          f"relative RMS = {rms:.3e}")
    assert ratio <= 1.0, f"{what}: max err/bound = {ratio:.3e}"
    if wl.dtype == torch.bfloat16:
        assert rms <= RMS_BF16, f"{what}: relative RMS error {rms:.3e}"
    return r


# ------------------------------------------------------------ named shapes --
@pytest.mark.parametrize("name", ["swiglu_tiny_fp32", "swiglu_decode"])
def test_named_full(name):
    wl = workloads.named_swiglu(name)
    out = run(wl)
    assert out.shape == (wl.T, wl.O) and out.dtype == wl.dtype
    r = check(out, wl, what=name)
    assert r["bad"] == 0


def test_decode_shape_fp32_tokens():
    wl = workloads.make_swiglu(T=8, E=128, K=4, I=2880, F=2880, O=2880, dtype=torch.float32,
                               seed=21, name="decode_fp32")
    check(run(wl), wl, what="decode shape, fp32 tokens")


def test_prefill_sampled_and_deterministic():
    wl = workloads.named_swiglu("swiglu_prefill")
    out = run(wl)
    rows = np.array(sorted({0, wl.T - 1, *np.random.default_rng(0).integers(0, wl.T, 10)}))
    check(out[torch.from_numpy(rows).cuda()], wl, rows=rows, what="swiglu_prefill sampled")
    assert torch.equal(run(wl), out)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,E,K,I,F,O", [(37, 9, 3, 320, 96, 100), (5, 3, 1, 32, 32, 1),
                                         (300, 6, 2, 256, 128, 192)])
def test_ragged_shapes(dtype, T, E, K, I, F, O):
    wl = workloads.make_swiglu(T=T, E=E, K=K, I=I, F=F, O=O, dtype=dtype, seed=T + F,
                               scale_lo=120, scale_hi=126)
    check(run(wl), wl, what=f"T={T} E={E} K={K} I={I} F={F} O={O} {dtype}")


# ------------------------------------------------ exact intermediate values --
def _exact_case(dtype, T=24, E=3, I=64, F=64, seed=5):
    """Integer tokens in [-4, 4] (max |x| = 4 per token) and gate/up weights
    in {0, +-0.5, +-1} x 1/8: every gate/up partial sum is exact in the
    kernels. Down: the identity (one 1.0 per row), K = 1, p = 1, no shared
    output, so out[t] = h of the token's pair, rounded to the token dtype."""
    rng = np.random.default_rng(seed)
    codes = rng.choice([0, 1, 2, 9, 10], size=(E, 2 * F, I))
    gu = np.zeros((E, 2 * F, I // 32, 16), dtype=np.uint8)
    for i in range(I):
        g, within = divmod(i, 32)
        j, high = divmod(within, 2)
        gu[:, :, g, j] |= (codes[:, :, i].astype(np.uint8) << (4 * high))
    gus = np.full((E, 2 * F, I // 32), 124, dtype=np.uint8)
    dn = np.zeros((E, F, F // 32, 16), dtype=np.uint8)
    for o in range(F):
        g, within = divmod(o, 32)
        dn[:, o, g, within // 2] = 0x02 if within % 2 == 0 else 0x20
    dns = np.full((E, F, F // 32), 127, dtype=np.uint8)
    x = rng.integers(-4, 5, size=(T, I)).astype(np.float32)
    x[:, 0] = 4.0
    sel = rng.integers(0, E, size=(T, 1)).astype(np.int32)
    return workloads.SwigluWorkload(
        name="exact", T=T, E=E, K=1, I=I, F=F, O=F, dtype=dtype,
        x=torch.from_numpy(x).to(dtype), gate_up_packed=torch.from_numpy(gu),
        gate_up_scales=torch.from_numpy(gus), down_packed=torch.from_numpy(dn),
        down_scales=torch.from_numpy(dns), sel=torch.from_numpy(sel),
        p=torch.ones((T, 1), dtype=torch.float32), y_shared=torch.zeros((T, F), dtype=dtype))


def test_exact_h_fp32():
    wl = _exact_case(torch.float32)
    out = run(wl).double().cpu().numpy()
    h = osw.swiglu_expert(*wl.args())["h"]
    assert np.all(np.abs(out - h) <= 2.0 ** -20 * np.abs(h)), np.max(np.abs(out - h))


def test_exact_h_bf16():
    wl = _exact_case(torch.bfloat16)
    out = run(wl).float().cpu()
    h = osw.swiglu_expert(*wl.args())["h"]
    h32 = torch.from_numpy(h.astype(np.float32))
    want = h32.to(torch.bfloat16).float()
    diff = (out != want).nonzero()
    # A mismatch is allowed only next to a rounding midpoint: the two values
    # are adjacent bf16 numbers and h lies within 2^-18 (relative) of the
    # point halfway between them.
    for t, f in diff.tolist():
        a, b = float(out[t, f]), float(want[t, f])
        mid = (a + b) / 2.0
        assert abs(a - b) <= 2.0 ** -7 * max(abs(a), abs(b)), (t, f, a, b)
        assert abs(h[t, f] - mid) <= 2.0 ** -18 * abs(mid), (t, f, a, b, h[t, f])
    assert len(diff) <= max(2, out.numel() // 1000)


# ------------------------------------------------------------- edge cases --
def test_invalid_ids_counted_once():
    wl = workloads.make_swiglu(T=6, E=5, K=3, I=64, F=64, O=40, dtype=torch.float32, seed=3)
    device_errors()
    sel = wl.sel.clone()
    sel[0, 1] = -1
    sel[2, 0] = 5
    sel[5, 2] = 1 << 20
    wl.sel = sel
    out = run(wl)
    assert device_errors() == 3
    r = check(out, wl, what="invalid ids")
    assert r["bad"] == 3


def test_k_zero_and_no_experts():
    wl = workloads.make_swiglu(T=4, E=3, K=0, I=32, F=32, O=16, dtype=torch.bfloat16, seed=1)
    out = run(wl)
    assert torch.equal(out.cpu(), wl.y_shared)
    wl = workloads.make_swiglu(T=4, E=3, K=2, I=32, F=32, O=16, dtype=torch.float32, seed=2)
    d = wl.device_tensors("cuda")
    device_errors()
    empty = torch.empty((0, 2 * 32, 1, 16), dtype=torch.uint8, device="cuda")
    out = mxfp4_swiglu_expert(d["x"], empty, torch.empty((0, 64, 1), dtype=torch.uint8,
                                                          device="cuda"),
                              torch.empty((0, 16, 1, 16), dtype=torch.uint8, device="cuda"),
                              torch.empty((0, 16, 1), dtype=torch.uint8, device="cuda"),
                              d["sel"], d["p"], d["y_shared"])
    assert torch.equal(out.cpu(), wl.y_shared)
    assert device_errors() == 8


def test_t_zero():
    wl = workloads.make_swiglu(T=0, E=3, K=2, I=32, F=32, O=16, dtype=torch.bfloat16, seed=1)
    out = run(wl)
    assert out.shape == (0, 16)


def test_int64_ids_and_entry_points_agree():
    wl = workloads.make_swiglu(T=24, E=16, K=4, I=256, F=128, O=96, dtype=torch.bfloat16,
                               seed=9)
    base = run(wl)
    d = wl.device_tensors("cuda")
    d["sel"] = d["sel"].long()
    assert torch.equal(mxfp4_swiglu_expert(*[d[k] for k in wl.ARGS]), base)
    # The library-owned-scratch entry point, through the C ABI.
    d = wl.device_tensors("cuda")
    out = torch.empty_like(base)
    lib = _native.load()
    stream = torch.cuda.current_stream().cuda_stream
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.mxfp4_swiglu_expert(ptr(d["x"]), ptr(d["gate_up_packed"]),
                                 ptr(d["gate_up_scales"]), ptr(d["down_packed"]),
                                 ptr(d["down_scales"]), ptr(d["sel"]), ptr(d["p"]),
                                 ptr(d["y_shared"]), ptr(out), wl.T, wl.E, wl.I, wl.F, wl.O,
                                 wl.K, _native.DTYPE_BF16, _native.INDEX_I32,
                                 ctypes.c_void_p(stream))
    assert rc == 0
    assert torch.equal(out, base)


@pytest.mark.parametrize("name", ["swiglu_decode", "swiglu_tiny_fp32"])
def test_poisoned_workspace(name):
    wl = workloads.named_swiglu(name)
    base = run(wl)
    n = swiglu_workspace_size(wl.T, wl.E, wl.I, wl.F, wl.O, wl.K, wl.dtype)
    for fill in (0x00, 0xFF, 0x7F):
        ws = torch.full((n,), fill, dtype=torch.uint8, device="cuda")
        assert torch.equal(run(wl, workspace=ws), base), fill


def test_alias_and_shape_checks():
    wl = workloads.make_swiglu(T=4, E=3, K=2, I=32, F=32, O=16, dtype=torch.float32, seed=4)
    d = wl.device_tensors("cuda")
    with pytest.raises(_native.MXFP4Error):
        mxfp4_swiglu_expert(*[d[k] for k in wl.ARGS], out=d["y_shared"])


# ------------------------------------------------ gate/up tiles (prefill) --
@pytest.mark.parametrize("T,E,K,I,F,O,bad,i64", [(300, 6, 2, 256, 128, 192, False, False),
                                                 (257, 5, 3, 64, 96, 80, False, True),
                                                 (1000, 16, 4, 320, 160, 128, False, False),
                                                 (400, 7, 2, 128, 64, 64, True, False)])
def test_gate_up_tiles_match_separate_swiglu(monkeypatch, T, E, K, I, F, O, bad, i64):
    # On the tensor cores the gate/up kernel forms h in tiles of 64 gate rows
    # and their 64 up rows (partial tiles when F is not a multiple of 64); the
    # separate SwiGLU kernel (MXFP4EL_SWIGLU_TILES=0) reads the partial
    # results instead. Same arithmetic, so the same bits.
    wl = workloads.make_swiglu(T=T, E=E, K=K, I=I, F=F, O=O, dtype=torch.bfloat16,
                               seed=T + F, scale_lo=120, scale_hi=126)
    if bad:
        sel = wl.sel.clone()
        sel[3, 0] = -1
        sel[10, 1] = E
        sel[T - 1, 0] = 1 << 20
        wl.sel = sel
    if i64:
        wl.sel = wl.sel.long()
    device_errors()
    out = run(wl)
    n_bad = device_errors()
    monkeypatch.setenv("MXFP4EL_SWIGLU_TILES", "0")
    ref = run(wl)
    assert device_errors() == n_bad == (3 if bad else 0)
    assert torch.equal(out, ref)
    rows = np.array(sorted({0, 3, 10, T - 1, *np.random.default_rng(T).integers(0, T, 8)}))
    r = check(out[torch.from_numpy(rows).cuda()], wl, rows=rows, what=f"tiles T={T} F={F}")
    assert r["bad"] == (3 if bad else 0)
