"""The C-ABI library: loads, exports what include/*.h declares, host checks.

These run without a GPU: only calls that return before any CUDA work
(argument checks, sizes, status strings) are made.
"""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M):
            if not m.group(0).lstrip().startswith(("#", "typedef")):
                names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from mxfp4_routed_expert_route_gb300 import _native, build
    build.build()
    return _native.load()


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert {"mxfp4_expert_linear", "mxfp4_expert_linear_with_workspace",
            "mxfp4_expert_linear_workspace_size"} <= declared
    for name in declared:
        assert hasattr(lib, name), name


def test_binding_covers_header(lib):
    from mxfp4_routed_expert_route_gb300 import _native
    assert _declared_functions() == set(_native.SIGNATURES)


def test_status_strings(lib):
    from mxfp4_routed_expert_route_gb300 import _native as n
    for code in (n.OK, n.ERR_INVALID_ARGUMENT, n.ERR_UNSUPPORTED_DTYPE, n.ERR_ALIAS,
                 n.ERR_WORKSPACE, n.ERR_CUDA, n.ERR_TOO_LARGE):
        assert lib.mxfp4el_status_string(code) not in (None, b"unknown status")
    assert lib.mxfp4el_status_string(12345) == b"unknown status"
    assert lib.mxfp4el_version() >= 100


def test_header_constants_match_binding():
    from mxfp4_routed_expert_route_gb300 import _native as n
    text = open(os.path.join(ROOT, "include", "mxfp4_expert_linear.h")).read()
    defs = dict(re.findall(r"#define\s+MXFP4EL_(\w+)\s+(-?\d+)", text))
    for name, val in defs.items():
        assert getattr(n, name) == int(val), name


def test_workspace_size(lib):
    ws = lib.mxfp4_expert_linear_workspace_size
    bad = ctypes.c_size_t(-1).value
    assert ws(0, 4, 64, 8, 2, 0) == 0
    assert ws(4, 4, 64, 0, 2, 0) == 0
    assert ws(4, 4, 60, 8, 2, 0) == bad            # I not a multiple of 32
    assert ws(4, 4, 64, 8, 2, 7) == bad            # unknown dtype
    assert ws(-1, 4, 64, 8, 2, 0) == bad
    assert ws(1 << 40, 4, 64, 8, 2, 0) == bad       # too large
    n = ws(8, 128, 2880, 5760, 4, 1)
    assert n >= 8 * 4 * 5760 * 4 and n % 256 == 0
    # decode-size batches route and scale the tokens inside the GEMV: no
    # f16 copy of the tokens, so bf16 and fp32 tokens need the same scratch
    assert n == ws(8, 128, 2880, 5760, 4, 0)
    # larger GEMV batches keep a power-of-two scaled f16 copy of the tokens
    m = ws(400, 128, 2880, 5760, 4, 1)
    assert m >= ws(400, 128, 2880, 5760, 4, 0) + 400 * 2880 * 2


def test_argument_checks_return_before_gpu_work(lib):
    from mxfp4_routed_expert_route_gb300 import _native as n
    f = lib.mxfp4_expert_linear
    fake = ctypes.c_void_p(1 << 20)
    args = [fake] * 7
    assert f(*args, 4, 4, 60, 8, 2, 0, 0, None) == n.ERR_INVALID_ARGUMENT
    assert f(*args, 4, 4, 64, 8, 2, 9, 0, None) == n.ERR_UNSUPPORTED_DTYPE
    assert f(*args, 4, 4, 64, 8, 2, 0, 5, None) == n.ERR_UNSUPPORTED_DTYPE
    assert f(*args, -4, 4, 64, 8, 2, 0, 0, None) == n.ERR_INVALID_ARGUMENT
    assert f(*args, 0, 4, 64, 8, 2, 0, 0, None) == n.OK            # T == 0: no-op
    assert f(*args, 4, 4, 64, 0, 2, 0, 0, None) == n.OK            # O == 0: no-op
    nulls = [None] * 7
    assert f(*nulls, 4, 4, 64, 8, 2, 0, 0, None) == n.ERR_INVALID_ARGUMENT
    # out aliasing the shared output is refused
    x = ctypes.c_void_p(1 << 24)
    w = ctypes.c_void_p(1 << 28)
    ys = ctypes.c_void_p(1 << 32)
    assert f(x, w, fake, fake, fake, ys, ys, 4, 4, 64, 8, 2, 0, 0, None) == n.ERR_ALIAS
    # misaligned token pointer
    assert f(ctypes.c_void_p((1 << 24) + 4), w, fake, fake, fake, ys,
             ctypes.c_void_p(1 << 36), 4, 4, 64, 8, 2, 0, 0, None) == n.ERR_INVALID_ARGUMENT
    g = lib.mxfp4_expert_linear_with_workspace
    out = ctypes.c_void_p(1 << 36)
    assert g(x, w, fake, fake, fake, ys, out, 4, 4, 64, 8, 2, 0, 0, None, 0,
             None) == n.ERR_WORKSPACE
    assert g(x, w, fake, fake, fake, ys, out, 4, 4, 64, 8, 2, 0, 0,
             ctypes.c_void_p((1 << 40) + 16), 1 << 20, None) == n.ERR_WORKSPACE


def test_product_path_has_no_oracle_reference():
    pkg = os.path.join(ROOT, "mxfp4_routed_expert_route_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text, f


def test_linear_path_choice(lib):
    # Tensor cores for bf16 tokens once experts average 16 tokens (and the
    # shapes fit the kernel), the GEMV otherwise; no GPU needed to ask.
    from mxfp4_routed_expert_route_gb300 import _native as n
    path = lib.mxfp4el_linear_path
    assert path(8, 128, 2880, 5760, 4, n.DTYPE_BF16) == n.PATH_GEMV        # decode
    assert path(4096, 128, 2880, 5760, 4, n.DTYPE_BF16) == n.PATH_GEMM     # prefill
    assert path(4096, 128, 2880, 5760, 4, n.DTYPE_F32) == n.PATH_GEMV      # fp32 tokens
    assert path(4096, 128, 2848, 5760, 4, n.DTYPE_BF16) == n.PATH_GEMV     # G odd
    assert path(640, 512, 64, 48, 16, n.DTYPE_BF16) == n.PATH_GEMM
    assert path(640, 600, 64, 48, 16, n.DTYPE_BF16) == n.PATH_GEMV         # > 512 experts
    assert path(640, 0, 64, 48, 16, n.DTYPE_BF16) == n.PATH_GEMV           # no experts


def test_router_argument_checks(lib):
    # Checked before anything is enqueued: no GPU needed. Codes: -1 invalid
    # argument, -3 alias, -6 too large.
    P = ctypes.c_void_p
    f = ctypes.c_float(1.0)
    # K > E
    assert lib.mxfp4_router_topk(P(4096), None, 4, 3, 4, f, P(8192), P(16384), None) == -1
    # missing outputs
    assert lib.mxfp4_router_topk(P(4096), None, 4, 8, 2, f, None, P(16384), None) == -1
    # the weights overlap the logits
    assert lib.mxfp4_router_topk(P(4096), None, 4, 8, 2, f, P(1 << 20), P(4096 + 16), None) == -3
    # E + K beyond the shared-memory limit
    assert lib.mxfp4_router_topk(P(4096), None, 1, 20000, 4, f, P(1 << 30), P(1 << 31), None) == -6
    # nothing to do
    assert lib.mxfp4_router_topk(None, None, 0, 8, 2, f, None, None, None) == 0
    assert lib.mxfp4_router_topk(None, None, 5, 8, 0, f, None, None, None) == 0


def test_swiglu_argument_checks(lib):
    # Checked before anything is enqueued: no GPU needed.
    from mxfp4_routed_expert_route_gb300 import _native as n
    f = lib.mxfp4_swiglu_expert
    P = ctypes.c_void_p
    x, gu, gs, dn, ds = P(1 << 24), P(1 << 28), P(1 << 29), P(1 << 30), P(1 << 31)
    sel, p, ys, out = P(1 << 32), P(1 << 33), P(1 << 34), P(1 << 35)
    ok = [x, gu, gs, dn, ds, sel, p, ys, out]
    assert f(*ok, 4, 4, 64, 48, 8, 2, 0, 0, None) == n.ERR_INVALID_ARGUMENT   # F % 32
    assert f(*ok, 4, 4, 60, 64, 8, 2, 0, 0, None) == n.ERR_INVALID_ARGUMENT   # I % 32
    assert f(*ok, 4, 4, 64, 0, 8, 2, 0, 0, None) == n.ERR_INVALID_ARGUMENT    # F == 0
    assert f(*ok, 4, 4, 64, 64, 8, 2, 3, 0, None) == n.ERR_UNSUPPORTED_DTYPE
    assert f(*ok, 4, 4, 64, 64, 8, 2, 0, 2, None) == n.ERR_UNSUPPORTED_DTYPE
    assert f(*ok, 0, 4, 64, 64, 8, 2, 0, 0, None) == n.OK                    # T == 0
    assert f(*ok, 4, 4, 64, 64, 0, 2, 0, 0, None) == n.OK                    # O == 0
    assert f(*ok, 1 << 40, 4, 64, 64, 8, 2, 0, 0, None) == n.ERR_TOO_LARGE
    # a missing down matrix
    assert f(x, gu, gs, None, ds, sel, p, ys, out, 4, 4, 64, 64, 8, 2, 0, 0,
             None) == n.ERR_INVALID_ARGUMENT
    # misaligned down matrix
    assert f(x, gu, gs, P((1 << 30) + 8), ds, sel, p, ys, out, 4, 4, 64, 64, 8, 2, 0, 0,
             None) == n.ERR_INVALID_ARGUMENT
    # out overlapping the down scales
    assert f(x, gu, gs, dn, ds, sel, p, ys, P((1 << 31) + 4), 4, 4, 64, 64, 8, 2, 0, 0,
             None) == n.ERR_ALIAS
    ws = lib.mxfp4_swiglu_expert_workspace_size
    bad = ctypes.c_size_t(-1).value
    assert ws(4, 4, 64, 48, 8, 2, 0) == bad
    assert ws(0, 4, 64, 64, 8, 2, 0) == 0
    # gate/up scratch (T K pairs x 2F) + down scratch (T K pairs x O) + h
    n1 = ws(8, 128, 2880, 2880, 2880, 4, 1)
    assert n1 >= 32 * 5760 * 4 + 32 * 2880 * 4 + 32 * 2880 * 2 and n1 % 256 == 0
    g = lib.mxfp4_swiglu_expert_with_workspace
    assert g(*ok, 4, 4, 64, 64, 8, 2, 0, 0, None, 0, None) == n.ERR_WORKSPACE


def test_swiglu_scratch_follows_the_gate_up_tiles(lib, monkeypatch):
    # Prefill shape on the tensor cores: the gate/up tiles write h directly,
    # so the call needs no float32 partial results for the gate/up
    # projection (T*K*2F*4 bytes); the separate-kernel path (test knob) does.
    ws = lib.mxfp4_swiglu_expert_workspace_size
    T, E, I, F, O, K = 4096, 128, 2880, 2880, 2880, 4
    tiles, fp32, decode = ws(T, E, I, F, O, K, 1), ws(T, E, I, F, O, K, 0), ws(8, E, I, F, O, K, 1)
    monkeypatch.setenv("MXFP4EL_SWIGLU_TILES", "0")
    separate = ws(T, E, I, F, O, K, 1)
    assert separate - tiles >= T * K * 2 * F * 4
    # fp32 tokens and decode batches never take the tensor cores: the knob
    # changes nothing there.
    assert ws(T, E, I, F, O, K, 0) == fp32 and ws(8, E, I, F, O, K, 1) == decode


def test_static_scratch_checks_like_the_other_entry_points(lib):
    # The allocation-free entry point runs the same argument checks, in the
    # same order, before its own size limit: a call with another error gets
    # that error's code even when it is also too large for the fixed array.
    # Every case returns before any GPU work.
    from mxfp4_routed_expert_route_gb300 import _native as n
    static, main = lib.mxfp4_expert_linear_static_scratch, lib.mxfp4_expert_linear
    assert lib.mxfp4_expert_linear_static_scratch_bytes() == 8 << 20
    P = ctypes.c_void_p
    x, w, s, sel, p, ys = P(1 << 24), P(1 << 28), P(1 << 29), P(1 << 30), P(1 << 31), P(1 << 32)
    out = P(1 << 40)
    # 64 tokens x 8 slots x 8192 rows of float32 partial results: 16 MiB of
    # scratch, over the 8 MiB array.
    big = (64, 16, 256, 8192, 8)
    cases = [
        ((x, w, s, sel, p, ys, out) + big + (n.DTYPE_BF16, 7), n.ERR_UNSUPPORTED_DTYPE),
        ((x, w, s, sel, p, ys, out) + big + (5, n.INDEX_I32), n.ERR_UNSUPPORTED_DTYPE),
        ((x, w, s, sel, p, ys, ys) + big + (n.DTYPE_BF16, n.INDEX_I32), n.ERR_ALIAS),
        ((P((1 << 24) + 8), w, s, sel, p, ys, out) + big + (n.DTYPE_BF16, n.INDEX_I32),
         n.ERR_INVALID_ARGUMENT),
        ((None, w, s, sel, p, ys, out) + big + (n.DTYPE_BF16, n.INDEX_I32),
         n.ERR_INVALID_ARGUMENT),
        ((x, w, s, sel, p, ys, out, 64, 16, 250, 8192, 8, n.DTYPE_BF16, n.INDEX_I32),
         n.ERR_INVALID_ARGUMENT),
        ((x, w, s, sel, p, ys, out, 0) + big[1:] + (n.DTYPE_BF16, n.INDEX_I32), n.OK),
        ((x, w, s, sel, p, ys, out, 1 << 40) + big[1:] + (n.DTYPE_BF16, n.INDEX_I32),
         n.ERR_TOO_LARGE),
    ]
    for args, code in cases:
        assert main(*args, None) == code, args
        assert static(*args, None) == code, args
    # Valid for the other entry points, too large only for the fixed array.
    assert static(x, w, s, sel, p, ys, out, *big, n.DTYPE_BF16, n.INDEX_I32,
                  None) == n.ERR_TOO_LARGE


def _a256(n):
    return (n + 255) // 256 * 256


def test_prepared_bytes_follow_the_documented_layout(lib):
    # One 4352-byte block per (expert, 128-row tile, 64-wide K chunk), then the
    # int16 [E][O] and uint8 [E][mtiles] parts, each 256-byte aligned.
    for E, I, O in [(1, 32, 1), (3, 96, 200), (128, 2880, 5760), (384, 7168, 4096)]:
        G = I // 32
        nk, mt = (G + 1) // 2, (O + 127) // 128
        want = _a256(E * mt * nk * 4352) + _a256(E * O * 2) + _a256(E * mt)
        assert lib.mxfp4_expert_linear_prepared_bytes(E, I, O) == want
    bad = ctypes.c_size_t(-1).value
    assert lib.mxfp4_expert_linear_prepared_bytes(2, 48, 8) == bad      # I % 32
    assert lib.mxfp4_expert_linear_prepared_bytes(-1, 64, 8) == bad
    assert lib.mxfp4_expert_linear_prepared_bytes(2, 15360 + 32, 8) == bad   # beyond the limit
    assert lib.mxfp4_expert_linear_prepared_bytes(2, 15360, 8) != bad


def test_prepared_argument_checks_return_before_gpu_work(lib):
    from mxfp4_routed_expert_route_gb300 import _native as n
    prep = lib.mxfp4_expert_linear_prepare
    w, s = ctypes.c_void_p(1 << 24), ctypes.c_void_p(1 << 28)
    buf = ctypes.c_void_p(1 << 36)
    need = lib.mxfp4_expert_linear_prepared_bytes(4, 64, 8)
    assert prep(w, s, 4, 60, 8, buf, need, None) == n.ERR_INVALID_ARGUMENT
    assert prep(w, s, 4, 64 * 1024, 8, buf, 1 << 40, None) == n.ERR_TOO_LARGE
    assert prep(None, s, 4, 64, 8, buf, need, None) == n.ERR_INVALID_ARGUMENT
    assert prep(w, s, 4, 64, 8, None, need, None) == n.ERR_INVALID_ARGUMENT
    assert prep(w, s, 0, 64, 8, None, 0, None) == n.OK               # E == 0: no-op
    assert prep(w, s, 4, 64, 8, buf, need - 1, None) == n.ERR_WORKSPACE
    assert prep(w, s, 4, 64, 8, ctypes.c_void_p((1 << 36) + 16), need, None) == n.ERR_WORKSPACE
    assert prep(ctypes.c_void_p((1 << 24) + 4), s, 4, 64, 8, buf, need,
                None) == n.ERR_INVALID_ARGUMENT
    assert prep(w, s, 4, 64, 8, ctypes.c_void_p((1 << 24) - 256), need, None) == n.ERR_ALIAS
    f = lib.mxfp4_expert_linear_prepared
    fake = ctypes.c_void_p(1 << 20)
    x, ys, out = ctypes.c_void_p(1 << 32), ctypes.c_void_p(1 << 33), ctypes.c_void_p(1 << 34)
    assert f(x, buf, fake, fake, ys, out, 4, 4, 60, 8, 2, 0, 0, None) == n.ERR_INVALID_ARGUMENT
    assert f(x, buf, fake, fake, ys, out, 4, 4, 64, 8, 2, 9, 0, None) == n.ERR_UNSUPPORTED_DTYPE
    assert f(x, buf, fake, fake, ys, out, 4, 4, 64 * 1024, 8, 2, 0, 0,
             None) == n.ERR_TOO_LARGE
    assert f(x, None, fake, fake, ys, out, 4, 4, 64, 8, 2, 0, 0, None) == n.ERR_INVALID_ARGUMENT
    assert f(x, ctypes.c_void_p((1 << 36) + 16), fake, fake, ys, out, 4, 4, 64, 8, 2, 0, 0,
             None) == n.ERR_INVALID_ARGUMENT
    assert f(x, buf, fake, fake, ys, ys, 4, 4, 64, 8, 2, 0, 0, None) == n.ERR_ALIAS
    assert f(x, buf, fake, fake, ys, out, 0, 4, 64, 8, 2, 0, 0, None) == n.OK
    g = lib.mxfp4_expert_linear_prepared_with_workspace
    assert g(x, buf, fake, fake, ys, out, 4, 4, 64, 8, 2, 0, 0, None, 0,
             None) == n.ERR_WORKSPACE
    ws = lib.mxfp4_expert_linear_prepared_workspace_size
    assert ws(4, 4, 64, 8, 2, 0) not in (0, ctypes.c_size_t(-1).value)
    assert ws(4, 4, 64 * 1024, 8, 2, 0) == ctypes.c_size_t(-1).value
