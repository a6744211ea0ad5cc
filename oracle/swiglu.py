"""TEST INFRASTRUCTURE: the CPU oracle for the routed MXFP4 SwiGLU expert.

Only the tests and the benchmark import this module; the product path never
does, and the two share no code.

The expert as the pages define it:

* "MoE Expert Kernels: Grouped Prefill and Mixed-Quant Compact Experts",
  section 1 (the shared building blocks: the SwiGLU expert shape): every
  routed expert computes down(silu(gate(x)) * up(x)); the per-slot results
  are added into the token's output scaled by the routing weight, in float32
  there (float64 here, never rounded).
* The Hy3 decode write-up, "Decode: fewer, fused kernels" (the gate and up
  projections stacked along their output rows, one gathered row per
  token-expert pair): the stacked gate/up matrix holds the gate rows first,
  then the up rows.
* Every matrix is an MXFP4 expert matrix decoded as in "MXFP4 Routed Expert
  Linear" (Kimi K3); the decoding and the matrix-vector products are the
  pinned linear oracle (``oracle.expert_linear``), used here as a library
  step: one call per projection with every (token, slot) pair as its own
  token, weight 1 and no shared output.

silu(v) = v * sigmoid(v) = v / (1 + exp(-v)), evaluated in float64.

The intermediate h is the down projection's input, "rounded once to the
token dtype". ``swiglu_expert(..., h_round="bf16")`` takes that step:
each exact h is rounded to the nearest bf16 value, ties to even
(``round_to_bf16``), before the down projection; without it h stays exact.

Besides the result, ``swiglu_expert`` returns the terms the comparison
tolerance is built from (each summed over the token's slots with |p|):
  abs_terms = |y_shared| + sum_k |p| |Wd| |h|       (the down stage's sum of |terms|)
  s_first   = sum_k |p| |Wd| (1.1 Ag |u| + |g| Au)   (first-order effect of gate/up errors)
  s_second  = sum_k |p| |Wd| (Ag Au)                 (their product term)
  s_h       = sum_k |p| |Wd| |h|                     (effect of relative errors in h)
where Ag = |Wg| |x| and Au = |Wu| |x| are the gate/up rows' sums of |terms|
and 1.1 bounds |silu'| (its maximum is about 1.0998, at v near 2.4).
Parity: pinned; tests/test_swiglu_oracle.py.
"""
from __future__ import annotations

import numpy as np

from .reference import expert_linear

SILU_SLOPE_MAX = 1.1


def silu(v):
    """v / (1 + exp(-v)) in float64 (exp(-v) may overflow to inf: silu -> -0)."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def round_to_bf16(v):
    """Round float64 values to the nearest bf16 value, ties to even, in one
    step from the exact value: 8 significant bits for normal values (exponent
    down to -126, float32's range), then the subnormal grid 2^-133; values
    that round to 2^128 or beyond become +-inf; zeros, infinities and NaN
    pass through."""
    v = np.asarray(v, dtype=np.float64)
    out = v.copy()
    fin = np.isfinite(v) & (v != 0.0)
    x = v[fin]
    _, e = np.frexp(x)                          # |x| = m 2^e, 1/2 <= m < 1
    quantum_exp = np.maximum(e - 8, -133)       # 8 bits: leading bit 2^(e-1) ... 2^(e-8)
    r = np.ldexp(np.rint(np.ldexp(x, -quantum_exp)), quantum_exp)   # rint: ties to even
    r = np.where(np.abs(r) >= np.ldexp(1.0, 128), np.copysign(np.inf, r), r)
    out[fin] = r
    return out


def _pairs(x, sel, rows):
    """Tokens (one per (token, slot) pair, slot-major within a token) and the
    pairs' expert ids as a (pairs, 1) selection."""
    x = np.asarray(x.detach().cpu().double().numpy() if hasattr(x, "detach") else x,
                   dtype=np.float64)
    sel = np.asarray(sel.detach().cpu().numpy() if hasattr(sel, "detach") else sel,
                     dtype=np.int64)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64).reshape(-1)
        x, sel = x[rows], sel[rows]
    K = sel.shape[1]
    return np.repeat(x, K, axis=0), sel.reshape(-1, 1), K


def projection(tokens, packed, scales, sel_pairs):
    """Per pair j: (W_{sel[j]} tokens[j], |W_{sel[j]}| |tokens[j]|, invalid ids),
    both (pairs, rows) float64; an invalid id gives a zero row."""
    n = tokens.shape[0]
    rows = packed.shape[1]
    one = np.ones((n, 1), dtype=np.float64)
    zero = np.zeros((n, rows), dtype=np.float64)
    return expert_linear(tokens, packed, scales, sel_pairs, one, zero)


def swiglu_expert(x, gate_up_packed, gate_up_scales, down_packed, down_scales, sel, p,
                  y_shared, rows=None, h_round=None):
    """The SwiGLU expert for every token (or the token ids in ``rows``).

    Shapes: x (T, I); gate_up_packed (E, 2F, I/32, 16) with the gate rows
    first; down_packed (E, O, F/32, 16); sel, p (T, K); y_shared (T, O).
    Returns a dict with ``out`` (n, O) float64, the tolerance terms named in
    the module docstring, ``bad`` (invalid ids seen) and, per pair (n*K rows,
    slot-major within a token), ``g``, ``u``, ``ag``, ``au`` and ``h`` (the
    exact h). h_round="bf16" runs the down projection on h rounded to bf16
    (``h_used``; the tolerance terms then use it too)."""
    tokens, sel_pairs, K = _pairs(x, sel, rows)
    F = gate_up_packed.shape[1] // 2
    gu, gu_abs, bad = projection(tokens, gate_up_packed, gate_up_scales, sel_pairs)
    g, u = gu[:, :F], gu[:, F:]
    ag, au = gu_abs[:, :F], gu_abs[:, F:]
    h = silu(g) * u
    if h_round not in (None, "bf16"):
        raise ValueError(f"unknown h_round {h_round!r}")
    h_used = round_to_bf16(h) if h_round == "bf16" else h
    d, d_abs_h, _ = projection(h_used, down_packed, down_scales, sel_pairs)
    # |Wd| v for the non-negative vectors v of the tolerance terms: the linear
    # oracle's sum of |terms| for token v is exactly |Wd| v.
    _, d_first, _ = projection(SILU_SLOPE_MAX * ag * np.abs(u) + np.abs(g) * au,
                               down_packed, down_scales, sel_pairs)
    _, d_second, _ = projection(ag * au, down_packed, down_scales, sel_pairs)

    p = np.asarray(p.detach().cpu().numpy() if hasattr(p, "detach") else p, dtype=np.float64)
    ys = np.asarray(y_shared.detach().cpu().double().numpy()
                    if hasattr(y_shared, "detach") else y_shared, dtype=np.float64)
    if rows is not None:
        r = np.asarray(rows, dtype=np.int64).reshape(-1)
        p, ys = p[r], ys[r]
    n, O = ys.shape
    out = ys.copy()
    s_h = np.zeros((n, O))
    s_first = np.zeros((n, O))
    s_second = np.zeros((n, O))
    for k in range(K):                         # slot order
        j = np.arange(n) * K + k
        pk = p[:, k:k + 1]
        out += pk * d[j]
        s_h += np.abs(pk) * d_abs_h[j]
        s_first += np.abs(pk) * d_first[j]
        s_second += np.abs(pk) * d_second[j]
    return {"out": out, "abs_terms": np.abs(ys) + s_h, "s_first": s_first,
            "s_second": s_second, "s_h": s_h, "bad": int(bad),
            "g": g, "u": u, "ag": ag, "au": au, "h": h, "h_used": h_used, "p": p, "K": K}


def tolerance(terms, tau, tau1, rho):
    """Elementwise bound on |computed - out| from the tolerance terms.

    tau bounds the down projection plus combine (relative to their sum of
    |terms|), tau1 the gate/up projections' errors (relative to Ag, Au), rho
    the relative error of evaluating silu(g) u and rounding it to the token
    dtype. With g' = g + dg, |dg| <= tau1 Ag (likewise u):
      |h' - h| <= 1.1 |dg| (|u| + |du|) + |g| |du|, plus rho |h'|,
    so the h error is at most dh = (1 + rho)(tau1 S1 + 1.1 tau1^2 S2) + rho |h|,
    and the result's error at most tau (A + |p||Wd| dh) + |p||Wd| dh."""
    dh = ((1.0 + rho) * (tau1 * terms["s_first"]
                         + SILU_SLOPE_MAX * tau1 * tau1 * terms["s_second"])
          + rho * terms["s_h"])
    return tau * terms["abs_terms"] + (1.0 + tau) * dh
