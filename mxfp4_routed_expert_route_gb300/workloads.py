"""Seeded synthetic inputs for the MXFP4 routed expert linear.

This module only draws random inputs. It holds none of the layer's arithmetic
(no nibble decode, no scale, no dot product), so the CUDA path and the CPU
oracle can both be fed from it without sharing any of the method.

Shapes follow the problem statement ("MXFP4 Routed Expert Linear", Kimi K3,
tensortonic formal statement): tokens (T, I), packed weights (E, O, G, 16)
uint8, scale bytes (E, O, G) uint8, selected experts (T, K), mixture weights
(T, K), shared output (T, O), with I = 32 G.

Recipe (the same for every named workload):
  * numpy ``default_rng(seed)``; bytes are drawn on the host, then uploaded.
  * packed bytes uniform over 0..255 and scale bytes uniform over the stated
    inclusive range, each array drawn in 64 MiB chunks: chunk c of stream s
    comes from ``default_rng((seed, s, c)).integers(lo, hi + 1, uint8)``
    (s = 1 packed bytes, 2 scale bytes; for the SwiGLU expert 1 and 2 are the
    gate/up matrix, 3 and 4 the down matrix), so the bytes do not depend on
    how many threads draw them;
  * x and y_shared ~ N(0, 1), rounded to nearest-even bf16 where the
    workload is bf16;
  * mixture weights = softmax of N(0, 1) logits over the K picks, stored fp32;
  * uniform picks: K distinct experts per token, uniformly at random;
  * Zipf picks: popularity r^-s over ranks 1..E, ranks mapped to expert ids by
    a seeded permutation, K distinct picks per token by Gumbel-top-K (the
    same law as successive sampling without replacement).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass
class Workload:
    name: str
    T: int
    E: int
    K: int
    I: int
    O: int
    dtype: torch.dtype            # token / shared-output / output dtype
    x: torch.Tensor               # (T, I) dtype, CPU
    packed: torch.Tensor          # (E, O, G, 16) uint8, CPU
    scales: torch.Tensor          # (E, O, G) uint8, CPU
    sel: torch.Tensor             # (T, K) int32, CPU
    p: torch.Tensor               # (T, K) float32, CPU
    y_shared: torch.Tensor        # (T, O) dtype, CPU
    meta: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.I // 32

    def device_tensors(self, device) -> dict:
        """Copies of every input on ``device`` (weights included)."""
        return {k: getattr(self, k).to(device) for k in
                ("x", "packed", "scales", "sel", "p", "y_shared")}


# The five named workloads: (T, E, K, I, O, dtype, scale range, pick law).
CONFIGS = {
    "tiny_fp32": dict(T=4, E=4, K=2, I=64, O=8, dtype=torch.float32,
                      scale_lo=120, scale_hi=134, picks="uniform", seed=0),
    "decode": dict(T=8, E=128, K=4, I=2880, O=5760, dtype=torch.bfloat16,
                   scale_lo=118, scale_hi=124, picks="uniform", seed=1),
    "prefill": dict(T=4096, E=128, K=4, I=2880, O=5760, dtype=torch.bfloat16,
                    scale_lo=118, scale_hi=124, picks="uniform", seed=2),
    "wide_decode": dict(T=16, E=384, K=8, I=7168, O=4096, dtype=torch.bfloat16,
                        scale_lo=116, scale_hi=124, picks="uniform", seed=3),
    "skewed_prefill": dict(T=8192, E=384, K=8, I=7168, O=4096,
                           dtype=torch.bfloat16, scale_lo=116, scale_hi=124,
                           picks="zipf", zipf_s=1.2, seed=4),
}


def _normal(rng, shape, dtype):
    a = rng.standard_normal(shape, dtype=np.float32)
    t = torch.from_numpy(a)
    return t.to(dtype) if dtype != torch.float32 else t


def uniform_picks(rng, T: int, E: int, K: int) -> np.ndarray:
    """K distinct expert ids per token, uniformly at random."""
    if K == 0 or T == 0:
        return np.zeros((T, K), dtype=np.int32)
    keys = rng.random((T, E))
    return np.argsort(keys, axis=1, kind="stable")[:, :K].astype(np.int32)


def zipf_picks(rng, T: int, E: int, K: int, s: float) -> np.ndarray:
    """K distinct picks per token from Zipf(s) popularity (Gumbel-top-K)."""
    ranks = np.arange(1, E + 1, dtype=np.float64)
    logw = -s * np.log(ranks)
    perm = rng.permutation(E)              # rank r -> expert id perm[r]
    logw_by_id = np.empty(E)
    logw_by_id[perm] = logw
    g = rng.gumbel(size=(T, E))
    keys = logw_by_id[None, :] + g
    return np.argsort(-keys, axis=1, kind="stable")[:, :K].astype(np.int32)


def softmax_weights(rng, T: int, K: int) -> np.ndarray:
    logits = rng.standard_normal((T, K))
    if K == 0:
        return np.zeros((T, 0), dtype=np.float32)
    z = np.exp(logits - logits.max(axis=1, keepdims=True))
    return (z / z.sum(axis=1, keepdims=True)).astype(np.float32)


CHUNK = 64 << 20


def uniform_bytes(seed: int, stream: int, n: int, lo: int = 0, hi: int = 255) -> np.ndarray:
    """n bytes uniform over [lo, hi]: chunk c of CHUNK bytes is drawn by
    default_rng((seed, stream, c)), the chunks in parallel threads."""
    out = np.empty(n, dtype=np.uint8)

    def fill(c):
        a, b = c * CHUNK, min(n, (c + 1) * CHUNK)
        out[a:b] = np.random.default_rng((seed, stream, c)).integers(
            lo, hi + 1, size=b - a, dtype=np.uint8)

    nchunks = (n + CHUNK - 1) // CHUNK
    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def make(T: int, E: int, K: int, I: int, O: int, dtype=torch.bfloat16,
         scale_lo: int = 118, scale_hi: int = 124, picks: str = "uniform",
         seed: int = 0, zipf_s: float = 1.2, name: str = "custom",
         sel: np.ndarray | None = None) -> Workload:
    """Draw one workload. ``sel`` may be supplied to fix the routing."""
    if I % 32:
        raise ValueError("I must be a multiple of 32")
    G = I // 32
    rng = np.random.default_rng(seed)
    packed = uniform_bytes(seed, 1, E * O * G * 16).reshape(E, O, G, 16)
    scales = uniform_bytes(seed, 2, E * O * G, scale_lo, scale_hi).reshape(E, O, G)
    x = _normal(rng, (T, I), dtype)
    y_shared = _normal(rng, (T, O), dtype)
    if sel is None:
        if picks == "uniform":
            sel = uniform_picks(rng, T, E, K)
        elif picks == "zipf":
            sel = zipf_picks(rng, T, E, K, zipf_s)
        else:
            raise ValueError(picks)
    p = softmax_weights(rng, T, K)
    return Workload(name=name, T=T, E=E, K=K, I=I, O=O, dtype=dtype, x=x,
                    packed=torch.from_numpy(packed),
                    scales=torch.from_numpy(scales),
                    sel=torch.from_numpy(np.ascontiguousarray(sel, dtype=np.int32)),
                    p=torch.from_numpy(p), y_shared=y_shared,
                    meta=dict(seed=seed, picks=picks, scale_range=(scale_lo, scale_hi)))


def named(name: str) -> Workload:
    cfg = dict(CONFIGS[name])
    return make(name=name, **cfg)


def experts_touched(sel: torch.Tensor, E: int) -> int:
    """Number of distinct expert ids in ``sel`` (a count, not layer math)."""
    s = sel.reshape(-1).to(torch.int64)
    s = s[(s >= 0) & (s < E)]
    return int(torch.unique(s).numel())


# ------------------------------------------------------- the SwiGLU expert --
@dataclass
class SwigluWorkload:
    """Inputs of the routed SwiGLU expert: the gate and up matrices stacked
    along their rows (gate rows first), the down matrix, routing and the
    shared output."""
    name: str
    T: int
    E: int
    K: int
    I: int
    F: int
    O: int
    dtype: torch.dtype
    x: torch.Tensor               # (T, I)
    gate_up_packed: torch.Tensor  # (E, 2F, I/32, 16) uint8
    gate_up_scales: torch.Tensor  # (E, 2F, I/32) uint8
    down_packed: torch.Tensor     # (E, O, F/32, 16) uint8
    down_scales: torch.Tensor     # (E, O, F/32) uint8
    sel: torch.Tensor             # (T, K) int32
    p: torch.Tensor               # (T, K) float32
    y_shared: torch.Tensor        # (T, O)
    meta: dict = field(default_factory=dict)

    ARGS = ("x", "gate_up_packed", "gate_up_scales", "down_packed", "down_scales", "sel",
            "p", "y_shared")

    def device_tensors(self, device) -> dict:
        return {k: getattr(self, k).to(device) for k in self.ARGS}

    def args(self) -> list:
        return [getattr(self, k) for k in self.ARGS]


# The SwiGLU expert at the layer shape of the named linear workloads: hidden
# width I = 2880 and intermediate width F = 2880, so the stacked gate/up
# matrix has the linear workloads' 5760 rows and the down matrix maps 2880
# back to 2880.
SWIGLU_CONFIGS = {
    "swiglu_tiny_fp32": dict(T=4, E=4, K=2, I=64, F=64, O=32, dtype=torch.float32, seed=10),
    "swiglu_decode": dict(T=8, E=128, K=4, I=2880, F=2880, O=2880, dtype=torch.bfloat16,
                          seed=11),
    "swiglu_prefill": dict(T=4096, E=128, K=4, I=2880, F=2880, O=2880,
                           dtype=torch.bfloat16, seed=12),
}


def make_swiglu(T: int, E: int, K: int, I: int, F: int, O: int, dtype=torch.bfloat16,
                scale_lo: int = 118, scale_hi: int = 124, picks: str = "uniform",
                seed: int = 0, zipf_s: float = 1.2, name: str = "custom") -> SwigluWorkload:
    """Draw one SwiGLU workload with the recipe of :func:`make` (uniform
    bytes, uniform scale bytes in [scale_lo, scale_hi] for both matrices,
    N(0, 1) tokens and shared output, softmax weights)."""
    if I % 32 or F % 32:
        raise ValueError("I and F must be multiples of 32")
    rng = np.random.default_rng(seed)
    gu = uniform_bytes(seed, 1, E * 2 * F * (I // 32) * 16).reshape(E, 2 * F, I // 32, 16)
    gus = uniform_bytes(seed, 2, E * 2 * F * (I // 32), scale_lo, scale_hi).reshape(
        E, 2 * F, I // 32)
    dn = uniform_bytes(seed, 3, E * O * (F // 32) * 16).reshape(E, O, F // 32, 16)
    dns = uniform_bytes(seed, 4, E * O * (F // 32), scale_lo, scale_hi).reshape(E, O, F // 32)
    x = _normal(rng, (T, I), dtype)
    y_shared = _normal(rng, (T, O), dtype)
    if picks == "uniform":
        sel = uniform_picks(rng, T, E, K)
    elif picks == "zipf":
        sel = zipf_picks(rng, T, E, K, zipf_s)
    else:
        raise ValueError(picks)
    p = softmax_weights(rng, T, K)
    return SwigluWorkload(name=name, T=T, E=E, K=K, I=I, F=F, O=O, dtype=dtype, x=x,
                          gate_up_packed=torch.from_numpy(gu),
                          gate_up_scales=torch.from_numpy(gus),
                          down_packed=torch.from_numpy(dn), down_scales=torch.from_numpy(dns),
                          sel=torch.from_numpy(np.ascontiguousarray(sel, dtype=np.int32)),
                          p=torch.from_numpy(p), y_shared=y_shared,
                          meta=dict(seed=seed, picks=picks, scale_range=(scale_lo, scale_hi)))


def named_swiglu(name: str) -> SwigluWorkload:
    return make_swiglu(name=name, **SWIGLU_CONFIGS[name])
