"""Helpers for the GPU parity tests: run the library, compare with the oracle."""
from __future__ import annotations

import hashlib

import numpy as np
import torch

import oracle
from mxfp4_routed_expert_route_gb300 import mxfp4_expert_linear, workloads

# Tolerances on max |gpu - oracle| / abs_terms, abs_terms = |y_shared| +
# sum |p w x| per output element.
TOL = {torch.float32: 1e-5, torch.bfloat16: 8e-3}


def run_gpu(wl: workloads.Workload, device="cuda", sel=None, **kw) -> torch.Tensor:
    d = wl.device_tensors(device)
    if sel is not None:
        d["sel"] = sel.to(device)
    return mxfp4_expert_linear(d["x"], d["packed"], d["scales"], d["sel"], d["p"],
                               d["y_shared"], **kw)


def oracle_rows(wl: workloads.Workload, rows=None, sel=None):
    return oracle.expert_linear(wl.x, wl.packed, wl.scales,
                                wl.sel if sel is None else sel, wl.p, wl.y_shared,
                                rows=rows)


def worst_ratio(gpu_rows: torch.Tensor, want: np.ndarray, abs_terms: np.ndarray) -> float:
    got = gpu_rows.detach().cpu().double().numpy()
    err = np.abs(got - want)
    scale = np.maximum(abs_terms, np.finfo(np.float64).tiny)
    r = err / scale
    r[(err == 0)] = 0.0
    return float(r.max()) if r.size else 0.0


def assert_parity(gpu_rows, want, abs_terms, dtype, what=""):
    assert np.all(np.isfinite(gpu_rows.detach().cpu().double().numpy())), what
    ratio = worst_ratio(gpu_rows, want, abs_terms)
    print(f"[parity] {what or 'case'}: max err/abs_terms = {ratio:.3e} (tol {TOL[dtype]:.0e})")
    assert ratio <= TOL[dtype], f"{what}: max err/abs_terms = {ratio:.3e} > {TOL[dtype]}"
    return ratio


def digest(*tensors) -> str:
    h = hashlib.sha256()
    for t in tensors:
        h.update(t.detach().contiguous().cpu().view(torch.uint8).numpy().tobytes())
    return h.hexdigest()


def parity_rows(wl: workloads.Workload, n_random: int = 256, seed: int = 0) -> np.ndarray:
    """Token rows for an element-by-element check of a full-size batch whose
    every row the oracle cannot afford: every token of the least-loaded
    expert, the first 192 tokens of the most-loaded expert (which cover its
    first token block of the tensor-core kernel, at most 192 tokens) and its
    last 64 (its last block), the first and last token, and n_random more
    drawn at random."""
    rng = np.random.default_rng(seed)
    sel = wl.sel.numpy()
    counts = np.bincount(sel[(sel >= 0) & (sel < wl.E)].reshape(-1), minlength=wl.E)
    hot = int(counts.argmax())
    used = np.nonzero(counts)[0]
    cold = int(used[counts[used].argmin()])
    hot_tokens = np.nonzero((sel == hot).any(1))[0]
    pick = {0, wl.T - 1}
    pick.update(np.nonzero((sel == cold).any(1))[0].tolist())
    pick.update(hot_tokens[:192].tolist())
    pick.update(hot_tokens[-64:].tolist())
    target = len(pick) + min(n_random, wl.T - len(pick))
    while len(pick) < target:
        pick.add(int(rng.integers(0, wl.T)))
    return np.array(sorted(pick), dtype=np.int64)


def sample_rows(wl: workloads.Workload, n: int, seed: int = 0) -> np.ndarray:
    """Tokens for a sampled full-size check: the first and last token, tokens of
    the most and least loaded experts, and random ones."""
    rng = np.random.default_rng(seed)
    sel = wl.sel.numpy()
    T = wl.T
    counts = np.bincount(sel.reshape(-1), minlength=wl.E)
    hot = int(counts.argmax())
    used = np.nonzero(counts)[0]
    cold = int(used[counts[used].argmin()])
    pick = {0, T - 1}
    pick.update(np.nonzero((sel == hot).any(1))[0][:2].tolist())
    pick.update(np.nonzero((sel == cold).any(1))[0][:2].tolist())
    while len(pick) < min(n, T):
        pick.add(int(rng.integers(0, T)))
    return np.array(sorted(pick), dtype=np.int64)
