"""TEST INFRASTRUCTURE: the CPU oracle for the sigmoid top-K router.

Only the tests and the benchmark import this module; the product path never
does, and the two share no code.

The router feeding the routed expert linear, as the pages define it:

* "MoE Expert Kernels: Grouped Prefill and Mixed-Quant Compact Experts",
  section 1 (the shared building blocks, the sigmoid router): the choice
  score is sigmoid(logit) plus a per-expert correction bias; the bias steers
  which experts are chosen only, and the weights are gathered from the raw
  sigmoid scores, not the biased ones.
* The Hy3 decode write-up, "Decode: fewer, fused kernels" and "How exactness
  was established" (the router after its logits): the top K are taken in the
  order a stable descending sort gives them (highest first, ties to the lower
  expert index); the K chosen scores are summed left to right, each is divided
  by that sum plus 1e-20 and multiplied by the routing scaling factor.

Readings: the selection is decided in float32, the precision the pages
compute it in (a float32 sigmoid of the float32 logit, plus the float32
bias); the weights are computed here in float64 from those float32 scores.
Parity: pinned; tests/test_router_oracle.py.
"""
from __future__ import annotations

import numpy as np


def choice_scores(logits, bias):
    """(raw, choice): float32 sigmoid scores and the float32 biased scores."""
    x = np.asarray(logits, dtype=np.float32)
    b = np.asarray(bias, dtype=np.float32)
    one = np.float32(1.0)
    raw = (one / (one + np.exp(-x))).astype(np.float32)
    choice = (raw + b[None, :]).astype(np.float32)
    return raw, choice


def topk_order(choice, K):
    """Expert ids of the K highest choice scores per row, highest first, ties
    to the lower index (the first K of a stable descending sort)."""
    choice = np.asarray(choice)
    T, E = choice.shape
    idx = np.arange(E)
    out = np.empty((T, K), dtype=np.int64)
    for t in range(T):
        order = np.lexsort((idx, -choice[t].astype(np.float64)))   # key -choice, then index
        out[t] = order[:K]
    return out


def router(logits, bias, K, scaling=1.0):
    """(sel, p): the chosen expert ids (T, K) int64 and their weights (T, K)
    float64, raw scores over their left-to-right sum plus 1e-20, times the
    scaling factor."""
    raw, choice = choice_scores(logits, bias)
    sel = topk_order(choice, K)
    p = np.empty(sel.shape, dtype=np.float64)
    for t in range(sel.shape[0]):
        s = [float(raw[t, e]) for e in sel[t]]
        total = 0.0
        for v in s:                     # left to right
            total += v
        for k, v in enumerate(s):
            p[t, k] = v / (total + 1e-20) * float(scaling)
    return sel, p
