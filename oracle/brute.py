"""TEST INFRASTRUCTURE: numpy brute force for tiny inputs.

An implementation independent of ``oracle.c``: it decodes each selected
expert's whole matrix at once with array operations (nibble split, interleave,
table lookup, ``np.ldexp`` by s - 127), as the problem statement "MXFP4
Routed Expert Linear" (Kimi K3) describes, then uses the library product
``W @ x``. It caches a decoded expert the first time it is selected, as the
page's "Decode only selected experts" section allows. Parity: pinned
(tests/oracle_pins.py) and cross-checked against ``oracle.c``.
"""
from __future__ import annotations

import numpy as np

# The E2M1 value table printed on the problem page.
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                 -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def dequantize(packed_e: np.ndarray, scales_e: np.ndarray) -> np.ndarray:
    """(O, G, 16) bytes + (O, G) scale bytes -> (O, 32 G) float64."""
    packed_e = np.asarray(packed_e, dtype=np.uint8)
    O, G, _ = packed_e.shape
    low = packed_e & 0x0F
    high = packed_e >> 4
    codes = np.stack([low, high], axis=-1).reshape(O, G, 32)   # low first
    values = E2M1[codes]
    exps = np.asarray(scales_e, dtype=np.int64)[:, :, None] - 127
    return np.ldexp(values, exps).reshape(O, G * 32)


def expert_linear(x, packed, scales, sel, p, y_shared):
    """float64 result (T, O) for valid expert indices."""
    x = np.asarray(x, dtype=np.float64)
    p = np.asarray(p, dtype=np.float64)
    out = np.array(y_shared, dtype=np.float64, copy=True)
    sel = np.asarray(sel, dtype=np.int64)
    cache = {}
    for t in range(x.shape[0]):
        for k in range(sel.shape[1]):
            e = int(sel[t, k])
            if e not in cache:
                cache[e] = dequantize(packed[e], scales[e])
            out[t] += p[t, k] * (cache[e] @ x[t])
    return out
