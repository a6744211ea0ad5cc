"""TEST INFRASTRUCTURE: ctypes wrapper around the float64 C oracle.

``expert_linear`` follows the problem statement "MXFP4 Routed Expert Linear"
(Kimi K3): y_t = y_shared_t + sum_k p[t,k] W_{sel[t,k]} x_t, every weight
decoded as LUT[nibble] * 2^(s-127), low nibble first. It returns the result in
float64 (never rounded) and abs_terms = |y_shared| + sum |p w x|, the scale of
the comparison tolerance. Parity: pinned (tests/oracle_pins.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``oracle.c`` with gcc (OpenMP) into a shared library."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-Wall", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (and if needed build) the oracle library; returns a ctypes CDLL."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _bind(lib):
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.oracle_expert_linear.restype = i64
    lib.oracle_expert_linear.argtypes = [P, P, P, P, P, P, i64, i64, i64, i64,
                                         i64, P, i64, P, P]
    lib.oracle_decode_expert.restype = ctypes.c_int
    lib.oracle_decode_expert.argtypes = [P, P, i64, i64, i64, i64, P]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    return lib


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):                      # torch tensor (CPU)
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _u8(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.uint8)


def _i64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def expert_linear(x, packed, scales, sel, p, y_shared, rows=None, lib=None):
    """Oracle result for every token (or the token ids in ``rows``).

    Inputs may be numpy arrays or CPU torch tensors of any float dtype; they
    are widened to float64 exactly. Returns ``(out, abs_terms, bad_pairs)``,
    both arrays (n_rows, O) float64.
    """
    lib = lib or load()
    x, p, ys = _f64(x), _f64(p), _f64(y_shared)
    packed, scales, sel = _u8(packed), _u8(scales), _i64(sel)
    T, I = x.shape
    E, O, G, sixteen = packed.shape
    K = sel.shape[1] if sel.ndim == 2 else 0
    if sixteen != 16 or G * 32 != I or scales.shape != (E, O, G):
        raise ValueError("shape mismatch")
    if rows is None:
        n = T
        rows_arr = None
    else:
        rows_arr = _i64(rows).reshape(-1)
        n = rows_arr.size
    out = np.zeros((n, O), dtype=np.float64)
    absm = np.zeros((n, O), dtype=np.float64)
    bad = lib.oracle_expert_linear(
        _ptr(x), _ptr(packed), _ptr(scales), _ptr(sel), _ptr(p), _ptr(ys),
        T, E, I, O, K, _ptr(rows_arr) if rows_arr is not None else None, n,
        _ptr(out), _ptr(absm))
    if bad < 0:
        raise ValueError("oracle rejected the call")
    return out, absm, int(bad)


def decode_expert(packed, scales, e, lib=None) -> np.ndarray:
    """The reconstructed (O, I) float64 matrix of expert ``e``."""
    lib = lib or load()
    packed, scales = _u8(packed), _u8(scales)
    E, O, G, _ = packed.shape
    W = np.zeros((O, G * 32), dtype=np.float64)
    rc = lib.oracle_decode_expert(_ptr(packed), _ptr(scales), E, O, G * 32,
                                  int(e), _ptr(W))
    if rc != 0:
        raise ValueError("bad expert index")
    return W


def num_threads(lib=None) -> int:
    return int((lib or load()).oracle_num_threads())
