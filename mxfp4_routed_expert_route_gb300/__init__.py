"""MXFP4 routed expert linear on GB300 (sm_103a).

    y_t = y_shared_t + sum_k p[t, k] * W_{sel[t, k]} x_t

with every expert matrix stored as packed E2M1 nibbles (low nibble first)
and one E8M0 scale byte per (expert, output row, 32-value group), as in the
problem statement "MXFP4 Routed Expert Linear" (Kimi K3).

This module is the thin Python face of the C library
``lib/libmxfp4_expert_linear.so`` (header ``include/mxfp4_expert_linear.h``):
it checks and marshals arguments and passes raw device pointers and the
current CUDA stream. Every step of the computation runs in the library's
CUDA kernels; there is no CPU path.
"""
from __future__ import annotations

import ctypes

import torch

from . import _native

__all__ = ["mxfp4_expert_linear", "workspace_size", "device_errors", "wait_timeouts",
           "LibraryNotBuilt", "MXFP4Error", "router_topk", "mxfp4_expert_linear_routed",
           "mxfp4_swiglu_expert", "swiglu_workspace_size", "PreparedWeights",
           "prepare_weights", "prepared_bytes", "mxfp4_expert_linear_prepared",
           "prepared_workspace_size"]

LibraryNotBuilt = _native.LibraryNotBuilt
MXFP4Error = _native.MXFP4Error

_TOKEN_DTYPES = {torch.float32: _native.DTYPE_F32,
                 torch.bfloat16: _native.DTYPE_BF16}
_INDEX_DTYPES = {torch.int32: _native.INDEX_I32, torch.int64: _native.INDEX_I64}


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() else None


def workspace_size(T: int, E: int, I: int, O: int, K: int,
                   dtype: torch.dtype = torch.bfloat16) -> int:
    """Bytes of scratch a call of these sizes needs (caller-owned form)."""
    n = _native.load().mxfp4_expert_linear_workspace_size(
        T, E, I, O, K, _TOKEN_DTYPES[dtype])
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("sizes rejected by the library")
    return n


def mxfp4_expert_linear(latent_tokens: torch.Tensor, packed_weights: torch.Tensor,
                        scale_bytes: torch.Tensor, selected_experts: torch.Tensor,
                        mixture_weights: torch.Tensor, shared_output: torch.Tensor,
                        out: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None) -> torch.Tensor:
    """The routed and shared expert output, shaped like ``shared_output``.

    Shapes: latent_tokens (T, I) fp32 or bf16; packed_weights (E, O, I/32, 16)
    uint8; scale_bytes (E, O, I/32) uint8; selected_experts (T, K) int32 or
    int64; mixture_weights (T, K) fp32; shared_output (T, O) in the token
    dtype. All on one CUDA device. The result has the token's dtype and device
    and is a new tensor unless ``out`` is given. Inputs are not modified.
    ``workspace`` (uint8, at least :func:`workspace_size` bytes) may be
    passed to reuse scratch; otherwise one is taken from torch's allocator.
    """
    x, w, s = latent_tokens, packed_weights, scale_bytes
    sel, p, ys = selected_experts, mixture_weights, shared_output
    if not x.is_cuda:
        raise ValueError("latent_tokens must be a CUDA tensor")
    dev = x.device
    for name, t in (("packed_weights", w), ("scale_bytes", s),
                    ("selected_experts", sel), ("mixture_weights", p),
                    ("shared_output", ys)):
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, tokens on {dev}")
    if x.dtype not in _TOKEN_DTYPES:
        raise TypeError(f"unsupported token dtype {x.dtype}")
    if ys.dtype != x.dtype:
        raise TypeError("shared_output must have the token dtype")
    if w.dtype != torch.uint8 or s.dtype != torch.uint8:
        raise TypeError("packed_weights and scale_bytes must be uint8")
    if sel.dtype not in _INDEX_DTYPES:
        raise TypeError(f"unsupported index dtype {sel.dtype}")
    if p.dtype != torch.float32:
        raise TypeError("mixture_weights must be float32")
    if x.dim() != 2 or w.dim() != 4 or s.dim() != 3 or sel.dim() != 2:
        raise ValueError("expected x (T,I), packed (E,O,G,16), scales (E,O,G), sel (T,K)")
    T, I = x.shape
    E, O, G, sixteen = w.shape
    K = sel.shape[1]
    if sixteen != 16 or I != 32 * G or tuple(s.shape) != (E, O, G):
        raise ValueError("packed/scale shapes do not match the token width")
    if tuple(sel.shape) != (T, K) or tuple(p.shape) != (T, K) or tuple(ys.shape) != (T, O):
        raise ValueError("routing or shared-output shape mismatch")
    x, w, s, sel, p, ys = (t.contiguous() for t in (x, w, s, sel, p, ys))
    if out is None:
        out = torch.empty((T, O), dtype=x.dtype, device=dev)
    elif out.shape != (T, O) or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous (T, O) tensor of the token dtype")
    lib = _native.load()
    ws_bytes = workspace_size(T, E, I, O, K, x.dtype)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        rc = lib.mxfp4_expert_linear_with_workspace(
            _ptr(x), _ptr(w), _ptr(s), _ptr(sel), _ptr(p), _ptr(ys), _ptr(out),
            T, E, I, O, K, _TOKEN_DTYPES[x.dtype], _INDEX_DTYPES[sel.dtype],
            _ptr(workspace), workspace.numel(), ctypes.c_void_p(stream))
    _native.check(rc, "mxfp4_expert_linear")
    return out


def prepared_bytes(E: int, I: int, O: int) -> int:
    """Bytes of the prepared copy of (E, O, I/32) experts' weights."""
    n = _native.load().mxfp4_expert_linear_prepared_bytes(E, I, O)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("sizes rejected by the library")
    return n


class PreparedWeights:
    """The experts' weights laid out once for the kernels.

    ``buffer`` is the uint8 device tensor the library wrote (see
    ``mxfp4_expert_linear_prepare`` in the header for the layout); E, I, O
    are the sizes it was prepared for.
    """

    def __init__(self, buffer: torch.Tensor, E: int, I: int, O: int):
        self.buffer, self.E, self.I, self.O = buffer, E, I, O

    @property
    def device(self):
        return self.buffer.device


def prepare_weights(packed_weights: torch.Tensor, scale_bytes: torch.Tensor) -> PreparedWeights:
    """Lay out packed_weights (E, O, I/32, 16) and scale_bytes (E, O, I/32)
    for :func:`mxfp4_expert_linear_prepared`, on the current stream."""
    w, s = packed_weights, scale_bytes
    if not w.is_cuda or s.device != w.device:
        raise ValueError("packed_weights and scale_bytes must be on one CUDA device")
    if w.dtype != torch.uint8 or s.dtype != torch.uint8:
        raise TypeError("packed_weights and scale_bytes must be uint8")
    if w.dim() != 4 or s.dim() != 3 or w.shape[3] != 16 or tuple(s.shape) != tuple(w.shape[:3]):
        raise ValueError("expected packed (E,O,G,16) and scales (E,O,G)")
    E, O, G, _ = w.shape
    I = 32 * G
    w, s = w.contiguous(), s.contiguous()
    nbytes = prepared_bytes(E, I, O)
    buf = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=w.device)
    stream = torch.cuda.current_stream(w.device).cuda_stream
    with torch.cuda.device(w.device):
        rc = _native.load().mxfp4_expert_linear_prepare(
            _ptr(w), _ptr(s), E, I, O, _ptr(buf), buf.numel(), ctypes.c_void_p(stream))
    _native.check(rc, "mxfp4_expert_linear_prepare")
    return PreparedWeights(buf, E, I, O)


def prepared_workspace_size(T: int, E: int, I: int, O: int, K: int,
                            dtype: torch.dtype = torch.bfloat16) -> int:
    """Bytes of scratch a call on prepared weights of these sizes needs."""
    n = _native.load().mxfp4_expert_linear_prepared_workspace_size(
        T, E, I, O, K, _TOKEN_DTYPES[dtype])
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("sizes rejected by the library")
    return n


def mxfp4_expert_linear_prepared(latent_tokens: torch.Tensor, prepared: PreparedWeights,
                                 selected_experts: torch.Tensor,
                                 mixture_weights: torch.Tensor, shared_output: torch.Tensor,
                                 out: torch.Tensor | None = None,
                                 workspace: torch.Tensor | None = None) -> torch.Tensor:
    """:func:`mxfp4_expert_linear` on weights from :func:`prepare_weights`:
    the same result, bit for bit."""
    x, sel, p, ys = latent_tokens, selected_experts, mixture_weights, shared_output
    if not x.is_cuda:
        raise ValueError("latent_tokens must be a CUDA tensor")
    dev = x.device
    for name, t in (("prepared", prepared.buffer), ("selected_experts", sel),
                    ("mixture_weights", p), ("shared_output", ys)):
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, tokens on {dev}")
    if x.dtype not in _TOKEN_DTYPES:
        raise TypeError(f"unsupported token dtype {x.dtype}")
    if ys.dtype != x.dtype:
        raise TypeError("shared_output must have the token dtype")
    if sel.dtype not in _INDEX_DTYPES:
        raise TypeError(f"unsupported index dtype {sel.dtype}")
    if p.dtype != torch.float32:
        raise TypeError("mixture_weights must be float32")
    if x.dim() != 2 or sel.dim() != 2:
        raise ValueError("expected x (T,I) and sel (T,K)")
    T, I = x.shape
    E, O, K = prepared.E, prepared.O, sel.shape[1]
    if I != prepared.I:
        raise ValueError("the weights were prepared for another token width")
    if tuple(sel.shape) != (T, K) or tuple(p.shape) != (T, K) or tuple(ys.shape) != (T, O):
        raise ValueError("routing or shared-output shape mismatch")
    x, sel, p, ys = (t.contiguous() for t in (x, sel, p, ys))
    if out is None:
        out = torch.empty((T, O), dtype=x.dtype, device=dev)
    elif out.shape != (T, O) or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous (T, O) tensor of the token dtype")
    lib = _native.load()
    ws_bytes = prepared_workspace_size(T, E, I, O, K, x.dtype)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        rc = lib.mxfp4_expert_linear_prepared_with_workspace(
            _ptr(x), _ptr(prepared.buffer), _ptr(sel), _ptr(p), _ptr(ys), _ptr(out),
            T, E, I, O, K, _TOKEN_DTYPES[x.dtype], _INDEX_DTYPES[sel.dtype],
            _ptr(workspace), workspace.numel(), ctypes.c_void_p(stream))
    _native.check(rc, "mxfp4_expert_linear_prepared")
    return out


def _router_args(router_logits, router_bias, K):
    lg = router_logits
    if not lg.is_cuda or lg.dtype != torch.float32 or lg.dim() != 2:
        raise ValueError("router_logits must be a (T, E) float32 CUDA tensor")
    T, E = lg.shape
    if router_bias is not None:
        if (router_bias.device != lg.device or router_bias.dtype != torch.float32
                or tuple(router_bias.shape) != (E,)):
            raise ValueError("router_bias must be an (E,) float32 tensor on the logits' device")
        router_bias = router_bias.contiguous()
    if not 0 <= K <= E:
        raise ValueError("need 0 <= K <= E")
    return lg.contiguous(), router_bias, T, E


def router_topk(router_logits: torch.Tensor, router_bias: torch.Tensor | None, K: int,
                scaling: float = 1.0) -> tuple[torch.Tensor, torch.Tensor]:
    """(selected_experts (T, K) int32, mixture_weights (T, K) float32): the K
    experts of highest sigmoid(logit) + bias per token, highest first, ties to
    the lower index, weighted by their raw scores normalised to sum to
    ``scaling`` (see mxfp4_router_topk in the C header)."""
    lg, b, T, E = _router_args(router_logits, router_bias, K)
    sel = torch.empty((T, K), dtype=torch.int32, device=lg.device)
    p = torch.empty((T, K), dtype=torch.float32, device=lg.device)
    stream = torch.cuda.current_stream(lg.device).cuda_stream
    with torch.cuda.device(lg.device):
        rc = _native.load().mxfp4_router_topk(_ptr(lg), _ptr(b), T, E, K, ctypes.c_float(scaling),
                                              _ptr(sel), _ptr(p), ctypes.c_void_p(stream))
    _native.check(rc, "mxfp4_router_topk")
    return sel, p


def mxfp4_expert_linear_routed(latent_tokens: torch.Tensor, packed_weights: torch.Tensor,
                               scale_bytes: torch.Tensor, router_logits: torch.Tensor,
                               router_bias: torch.Tensor | None, K: int,
                               shared_output: torch.Tensor, scaling: float = 1.0,
                               out: torch.Tensor | None = None
                               ) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """(out, selected_experts, mixture_weights): the router, then the routed
    expert linear on its selection, in one library call on the current
    stream. Shapes as in :func:`mxfp4_expert_linear` and :func:`router_topk`."""
    lg, b, T, E = _router_args(router_logits, router_bias, K)
    x, w, s, ys = latent_tokens, packed_weights, scale_bytes, shared_output
    if x.dtype not in _TOKEN_DTYPES or ys.dtype != x.dtype:
        raise TypeError("tokens and shared_output must share a supported dtype")
    if w.dim() != 4 or tuple(w.shape[:1]) != (E,) or x.dim() != 2 or x.shape[0] != T:
        raise ValueError("expected x (T, I) and packed (E, O, I/32, 16) matching the logits")
    if w.dtype != torch.uint8 or s.dtype != torch.uint8:
        raise TypeError("packed_weights and scale_bytes must be uint8")
    I = x.shape[1]
    O = w.shape[1]
    if tuple(w.shape) != (E, O, I // 32, 16) or tuple(s.shape) != (E, O, I // 32) \
            or tuple(ys.shape) != (T, O):
        raise ValueError("packed, scale or shared-output shape mismatch")
    for t in (w, s, ys):
        if t.device != lg.device or not x.is_cuda or x.device != lg.device:
            raise ValueError("all tensors must be on the logits' CUDA device")
    x, w, s, ys = (t.contiguous() for t in (x, w, s, ys))
    if out is None:
        out = torch.empty((T, O), dtype=x.dtype, device=x.device)
    elif out.shape != (T, O) or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous (T, O) tensor of the token dtype")
    sel = torch.empty((T, K), dtype=torch.int32, device=x.device)
    p = torch.empty((T, K), dtype=torch.float32, device=x.device)
    stream = torch.cuda.current_stream(x.device).cuda_stream
    with torch.cuda.device(x.device):
        rc = _native.load().mxfp4_expert_linear_routed(
            _ptr(x), _ptr(w), _ptr(s), _ptr(lg), _ptr(b), ctypes.c_float(scaling), _ptr(ys),
            _ptr(out), _ptr(sel), _ptr(p), T, E, I, O, K, _TOKEN_DTYPES[x.dtype],
            ctypes.c_void_p(stream))
    _native.check(rc, "mxfp4_expert_linear_routed")
    return out, sel, p


def swiglu_workspace_size(T: int, E: int, I: int, F: int, O: int, K: int,
                          dtype: torch.dtype) -> int:
    """Scratch bytes of one :func:`mxfp4_swiglu_expert` call of these sizes."""
    n = _native.load().mxfp4_swiglu_expert_workspace_size(T, E, I, F, O, K,
                                                          _TOKEN_DTYPES[dtype])
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("sizes rejected by the library")
    return int(n)


def mxfp4_swiglu_expert(latent_tokens: torch.Tensor, gate_up_packed: torch.Tensor,
                        gate_up_scales: torch.Tensor, down_packed: torch.Tensor,
                        down_scales: torch.Tensor, selected_experts: torch.Tensor,
                        mixture_weights: torch.Tensor, shared_output: torch.Tensor,
                        out: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None) -> torch.Tensor:
    """The routed SwiGLU expert: out[t] = shared_output[t] + sum_k p[t,k] *
    Wd_e (silu(Wg_e x_t) * (Wu_e x_t)), e = selected_experts[t, k].

    Shapes: latent_tokens (T, I); gate_up_packed (E, 2F, I/32, 16) uint8 with
    the gate rows first, gate_up_scales (E, 2F, I/32); down_packed
    (E, O, F/32, 16), down_scales (E, O, F/32); routing and shared output as
    in :func:`mxfp4_expert_linear`. All on one CUDA device."""
    x, gw, gs, dw, ds = latent_tokens, gate_up_packed, gate_up_scales, down_packed, down_scales
    sel, p, ys = selected_experts, mixture_weights, shared_output
    if not x.is_cuda:
        raise ValueError("latent_tokens must be a CUDA tensor")
    dev = x.device
    for name, t in (("gate_up_packed", gw), ("gate_up_scales", gs), ("down_packed", dw),
                    ("down_scales", ds), ("selected_experts", sel),
                    ("mixture_weights", p), ("shared_output", ys)):
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, tokens on {dev}")
    if x.dtype not in _TOKEN_DTYPES or ys.dtype != x.dtype:
        raise TypeError("tokens and shared_output must share a supported dtype")
    if any(t.dtype != torch.uint8 for t in (gw, gs, dw, ds)):
        raise TypeError("packed weights and scale bytes must be uint8")
    if sel.dtype not in _INDEX_DTYPES or p.dtype != torch.float32:
        raise TypeError("selected_experts must be int32/int64, mixture_weights float32")
    if x.dim() != 2 or gw.dim() != 4 or dw.dim() != 4 or sel.dim() != 2:
        raise ValueError("expected x (T,I), packed (E,2F,I/32,16), (E,O,F/32,16), sel (T,K)")
    T, I = x.shape
    E, F2, Gi, _ = gw.shape
    F = F2 // 2
    O, Gf = dw.shape[1], dw.shape[2]
    K = sel.shape[1]
    if (F2 % 2 or tuple(gw.shape) != (E, 2 * F, I // 32, 16) or I % 32
            or tuple(gs.shape) != (E, 2 * F, I // 32)
            or tuple(dw.shape) != (E, O, F // 32, 16) or F % 32 or Gf * 32 != F
            or tuple(ds.shape) != (E, O, F // 32)):
        raise ValueError("gate/up or down weight shapes do not match")
    if tuple(sel.shape) != (T, K) or tuple(p.shape) != (T, K) or tuple(ys.shape) != (T, O):
        raise ValueError("routing or shared-output shape mismatch")
    x, gw, gs, dw, ds, sel, p, ys = (t.contiguous() for t in (x, gw, gs, dw, ds, sel, p, ys))
    if out is None:
        out = torch.empty((T, O), dtype=x.dtype, device=dev)
    elif out.shape != (T, O) or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous (T, O) tensor of the token dtype")
    lib = _native.load()
    ws_bytes = swiglu_workspace_size(T, E, I, F, O, K, x.dtype)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        rc = lib.mxfp4_swiglu_expert_with_workspace(
            _ptr(x), _ptr(gw), _ptr(gs), _ptr(dw), _ptr(ds), _ptr(sel), _ptr(p), _ptr(ys),
            _ptr(out), T, E, I, F, O, K, _TOKEN_DTYPES[x.dtype], _INDEX_DTYPES[sel.dtype],
            _ptr(workspace), workspace.numel(), ctypes.c_void_p(stream))
    _native.check(rc, "mxfp4_swiglu_expert")
    return out


def device_errors(device=None) -> int:
    """Pairs with an out-of-range expert id since the last query (syncs)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    n = ctypes.c_int64(0)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        _native.check(_native.load().mxfp4el_device_errors(ctypes.c_void_p(stream),
                                                           ctypes.byref(n)),
                      "mxfp4el_device_errors")
    return int(n.value)


def wait_timeouts(device=None) -> int:
    """Kernel waits that gave up after their time limit since the last query
    (syncs). Always 0 on a healthy device; a nonzero count means the outputs
    of the calls since the last query are not valid."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    n = ctypes.c_int64(0)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        _native.check(_native.load().mxfp4el_wait_timeouts(ctypes.c_void_p(stream),
                                                           ctypes.byref(n)),
                      "mxfp4el_wait_timeouts")
    return int(n.value)
