"""KDA (Kimi Delta Attention) recurrence for NVIDIA GB300 (sm_103a).

Thin Python binding of ``libkda_gb300.so`` (the C ABI in ``include/kda.h``):
it checks and marshals torch tensors into pointers and sizes and calls the
library on torch's current CUDA stream.  Every step of the computation runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback, and the
calls raise if the library has not been built.

    o, S_out = prefill_chunked(q, k, v, g, beta, cu_seqlens, S0=None, chunk=64)
    o, S_out = prefill_chunked_noalloc(...)      # same, no device allocation
    ws = torch.empty(prefill_workspace_bytes(N, T, H), dtype=torch.uint8, device="cuda")
    o, S_out = prefill_chunked(..., workspace=ws) # same, in a workspace the caller owns
    o = decode_step(q, k, v, g, beta, S)          # S updated in place

The layer around the recurrence (conv1d + SiLU + L2 norm before it, gated
RMSNorm after it):

    q, k, v, conv_out = conv_prologue(xq, xk, xv, conv_w, cu_seqlens, conv_in=None)
    out, S_out = prefill_chunked_gated(q, k, v, g, beta, cu_seqlens, gate, norm_w)
    out, S_out, conv_out = prefill_layer(xq, xk, xv, conv_w, g, beta, gate, norm_w, cu_seqlens)
    out = decode_layer_step(xq, xk, xv, conv_w, conv_pool, g, beta, gate, norm_w, S_pool)

Shapes (token-major): q, k, g [T, H, 128]; v [T, H, 128]; beta [T, H];
S [N, H, 128, 128] fp32; q/k/v bf16 or fp32, g/beta fp32.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

__all__ = ["prefill_chunked", "prefill_chunked_noalloc", "prefill_chunked_events",
           "prefill_workspace_bytes", "decode_step",
           "decode_step_pool", "conv_prologue", "prefill_chunked_gated", "prefill_layer",
           "decode_layer_step", "device_error", "lib",
           "KDAError", "KDA_BF16", "KDA_F32", "library_path"]

_PKG = os.path.dirname(os.path.abspath(__file__))
# KDA_GB300_DEBUG=1 loads the debug build (python -m kda_linear_attention_gb300.build
# --debug): the same kernels with index checks that flag bit 3 of the device
# error word instead of touching memory outside a buffer.
_LIB_PATH = os.path.join(_PKG, "libkda_gb300_debug.so" if os.environ.get("KDA_GB300_DEBUG") == "1"
                         else "libkda_gb300.so")
_lib = None

KDA_BF16 = 0
KDA_F32 = 1
DK = 128
DV = 128


class KDAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed with status %d (%s)" % (what, status,
                                                            lib().kda_status_string(status).decode()))


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                "%s is not built (python -m kda_linear_attention_gb300.build%s); "
                "this package has no CPU fallback"
                % (os.path.basename(_LIB_PATH), " --debug" if "debug" in _LIB_PATH else ""))
        L = ctypes.CDLL(_LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.kda_version.argtypes = []
        L.kda_version.restype = i32
        L.kda_status_string.argtypes = [i32]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_prefill_chunked.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                          i32, i64, i32, i32, i32, i32, i32, vp]
        L.kda_prefill_chunked.restype = i32
        L.kda_prefill_chunked_noalloc.argtypes = L.kda_prefill_chunked.argtypes
        L.kda_prefill_chunked_noalloc.restype = i32
        L.kda_prefill_chunked_events.argtypes = L.kda_prefill_chunked.argtypes + [
            ctypes.POINTER(ctypes.c_void_p)]
        L.kda_prefill_chunked_events.restype = i32
        L.kda_prefill_chunked_ws.argtypes = L.kda_prefill_chunked.argtypes[:-1] + [
            vp, ctypes.c_size_t, vp]
        L.kda_prefill_chunked_ws.restype = i32
        L.kda_prefill_workspace_bytes.argtypes = [i32, i64, i32, i32, i32, i32, i32]
        L.kda_prefill_workspace_bytes.restype = ctypes.c_size_t
        L.kda_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
        L.kda_decode_step.restype = i32
        L.kda_decode_step_pool.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, vp, i32, i32,
                                           i32, i32, i32, vp]
        L.kda_decode_step_pool.restype = i32
        f32 = ctypes.c_float
        L.kda_conv_prologue.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32,
                                        f32, f32, vp]
        L.kda_conv_prologue.restype = i32
        L.kda_prefill_chunked_gated.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, f32, vp, vp, vp,
                                                i32, i64, i32, i32, i32, i32, i32, vp]
        L.kda_prefill_chunked_gated.restype = i32
        L.kda_layer_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, f32, f32,
                                        vp, vp, vp, i32, i64, i32, i32, i32, vp]
        L.kda_layer_prefill.restype = i32
        L.kda_decode_layer_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32,
                                            vp, i32, i32, i32, i32, f32, f32, f32, vp]
        L.kda_decode_layer_step.restype = i32
        L.kda_workspace_release.argtypes = []
        L.kda_workspace_release.restype = i32
        L.kda_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint), i32]
        L.kda_device_error.restype = i32
        _lib = L
    return _lib


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _qkv_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError("q, k, v must be bfloat16 or float32, got %s" % t.dtype)


def _check(name: str, t: torch.Tensor, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _stream(device: torch.device, stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _prefill(fn_name: str, q, k, v, g, beta, cu_seqlens, S0, chunk, o, S_out, stream, extra=(),
             gated=None, ws=None):
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    T, H = q.shape[0], q.shape[1]
    N = cu_seqlens.numel() - 1
    dt = _qkv_dtype(q)
    _check("q", q, q.dtype, (T, H, DK), dev)
    _check("k", k, q.dtype, (T, H, DK), dev)
    _check("v", v, q.dtype, (T, H, DV), dev)
    _check("g", g, torch.float32, (T, H, DK), dev)
    _check("beta", beta, torch.float32, (T, H), dev)
    _check("cu_seqlens", cu_seqlens, torch.int32, (N + 1,), dev)
    if S0 is not None:
        _check("S0", S0, torch.float32, (N, H, DK, DV), dev)
    if o is None:
        o = torch.empty((T, H, DV), dtype=torch.float32, device=dev)
    if S_out is None:
        S_out = torch.empty((N, H, DK, DV), dtype=torch.float32, device=dev)
    _check("o", o, torch.float32, (T, H, DV), dev)
    _check("S_out", S_out, torch.float32, (N, H, DK, DV), dev)
    if gated is not None:
        gate, norm_w, eps = gated
        rc = getattr(lib(), fn_name)(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0), _p(gate),
                                     _p(norm_w), float(eps), _p(o), _p(S_out), _p(cu_seqlens), N,
                                     T, H, DK, DV, int(chunk), dt, _stream(dev, stream))
    elif ws is not None:
        rc = getattr(lib(), fn_name)(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0), _p(o),
                                     _p(S_out), _p(cu_seqlens), N, T, H, DK, DV, int(chunk), dt,
                                     ws[0], ctypes.c_size_t(ws[1]), _stream(dev, stream))
    else:
        rc = getattr(lib(), fn_name)(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0), _p(o),
                                     _p(S_out), _p(cu_seqlens), N, T, H, DK, DV, int(chunk), dt,
                                     _stream(dev, stream), *extra)
    if rc != 0:
        raise KDAError(rc, fn_name)
    return o, S_out


def prefill_workspace_bytes(N: int, T: int, H: int, chunk: int = 64, dtype: int = None) -> int:
    """Bytes of workspace ``prefill_chunked(..., workspace=...)`` needs
    (``kda_prefill_workspace_bytes``); 0 where the call needs none."""
    dt = KDA_BF16 if dtype is None else int(dtype)
    return int(lib().kda_prefill_workspace_bytes(int(N), int(T), int(H), DK, DV, int(chunk), dt))


def prefill_chunked(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                    beta: torch.Tensor, cu_seqlens: torch.Tensor,
                    S0: Optional[torch.Tensor] = None, chunk: int = 64,
                    o: Optional[torch.Tensor] = None, S_out: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None,
                    workspace: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Chunked KDA prefill over packed varlen sequences (``kda_prefill_chunked``).

    Returns (o [T, H, 128] fp32, S_out [N, H, 128, 128] fp32).  ``S_out`` may
    be ``S0`` itself to update the states in place.  With ``workspace`` (a
    contiguous CUDA tensor of at least ``prefill_workspace_bytes`` bytes) the
    call runs in that buffer (``kda_prefill_chunked_ws``) instead of the
    library's own pool.
    """
    if workspace is not None:
        if workspace.device != q.device or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on the inputs' device")
        nbytes = workspace.numel() * workspace.element_size()
        return _prefill("kda_prefill_chunked_ws", q, k, v, g, beta, cu_seqlens, S0, chunk, o,
                        S_out, stream, ws=(_p(workspace), nbytes))
    return _prefill("kda_prefill_chunked", q, k, v, g, beta, cu_seqlens, S0, chunk, o, S_out,
                    stream)


def prefill_chunked_events(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                           beta: torch.Tensor, cu_seqlens: torch.Tensor, events,
                           S0: Optional[torch.Tensor] = None,
                           o: Optional[torch.Tensor] = None, S_out: Optional[torch.Tensor] = None,
                           stream: Optional[torch.cuda.Stream] = None
                           ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Tensor-core ``prefill_chunked`` (bf16, chunk 64) that also records four
    ``torch.cuda.Event`` (timing enabled) around its kernels: before the chunk
    plan, before the intra-chunk kernel, before the state pass, after it
    (``kda_prefill_chunked_events``)."""
    if len(events) != 4:
        raise ValueError("need four events")
    s = torch.cuda.current_stream(q.device) if stream is None else stream
    for e in events:
        if not e.cuda_event:          # torch creates the CUDA event at its first record
            e.record(s)
    evs = [ctypes.c_void_p(e.cuda_event) for e in events]
    arr = (ctypes.c_void_p * 4)(*evs)
    return _prefill("kda_prefill_chunked_events", q, k, v, g, beta, cu_seqlens, S0, 64, o, S_out,
                    stream, extra=(ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)),))


def prefill_chunked_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                            beta: torch.Tensor, cu_seqlens: torch.Tensor,
                            S0: Optional[torch.Tensor] = None, chunk: int = 64,
                            o: Optional[torch.Tensor] = None, S_out: Optional[torch.Tensor] = None,
                            stream: Optional[torch.cuda.Stream] = None
                            ) -> Tuple[torch.Tensor, torch.Tensor]:
    """``prefill_chunked`` through ``kda_prefill_chunked_noalloc``: the library
    allocates nothing (its fixed scratch array bounds the input size; pass
    ``o`` and ``S_out`` to keep this binding from allocating them either)."""
    return _prefill("kda_prefill_chunked_noalloc", q, k, v, g, beta, cu_seqlens, S0, chunk, o,
                    S_out, stream)


def decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                beta: torch.Tensor, S: torch.Tensor, o: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """One decode token per sequence (``kda_decode_step``); ``S`` is updated in place.

    q, k, g [B, H, 128]; v [B, H, 128]; beta [B, H]; S [B, H, 128, 128] fp32.
    Returns o [B, H, 128] fp32.
    """
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, H = q.shape[0], q.shape[1]
    dt = _qkv_dtype(q)
    _check("q", q, q.dtype, (B, H, DK), dev)
    _check("k", k, q.dtype, (B, H, DK), dev)
    _check("v", v, q.dtype, (B, H, DV), dev)
    _check("g", g, torch.float32, (B, H, DK), dev)
    _check("beta", beta, torch.float32, (B, H), dev)
    _check("S", S, torch.float32, (B, H, DK, DV), dev)
    if o is None:
        o = torch.empty((B, H, DV), dtype=torch.float32, device=dev)
    _check("o", o, torch.float32, (B, H, DV), dev)
    rc = lib().kda_decode_step(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S), _p(o), B, H, DK, DV,
                               dt, _stream(dev, stream))
    if rc != 0:
        raise KDAError(rc, "kda_decode_step")
    return o


def decode_step_pool(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                     beta: torch.Tensor, S_pool: torch.Tensor,
                     state_indices: Optional[torch.Tensor] = None,
                     o: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """One decode token per sequence on a state pool (``kda_decode_step_pool``).

    S_pool [P, H, 128, 128] fp32 or bf16 is updated in place at rows
    ``state_indices`` ([B] int32; negative = padding, o row zero), or at rows
    0..B-1 when it is None.  Returns o [B, H, 128] fp32.
    """
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, H = q.shape[0], q.shape[1]
    dt = _qkv_dtype(q)
    _check("q", q, q.dtype, (B, H, DK), dev)
    _check("k", k, q.dtype, (B, H, DK), dev)
    _check("v", v, q.dtype, (B, H, DV), dev)
    _check("g", g, torch.float32, (B, H, DK), dev)
    _check("beta", beta, torch.float32, (B, H), dev)
    if S_pool.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("S_pool must be float32 or bfloat16")
    P = S_pool.shape[0]
    _check("S_pool", S_pool, S_pool.dtype, (P, H, DK, DV), dev)
    if state_indices is not None:
        _check("state_indices", state_indices, torch.int32, (B,), dev)
    if o is None:
        o = torch.empty((B, H, DV), dtype=torch.float32, device=dev)
    _check("o", o, torch.float32, (B, H, DV), dev)
    sdt = KDA_BF16 if S_pool.dtype == torch.bfloat16 else KDA_F32
    rc = lib().kda_decode_step_pool(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S_pool), sdt,
                                    _p(state_indices), P, _p(o), B, H, DK, DV, dt,
                                    _stream(dev, stream))
    if rc != 0:
        raise KDAError(rc, "kda_decode_step_pool")
    return o


# ------------------------------------------------------------ the layer
CONV_K = 4
Q_SCALE = DK ** -0.5          # the pages' q scale, 1/sqrt(head width)
L2_EPS = 1e-6
NORM_EPS = 1e-6


def conv_prologue(xq: torch.Tensor, xk: torch.Tensor, xv: torch.Tensor, conv_w: torch.Tensor,
                  cu_seqlens: torch.Tensor, conv_in: Optional[torch.Tensor] = None,
                  conv_out: Optional[torch.Tensor] = None, q_scale: float = Q_SCALE,
                  eps: float = L2_EPS, q=None, k=None, v=None,
                  stream: Optional[torch.cuda.Stream] = None):
    """conv1d + SiLU + L2 norm of the raw projections (``kda_conv_prologue``).

    xq, xk, xv [T, H, 128] bf16; conv_w [3, H, 128, 4] fp32; conv_in / conv_out
    [N, 3, 3, H, 128] bf16 windows (conv_in None = zeros; conv_out allocated
    if None).  Returns (q, k, v [T, H, 128] bf16, conv_out).
    """
    dev = xq.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    T, H = xq.shape[0], xq.shape[1]
    N = cu_seqlens.numel() - 1
    bf = torch.bfloat16
    for n, t in (("xq", xq), ("xk", xk), ("xv", xv)):
        _check(n, t, bf, (T, H, DK), dev)
    _check("conv_w", conv_w, torch.float32, (3, H, DK, CONV_K), dev)
    _check("cu_seqlens", cu_seqlens, torch.int32, (N + 1,), dev)
    wshape = (N, 3, CONV_K - 1, H, DK)
    if conv_in is not None:
        _check("conv_in", conv_in, bf, wshape, dev)
    if conv_out is None:
        conv_out = torch.empty(wshape, dtype=bf, device=dev)
    _check("conv_out", conv_out, bf, wshape, dev)
    q = torch.empty((T, H, DK), dtype=bf, device=dev) if q is None else q
    k = torch.empty((T, H, DK), dtype=bf, device=dev) if k is None else k
    v = torch.empty((T, H, DV), dtype=bf, device=dev) if v is None else v
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check(n, t, bf, (T, H, DK), dev)
    rc = lib().kda_conv_prologue(_p(xq), _p(xk), _p(xv), _p(conv_w), _p(conv_in), _p(conv_out),
                                 _p(q), _p(k), _p(v), _p(cu_seqlens), N, T, H, DK,
                                 float(q_scale), float(eps), _stream(dev, stream))
    if rc != 0:
        raise KDAError(rc, "kda_conv_prologue")
    return q, k, v, conv_out


def prefill_chunked_gated(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                          beta: torch.Tensor, cu_seqlens: torch.Tensor, gate: torch.Tensor,
                          norm_w: torch.Tensor, S0: Optional[torch.Tensor] = None,
                          chunk: int = 64, eps: float = NORM_EPS,
                          out: Optional[torch.Tensor] = None, S_out: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None
                          ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Chunked prefill whose output is RMSNorm(o) * norm_w * sigmoid(gate)
    (``kda_prefill_chunked_gated``).  gate [T, H, 128] bf16, norm_w [128] fp32.
    Returns (out [T, H, 128] fp32, S_out)."""
    dev = q.device
    T, H = q.shape[0], q.shape[1]
    _check("gate", gate, torch.bfloat16, (T, H, DV), dev)
    _check("norm_w", norm_w, torch.float32, (DV,), dev)
    return _prefill("kda_prefill_chunked_gated", q, k, v, g, beta, cu_seqlens, S0, chunk, out,
                    S_out, stream, gated=(gate, norm_w, eps))


def prefill_layer(xq, xk, xv, conv_w, g, beta, gate, norm_w, cu_seqlens,
                  conv_in: Optional[torch.Tensor] = None, S0: Optional[torch.Tensor] = None,
                  q_scale: float = Q_SCALE, l2_eps: float = L2_EPS, norm_eps: float = NORM_EPS,
                  out: Optional[torch.Tensor] = None, S_out: Optional[torch.Tensor] = None,
                  conv_out: Optional[torch.Tensor] = None, one_call: bool = True,
                  stream: Optional[torch.cuda.Stream] = None):
    """The layer's prefill from raw projections in one C call
    (``kda_layer_prefill``: the conv + SiLU + L2-norm prologue, then the
    gated prefill, q, k, v in the library's workspace).  one_call=False runs
    the same layer as the two public calls, ``conv_prologue`` (q, k, v in
    tensors of this binding) then ``prefill_chunked_gated``.  Returns
    (out [T, H, 128] fp32, S_out [N, H, 128, 128] fp32,
    conv_out [N, 3, 3, H, 128] bf16)."""
    if not one_call:
        q, k, v, conv_out = conv_prologue(xq, xk, xv, conv_w, cu_seqlens, conv_in=conv_in,
                                          conv_out=conv_out, q_scale=q_scale, eps=l2_eps,
                                          stream=stream)
        out, S_out = prefill_chunked_gated(q, k, v, g, beta, cu_seqlens, gate, norm_w, S0=S0,
                                           eps=norm_eps, out=out, S_out=S_out, stream=stream)
        return out, S_out, conv_out
    dev = xq.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    T, H = xq.shape[0], xq.shape[1]
    N = cu_seqlens.numel() - 1
    bf = torch.bfloat16
    for n, t in (("xq", xq), ("xk", xk), ("xv", xv), ("gate", gate)):
        _check(n, t, bf, (T, H, DK), dev)
    _check("conv_w", conv_w, torch.float32, (3, H, DK, CONV_K), dev)
    _check("g", g, torch.float32, (T, H, DK), dev)
    _check("beta", beta, torch.float32, (T, H), dev)
    _check("norm_w", norm_w, torch.float32, (DV,), dev)
    _check("cu_seqlens", cu_seqlens, torch.int32, (N + 1,), dev)
    wshape = (N, 3, CONV_K - 1, H, DK)
    if conv_in is not None:
        _check("conv_in", conv_in, bf, wshape, dev)
    if conv_out is None:
        conv_out = torch.empty(wshape, dtype=bf, device=dev)
    _check("conv_out", conv_out, bf, wshape, dev)
    if S0 is not None:
        _check("S0", S0, torch.float32, (N, H, DK, DV), dev)
    if out is None:
        out = torch.empty((T, H, DV), dtype=torch.float32, device=dev)
    if S_out is None:
        S_out = torch.empty((N, H, DK, DV), dtype=torch.float32, device=dev)
    _check("out", out, torch.float32, (T, H, DV), dev)
    _check("S_out", S_out, torch.float32, (N, H, DK, DV), dev)
    rc = lib().kda_layer_prefill(_p(xq), _p(xk), _p(xv), _p(conv_w), _p(conv_in), _p(conv_out),
                                 _p(g), _p(beta), _p(S0), _p(gate), _p(norm_w), float(q_scale),
                                 float(l2_eps), float(norm_eps), _p(out), _p(S_out),
                                 _p(cu_seqlens), N, T, H, DK, DV, _stream(dev, stream))
    if rc != 0:
        raise KDAError(rc, "kda_layer_prefill")
    return out, S_out, conv_out


def decode_layer_step(xq: torch.Tensor, xk: torch.Tensor, xv: torch.Tensor, conv_w: torch.Tensor,
                      conv_pool: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                      gate: torch.Tensor, norm_w: torch.Tensor, S_pool: torch.Tensor,
                      state_indices: Optional[torch.Tensor] = None, q_scale: float = Q_SCALE,
                      l2_eps: float = L2_EPS, norm_eps: float = NORM_EPS,
                      out: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """One token of the whole layer per sequence (``kda_decode_layer_step``):
    conv windows (conv_pool [P, 3, 3, H, 128] bf16) and states (S_pool
    [P, H, 128, 128] fp32 or bf16) updated in place at rows state_indices.
    Returns out [B, H, 128] fp32."""
    dev = xq.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, H = xq.shape[0], xq.shape[1]
    bf = torch.bfloat16
    for n, t in (("xq", xq), ("xk", xk), ("xv", xv), ("gate", gate)):
        _check(n, t, bf, (B, H, DK), dev)
    _check("conv_w", conv_w, torch.float32, (3, H, DK, CONV_K), dev)
    _check("g", g, torch.float32, (B, H, DK), dev)
    _check("beta", beta, torch.float32, (B, H), dev)
    _check("norm_w", norm_w, torch.float32, (DV,), dev)
    if S_pool.dtype not in (torch.float32, bf):
        raise TypeError("S_pool must be float32 or bfloat16")
    P = S_pool.shape[0]
    _check("S_pool", S_pool, S_pool.dtype, (P, H, DK, DV), dev)
    _check("conv_pool", conv_pool, bf, (P, 3, CONV_K - 1, H, DK), dev)
    if state_indices is not None:
        _check("state_indices", state_indices, torch.int32, (B,), dev)
    if out is None:
        out = torch.empty((B, H, DV), dtype=torch.float32, device=dev)
    _check("out", out, torch.float32, (B, H, DV), dev)
    sdt = KDA_BF16 if S_pool.dtype == bf else KDA_F32
    rc = lib().kda_decode_layer_step(_p(xq), _p(xk), _p(xv), _p(conv_w), _p(conv_pool), _p(g),
                                     _p(beta), _p(gate), _p(norm_w), _p(S_pool), sdt,
                                     _p(state_indices), P, _p(out), B, H, DK, DV, float(q_scale),
                                     float(l2_eps), float(norm_eps), _stream(dev, stream))
    if rc != 0:
        raise KDAError(rc, "kda_decode_layer_step")
    return out


def device_error(reset: bool = True) -> int:
    """The library's device-side error word (``kda_device_error``); nonzero if
    a bounded wait inside a kernel gave up since the last reset."""
    code = ctypes.c_uint(0)
    rc = lib().kda_device_error(ctypes.byref(code), int(reset))
    if rc != 0:
        raise KDAError(rc, "kda_device_error")
    return int(code.value)


def workspace_release() -> None:
    """Give the library's workspace pool memory on the current device back to
    the driver (``kda_workspace_release``); synchronise the streams that ran
    prefills first."""
    rc = lib().kda_workspace_release()
    if rc != 0:
        raise KDAError(rc, "kda_workspace_release")
