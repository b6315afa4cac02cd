"""Exact attention for one GB300 (sm_103a): Python binding of libfa.

The functions named like the C ABI (``fa_fwd``, ``fa_bwd``, ``fa_get_status``,
``fa_status_string``, ``fa_debug_set``, ``fa_debug_exp2``) only marshal
arguments: pointers may be given as ints or as CUDA tensors, the stream as an
int, a ``torch.cuda.Stream`` or None (the current stream). They return the
library's integer status. ``forward`` and ``backward`` allocate outputs with
torch, call the C ABI and raise ``FAError`` on a non-zero status.

Every computation runs in the CUDA kernels of libfa.so; there is no fallback.
If the library is missing the import of this module still succeeds (so it can
be built), but every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

__all__ = ["FAError", "lib", "fa_fwd", "fa_bwd", "fa_bwd_noalloc", "fa_bwd_launches", "fa_get_status", "fa_status_string", "fa_debug_set",
           "fa_debug_exp2", "fa_tune", "TUNE_EXP2_SPLIT", "TUNE_CTA_PAIRS", "TUNE_BWD_SPLIT", "fa_profile_events", "fa_trace", "forward", "backward", "STATUS"]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

STATUS = {
    0: "FA_OK",
    1: "FA_ERR_INVALID_ARG",
    2: "FA_ERR_UNSUPPORTED",
    3: "FA_ERR_ALLOC",
    4: "FA_ERR_LAUNCH",
    5: "FA_ERR_TIMEOUT",
    6: "FA_ERR_NO_DEVICE",
}


class FAError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Load libfa.so (built in-tree). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libfa.so is not built ({LIB_PATH}); run exact_attention_99_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, ull = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_ulonglong
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        L.fa_fwd.restype = i
        L.fa_fwd_window.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp]
        L.fa_fwd_window.restype = i
        L.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp]
        L.fa_fwd_fp8.restype = i
        L.fa_bwd.argtypes = [vp] * 9 + [i, i, i, i, i, i, f, i, vp]
        L.fa_step_host.argtypes = [vp] * 9 + [i, i, i, i, i, i, f, i, vp]
        L.fa_step_host.restype = i
        L.fa_bwd.restype = i
        L.fa_bwd_window.argtypes = [vp] * 9 + [i, i, i, i, i, i, f, i, i, vp]
        L.fa_bwd_window.restype = i
        L.fa_bwd_noalloc.argtypes = [vp] * 9 + [i, i, i, i, i, i, f, i, vp]
        L.fa_bwd_noalloc.restype = i
        L.fa_bwd_launches.argtypes = [i] * 7
        L.fa_bwd_launches.restype = i
        L.fa_get_status.argtypes = [vp]
        L.fa_get_status.restype = i
        L.fa_status_string.argtypes = [i]
        L.fa_status_string.restype = ctypes.c_char_p
        L.fa_debug_set.argtypes = [ull, i]
        L.fa_debug_set.restype = i
        L.fa_profile_events.argtypes = [vp, vp]
        L.fa_profile_events.restype = i
        L.fa_trace.argtypes = [vp]
        L.fa_trace.restype = i
        L.fa_debug_exp2.argtypes = [vp, vp, i, i, vp]
        L.fa_debug_exp2.restype = i
        L.fa_tune.argtypes = [i, i]
        L.fa_tune.restype = i
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def fa_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, stream=None) -> int:
    return lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d, float(scale),
                        int(causal), _stream(stream))


def fa_fwd_window(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, window_left, window_right, stream=None) -> int:
    return lib().fa_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d, float(scale),
                               int(window_left), int(window_right), _stream(stream))


def fa_step_host(q, k, v, dout, o, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, scale, causal, stream=None) -> int:
    """Forward + backward on host (CPU, preferably pinned) tensors; see fa.h fa_step_host."""
    return lib().fa_step_host(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(o), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                              B, Hq, Hkv, Nq, Nk, d, float(scale), int(causal), _stream(stream))


def fa_fwd_fp8(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, incoherent=1, stream=None) -> int:
    return lib().fa_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d, float(scale),
                            int(causal), int(incoherent), _stream(stream))


def forward_fp8(q, k, v, causal: bool = False, scale: float | None = None, incoherent: bool = True, stream=None):
    """O, LSE of the e4m3 forward (d = 128; see fa.h fa_fwd_fp8)."""
    import torch
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    _check_bshd("q", q, B, Nq, Hq, d)
    _check_bshd("k", k, B, Nk, Hkv, d)
    _check_bshd("v", v, B, Nk, Hkv, d)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), device=q.device, dtype=torch.float32)
    st = fa_fwd_fp8(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, int(incoherent), stream)
    if st != 0:
        raise FAError(st, "fa_fwd_fp8")
    return o, lse


def _window_args(causal, window):
    """(left, right) bounds for the *_window calls; causal caps right at 0."""
    wl, wr = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    if causal:
        wr = 0 if wr < 0 else min(wr, 0)
    return wl, wr


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, scale, causal, stream=None) -> int:
    return lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                        B, Hq, Hkv, Nq, Nk, d, float(scale), int(causal), _stream(stream))


def fa_bwd_window(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, scale, window_left, window_right,
                  stream=None) -> int:
    return lib().fa_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                               _ptr(dv), B, Hq, Hkv, Nq, Nk, d, float(scale), int(window_left), int(window_right),
                               _stream(stream))


def fa_bwd_launches(B, Hq, Hkv, Nq, Nk, d, causal) -> int:
    """Kernels fa_bwd launches for this problem (see fa.h), or minus a status."""
    return lib().fa_bwd_launches(int(B), int(Hq), int(Hkv), int(Nq), int(Nk), int(d), int(causal))


def fa_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, scale, causal, stream=None) -> int:
    """fa_bwd with its workspace in the library's fixed device array (no
    device allocation during the call; see fa.h for the size limit)."""
    return lib().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                _ptr(dv), B, Hq, Hkv, Nq, Nk, d, float(scale), int(causal), _stream(stream))


def fa_get_status(stream=None) -> int:
    return lib().fa_get_status(_stream(stream))


def fa_status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def fa_debug_set(wait_limit_ns: int = 0, inject: int = 0) -> int:
    return lib().fa_debug_set(int(wait_limit_ns), int(inject))


def fa_profile_events(begin=None, end=None) -> int:
    """begin/end: torch.cuda.Event (created with enable_timing) or None."""
    b = None if begin is None else begin.cuda_event
    e = None if end is None else end.cuda_event
    return lib().fa_profile_events(b, e)


TRACE_CTAS, TRACE_STEPS, TRACE_POINTS = 4, 64, 16


def fa_trace(buf=None) -> int:
    """buf: CUDA int64 tensor of TRACE_CTAS*TRACE_STEPS*TRACE_POINTS words, or None."""
    return lib().fa_trace(_ptr(buf))


TUNE_EXP2_SPLIT = 1
TUNE_CTA_PAIRS = 2
TUNE_BWD_SPLIT = 3


def fa_tune(knob: int, value: int) -> int:
    """Process-wide tuning knob (see fa.h fa_tune); TUNE_EXP2_SPLIT: 0 = every
    forward exponential on the special-function unit, N in {1, 2, 4, 8} = one
    column pair in every N on the FMA-pipe polynomial; TUNE_CTA_PAIRS: 1 = the
    d = 128 forward on pairs of CTAs (cta_group::2), 0 = one CTA per SM;
    TUNE_BWD_SPLIT: -1 = the causal backward's split count from its model,
    m >= 0 = that many pairs per kv head run as single tiles."""
    return lib().fa_tune(int(knob), int(value))


def fa_debug_exp2(x, y, n, mode, stream=None) -> int:
    return lib().fa_debug_exp2(_ptr(x), _ptr(y), int(n), int(mode), _stream(stream))


def _check_bshd(name, t, B, N, H, d):
    import torch
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (B, N, H, d):
        raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor of shape {(B, N, H, d)}")


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, stream=None, window=None):
    """O, LSE for q [B,Nq,Hq,d], k/v [B,Nk,Hkv,d] (bf16, CUDA, contiguous).
    window: optional (left, right) sliding-window bounds (see fa.h)."""
    import torch
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    _check_bshd("q", q, B, Nq, Hq, d)
    _check_bshd("k", k, B, Nk, Hkv, d)
    _check_bshd("v", v, B, Nk, Hkv, d)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if out is None:
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, Nq), device=q.device, dtype=torch.float32)
    else:
        o, lse = out
    if window is None:
        st = fa_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, stream)
    else:
        st = fa_fwd_window(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, *_window_args(causal, window), stream)
    if st != 0:
        raise FAError(st, "fa_fwd")
    return o, lse


def backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, out=None, stream=None,
             window=None):
    """dQ, dK, dV for the forward that produced o and lse (same causal flag
    and window)."""
    import torch
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    for name, t, N, H in (("q", q, Nq, Hq), ("k", k, Nk, Hkv), ("v", v, Nk, Hkv), ("o", o, Nq, Hq),
                          ("dout", dout, Nq, Hq)):
        _check_bshd(name, t, B, N, H, d)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = out
    if window is None:
        st = fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, scale, causal, stream)
    else:
        st = fa_bwd_window(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, scale,
                           *_window_args(causal, window), stream)
    if st != 0:
        raise FAError(st, "fa_bwd")
    return dq, dk, dv
