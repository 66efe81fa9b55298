"""GB300 (sm_103a) fused exact attention: forward and backward.

A thin ctypes binding of the C ABI in ``include/attn_fwd.h``,
``include/attn_bwd.h`` and ``include/attn_fp8.h`` (the library
``_build/libattn_fwd.so``, built by ``build.py``).  The functions here only
marshal arguments: every step of the computation runs in the library's CUDA
kernels.  There is no CPU path: calling the library without it built, or on a
device other than sm_103, raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

__all__ = ["attn_fwd", "attn_bwd", "attn_bwd_window", "attn_fwd_fp8", "attn_fwd_fp8_codes", "attn_fp8_quantize_qk", "attn_fp8_quantize_v",
           "attn_fwd_ex", "attn_fwd_host", "attn_fwd_noalloc", "attn_fwd_noalloc_ex",
           "attn_fwd_noalloc_last_device_error", "attn_device_bytes", "attn_fwd_window", "attn_fwd_kvsplit", "attn_fwd_decode", "attn_last_device_error", "attn_last_error_site",
           "attn_status_string", "AttnError", "AttnFwdOptions", "lib", "forward", "backward", "decode",
           "EXPORTED_SYMBOLS"]

# Every symbol the headers under include/ declare.
EXPORTED_SYMBOLS = ("attn_fwd", "attn_fwd_ex", "attn_fwd_host", "attn_fwd_decode", "attn_last_device_error", "attn_last_error_site",
                    "attn_last_cuda_error", "attn_status_string", "attn_fwd_noalloc",
                    "attn_fwd_noalloc_ex", "attn_fwd_noalloc_last_device_error", "attn_device_bytes",
                    "attn_fwd_window", "attn_fwd_kvsplit", "attn_bwd", "attn_bwd_window",
                    "attn_fwd_fp8", "attn_fwd_fp8_codes",
                    "attn_fp8_quantize_qk", "attn_fp8_quantize_v")

ATTN_OK = 0


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str = "attn_fwd"):
        self.status = status
        extra = f" (cudaError {lib().attn_last_cuda_error()})" if status == -6 else ""
        super().__init__(f"{what} failed: {attn_status_string(status)} [{status}]{extra}")


class AttnFwdOptions(ctypes.Structure):
    _fields_ = [("wait_timeout_ns", ctypes.c_uint64),
                ("fault_inject", ctypes.c_int),
                ("max_ctas", ctypes.c_int),
                ("kernel", ctypes.c_int)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} is missing "
                               "(run `python -m io_aware_exact_06_gb300.build`)")
        L = ctypes.CDLL(path)
        vp, i = ctypes.c_void_p, ctypes.c_int
        sig = [vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float, i, vp, vp]
        L.attn_fwd.argtypes = sig
        L.attn_fwd.restype = i
        L.attn_fwd_ex.argtypes = sig + [ctypes.POINTER(AttnFwdOptions)]
        L.attn_fwd_ex.restype = i
        L.attn_fwd_window.argtypes = sig[:11] + [i, i] + sig[11:]
        L.attn_fwd_window.restype = i
        L.attn_fwd_kvsplit.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, i, vp]
        L.attn_fwd_kvsplit.restype = i
        L.attn_fwd_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, ctypes.c_float, vp, i, i, vp]
        L.attn_fwd_decode.restype = i
        L.attn_bwd.argtypes = [vp] * 9 + [i, i, i, i, ctypes.c_float, i, vp, vp]
        L.attn_bwd.restype = i
        L.attn_bwd_window.argtypes = [vp] * 9 + [i, i, i, i, ctypes.c_float, i, i, i, vp, vp]
        L.attn_bwd_window.restype = i
        L.attn_fwd_fp8.argtypes = sig[:11] + [vp, vp, vp]
        L.attn_fwd_fp8.restype = i
        L.attn_fwd_fp8_codes.argtypes = [vp] * 8 + [i, i, i, i, ctypes.c_float, i, i, vp, vp]
        L.attn_fwd_fp8_codes.restype = i
        L.attn_fp8_quantize_qk.argtypes = [vp, vp, vp, i, i, i, i, vp, vp, vp]
        L.attn_fp8_quantize_qk.restype = i
        L.attn_fp8_quantize_v.argtypes = [vp, vp, vp, i, i, i, i, vp, vp]
        L.attn_fp8_quantize_v.restype = i
        L.attn_fwd_noalloc.argtypes = sig
        L.attn_fwd_noalloc.restype = i
        L.attn_fwd_noalloc_ex.argtypes = sig + [ctypes.POINTER(AttnFwdOptions)]
        L.attn_fwd_noalloc_ex.restype = i
        L.attn_fwd_noalloc_last_device_error.argtypes = [vp]
        L.attn_fwd_noalloc_last_device_error.restype = i
        L.attn_device_bytes.argtypes = []
        L.attn_device_bytes.restype = ctypes.c_size_t
        L.attn_fwd_host.argtypes = sig
        L.attn_fwd_host.restype = i
        L.attn_last_device_error.argtypes = [vp]
        L.attn_last_device_error.restype = i
        L.attn_last_error_site.restype = i
        L.attn_last_cuda_error.restype = i
        L.attn_status_string.argtypes = [i]
        L.attn_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _ptr(x) -> int | None:
    """A buffer address from a torch tensor, an int address or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None or isinstance(stream, int):
        return stream
    return stream.cuda_stream  # torch.cuda.Stream


def attn_status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def attn_fwd(q, k, v, o, lse, B: int, H: int, N: int, d: int, scale: float, causal: bool,
             cu_seqlens=None, stream=None) -> int:
    """The C call ``attn_fwd`` with the same arguments (tensors or addresses).

    Raises AttnError on a non-zero status; returns 0."""
    st = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N),
                        int(d), float(scale), int(bool(causal)), _ptr(cu_seqlens), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st)
    return st


def attn_fwd_host(q, k, v, o, lse, B: int, H: int, N: int, d: int, scale: float, causal: bool,
                  cu_seqlens=None, stream=None) -> int:
    """The C call ``attn_fwd_host``: attn_fwd on host buffers (CPU tensors,
    page-locked for overlapped copies, or addresses), cu_seqlens included."""
    st = lib().attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N),
                             int(d), float(scale), int(bool(causal)), _ptr(cu_seqlens),
                             _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st)
    return st


def attn_fwd_ex(q, k, v, o, lse, B: int, H: int, N: int, d: int, scale: float, causal: bool,
                cu_seqlens=None, stream=None, wait_timeout_ns: int = 0, fault_inject: int = 0,
                max_ctas: int = 0, kernel: int = 0) -> int:
    """The C call ``attn_fwd_ex``; options as keyword arguments (kernel: 0 the
    library's choice, 1 one CTA per unit, 2 a pair of SMs, for d = 128)."""
    opts = AttnFwdOptions(int(wait_timeout_ns), int(fault_inject), int(max_ctas), int(kernel))
    st = lib().attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N),
                           int(d), float(scale), int(bool(causal)), _ptr(cu_seqlens),
                           _stream(stream), ctypes.byref(opts))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_ex")
    return st


def attn_fwd_window(q, k, v, o, lse, B: int, H: int, N: int, d: int, scale: float, causal: bool,
                    window_left: int, window_right: int, cu_seqlens=None, stream=None) -> int:
    """The C call ``attn_fwd_window``: keys i - window_left <= j <= i + window_right
    (-1: unbounded side)."""
    st = lib().attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                               int(N), int(d), float(scale), int(bool(causal)), int(window_left),
                               int(window_right), _ptr(cu_seqlens), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_window")
    return st


def attn_fwd_kvsplit(q, k, v, o, lse, B: int, H: int, Nq: int, Nk: int, d: int, scale: float,
                     causal: bool, num_splits: int = 0, stream=None) -> int:
    """The C call ``attn_fwd_kvsplit``: Nq queries against Nk keys, the keys cut
    into num_splits ranges (0: automatic) merged afterwards."""
    st = lib().attn_fwd_kvsplit(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                                int(Nq), int(Nk), int(d), float(scale), int(bool(causal)),
                                int(num_splits), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_kvsplit")
    return st


def attn_fwd_decode(q, k, v, o, lse, B: int, H: int, d: int, scale: float, cu_seqlens_k,
                    max_seqlen_k: int, num_splits: int = 0, stream=None) -> int:
    """The C call ``attn_fwd_decode``: one query per sequence against its packed keys."""
    st = lib().attn_fwd_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(d),
                               float(scale), _ptr(cu_seqlens_k), int(max_seqlen_k), int(num_splits),
                               _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_decode")
    return st


def attn_fwd_noalloc(q, k, v, o, lse, B: int, H: int, N: int, d: int, scale: float, causal: bool,
                     cu_seqlens=None, stream=None) -> int:
    """The C call ``attn_fwd_noalloc``: attn_fwd without any device allocation
    (fixed library scratch; for callers that cannot call cudaMalloc)."""
    st = lib().attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                                int(N), int(d), float(scale), int(bool(causal)),
                                _ptr(cu_seqlens), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_noalloc")
    return st


def attn_fwd_noalloc_ex(q, k, v, o, lse, B: int, H: int, N: int, d: int, scale: float,
                        causal: bool, cu_seqlens=None, stream=None, wait_timeout_ns: int = 0,
                        fault_inject: int = 0, max_ctas: int = 0) -> int:
    """The C call ``attn_fwd_noalloc_ex``: attn_fwd_noalloc with attn_fwd_ex's options."""
    opts = AttnFwdOptions(int(wait_timeout_ns), int(fault_inject), int(max_ctas), 0)
    st = lib().attn_fwd_noalloc_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                                   int(N), int(d), float(scale), int(bool(causal)),
                                   _ptr(cu_seqlens), _stream(stream), ctypes.byref(opts))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_noalloc_ex")
    return st


def attn_fwd_noalloc_last_device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error status
    of attn_fwd_noalloc's scratch."""
    return lib().attn_fwd_noalloc_last_device_error(_stream(stream))


def attn_device_bytes() -> int:
    """Bytes of device memory the library holds in its own workspaces."""
    return int(lib().attn_device_bytes())


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B: int, H: int, N: int, d: int, scale: float,
             causal: bool, cu_seqlens=None, stream=None) -> int:
    """The C call ``attn_bwd``: dQ, dK, dV of attn_fwd for the upstream gradient dout."""
    st = lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                        _ptr(dk), _ptr(dv), int(B), int(H), int(N), int(d), float(scale),
                        int(bool(causal)), _ptr(cu_seqlens), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")
    return st


def attn_bwd_window(q, k, v, o, dout, lse, dq, dk, dv, B: int, H: int, N: int, d: int,
                    scale: float, causal: bool, window_left: int, window_right: int,
                    cu_seqlens=None, stream=None) -> int:
    """The C call ``attn_bwd_window`` (the sliding window of attn_fwd_window)."""
    st = lib().attn_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                               _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(H), int(N), int(d),
                               float(scale), int(bool(causal)), int(window_left),
                               int(window_right), _ptr(cu_seqlens), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_window")
    return st


def _signs(signs, d: int):
    """A host int8[d] sign vector (kept alive by the caller) or None."""
    if signs is None:
        return None, None
    import numpy as np
    arr = np.ascontiguousarray(signs, dtype=np.int8)
    if arr.shape != (int(d),):
        raise ValueError(f"signs must hold d = {int(d)} entries of +1 / -1")
    return arr, arr.ctypes.data


def attn_fwd_fp8(q, k, v, o, lse, B: int, H: int, N: int, d: int, scale: float, causal: bool,
                 signs=None, cu_seqlens=None, stream=None) -> int:
    """The C call ``attn_fwd_fp8`` (e4m3 path; signs: d x +-1 or None)."""
    keep, sp = _signs(signs, d)
    st = lib().attn_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N),
                            int(d), float(scale), int(bool(causal)), _ptr(cu_seqlens), sp,
                            _stream(stream))
    del keep
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_fp8")
    return st


def attn_fwd_fp8_codes(q8, sq, k8, sk, vt, sv, o, lse, B: int, H: int, N: int, d: int,
                       scale: float, causal: bool, rotated: bool, cu_seqlens=None,
                       stream=None) -> int:
    """The C call ``attn_fwd_fp8_codes``: the FP8 attention on codes and scales
    from attn_fp8_quantize_qk / attn_fp8_quantize_v (d = 128)."""
    st = lib().attn_fwd_fp8_codes(_ptr(q8), _ptr(sq), _ptr(k8), _ptr(sk), _ptr(vt), _ptr(sv),
                                  _ptr(o), _ptr(lse), int(B), int(H), int(N), int(d),
                                  float(scale), int(bool(causal)), int(bool(rotated)),
                                  _ptr(cu_seqlens), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_fp8_codes")
    return st

def attn_fp8_quantize_qk(x, codes, scales, B: int, H: int, N: int, d: int, signs=None,
                         cu_seqlens=None, stream=None) -> int:
    """The C call ``attn_fp8_quantize_qk``."""
    keep, sp = _signs(signs, d)
    st = lib().attn_fp8_quantize_qk(_ptr(x), _ptr(codes), _ptr(scales), int(B), int(H), int(N),
                                    int(d), _ptr(cu_seqlens), sp, _stream(stream))
    del keep
    if st != ATTN_OK:
        raise AttnError(st, "attn_fp8_quantize_qk")
    return st


def attn_fp8_quantize_v(v, codes_t, scale, B: int, H: int, N: int, d: int, cu_seqlens=None,
                        stream=None) -> int:
    """The C call ``attn_fp8_quantize_v``."""
    st = lib().attn_fp8_quantize_v(_ptr(v), _ptr(codes_t), _ptr(scale), int(B), int(H), int(N),
                                   int(d), _ptr(cu_seqlens), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fp8_quantize_v")
    return st


def attn_last_device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error status."""
    return lib().attn_last_device_error(_stream(stream))


def attn_last_error_site() -> int:
    return lib().attn_last_error_site()


def forward(q, k, v, causal: bool, scale: float | None = None, cu_seqlens=None,
            max_seqlen: int | None = None, out=None, lse=None, stream=None):
    """Convenience call on torch CUDA tensors.

    Dense: q, k, v are [B, N, H, d] bf16.  Packed: [total, H, d] with
    cu_seqlens (int32 [B+1], on the device) and max_seqlen.  Returns (o, lse):
    o like q; lse [B, H, N] (dense) or [H, total] (packed), fp32.
    Output tensors are allocated by torch when not given.
    """
    import torch
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("q, k, v must be bf16")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    d = q.shape[-1]
    if cu_seqlens is None:
        B, N, H, _ = q.shape
        lse_shape = (B, H, N)
    else:
        total, H, _ = q.shape
        B = cu_seqlens.numel() - 1
        N = int(max_seqlen)
        lse_shape = (H, total)
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    attn_fwd(q, k, v, out, lse, B, H, N, d, scale, causal, cu_seqlens, stream)
    return out, lse


def _check_bf16(*ts):
    import torch
    for t in ts:
        if t.dtype != torch.bfloat16:
            raise TypeError("tensors must be bf16")
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")


def backward(q, k, v, o, dout, lse, causal: bool, scale: float | None = None, cu_seqlens=None,
             max_seqlen: int | None = None, window=(-1, -1), stream=None):
    """Convenience call of attn_bwd / attn_bwd_window on torch CUDA tensors.

    q, k, v, o, dout in the forward's layout (dense [B, N, H, d] or packed
    [total, H, d] with cu_seqlens and max_seqlen), lse as the forward returns
    it.  Returns (dq, dk, dv), allocated by torch.
    """
    import torch
    _check_bf16(q, k, v, o, dout)
    d = q.shape[-1]
    if cu_seqlens is None:
        B, N, H, _ = q.shape
    else:
        H = q.shape[1]
        B = cu_seqlens.numel() - 1
        N = int(max_seqlen)
    if scale is None:
        scale = d ** -0.5
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wl, wr = window
    attn_bwd_window(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, wl, wr,
                    cu_seqlens, stream)
    return dq, dk, dv


def decode(q, k, v, cu_seqlens_k, max_seqlen_k: int, scale: float | None = None,
           num_splits: int = 0, stream=None):
    """Convenience call of attn_fwd_decode on torch CUDA tensors: q [B, H, d]
    (one query per sequence), k, v [total, H, d] packed with cu_seqlens_k
    (int32 [B+1], on the device).  Returns (o [B, H, d] bf16, lse [B, H] fp32)."""
    import torch
    _check_bf16(q, k, v)
    B, H, d = q.shape
    if scale is None:
        scale = d ** -0.5
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    attn_fwd_decode(q, k, v, o, lse, B, H, d, scale, cu_seqlens_k, max_seqlen_k, num_splits, stream)
    return o, lse
