"""fp64 CPU oracle for exact softmax attention (forward and gradients).

TEST INFRASTRUCTURE ONLY.  Callers allowed: the tests, the package smoke check
and the benchmark's CPU-baseline leg.  The CUDA path never imports this package
and this package never imports the CUDA path; the two share only the seeded
input generators.

Every routine wraps ``oracle.c``, plain C in fp64.  See that file for the
definition it computes and the passages of the pages it follows.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

_c_i64p = ctypes.POINTER(ctypes.c_int64)
_c_dp = ctypes.POINTER(ctypes.c_double)
_c_u16p = ctypes.POINTER(ctypes.c_uint16)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
    return a


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """The oracle library at ``path`` (the built ``oracle.c``)."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        L.oracle_cpu_count.restype = ctypes.c_int
        L.oracle_attn_rows.restype = ctypes.c_int
        L.oracle_attn_rows.argtypes = [_c_u16p, _c_u16p, _c_u16p, _c_i64p, ctypes.c_int64,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                       _c_i64p, ctypes.c_int64, _c_dp, _c_dp, ctypes.c_int,
                                       ctypes.POINTER(ctypes.c_int)]
        L.oracle_attn_rows_window.restype = ctypes.c_int
        L.oracle_attn_rows_window.argtypes = [_c_u16p, _c_u16p, _c_u16p, _c_i64p, ctypes.c_int64,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                              ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                              _c_i64p, ctypes.c_int64, _c_dp, _c_dp, ctypes.c_int,
                                              ctypes.POINTER(ctypes.c_int)]
        L.oracle_attn_probs.restype = ctypes.c_int64
        L.oracle_attn_probs.argtypes = [_c_u16p, _c_u16p, _c_i64p, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                        ctypes.c_int64, ctypes.c_int, ctypes.c_int64, _c_dp]
        L.oracle_softmax_merge.restype = ctypes.c_int
        L.oracle_softmax_merge.argtypes = [_c_dp, ctypes.c_int64, _c_i64p, ctypes.c_int64,
                                           _c_dp, _c_dp, _c_dp]
        L.oracle_attn_online.restype = ctypes.c_int
        L.oracle_attn_online.argtypes = [_c_u16p, _c_u16p, _c_u16p, _c_i64p, ctypes.c_int64,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                         _c_i64p, ctypes.c_int64, ctypes.c_int64, _c_dp, _c_dp]
        L.oracle_attn_bwd_window.restype = ctypes.c_int
        L.oracle_attn_bwd_window.argtypes = [_c_u16p, _c_u16p, _c_u16p, _c_u16p, _c_i64p,
                                             ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_double, ctypes.c_int, ctypes.c_int64,
                                             ctypes.c_int64, _c_i64p, ctypes.c_int64, _c_dp, _c_dp,
                                             _c_dp, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
        L.oracle_attn_bwd.restype = ctypes.c_int
        L.oracle_attn_bwd.argtypes = [_c_u16p, _c_u16p, _c_u16p, _c_u16p, _c_i64p, ctypes.c_int64,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                      _c_i64p, ctypes.c_int64, _c_dp, _c_dp, _c_dp, ctypes.c_int,
                                      ctypes.POINTER(ctypes.c_int)]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_decode.restype = ctypes.c_double
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_fwht_f32.restype = None
        L.oracle_fwht_f32.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_int,
                                      ctypes.POINTER(ctypes.c_int8)]
        L.oracle_fp8_quantize.restype = ctypes.c_int
        L.oracle_fp8_quantize.argtypes = [_c_u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_int8),
                                          ctypes.POINTER(ctypes.c_uint8),
                                          ctypes.POINTER(ctypes.c_float)]
        L.oracle_fp8_quantize_tensor.restype = ctypes.c_int
        L.oracle_fp8_quantize_tensor.argtypes = [_c_u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                 ctypes.POINTER(ctypes.c_uint8),
                                                 ctypes.POINTER(ctypes.c_float)]
        L.oracle_attn_rows_f64.restype = ctypes.c_int
        L.oracle_attn_rows_f64.argtypes = [_c_dp, _c_dp, _c_dp, _c_i64p, ctypes.c_int64,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                           ctypes.c_int, _c_i64p, ctypes.c_int64, _c_dp, _c_dp]
        self.lib = L
        self.path = path

    def cpu_count(self) -> int:
        return int(self.lib.oracle_cpu_count())

    def attn_rows(self, q, k, v, cu_seqlens, rows, scale: float, causal: bool,
                  nthreads: int = 0, window=(-1, -1)):
        """O (fp64 [n, d]) and LSE (fp64 [n]) of the given (seq, head, row) triples.

        q, k, v: uint16 bf16 bits, [tokens, H, d].  window = (wl, wr): keys
        i - wl <= j <= i + wr only (negative: unbounded).  Returns (o, lse,
        threads_used).
        """
        q, k, v = _u16(q), _u16(k), _u16(v)
        tokens, H, d = q.shape
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
        n = rows.shape[0]
        o = np.zeros((n, d), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        used = ctypes.c_int(0)
        wl, wr = (int(window[0]), int(window[1]))
        st = self.lib.oracle_attn_rows_window(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                              _ptr(v, ctypes.c_uint16), _ptr(cu, ctypes.c_int64),
                                              len(cu) - 1, H, d, float(scale), int(bool(causal)),
                                              wl, wr, _ptr(rows, ctypes.c_int64), n,
                                              _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                                              int(nthreads), ctypes.byref(used))
        if st != 0:
            raise ValueError(f"oracle_attn_rows failed with status {st}")
        return o, lse, used.value

    def attn_bwd(self, q, k, v, dout, cu_seqlens, pairs, scale: float, causal: bool,
                 nthreads: int = 0, window=(-1, -1)):
        """dQ, dK, dV (fp64) of the given (seq, head) pairs.

        q, k, v, dout: uint16 bf16 bits, [tokens, H, d] (dout = dO, the
        gradient of the loss with respect to O).  window = (wl, wr): keys
        i - wl <= j <= i + wr only (negative: unbounded).  Returns (dq, dk, dv,
        threads_used); each gradient is a list with one [L_s, d] array per
        pair.
        """
        q, k, v, dout = _u16(q), _u16(k), _u16(v), _u16(dout)
        tokens, H, d = q.shape
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
        pairs = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
        lens = [int(cu[s + 1] - cu[s]) for s in pairs[:, 0]]
        n = sum(lens)
        dq = np.zeros((max(n, 1), d), dtype=np.float64)
        dk = np.zeros_like(dq)
        dv = np.zeros_like(dq)
        used = ctypes.c_int(0)
        st = self.lib.oracle_attn_bwd_window(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                      _ptr(v, ctypes.c_uint16), _ptr(dout, ctypes.c_uint16),
                                      _ptr(cu, ctypes.c_int64), len(cu) - 1, H, d, float(scale),
                                      int(bool(causal)), int(window[0]), int(window[1]),
                                      _ptr(pairs, ctypes.c_int64), len(pairs),
                                      _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double),
                                      _ptr(dv, ctypes.c_double), int(nthreads), ctypes.byref(used))
        if st != 0:
            raise ValueError(f"oracle_attn_bwd failed with status {st}")
        split = np.cumsum(lens)[:-1]
        return np.split(dq[:n], split), np.split(dk[:n], split), np.split(dv[:n], split), used.value

    def e4m3_encode(self, x) -> np.ndarray:
        """e4m3 codes (uint8) of fp32 values: nearest, ties to even, saturating."""
        x = np.ascontiguousarray(x, dtype=np.float32).ravel()
        return np.array([self.lib.oracle_e4m3_encode(float(v)) for v in x], dtype=np.uint8)

    def e4m3_decode(self, c) -> np.ndarray:
        c = np.ascontiguousarray(c, dtype=np.uint8).ravel()
        return np.array([self.lib.oracle_e4m3_decode(int(v)) for v in c], dtype=np.float64)

    def fwht_f32(self, x, signs=None) -> np.ndarray:
        """(x * signs) H_d in fp32 butterflies, for each row of x [..., d]."""
        x = np.array(x, dtype=np.float32)
        d = x.shape[-1]
        flat = x.reshape(-1, d)
        sg = None if signs is None else np.ascontiguousarray(signs, dtype=np.int8)
        for r in range(flat.shape[0]):
            row = np.ascontiguousarray(flat[r])
            self.lib.oracle_fwht_f32(_ptr(row, ctypes.c_float), d,
                                     None if sg is None else _ptr(sg, ctypes.c_int8))
            flat[r] = row
        return flat.reshape(x.shape)

    def fp8_quantize(self, x, B: int, N: int, block_rows: int, rotate: bool, signs=None):
        """Block e4m3 quantisation of bf16 bits x [B*N, H, d] (see oracle.c).

        Returns (codes uint8 [B*N, H, d], scales fp32 [B, H, nblocks])."""
        x = _u16(x)
        tokens, H, d = x.shape
        nblk = 1 if block_rows == 0 else -(-N // block_rows)
        codes = np.zeros(x.shape, dtype=np.uint8)
        scales = np.zeros((B, H, nblk), dtype=np.float32)
        sg = None if signs is None else np.ascontiguousarray(signs, dtype=np.int8)
        st = self.lib.oracle_fp8_quantize(_ptr(x, ctypes.c_uint16), int(B), int(N), H, d,
                                          int(block_rows), int(bool(rotate)),
                                          None if sg is None else _ptr(sg, ctypes.c_int8),
                                          _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_float))
        if st != 0:
            raise ValueError(f"oracle_fp8_quantize failed with status {st}")
        return codes, scales

    def fp8_quantize_tensor(self, x):
        """Per-tensor e4m3 quantisation (one scale per head) of bf16 bits x
        [tokens, H, d] (see oracle.c).  Returns (codes uint8 [tokens, H, d],
        scales fp32 [H])."""
        x = _u16(x)
        tokens, H, d = x.shape
        codes = np.zeros(x.shape, dtype=np.uint8)
        scales = np.zeros(H, dtype=np.float32)
        st = self.lib.oracle_fp8_quantize_tensor(_ptr(x, ctypes.c_uint16), int(tokens), H, d,
                                                 _ptr(codes, ctypes.c_uint8),
                                                 _ptr(scales, ctypes.c_float))
        if st != 0:
            raise ValueError(f"oracle_fp8_quantize_tensor failed with status {st}")
        return codes, scales

    def attn_rows_f64(self, q, k, v, cu_seqlens, rows, scale: float, causal: bool):
        """O and LSE of the given rows for fp64 inputs [tokens, H, d]."""
        q, k, v = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v))
        tokens, H, d = q.shape
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
        n = rows.shape[0]
        o = np.zeros((n, d), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        st = self.lib.oracle_attn_rows_f64(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                                           _ptr(v, ctypes.c_double), _ptr(cu, ctypes.c_int64),
                                           len(cu) - 1, H, d, float(scale), int(bool(causal)),
                                           _ptr(rows, ctypes.c_int64), n,
                                           _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
        if st != 0:
            raise ValueError(f"oracle_attn_rows_f64 failed with status {st}")
        return o, lse

    def attn_probs(self, q, k, cu_seqlens, seq: int, h: int, i: int, scale: float,
                   causal: bool):
        """The probability row P_i (fp64) of one query row."""
        q, k = _u16(q), _u16(k)
        tokens, H, d = q.shape
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
        L = int(cu[seq + 1] - cu[seq])
        p = np.zeros(max(L, 1), dtype=np.float64)
        n = self.lib.oracle_attn_probs(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                       _ptr(cu, ctypes.c_int64), len(cu) - 1, H, d,
                                       float(scale), int(bool(causal)), int(seq), int(h),
                                       int(i), _ptr(p, ctypes.c_double))
        if n < 0:
            raise ValueError(f"oracle_attn_probs failed with status {n}")
        return p[:n]

    def softmax_merge(self, x, cuts):
        """softmax(x) by segment-wise (m, l, f) merging at the given cut points.

        Returns (softmax, m, l)."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        cuts = np.ascontiguousarray(cuts, dtype=np.int64)
        out = np.zeros_like(x)
        m = ctypes.c_double(0)
        l = ctypes.c_double(0)
        st = self.lib.oracle_softmax_merge(_ptr(x, ctypes.c_double), x.size,
                                           _ptr(cuts, ctypes.c_int64) if cuts.size else None,
                                           cuts.size, _ptr(out, ctypes.c_double),
                                           ctypes.byref(m), ctypes.byref(l))
        if st != 0:
            raise ValueError(f"oracle_softmax_merge failed with status {st}")
        return out, m.value, l.value

    def attn_online(self, q, k, v, cu_seqlens, rows, scale: float, causal: bool, bc: int):
        """O and LSE of the given rows by the block-wise online loop (block size bc)."""
        q, k, v = _u16(q), _u16(k), _u16(v)
        tokens, H, d = q.shape
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
        n = rows.shape[0]
        o = np.zeros((n, d), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        st = self.lib.oracle_attn_online(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                         _ptr(v, ctypes.c_uint16), _ptr(cu, ctypes.c_int64),
                                         len(cu) - 1, H, d, float(scale), int(bool(causal)),
                                         _ptr(rows, ctypes.c_int64), n, int(bc),
                                         _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
        if st != 0:
            raise ValueError(f"oracle_attn_online failed with status {st}")
        return o, lse


_default = None


def default() -> Oracle:
    """The oracle built from this package's ``oracle.c``."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def cpu_count() -> int:
    return default().cpu_count()


def attn_rows(*a, **kw):
    return default().attn_rows(*a, **kw)


def attn_probs(*a, **kw):
    return default().attn_probs(*a, **kw)


def attn_bwd(*a, **kw):
    return default().attn_bwd(*a, **kw)


def e4m3_encode(*a, **kw):
    return default().e4m3_encode(*a, **kw)


def e4m3_decode(*a, **kw):
    return default().e4m3_decode(*a, **kw)


def fwht_f32(*a, **kw):
    return default().fwht_f32(*a, **kw)


def fp8_quantize(*a, **kw):
    return default().fp8_quantize(*a, **kw)


def fp8_quantize_tensor(*a, **kw):
    return default().fp8_quantize_tensor(*a, **kw)


def attn_rows_f64(*a, **kw):
    return default().attn_rows_f64(*a, **kw)


def softmax_merge(*a, **kw):
    return default().softmax_merge(*a, **kw)


def attn_online(*a, **kw):
    return default().attn_online(*a, **kw)
