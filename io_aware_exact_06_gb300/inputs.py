"""Seeded synthetic inputs for the attention forward workloads.

This module is shared by the CUDA path's tests/bench and by the fp64 oracle's
tests.  It holds none of the attention arithmetic: only a counter-based random
source, a normal transform, bf16 rounding, the variable-length batch layout and
the choice of rows to compare.

Random source: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style: draw ``i`` of stream
``seed`` is ``mix(seed + (i + 1) * 0x9E3779B97F4A7C15)``.

Normal transform: Box-Muller (Box & Muller, 1958).  Element ``i`` of a tensor
uses draws ``2i`` and ``2i + 1``:  u1 = ((x >> 11) + 1) * 2**-53 in (0, 1],
u2 = (y >> 11) * 2**-53 in [0, 1), z = sqrt(-2 ln u1) * cos(2 pi u2).

bf16: every value is drawn in fp64, scaled by its standard deviation in fp64,
then rounded once, to nearest-even, straight from fp64 to bf16 (no fp32 step).
Both sides of every comparison read the same rounded bits.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1

# Config k of the workload table is drawn from seed CONFIG_SEED_BASE + k.
CONFIG_SEED_BASE = 0xA77E0000


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the SplitMix64 stream ``seed``."""
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & _MASK64) + idx * GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _normals_chunk(seed: int, start: int, count: int) -> np.ndarray:
    raw = splitmix64(seed, 2 * start, 2 * count)
    x = raw[0::2]
    y = raw[1::2]
    u1 = ((x >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (y >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Rounds fp64 values to bf16 (nearest, ties to even) and returns the bits.

    Handles zero, normal values in bf16 range, +-inf and NaN; values below the
    bf16 normal range are flushed to signed zero (the generators here never
    produce them: |z| < 2**-126 has probability ~0).
    """
    b = np.ascontiguousarray(x, dtype=np.float64).view(np.uint64)
    sign = ((b >> np.uint64(63)) & np.uint64(1)).astype(np.uint16)
    exp = ((b >> np.uint64(52)) & np.uint64(0x7FF)).astype(np.int64)
    mant = b & np.uint64((1 << 52) - 1)
    # round the 52-bit mantissa to 7 bits, nearest-even; a carry bumps the exponent
    lsb = (mant >> np.uint64(45)) & np.uint64(1)
    rounded = (mant + np.uint64((1 << 44) - 1) + lsb) >> np.uint64(45)
    carry = (rounded >> np.uint64(7)).astype(np.int64)
    m7 = (rounded & np.uint64(0x7F)).astype(np.uint16)
    e = exp - 1023 + 127 + carry
    out = np.empty(b.shape, dtype=np.uint16)
    normal = (exp > 0) & (exp < 0x7FF)
    e_ok = normal & (e > 0) & (e < 255)
    out[...] = (sign << np.uint16(15))  # zero / underflow
    out[e_ok] = (sign[e_ok] << np.uint16(15)) | (e[e_ok].astype(np.uint16) << np.uint16(7)) | m7[e_ok]
    over = normal & (e >= 255)
    out[over] = (sign[over] << np.uint16(15)) | np.uint16(0x7F80)
    special = exp == 0x7FF
    is_nan = special & (mant != 0)
    out[special & ~is_nan] = (sign[special & ~is_nan] << np.uint16(15)) | np.uint16(0x7F80)
    out[is_nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    u = (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16))
    return u.view(np.float32).astype(np.float64)


def normal_bf16(seed: int, count: int, std: float = 1.0, threads: int | None = None) -> np.ndarray:
    """``count`` draws of N(0, std**2), rounded to bf16; returns uint16 bits."""
    out = np.empty(count, dtype=np.uint16)
    chunk = 1 << 22
    starts = list(range(0, count, chunk))

    def work(s: int) -> None:
        n = min(chunk, count - s)
        out[s:s + n] = f64_to_bf16_bits(_normals_chunk(seed, s, n) * std)

    nthreads = threads or min(len(starts), os.cpu_count() or 1) or 1
    if nthreads <= 1 or len(starts) <= 1:
        for s in starts:
            work(s)
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(work, starts))
    return out


def uniform_ints(seed: int, count: int, lo: int, hi: int) -> np.ndarray:
    """``count`` integers uniform on [lo, hi] (inclusive), by rejection-free
    multiply-shift on the top 32 bits of each draw (bias < 2**-17 here)."""
    span = hi - lo + 1
    top = splitmix64(seed, 0, count) >> np.uint64(32)
    return (lo + ((top * np.uint64(span)) >> np.uint64(32)).astype(np.int64)).astype(np.int64)


class Workload:
    """One synthetic attention forward problem in the packed [tokens, H, d] layout.

    ``cu_seqlens`` (int32, nseq+1) always describes the batch; a dense batch of B
    sequences of length N is cu_seqlens = [0, N, 2N, ..., BN].
    """

    def __init__(self, name, q, k, v, cu_seqlens, H, d, scale, causal, varlen, max_seqlen):
        self.name = name
        self.q, self.k, self.v = q, k, v          # uint16 bf16 bits, shape [tokens, H, d]
        self.cu_seqlens = cu_seqlens              # int32 [nseq + 1]
        self.H, self.d = H, d
        self.scale = scale
        self.causal = causal
        self.varlen = varlen
        self.max_seqlen = max_seqlen

    @property
    def nseq(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    def seqlens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens.astype(np.int64))

    def flops(self) -> float:
        """4*H*L^2*d per sequence, halved when causal (the metric's convention)."""
        L = self.seqlens().astype(np.float64)
        f = float(np.sum(4.0 * self.H * L * L * self.d))
        return f / 2 if self.causal else f


def make_workload(name: str, seed: int, seqlens, H: int, d: int, causal: bool,
                  qk_std: float = 1.0, v_std: float = 1.0, varlen: bool = False,
                  scale: float | None = None) -> Workload:
    seqlens = np.asarray(seqlens, dtype=np.int64)
    cu = np.zeros(len(seqlens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(seqlens)
    tokens = int(cu[-1])
    n = tokens * H * d
    # three independent streams derived from the config seed, one per tensor
    q = normal_bf16(seed * 4 + 1, n, qk_std).reshape(tokens, H, d)
    k = normal_bf16(seed * 4 + 2, n, qk_std).reshape(tokens, H, d)
    v = normal_bf16(seed * 4 + 3, n, v_std).reshape(tokens, H, d)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return Workload(name, q, k, v, cu.astype(np.int32), H, d, float(scale), causal,
                    varlen, int(seqlens.max()) if len(seqlens) else 0)


# The five workloads: shapes and distributions of the attention forward configs.
CONFIGS = {
    "tiny":        dict(k=0, B=1, H=1, N=256, d=64, causal=False),
    "gpt2_causal": dict(k=1, B=8, H=12, N=1024, d=64, causal=True),
    "long_causal": dict(k=2, B=2, H=16, N=8192, d=128, causal=True),
    "long_full":   dict(k=2, B=2, H=16, N=8192, d=128, causal=False),
    "stress":      dict(k=3, B=1, H=16, N=16384, d=128, causal=False, qk_std=3.0),
    "varlen":      dict(k=4, nseq=16, Lmin=512, Lmax=16384, H=16, d=128, causal=True),
}


def varlen_lengths(seed: int, nseq: int, lo: int, hi: int) -> np.ndarray:
    """Sequence lengths of the packed batch, drawn before any tensor value."""
    return uniform_ints(seed * 4 + 0, nseq, lo, hi)


def config_workload(name: str) -> Workload:
    c = CONFIGS[name]
    seed = CONFIG_SEED_BASE + c["k"]
    if "nseq" in c:
        lens = varlen_lengths(seed, c["nseq"], c["Lmin"], c["Lmax"])
        return make_workload(name, seed, lens, c["H"], c["d"], c["causal"], varlen=True)
    return make_workload(name, seed, [c["N"]] * c["B"], c["H"], c["d"], c["causal"],
                         qk_std=c.get("qk_std", 1.0))


def sample_rows(cu_seqlens, H: int, count: int, seed: int) -> np.ndarray:
    """A seeded set of (seq, head, row) triples to compare, int64 [n, 3].

    Always holds, for every sequence and every head: the first and last row and
    the tile-edge rows 127, 128, 255, 256 (where they exist); the rest are drawn
    uniformly over (seq, head, row), without repeats, until ``count`` rows (or
    every row) are held.  The result is sorted.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    lens = np.diff(cu)
    fixed = []
    for s in range(len(cu) - 1):
        L = int(lens[s])
        if L == 0:
            continue
        rr = sorted({0, L - 1} | {r for r in (127, 128, 255, 256) if r < L})
        fixed.extend(int(cu[s]) + r for r in rr)
    fixed = np.asarray(fixed, dtype=np.int64)
    # key = token * H + head over the packed (token, head) grid
    fixed_keys = np.unique((fixed[:, None] * H + np.arange(H, dtype=np.int64)[None, :]).ravel())
    total = int(lens.sum()) * H
    target = min(max(count, fixed_keys.size), total)
    if target >= total:
        keys = np.arange(total, dtype=np.int64)
    else:
        # the rest: the keys with the smallest SplitMix64 hash (a seeded
        # sample without repeats, no rejection loop)
        prio = splitmix64(seed, 0, total)
        prio[fixed_keys] = 0
        extra = target - fixed_keys.size
        free = np.ones(total, dtype=bool)
        free[fixed_keys] = False
        cand = np.flatnonzero(free)
        pick = cand[np.argpartition(prio[cand], extra - 1)[:extra]] if extra > 0 else cand[:0]
        keys = np.concatenate([fixed_keys, pick])
    tok = keys // H
    hh = keys % H
    seq = np.searchsorted(cu, tok, side="right") - 1
    out = np.stack([seq, hh, tok - cu[seq]], axis=1).astype(np.int64)
    return out[np.lexsort((out[:, 2], out[:, 1], out[:, 0]))]


def all_rows(cu_seqlens, H: int) -> np.ndarray:
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = []
    for s in range(len(cu) - 1):
        L = int(cu[s + 1] - cu[s])
        hh, rr = np.meshgrid(np.arange(H), np.arange(L), indexing="ij")
        block = np.stack([np.full(H * L, s), hh.ravel(), rr.ravel()], axis=1)
        out.append(block)
    return np.concatenate(out).astype(np.int64) if out else np.zeros((0, 3), np.int64)
