"""Backward pass (attn_bwd) against the fp64 oracle's gradients.

The CUDA side runs its own forward (attn_fwd) for O and the LSE, then
attn_bwd; the oracle computes dQ, dK, dV from Q, K, V and dO alone.

Tolerance (derived from the arithmetic, per gradient tensor over the compared
(sequence, head) pairs): every output is a sum of products in which one factor
(P or dS) is rounded to bf16 (relative error <= 2^-9 each, independent
signs), D_i comes from the bf16-rounded O, and the result is rounded to bf16
once more; with random-sign terms each source adds about 2^-9 / sqrt(3) ~ 1.1e-3
to the relative L2 error of the whole tensor.  Bound: rel-L2 <= 1e-2 (about
3x the sum of three such sources) and max-abs <= 2.5e-2 * max |ref| (four
standard deviations of the per-element error of the largest elements), plus
an absolute floor of 1e-3 for gradients whose exact value is 0 (a single
visible key: dS = dP - D with both dot products of d = 128 bf16 pairs summed
in fp32, whose difference is bounded by 2 d 2^-24 sum|dO_c v_c| ~ 1.3e-3 for
unit-variance inputs; the relative L2 test is skipped when the reference
tensor is exactly zero).
"""
import json
import os

import numpy as np
import pytest

import oracle
from io_aware_exact_06_gb300 import inputs

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_ABS_REL = 2.5e-2
ABS_FLOOR = 1e-3


@pytest.fixture(scope="module")
def dev():
    import torch
    import __graft_entry__
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    __graft_entry__.build()
    return torch.device("cuda:0")


def run_bwd(dev, wl, dout_bits, stream=None):
    """CUDA forward then backward on a dense workload; returns dq, dk, dv as
    fp64 numpy arrays [tokens, H, d]."""
    import torch
    import io_aware_exact_06_gb300 as fa
    B, N, H, d = wl.nseq, int(wl.seqlens()[0]), wl.H, wl.d
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    q, k, v, do = t(wl.q), t(wl.k), t(wl.v), t(dout_bits)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fa.attn_fwd(q, k, v, o, lse, B, H, N, d, wl.scale, wl.causal, None, stream)
    dq = torch.full_like(q, float("nan"))
    dk = torch.full_like(q, float("nan"))
    dv = torch.full_like(q, float("nan"))
    fa.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, wl.scale, wl.causal, None, stream)
    assert fa.attn_last_device_error(stream) == 0
    return tuple(x.float().cpu().numpy().astype(np.float64) for x in (dq, dk, dv))


def compare(wl, dout_bits, got, pairs, what):
    ref = oracle.attn_bwd(wl.q, wl.k, wl.v, dout_bits, wl.cu_seqlens, pairs, wl.scale, wl.causal)
    stats = {}
    for t, name in enumerate(("dq", "dk", "dv")):
        r = np.concatenate(ref[t]) if pairs else np.zeros((0, wl.d))
        g = np.concatenate([got[t][int(wl.cu_seqlens[s]):int(wl.cu_seqlens[s + 1]), h]
                            for s, h in pairs])
        assert np.isfinite(g).all(), (what, name, "non-finite output")
        diff = g - r
        stats[name] = {"rel_l2": float(np.linalg.norm(diff) / max(np.linalg.norm(r), 1e-300)),
                       "max_abs": float(np.abs(diff).max()),
                       "max_ref": float(np.abs(r).max())}
    log = os.environ.get("PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"test": "bwd", "what": what, **stats}) + "\n")
    for name, s in stats.items():
        if s["max_ref"] > 0:
            assert s["rel_l2"] <= REL_L2, (what, name, s)
        assert s["max_abs"] <= MAX_ABS_REL * s["max_ref"] + ABS_FLOOR, (what, name, s)


def make(seed, B, N, H, d, causal, qk_std=1.0):
    wl = inputs.make_workload("bwd", seed, [N] * B, H, d, causal, qk_std=qk_std)
    dout = inputs.normal_bf16(4 * seed + 7, wl.q.size).reshape(wl.q.shape)
    return wl, dout


def all_pairs(wl):
    return [(s, h) for s in range(wl.nseq) for h in range(wl.H)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_small_all_pairs(dev, d, causal):
    wl, dout = make(2001 + d + causal, 1, 256, 2, d, causal)
    compare(wl, dout, run_bwd(dev, wl, dout), all_pairs(wl), f"N=256 d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_tail(dev, d, causal):
    # N = 1000: eight 128-row tiles, the last pulled back over the seventh
    wl, dout = make(2101 + d + causal, 2, 1000, 3, d, causal)
    compare(wl, dout, run_bwd(dev, wl, dout), all_pairs(wl), f"N=1000 d={d} causal={causal}")


@pytest.mark.parametrize("N", [1, 77, 129, 384])
def test_short_and_odd_lengths(dev, N):
    # shorter than a tile (rows before the sequence start are loaded and
    # dropped), one row past a tile, exact multiple
    for causal in (False, True):
        wl, dout = make(2201 + N + causal, 3, N, 2, 128, causal)
        compare(wl, dout, run_bwd(dev, wl, dout), all_pairs(wl), f"N={N} causal={causal}")


def test_peaky_softmax(dev):
    # Q, K ~ N(0, 3^2): scores with a spread of tens, P close to one-hot
    wl, dout = make(2301, 1, 2048, 4, 128, False, qk_std=3.0)
    compare(wl, dout, run_bwd(dev, wl, dout), all_pairs(wl), "Q/K std 3")


def test_long_causal_sampled(dev):
    # the long causal shape (B=2, H=16, N=8192, d=128); the oracle recomputes
    # two whole (sequence, head) pairs
    wl = inputs.config_workload("long_causal")
    dout = inputs.normal_bf16(0xD0D0, wl.q.size).reshape(wl.q.shape)
    compare(wl, dout, run_bwd(dev, wl, dout), [(0, 3), (1, 14)], "long causal sampled")


def run_bwd_packed(dev, wl, dout_bits, N=None):
    """CUDA forward then backward on a packed batch (cu_seqlens on the device;
    N: the length bound, by default the longest length)."""
    import torch
    import io_aware_exact_06_gb300 as fa
    H, d = wl.H, wl.d
    lens = wl.seqlens()
    if N is None:
        N = int(lens.max()) if len(lens) else 0
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    q, k, v, do = t(wl.q), t(wl.k), t(wl.v), t(dout_bits)
    cu = torch.from_numpy(wl.cu_seqlens.astype(np.int32)).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((H, wl.tokens), dtype=torch.float32, device=dev)
    fa.attn_fwd(q, k, v, o, lse, wl.nseq, H, N, d, wl.scale, wl.causal, cu)
    grads = [torch.full_like(q, float("nan")) for _ in range(3)]
    fa.attn_bwd(q, k, v, o, do, lse, *grads, wl.nseq, H, N, d, wl.scale, wl.causal, cu)
    assert fa.attn_last_device_error() == 0
    return tuple(x.float().cpu().numpy().astype(np.float64) for x in grads)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_lengths(dev, d, causal):
    # an empty sequence, a single row, tails of every kind, several tiles
    lens = [0, 1, 77, 128, 129, 300, 1000, 513]
    wl = inputs.make_workload("bwd_packed", 2600 + d + causal, lens, 2, d, causal, varlen=True)
    dout = inputs.normal_bf16(2650 + d, wl.q.size).reshape(wl.q.shape)
    pairs = [(s, h) for s in range(wl.nseq) for h in range(wl.H) if lens[s] > 0]
    compare(wl, dout, run_bwd_packed(dev, wl, dout), pairs, f"packed d={d} causal={causal}")


def test_packed_equals_dense(dev):
    # the same equal-length batch through both layouts gives the same bits
    wl, dout = make(2701, 3, 384, 2, 128, True)
    a = run_bwd(dev, wl, dout)
    b = run_bwd_packed(dev, wl, dout)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def run_bwd_window(dev, wl, dout_bits, window, packed=False):
    """CUDA windowed forward then windowed backward (dense or packed)."""
    import torch
    import io_aware_exact_06_gb300 as fa
    H, d = wl.H, wl.d
    lens = wl.seqlens()
    N = int(lens.max())
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    q, k, v, do = t(wl.q), t(wl.k), t(wl.v), t(dout_bits)
    cu = torch.from_numpy(wl.cu_seqlens.astype(np.int32)).to(dev) if packed else None
    B = wl.nseq
    o = torch.empty_like(q)
    lse = (torch.empty((H, wl.tokens), dtype=torch.float32, device=dev) if packed
           else torch.empty((B, H, N), dtype=torch.float32, device=dev))
    fa.attn_fwd_window(q, k, v, o, lse, B, H, N, d, wl.scale, wl.causal, window[0], window[1], cu)
    grads = [torch.full_like(q, float("nan")) for _ in range(3)]
    fa.attn_bwd_window(q, k, v, o, do, lse, *grads, B, H, N, d, wl.scale, wl.causal, window[0],
                       window[1], cu)
    assert fa.attn_last_device_error() == 0
    return tuple(x.float().cpu().numpy().astype(np.float64) for x in grads)


def compare_window(wl, dout_bits, got, pairs, window, what):
    ref = oracle.attn_bwd(wl.q, wl.k, wl.v, dout_bits, wl.cu_seqlens, pairs, wl.scale, wl.causal,
                          window=window)
    for t, name in enumerate(("dq", "dk", "dv")):
        r = np.concatenate(ref[t])
        g = np.concatenate([got[t][int(wl.cu_seqlens[s]):int(wl.cu_seqlens[s + 1]), h]
                            for s, h in pairs])
        assert np.isfinite(g).all(), (what, name)
        rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)
        mx = np.abs(g - r).max()
        if np.abs(r).max() > 0:
            assert rel <= REL_L2, (what, name, rel)
        assert mx <= MAX_ABS_REL * np.abs(r).max() + ABS_FLOOR, (what, name, mx)


@pytest.mark.parametrize("window,causal", [((100, 0), True), ((64, 64), False), ((0, 300), False),
                                           ((200, -1), True), ((-1, 130), False), ((0, 0), False)])
@pytest.mark.parametrize("d", [64, 128])
def test_window_dense(dev, window, causal, d):
    wl, dout = make(2800 + d + window[0] + 3 * window[1], 2, 1000, 2, d, causal)
    compare_window(wl, dout, run_bwd_window(dev, wl, dout, window), all_pairs(wl), window,
                   f"window {window} causal={causal} d={d}")


def test_window_packed(dev):
    lens = [0, 1, 77, 300, 1000, 513]
    wl = inputs.make_workload("bwd_win_packed", 2900, lens, 2, 128, True, varlen=True)
    dout = inputs.normal_bf16(2901, wl.q.size).reshape(wl.q.shape)
    pairs = [(s, h) for s in range(wl.nseq) for h in range(wl.H) if lens[s] > 0]
    compare_window(wl, dout, run_bwd_window(dev, wl, dout, (150, -1), packed=True), pairs,
                   (150, -1), "packed window (150, -1)")


def test_unbounded_window_is_attn_bwd(dev):
    wl, dout = make(2950, 2, 700, 2, 128, True)
    a = run_bwd(dev, wl, dout)
    b = run_bwd_window(dev, wl, dout, (-1, -1))
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale(dev, causal):
    # scale 0: P is uniform over the visible keys, dQ = dK = 0 exactly
    wl = inputs.make_workload("bwd", 2501 + causal, [300] * 2, 2, 128, causal, scale=0.0)
    dout = inputs.normal_bf16(4 * 2501 + 7, wl.q.size).reshape(wl.q.shape)
    got = run_bwd(dev, wl, dout)
    assert not got[0].any() and not got[1].any()
    compare(wl, dout, got, all_pairs(wl), f"scale 0 causal={causal}")


def test_zero_upstream_gradient(dev):
    wl, _ = make(2401, 2, 300, 2, 64, True)
    zero = np.zeros_like(wl.q)
    dq, dk, dv = run_bwd(dev, wl, zero)
    assert not dq.any() and not dk.any() and not dv.any()


def test_deterministic(dev):
    wl, dout = make(2501, 2, 700, 4, 128, True)
    a = run_bwd(dev, wl, dout)
    b = run_bwd(dev, wl, dout)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_convenience_wrappers(dev):
    """fa.forward then fa.backward give what the C calls give."""
    import torch
    import io_aware_exact_06_gb300 as fa
    wl, dout = make(2601, 2, 640, 2, 128, True)
    ref = run_bwd(dev, wl, dout)
    tt = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    q = tt(wl.q).view(2, 640, 2, 128)
    k = tt(wl.k).view(2, 640, 2, 128)
    v = tt(wl.v).view(2, 640, 2, 128)
    o, lse = fa.forward(q, k, v, True, wl.scale)
    dq, dk, dv = fa.backward(q, k, v, o, tt(dout).view(2, 640, 2, 128), lse, True, wl.scale)
    assert fa.attn_last_device_error() == 0
    for a, b in zip(ref, (dq, dk, dv)):
        assert np.array_equal(a, b.float().cpu().numpy().astype(np.float64).reshape(a.shape))


@pytest.mark.parametrize("causal", [False, True])
def test_packed_head_group_order_same_result(dev, causal):
    """Packed calls with a large length bound take their units in head groups
    (causal: at least 64 units per SM counted from the bound); the result may
    not depend on the order.  The same sequences with N = their longest length
    and with N = 8192 (16 sequences x 20 heads x 64 tiles = 20480 units, one
    head per group on 152 SMs) give bit-identical gradients, and sampled
    (sequence, head) pairs match the oracle."""
    lens = inputs.uniform_ints(2750 + causal, 16, 1, 1200).tolist()
    wl = inputs.make_workload("bwd_groups", 2760 + causal, lens, 20, 128, causal, varlen=True)
    dout = inputs.normal_bf16(2770 + causal, wl.q.size).reshape(wl.q.shape)
    a = run_bwd_packed(dev, wl, dout)
    b = run_bwd_packed(dev, wl, dout, N=8192)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    pairs = [(s, h) for s, h in ((0, 0), (3, 7), (9, 19), (15, 11)) if lens[s] > 0]
    compare(wl, dout, b, pairs, f"packed head groups causal={causal}")
