"""Randomised library cross-checks of the oracle: packed batches of ragged
lengths, head counts and head dimensions, causal masks, sliding windows and
scales drawn by hypothesis.  The forward against torch's fp64 softmax and
logsumexp of the explicitly masked logits, the backward against torch
autograd through the same masked softmax (the independent references of the
fixed-shape library pins, over many more shapes).  Every row sees at least
its own key, so no row is empty."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from io_aware_exact_06_gb300 import inputs  # noqa: E402


@settings(max_examples=60, deadline=None)
@given(lens=st.lists(st.integers(1, 40), min_size=1, max_size=4),
       H=st.integers(1, 3), d=st.sampled_from([1, 2, 4, 8, 16]), causal=st.booleans(),
       wl=st.integers(-1, 12), wr=st.integers(-1, 12), scale=st.floats(0.05, 2.0),
       seed=st.integers(0, 1 << 20))
def test_oracle_matches_masked_softmax(lens, H, d, causal, wl, wr, scale, seed):
    import torch
    w = inputs.make_workload("rand", seed, lens, H, d, causal)
    rows = inputs.all_rows(w.cu_seqlens, H)
    o, lse, _ = oracle.attn_rows(w.q, w.k, w.v, w.cu_seqlens, rows, scale, causal, 1,
                                 window=(wl, wr))
    qf, kf, vf = (inputs.bf16_bits_to_f64(a) for a in (w.q, w.k, w.v))
    n = 0
    for s, L in enumerate(lens):
        b0 = int(w.cu_seqlens[s])
        i = torch.arange(L)[:, None]
        j = torch.arange(L)[None, :]
        vis = torch.ones(L, L, dtype=torch.bool)
        if causal:
            vis &= j <= i
        if wl >= 0:
            vis &= j >= i - wl
        if wr >= 0:
            vis &= j <= i + wr
        for h in range(H):
            qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(a[b0:b0 + L, h]))
                          for a in (qf, kf, vf))
            logits = (qt @ kt.T * scale).masked_fill(~vis, float("-inf"))
            ref_lse = torch.logsumexp(logits, dim=-1).numpy()
            ref_o = (torch.softmax(logits, dim=-1) @ vt).numpy()
            got_o, got_lse = o[n:n + L], lse[n:n + L]
            n += L
            err_o = np.max(np.abs(got_o - ref_o) / np.maximum(1.0, np.abs(ref_o)))
            err_l = np.max(np.abs(got_lse - ref_lse) / np.maximum(1.0, np.abs(ref_lse)))
            assert err_o <= 1e-12 and err_l <= 1e-12, (s, h, err_o, err_l)
    assert n == len(rows)


@settings(max_examples=40, deadline=None)
@given(lens=st.lists(st.integers(1, 30), min_size=1, max_size=3),
       H=st.integers(1, 2), d=st.sampled_from([1, 4, 8, 16]), causal=st.booleans(),
       wl=st.integers(-1, 10), wr=st.integers(-1, 10), scale=st.floats(0.05, 2.0),
       seed=st.integers(0, 1 << 20))
def test_oracle_gradients_match_autograd(lens, H, d, causal, wl, wr, scale, seed):
    """The backward oracle against torch autograd through the same masked
    softmax in fp64 (the loss is sum(dO * O))."""
    import torch
    w = inputs.make_workload("rand", seed, lens, H, d, causal)
    dout = inputs.normal_bf16(seed + 17, w.q.size).reshape(w.q.shape)
    pairs = [(s, h) for s in range(len(lens)) for h in range(H)]
    dq, dk, dv, _ = oracle.attn_bwd(w.q, w.k, w.v, dout, w.cu_seqlens, pairs, scale, causal, 1,
                                    window=(wl, wr))
    qf, kf, vf, df = (inputs.bf16_bits_to_f64(a) for a in (w.q, w.k, w.v, dout))
    for n, (s, h) in enumerate(pairs):
        b0, L = int(w.cu_seqlens[s]), lens[s]
        i = torch.arange(L)[:, None]
        j = torch.arange(L)[None, :]
        vis = torch.ones(L, L, dtype=torch.bool)
        if causal:
            vis &= j <= i
        if wl >= 0:
            vis &= j >= i - wl
        if wr >= 0:
            vis &= j <= i + wr
        qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(a[b0:b0 + L, h])).requires_grad_(True)
                      for a in (qf, kf, vf))
        logits = (qt @ kt.T * scale).masked_fill(~vis, float("-inf"))
        out = torch.softmax(logits, dim=-1) @ vt
        out.backward(torch.from_numpy(np.ascontiguousarray(df[b0:b0 + L, h])))
        for got, ref, name in ((dq[n], qt.grad, "dQ"), (dk[n], kt.grad, "dK"), (dv[n], vt.grad, "dV")):
            ref = ref.numpy()
            err = np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref)))
            assert err <= 1e-11, (s, h, name, err)


def _e4m3_grid():
    """(value, code) of every non-negative finite e4m3 code, from the bit fields."""
    out = []
    for c in range(128):
        e, m = (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue
        out.append((m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7), c))
    return sorted(out)


_GRID = _e4m3_grid()


def _nearest_e4m3(y):
    """Nearest e4m3 code by exhaustive search, ties to the even code, beyond
    448 saturating at 448 (y fp32)."""
    vals = np.array([v for v, _ in _GRID])
    codes = np.array([c for _, c in _GRID], dtype=np.uint8)
    a = np.minimum(np.abs(y.astype(np.float64)), 448.0)
    dist = np.abs(a[..., None] - vals)
    best = dist.min(axis=-1, keepdims=True)
    cand = dist == best
    # among equally near codes the even one
    even = cand & ((codes & 1) == 0)
    idx = np.where(even.any(axis=-1), even.argmax(axis=-1), cand.argmax(axis=-1))
    c = codes[idx]
    return np.where((y < 0) & (c != 0), c | 0x80, c).astype(np.uint8)


@settings(max_examples=30, deadline=None)
@given(B=st.integers(1, 2), N=st.integers(1, 300), H=st.integers(1, 2),
       d=st.sampled_from([8, 64]), rotate=st.booleans(),
       std=st.sampled_from([0.01, 1.0, 60.0]), zero_block=st.booleans(),
       outlier=st.booleans(), seed=st.integers(0, 1 << 20))
def test_fp8_quantize_matches_exhaustive_encoder(B, N, H, d, rotate, std, zero_block, outlier,
                                                seed):
    """Block scales and codes of the quantisation step against the definition:
    scale = max|x| / 448 (1 for an all-zero block), codes = nearest e4m3 of
    x * (448 / max|x|) in fp32, the last block pulled back to end at N; with
    rotation the block is that of the Hadamard-rotated rows."""
    rows = 128
    xf = inputs.bf16_bits_to_f64(inputs.normal_bf16(seed, B * N * H * d, std)).reshape(B * N, H, d)
    if outlier:
        xf[:, :, seed % d] *= 30.0
    if zero_block:
        xf[:min(N, rows)] = 0.0
    x = inputs.f64_to_bf16_bits(xf)
    xf = inputs.bf16_bits_to_f64(x).astype(np.float32)
    signs = np.where(inputs.splitmix64(seed + 5, 0, d) & np.uint64(1), -1, 1).astype(np.int8)
    codes, scales = oracle.fp8_quantize(x, B, N, rows, rotate, signs if rotate else None)
    nblk = -(-N // rows)
    assert scales.shape == (B, H, nblk)
    for b in range(B):
        for h in range(H):
            for t in range(nblk):
                r0 = max(0, min(t * rows, N - rows))
                blk = xf[b * N + r0:b * N + min(r0 + rows, N), h]
                if rotate:
                    blk = oracle.fwht_f32(blk, signs)
                amax = np.float32(np.max(np.abs(blk)))
                want_scale = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
                assert scales[b, h, t] == want_scale, (b, h, t)
                inv = np.float32(np.float32(448.0) / amax) if amax > 0 else np.float32(1.0)
                want = _nearest_e4m3((blk * inv).astype(np.float32))
                keep = np.arange(r0, r0 + len(blk)) >= t * rows
                got = codes[b * N + r0:b * N + r0 + len(blk), h][keep]
                assert np.array_equal(got & 0x7f, want[keep] & 0x7f), (b, h, t, rotate)
                nz = (want[keep] & 0x7f) != 0
                assert np.array_equal(got[nz], want[keep][nz]), (b, h, t, "sign")
