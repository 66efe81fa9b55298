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
