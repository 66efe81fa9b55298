"""Checks that pin the fp64 oracle to facts fixed outside the oracle itself.

Each check takes an ``oracle.Oracle`` and raises AssertionError when the oracle
disagrees with:
  - a brute-force high-precision (50-digit Decimal) evaluation of the
    definition on tiny inputs, without max subtraction;
  - a hand closed form on two keys;
  - rows of P summing to one;
  - constant V giving constant O;
  - Q = 0 (or K = 0) giving the column mean of V (causal: the prefix mean)
    with LSE = log(#visible keys);
  - a large-scale one-hot limit where O tends to one chosen value row;
  - torch's scaled_dot_product_attention and logsumexp in fp64 on CPU;
  - the two-segment merge identity of the online softmax;
  - the block-wise online loop, for several block sizes;
  - packing: a sequence inside a packed batch equals that sequence alone;
  - causal masking: the last row of a causal sequence sees every key;
  - gradients (dQ, dK, dV): central finite differences of sum(dO * O), torch
    autograd through SDPA in fp64, the sum rules (sum of dV = sum of dO, sum
    of dK = 0), constant V (no dQ, dK), dO = 0, and packing;
  - FP8: e4m3 decoding from the bit fields and encoding by exhaustive
    nearest search, the fp32 Hadamard butterflies against scipy's Hadamard
    matrix, block scales and codes against the exhaustive encoder, and the
    fp64-input attention against the bf16-input one.
The mutation tests run the same checks against deliberately broken copies of
the oracle and require each copy to fail at least one of them.
"""
from __future__ import annotations

import math
from decimal import Decimal, getcontext

import numpy as np

from io_aware_exact_06_gb300 import inputs


def _rand_workload(seed, seqlens, H, d, std=1.0):
    return inputs.make_workload("pin", seed, seqlens, H, d, causal=False, qk_std=std, v_std=std)


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.max(np.abs(a - b) / np.maximum(1.0, np.abs(b))) if a.size else 0.0
    assert err <= tol, f"{what}: max rel/abs error {err:.3e} > {tol:.1e}"


def check_brute_force_decimal(orc):
    """Tiny inputs, definition evaluated in 50-digit decimal arithmetic."""
    getcontext().prec = 50
    wl = _rand_workload(101, [3, 5, 1], H=2, d=4)
    rows = inputs.all_rows(wl.cu_seqlens, wl.H)
    qf = inputs.bf16_bits_to_f64(wl.q)
    kf = inputs.bf16_bits_to_f64(wl.k)
    vf = inputs.bf16_bits_to_f64(wl.v)
    for causal in (False, True):
        for scale in (0.5, 1.0 / math.sqrt(4), 1.7):
            o, lse, _ = orc.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, scale, causal, 1)
            for n, (s, h, i) in enumerate(rows):
                base = int(wl.cu_seqlens[s])
                L = int(wl.cu_seqlens[s + 1]) - base
                nvis = i + 1 if causal else L
                ds = Decimal(scale)
                e = []
                for j in range(nvis):
                    dot = sum(Decimal(qf[base + i, h, c]) * Decimal(kf[base + j, h, c])
                              for c in range(wl.d))
                    e.append((ds * dot).exp())
                z = sum(e)
                ref_o = [float(sum(e[j] * Decimal(vf[base + j, h, c]) for j in range(nvis)) / z)
                         for c in range(wl.d)]
                _close(o[n], ref_o, 1e-13, f"O brute force row {(s, h, i)} causal={causal}")
                _close(lse[n], float(z.ln()), 1e-13, f"LSE brute force row {(s, h, i)}")


def check_two_key_closed_form(orc):
    """N=2, d=1: O_0 = (e^{s00} v0 + e^{s01} v1) / (e^{s00} + e^{s01})."""
    bits = inputs.f64_to_bf16_bits
    qv = np.array([1.5, -0.75]); kv = np.array([0.5, 2.0]); vv = np.array([3.0, -1.0])
    q = bits(qv).reshape(2, 1, 1); k = bits(kv).reshape(2, 1, 1); v = bits(vv).reshape(2, 1, 1)
    cu = np.array([0, 2])
    scale = 0.8
    rows = np.array([[0, 0, 0], [0, 0, 1]])
    o, lse, _ = orc.attn_rows(q, k, v, cu, rows, scale, False, 1)
    for i in range(2):
        s0 = scale * qv[i] * kv[0]
        s1 = scale * qv[i] * kv[1]
        ref = (math.exp(s0) * vv[0] + math.exp(s1) * vv[1]) / (math.exp(s0) + math.exp(s1))
        _close(o[i, 0], ref, 1e-15, f"two-key O row {i}")
        _close(lse[i], math.log(math.exp(s0) + math.exp(s1)), 1e-15, f"two-key LSE row {i}")
    o, lse, _ = orc.attn_rows(q, k, v, cu, rows, scale, True, 1)
    _close(o[0, 0], vv[0], 0.0, "causal row 0 sees only key 0")
    _close(lse[0], scale * qv[0] * kv[0], 1e-15, "causal row 0 LSE = its single logit")


def check_probs_sum_to_one(orc):
    wl = _rand_workload(202, [37, 64], H=3, d=16, std=2.0)
    for causal in (False, True):
        for (s, h, i) in [(0, 0, 0), (0, 2, 36), (1, 1, 17), (1, 2, 63)]:
            p = orc.attn_probs(wl.q, wl.k, wl.cu_seqlens, s, h, i, 0.25, causal)
            L = int(wl.cu_seqlens[s + 1] - wl.cu_seqlens[s])
            assert p.size == (i + 1 if causal else L), "visible key count"
            assert np.all(p >= 0)
            _close(math.fsum(p), 1.0, 1e-14, "sum of P row")


def check_constant_v(orc):
    wl = _rand_workload(303, [50, 20], H=2, d=8, std=1.5)
    c = inputs.f64_to_bf16_bits(np.array([-2.625]))[0]
    v = np.full_like(wl.v, c)
    rows = inputs.all_rows(wl.cu_seqlens, wl.H)
    for causal in (False, True):
        o, _, _ = orc.attn_rows(wl.q, wl.k, v, wl.cu_seqlens, rows, 0.3, causal, 2)
        _close(o, np.full_like(o, -2.625), 1e-14, "constant V gives constant O")


def check_zero_q_or_k(orc):
    wl = _rand_workload(404, [33, 7], H=2, d=8)
    zero = np.zeros_like(wl.q)
    rows = inputs.all_rows(wl.cu_seqlens, wl.H)
    vf = inputs.bf16_bits_to_f64(wl.v)
    # Q = 0, K = 0 or scale = 0: every logit is 0
    for which in ("q", "k", "scale"):
        q = zero if which == "q" else wl.q
        k = zero if which == "k" else wl.k
        scale = 0.0 if which == "scale" else 0.7
        for causal in (False, True):
            o, lse, _ = orc.attn_rows(q, k, wl.v, wl.cu_seqlens, rows, scale, causal, 2)
            for n, (s, h, i) in enumerate(rows):
                base = int(wl.cu_seqlens[s]); L = int(wl.cu_seqlens[s + 1]) - base
                nvis = i + 1 if causal else L
                ref = vf[base:base + nvis, h, :].mean(axis=0)
                _close(o[n], ref, 1e-14, f"{which}=0 mean of visible V")
                _close(lse[n], math.log(nvis), 1e-14, f"{which}=0 LSE = log(#visible)")


def check_one_hot_limit(orc):
    """K rows are distinct one-hot vectors, q_i = e_r: S_ij = scale * [j == r].

    With scale t >= 60 the softmax puts all but ~L*e^-t of its mass on key r, so
    O_i = v_r and LSE_i = t + log(1 + (L-1) e^-t) to fp64 precision."""
    L, d, H = 12, 16, 2
    k = np.zeros((L, H, d)); q = np.zeros((L, H, d))
    for j in range(L):
        k[j, :, j] = 1.0
    targets = [(i * 5 + 3) % L for i in range(L)]
    for i, r in enumerate(targets):
        q[i, :, r] = 1.0
    wl = _rand_workload(505, [L], H=H, d=d)
    bits = inputs.f64_to_bf16_bits
    qb, kb = bits(q.ravel()).reshape(q.shape), bits(k.ravel()).reshape(k.shape)
    rows = inputs.all_rows(wl.cu_seqlens, H)
    vf = inputs.bf16_bits_to_f64(wl.v)
    # scale 800: exp(800) overflows fp64, so this also needs a true max subtraction
    for scale in (60.0, 800.0):
        o, lse, _ = orc.attn_rows(qb, kb, wl.v, wl.cu_seqlens, rows, scale, False, 1)
        for n, (s, h, i) in enumerate(rows):
            r = targets[i]
            _close(o[n], vf[r, h], 1e-14, f"one-hot limit picks v_r (scale {scale})")
            _close(lse[n], scale + math.log1p((L - 1) * math.exp(-scale)), 1e-14,
                   f"one-hot LSE (scale {scale})")


def check_torch_sdpa(orc):
    """Library cross-check: torch SDPA (fp64, CPU) and logsumexp of the masked logits."""
    import torch
    B, H, N, d = 2, 3, 45, 16
    wl = _rand_workload(606, [N] * B, H=H, d=d, std=1.3)
    rows = inputs.all_rows(wl.cu_seqlens, H)
    to_t = lambda a: torch.from_numpy(inputs.bf16_bits_to_f64(a).reshape(B, N, H, d)).permute(0, 2, 1, 3)
    qt, kt, vt = to_t(wl.q), to_t(wl.k), to_t(wl.v)
    for causal in (False, True):
        scale = 1.0 / math.sqrt(d)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)
        logits = (qt @ kt.transpose(-1, -2)) * scale
        if causal:
            mask = torch.ones(N, N, dtype=torch.bool).tril()
            logits = logits.masked_fill(~mask, float("-inf"))
        ref_lse = torch.logsumexp(logits, dim=-1)
        o, lse, _ = orc.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, scale, causal, 2)
        for n, (s, h, i) in enumerate(rows):
            _close(o[n], ref[s, h, i].numpy(), 1e-12, f"SDPA O causal={causal}")
            _close(lse[n], float(ref_lse[s, h, i]), 1e-12, f"logsumexp causal={causal}")


def check_merge_identity(orc):
    rng_bits = inputs.splitmix64(707, 0, 4096)
    x = ((rng_bits >> np.uint64(11)).astype(np.float64) * 2.0 ** -53 - 0.5) * 40.0
    for n, cuts in [(1, []), (2, [1]), (10, [3]), (100, [10, 11, 50, 99]),
                    (1000, list(range(128, 1000, 128))), (777, [5, 400])]:
        xs = x[:n]
        sm, m, l = orc.softmax_merge(xs, cuts)
        e = np.exp(xs - xs.max())
        _close(sm, e / e.sum(), 1e-14, f"merged softmax n={n} cuts={len(cuts)}")
        _close(m, xs.max(), 0.0, "merged max")
        _close(l, math.fsum(e), 1e-13, "merged sum")
    # the merge must not depend on where the row is cut
    a, _, _ = orc.softmax_merge(x[:500], [7, 300])
    b, _, _ = orc.softmax_merge(x[:500], [250])
    _close(a, b, 1e-14, "merge independent of cut points")


def check_online_loop(orc):
    wl = _rand_workload(808, [200, 129], H=2, d=16, std=2.5)
    rows = inputs.all_rows(wl.cu_seqlens, wl.H)
    for causal in (False, True):
        o, lse, _ = orc.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, 0.4, causal, 2)
        for bc in (1, 7, 64, 128, 1000):
            o2, lse2 = orc.attn_online(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, 0.4, causal, bc)
            _close(o2, o, 1e-12, f"online loop O bc={bc} causal={causal}")
            _close(lse2, lse, 1e-12, f"online loop LSE bc={bc}")


def check_packing(orc):
    wl = _rand_workload(909, [17, 40, 3], H=2, d=8)
    for causal in (False, True):
        rows = inputs.all_rows(wl.cu_seqlens, wl.H)
        o, lse, _ = orc.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, 0.35, causal, 2)
        for s in range(wl.nseq):
            a, b = int(wl.cu_seqlens[s]), int(wl.cu_seqlens[s + 1])
            cu1 = np.array([0, b - a])
            rows1 = inputs.all_rows(cu1, wl.H)
            o1, lse1, _ = orc.attn_rows(wl.q[a:b], wl.k[a:b], wl.v[a:b], cu1, rows1, 0.35, causal, 1)
            sel = rows[:, 0] == s
            _close(o[sel], o1, 0.0, "packed sequence equals the sequence alone")
            _close(lse[sel], lse1, 0.0, "packed LSE equals the sequence alone")


def check_causal_last_row(orc):
    wl = _rand_workload(1010, [31, 64], H=2, d=8)
    rows = np.array([[0, 0, 30], [0, 1, 30], [1, 0, 63], [1, 1, 63]])
    o1, l1, _ = orc.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, 0.5, True, 1)
    o2, l2, _ = orc.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, 0.5, False, 1)
    _close(o1, o2, 0.0, "last causal row sees every key")
    _close(l1, l2, 0.0, "last causal row LSE")
    # and a middle row does not: causal row 10 must differ from the full row 10
    rows = np.array([[1, 0, 10]])
    o1, _, _ = orc.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, 0.5, True, 1)
    o2, _, _ = orc.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, 0.5, False, 1)
    assert np.max(np.abs(o1 - o2)) > 1e-3, "causal mask has no effect on a middle row"


def _visible(i, L, causal, wl, wr):
    """Visible keys of row i written out directly from the window definition."""
    return [j for j in range(L)
            if (not causal or j <= i) and (wl < 0 or j >= i - wl) and (wr < 0 or j <= i + wr)]


WINDOWS = [(0, 0), (1, -1), (2, 1), (-1, 2), (3, 0), (0, 5), (-1, -1)]


def check_window_brute_force_decimal(orc):
    """Sliding windows on tiny inputs against 50-digit decimal evaluation."""
    getcontext().prec = 50
    wl_ = _rand_workload(111, [6, 9], H=2, d=4, std=1.2)
    rows = inputs.all_rows(wl_.cu_seqlens, wl_.H)
    qf, kf, vf = (inputs.bf16_bits_to_f64(a) for a in (wl_.q, wl_.k, wl_.v))
    for causal in (False, True):
        for (a, b) in WINDOWS:
            o, lse, _ = orc.attn_rows(wl_.q, wl_.k, wl_.v, wl_.cu_seqlens, rows, 0.6, causal, 1,
                                      window=(a, b))
            for n, (s, h, i) in enumerate(rows):
                base = int(wl_.cu_seqlens[s]); L = int(wl_.cu_seqlens[s + 1]) - base
                vis = _visible(i, L, causal, a, b)
                e = [(Decimal(0.6) * sum(Decimal(qf[base + i, h, c]) * Decimal(kf[base + j, h, c])
                                         for c in range(wl_.d))).exp() for j in vis]
                z = sum(e)
                ref = [float(sum(e[t] * Decimal(vf[base + j, h, c]) for t, j in enumerate(vis)) / z)
                       for c in range(wl_.d)]
                _close(o[n], ref, 1e-13, f"window {(a, b)} causal={causal} row {(s, h, i)}")
                _close(lse[n], float(z.ln()), 1e-13, f"window LSE {(a, b)}")


def check_window_closed_forms(orc):
    """A zero-width window sees only its own key: O_i = v_i, LSE_i = scale q_i.k_i.
    Q = 0 gives the mean of V over the window; a window wider than the
    sequence is no window."""
    wl_ = _rand_workload(112, [20, 7], H=2, d=8)
    rows = inputs.all_rows(wl_.cu_seqlens, wl_.H)
    qf, kf, vf = (inputs.bf16_bits_to_f64(a) for a in (wl_.q, wl_.k, wl_.v))
    for causal, win in ((True, (0, -1)), (False, (0, 0))):
        o, lse, _ = orc.attn_rows(wl_.q, wl_.k, wl_.v, wl_.cu_seqlens, rows, 0.4, causal, 1,
                                  window=win)
        for n, (s, h, i) in enumerate(rows):
            t = int(wl_.cu_seqlens[s]) + i
            _close(o[n], vf[t, h], 0.0, "zero window picks v_i")
            _close(lse[n], 0.4 * float(np.dot(qf[t, h], kf[t, h])), 1e-14, "zero window LSE")
    zero = np.zeros_like(wl_.q)
    for causal in (False, True):
        for (a, b) in WINDOWS:
            o, lse, _ = orc.attn_rows(zero, wl_.k, wl_.v, wl_.cu_seqlens, rows, 0.4, causal, 1,
                                      window=(a, b))
            for n, (s, h, i) in enumerate(rows):
                base = int(wl_.cu_seqlens[s]); L = int(wl_.cu_seqlens[s + 1]) - base
                vis = _visible(i, L, causal, a, b)
                _close(o[n], vf[[base + j for j in vis], h].mean(axis=0), 1e-14, "Q=0 window mean")
                _close(lse[n], math.log(len(vis)), 1e-14, "Q=0 window LSE")
        o1, l1, _ = orc.attn_rows(wl_.q, wl_.k, wl_.v, wl_.cu_seqlens, rows, 0.4, causal, 1,
                                  window=(100, 100))
        o2, l2, _ = orc.attn_rows(wl_.q, wl_.k, wl_.v, wl_.cu_seqlens, rows, 0.4, causal, 1)
        _close(o1, o2, 0.0, "wide window is no window")
        _close(l1, l2, 0.0, "wide window LSE")


def check_window_torch_sdpa(orc):
    """torch scaled_dot_product_attention (fp64, CPU) with the window as a boolean mask."""
    import torch
    B, H, N, d = 2, 2, 37, 8
    wl_ = _rand_workload(113, [N] * B, H=H, d=d, std=1.3)
    rows = inputs.all_rows(wl_.cu_seqlens, H)
    to_t = lambda a: torch.from_numpy(inputs.bf16_bits_to_f64(a).reshape(B, N, H, d)).permute(0, 2, 1, 3)
    qt, kt, vt = to_t(wl_.q), to_t(wl_.k), to_t(wl_.v)
    ii = torch.arange(N).view(N, 1)
    jj = torch.arange(N).view(1, N)
    for causal in (False, True):
        for (a, b) in [(4, 0), (2, 3), (10, -1), (-1, 1)]:
            mask = torch.ones(N, N, dtype=torch.bool)
            if causal:
                mask &= jj <= ii
            if a >= 0:
                mask &= jj >= ii - a
            if b >= 0:
                mask &= jj <= ii + b
            ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=0.3)
            o, _, _ = orc.attn_rows(wl_.q, wl_.k, wl_.v, wl_.cu_seqlens, rows, 0.3, causal, 2,
                                    window=(a, b))
            for n, (s, h, i) in enumerate(rows):
                _close(o[n], ref[s, h, i].numpy(), 1e-12, f"SDPA window {(a, b)} causal={causal}")


# ------------------------------------------------------------ backward --

def _all_pairs(wl):
    return [(s, h) for s in range(wl.nseq) for h in range(wl.H)]


def _np_forward(qf, kf, vf, scale, causal):
    """O of one (sequence, head) from fp64 arrays [L, d] (for finite differences)."""
    S = scale * (qf @ kf.T)
    if causal:
        S = np.where(np.tril(np.ones(S.shape, dtype=bool)), S, -np.inf)
    S = S - S.max(axis=1, keepdims=True)
    P = np.exp(S)
    P /= P.sum(axis=1, keepdims=True)
    return P @ vf


def check_bwd_finite_differences(orc):
    """Central differences of loss = sum(dO * O) agree with the oracle's dQ, dK,
    dV; the fp64 forward used for the differences is first tied to the pinned
    forward oracle."""
    wl = _rand_workload(1111, [3, 6], H=2, d=4)
    dout = inputs.normal_bf16(1112, wl.q.size).reshape(wl.q.shape)
    qf, kf, vf = (inputs.bf16_bits_to_f64(a) for a in (wl.q, wl.k, wl.v))
    dof = inputs.bf16_bits_to_f64(dout)
    scale = 0.6
    for causal in (False, True):
        pairs = _all_pairs(wl)
        dq, dk, dv, _ = orc.attn_bwd(wl.q, wl.k, wl.v, dout, wl.cu_seqlens, pairs, scale, causal)
        o_or, _, _ = orc.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens,
                                   inputs.all_rows(wl.cu_seqlens, wl.H), scale, causal, 1)
        for n, (s, h) in enumerate(pairs):
            a, b = int(wl.cu_seqlens[s]), int(wl.cu_seqlens[s + 1])
            X = [qf[a:b, h].copy(), kf[a:b, h].copy(), vf[a:b, h].copy()]
            G = dof[a:b, h]
            sel = [r for r, (ss, hh, _) in enumerate(inputs.all_rows(wl.cu_seqlens, wl.H))
                   if ss == s and hh == h]
            _close(_np_forward(*X, scale, causal), o_or[sel], 1e-13, "fp64 forward = oracle forward")
            eps = 1e-6
            for t, grad in enumerate((dq[n], dk[n], dv[n])):
                num = np.zeros_like(X[t])
                for idx in np.ndindex(*X[t].shape):
                    keep = X[t][idx]
                    X[t][idx] = keep + eps
                    up = float(np.sum(G * _np_forward(*X, scale, causal)))
                    X[t][idx] = keep - eps
                    dn = float(np.sum(G * _np_forward(*X, scale, causal)))
                    X[t][idx] = keep
                    num[idx] = (up - dn) / (2 * eps)
                _close(grad, num, 1e-7, f"finite differences of {'QKV'[t]} causal={causal}")


def check_bwd_window(orc):
    """Sliding-window gradients: central finite differences of a windowed fp64
    forward (tied to the pinned windowed forward oracle) and torch autograd
    through an attention with the window as an explicit boolean mask."""
    import torch
    wl_, H, d = [7, 12], 2, 4
    wlk = _rand_workload(1919, wl_, H=H, d=d)
    dout = inputs.normal_bf16(1920, wlk.q.size).reshape(wlk.q.shape)
    qf, kf, vf = (inputs.bf16_bits_to_f64(a) for a in (wlk.q, wlk.k, wlk.v))
    dof = inputs.bf16_bits_to_f64(dout)
    scale = 0.55
    for causal, (a, b) in [(False, (2, 1)), (True, (3, -1)), (False, (0, 0)), (True, (1, 5))]:
        pairs = _all_pairs(wlk)
        dq, dk, dv, _ = orc.attn_bwd(wlk.q, wlk.k, wlk.v, dout, wlk.cu_seqlens, pairs, scale, causal,
                                     window=(a, b))
        rows = inputs.all_rows(wlk.cu_seqlens, wlk.H)
        o_or, _, _ = orc.attn_rows(wlk.q, wlk.k, wlk.v, wlk.cu_seqlens, rows, scale, causal, 1,
                                   window=(a, b))
        for n, (sq, h) in enumerate(pairs):
            lo, hi = int(wlk.cu_seqlens[sq]), int(wlk.cu_seqlens[sq + 1])
            L = hi - lo
            vis = np.zeros((L, L), dtype=bool)
            for i in range(L):
                vis[i, _visible(i, L, causal, a, b)] = True

            def fwd(X):
                S = scale * (X[0] @ X[1].T)
                S = np.where(vis, S, -np.inf)
                S = S - S.max(axis=1, keepdims=True)
                P = np.exp(S)
                P /= P.sum(axis=1, keepdims=True)
                return P @ X[2]

            X = [qf[lo:hi, h].copy(), kf[lo:hi, h].copy(), vf[lo:hi, h].copy()]
            sel = [r for r, (s2, h2, _) in enumerate(rows) if s2 == sq and h2 == h]
            _close(fwd(X), o_or[sel], 1e-13, "windowed fp64 forward = oracle forward")
            G = dof[lo:hi, h]
            eps = 1e-6
            for t, grad in enumerate((dq[n], dk[n], dv[n])):
                num = np.zeros_like(X[t])
                for idx in np.ndindex(*X[t].shape):
                    keep = X[t][idx]
                    X[t][idx] = keep + eps
                    up = float(np.sum(G * fwd(X)))
                    X[t][idx] = keep - eps
                    dn = float(np.sum(G * fwd(X)))
                    X[t][idx] = keep
                    num[idx] = (up - dn) / (2 * eps)
                _close(grad, num, 1e-7, f"window {(a, b)} finite differences of {'QKV'[t]}")
            # torch autograd with the mask
            qt, kt, vt = (torch.from_numpy(x.copy()).requires_grad_(True) for x in X)
            out = torch.nn.functional.scaled_dot_product_attention(
                qt[None], kt[None], vt[None], attn_mask=torch.from_numpy(vis)[None], scale=scale)[0]
            out.backward(torch.from_numpy(G.copy()))
            _close(dq[n], qt.grad.numpy(), 1e-11, f"window {(a, b)} autograd dQ")
            _close(dk[n], kt.grad.numpy(), 1e-11, f"window {(a, b)} autograd dK")
            _close(dv[n], vt.grad.numpy(), 1e-11, f"window {(a, b)} autograd dV")


def check_bwd_torch_autograd(orc):
    """Library cross-check: torch autograd through SDPA, fp64 on CPU."""
    import torch
    B, H, N, d = 2, 3, 37, 16
    wl = _rand_workload(1212, [N] * B, H=H, d=d, std=1.2)
    dout = inputs.normal_bf16(1213, wl.q.size).reshape(wl.q.shape)
    to_t = lambda a: torch.from_numpy(inputs.bf16_bits_to_f64(a).reshape(B, N, H, d)).permute(0, 2, 1, 3)
    for causal in (False, True):
        qt, kt, vt = (to_t(a).clone().requires_grad_(True) for a in (wl.q, wl.k, wl.v))
        scale = 1.0 / math.sqrt(d)
        out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)
        out.backward(to_t(dout))
        pairs = _all_pairs(wl)
        dq, dk, dv, _ = orc.attn_bwd(wl.q, wl.k, wl.v, dout, wl.cu_seqlens, pairs, scale, causal, 2)
        for n, (s, h) in enumerate(pairs):
            _close(dq[n], qt.grad[s, h].numpy(), 1e-11, f"autograd dQ causal={causal}")
            _close(dk[n], kt.grad[s, h].numpy(), 1e-11, f"autograd dK causal={causal}")
            _close(dv[n], vt.grad[s, h].numpy(), 1e-11, f"autograd dV causal={causal}")


def check_bwd_invariants(orc):
    """Rows of P sum to one, so sum_j dV_j = sum_i dO_i and sum_j dS_ij = 0,
    so sum_j dK_j = 0; constant V rows make dP constant along a row, so
    dS = 0 and dQ = dK = 0; dO = 0 gives no gradient at all."""
    wl = _rand_workload(1313, [9, 30, 1], H=2, d=8)
    dout = inputs.normal_bf16(1314, wl.q.size).reshape(wl.q.shape)
    dof = inputs.bf16_bits_to_f64(dout)
    pairs = _all_pairs(wl)
    for causal in (False, True):
        dq, dk, dv, _ = orc.attn_bwd(wl.q, wl.k, wl.v, dout, wl.cu_seqlens, pairs, 0.45, causal)
        for n, (s, h) in enumerate(pairs):
            a, b = int(wl.cu_seqlens[s]), int(wl.cu_seqlens[s + 1])
            _close(dv[n].sum(axis=0), dof[a:b, h].sum(axis=0), 1e-12, "sum of dV = sum of dO")
            _close(dk[n].sum(axis=0), np.zeros(wl.d), 1e-12, "sum of dK = 0")
        vconst = np.tile(inputs.f64_to_bf16_bits(np.linspace(-2, 2, wl.d)), (wl.q.shape[0], wl.H, 1))
        dq, dk, dv, _ = orc.attn_bwd(wl.q, wl.k, vconst, dout, wl.cu_seqlens, pairs, 0.45, causal)
        for n in range(len(pairs)):
            _close(dq[n], 0 * dq[n], 1e-12, "constant V: dQ = 0")
            _close(dk[n], 0 * dk[n], 1e-12, "constant V: dK = 0")
        zero = np.zeros_like(dout)
        dq, dk, dv, _ = orc.attn_bwd(wl.q, wl.k, wl.v, zero, wl.cu_seqlens, pairs, 0.45, causal)
        for n in range(len(pairs)):
            assert not dq[n].any() and not dk[n].any() and not dv[n].any(), "dO = 0: no gradient"


def check_bwd_packing(orc):
    """A sequence inside a packed batch has the gradients it has alone."""
    wl = _rand_workload(1414, [13, 21, 2], H=2, d=8)
    dout = inputs.normal_bf16(1415, wl.q.size).reshape(wl.q.shape)
    pairs = _all_pairs(wl)
    for causal in (False, True):
        dq, dk, dv, _ = orc.attn_bwd(wl.q, wl.k, wl.v, dout, wl.cu_seqlens, pairs, 0.3, causal, 3)
        for n, (s, h) in enumerate(pairs):
            a, b = int(wl.cu_seqlens[s]), int(wl.cu_seqlens[s + 1])
            g = orc.attn_bwd(wl.q[a:b], wl.k[a:b], wl.v[a:b], dout[a:b], np.array([0, b - a]),
                             [(0, h)], 0.3, causal, 1)
            for t in range(3):
                _close((dq, dk, dv)[t][n], g[t][0], 1e-13, f"packed gradient {'QKV'[t]}")


# ---------------------------------------------------------------- FP8 --

def _e4m3_table():
    """Every finite e4m3 value from its bit fields (sign, 4-bit exponent with
    bias 7, 3-bit mantissa; exponent 15 with mantissa 7 is NaN)."""
    vals = {}
    for c in range(256):
        sgn = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue
        vals[c] = sgn * (m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return vals


def check_e4m3_brute_force(orc):
    """Decoding matches the bit fields; encoding is the nearest finite value
    by exhaustive search (ties to the even code, beyond 448 saturating)."""
    table = _e4m3_table()
    codes = np.array(sorted(table), dtype=np.uint8)
    _close(orc.e4m3_decode(codes), [table[c] for c in codes], 0.0, "e4m3 decode")
    assert math.isnan(orc.e4m3_decode([0x7f])[0]) and math.isnan(orc.e4m3_decode([0xff])[0])
    assert table[0x7e] == 448.0 and table[0x08] == 2.0 ** -6 and table[0x01] == 2.0 ** -9
    pos = sorted((v, c) for c, v in table.items() if v >= 0 and c != 0x80)
    bits = inputs.splitmix64(1515, 0, 4000)
    xs = list(((bits >> np.uint64(40)).astype(np.float64) / 2.0 ** 24 - 0.5) * 1100.0)
    xs += [v for v, _ in pos] + [(pos[i][0] + pos[i + 1][0]) / 2 for i in range(len(pos) - 1)]
    xs += [1e-12, 2.0 ** -10, 447.9, 448.0, 463.9, 464.0, 1e6]
    xs = np.array([np.float32(x) for x in xs] + [-np.float32(x) for x in xs], dtype=np.float32)
    got = orc.e4m3_encode(xs)
    for x, c in zip(xs, got):
        a = abs(float(x))
        best = min(pos, key=lambda vc: (abs(vc[0] - a), vc[1] & 1))  # nearest, then even code
        want = best[1] if a < 448.0 else 0x7e
        if x < 0 and not (want == 0 and a < 2.0 ** -10 + 0.0):
            want |= 0x80
        if want & 0x7f == 0:  # +-0: either sign bit
            assert c & 0x7f == 0, f"e4m3({x}) = {c:#x}, want zero"
            continue
        assert c == want, f"e4m3({x}) = {c:#x}, want {want:#x}"


def check_fwht(orc):
    """The fp32 butterflies equal (x * signs) H_d with H_d from scipy (the
    Sylvester construction): exactly on small integers (every partial sum is
    exact in fp32), within fp32 rounding on normal draws; H_d H_d = d I."""
    from scipy.linalg import hadamard
    for d in (8, 64, 128):
        Hd = hadamard(d).astype(np.float64)
        signs = np.where(inputs.splitmix64(1616 + d, 0, d) & np.uint64(1), -1, 1).astype(np.int8)
        ints = ((inputs.splitmix64(1617 + d, 0, 4 * d) % np.uint64(201)).astype(np.float64) - 100).reshape(4, d)
        got = orc.fwht_f32(ints, signs)
        _close(got, (ints * signs) @ Hd, 0.0, f"integer Hadamard d={d}")
        x = inputs.bf16_bits_to_f64(inputs.normal_bf16(1618 + d, 8 * d)).reshape(8, d)
        got = orc.fwht_f32(x, signs).astype(np.float64)
        ref = (x * signs) @ Hd
        assert np.max(np.abs(got - ref)) <= 1e-5 * np.max(np.abs(ref)), f"fp32 Hadamard d={d}"
        twice = orc.fwht_f32(orc.fwht_f32(x, None), None).astype(np.float64)
        assert np.max(np.abs(twice - d * x)) <= 1e-4 * d * np.max(np.abs(x)), "H H = d I"


def check_fp8_block_quantize(orc):
    """Per-block scale = max|x| / 448 and codes = nearest e4m3 of x * (448 /
    max|x|) (fp32), by exhaustive search; the last block of a ragged sequence
    is pulled back and leaves the rows it shares to the block before it; with
    rotation the block is that of the Hadamard-rotated rows."""
    table = _e4m3_table()
    pos = sorted((v, c) for c, v in table.items() if v >= 0 and c != 0x80)
    grid = np.array([v for v, _ in pos])

    def nearest(y):
        a = np.abs(y.astype(np.float64))
        idx = np.abs(a[..., None] - grid[None, :]).argmin(axis=-1)
        # ties to the even code: if the next code is equally near and even, take it
        nxt = np.minimum(idx + 1, len(grid) - 1)
        tie = np.abs(a - grid[nxt]) == np.abs(a - grid[idx])
        odd = np.array([pos[i][1] & 1 for i in range(len(pos))])[idx] == 1
        idx = np.where(tie & odd & (nxt != idx), nxt, idx)
        c = np.array([pos[i][1] for i in range(len(pos))], dtype=np.uint8)[idx]
        return np.where((y < 0) & (c != 0), c | 0x80, c).astype(np.uint8)

    B, N, H, d, rows = 2, 300, 2, 8, 128
    x = inputs.normal_bf16(1717, B * N * H * d, 2.0).reshape(B * N, H, d)
    xf = inputs.bf16_bits_to_f64(x).astype(np.float32)
    for rotate in (False, True):
        signs = np.array([1, -1, 1, 1, -1, -1, 1, -1], dtype=np.int8)
        codes, scales = orc.fp8_quantize(x, B, N, rows, rotate, signs)
        nblk = -(-N // rows)
        assert scales.shape == (B, H, nblk)
        for b in range(B):
            for h in range(H):
                for t in range(nblk):
                    r0 = min(t * rows, N - rows)
                    blk = xf[b * N + r0:b * N + r0 + rows, h]
                    if rotate:
                        blk = orc.fwht_f32(blk, signs)
                    amax = np.float32(np.max(np.abs(blk)))
                    assert scales[b, h, t] == np.float32(amax / np.float32(448.0)), "block scale"
                    inv = np.float32(np.float32(448.0) / amax)
                    want = nearest((blk * inv).astype(np.float32))
                    keep = np.arange(r0, r0 + rows) >= t * rows
                    got = codes[b * N + r0:b * N + r0 + rows, h][keep]
                    assert np.array_equal(got, want[keep]), f"codes b={b} h={h} t={t} rotate={rotate}"


def check_fp8_tensor_quantize(orc):
    """Per-tensor quantisation: one scale per head = max|x| over every token of
    the head / 448, codes = nearest e4m3 of x * (448 / max|x|) (fp32), by
    exhaustive search; an all-zero head gets scale 1 and zero codes."""
    table = _e4m3_table()
    pos = sorted((v, c) for c, v in table.items() if v >= 0 and c != 0x80)
    grid = np.array([v for v, _ in pos])
    codes_of = np.array([c for _, c in pos], dtype=np.uint8)
    tokens, H, d = 301, 3, 8
    x = inputs.normal_bf16(1719, tokens * H * d, 1.5).reshape(tokens, H, d)
    xf = inputs.bf16_bits_to_f64(x).astype(np.float32)
    # head 1 carries one large entry late in the tensor (the scale must see it);
    # head 2 is all zero
    x[250, 1, 5] = inputs.f64_to_bf16_bits(np.array([37.0]))[0]
    xf[250, 1, 5] = 37.0
    x[:, 2] = 0
    xf[:, 2] = 0
    codes, scales = orc.fp8_quantize_tensor(x)
    assert scales.shape == (H,) and codes.shape == (tokens, H, d)
    for h in range(H):
        amax = np.float32(np.max(np.abs(xf[:, h])))
        if amax == 0:
            assert scales[h] == 1.0 and not codes[:, h].any(), "all-zero head"
            continue
        assert scales[h] == np.float32(amax / np.float32(448.0)), f"tensor scale h={h}"
        y = (xf[:, h] * np.float32(np.float32(448.0) / amax)).astype(np.float32)
        a = np.abs(y.astype(np.float64))
        dist = np.abs(a[..., None] - grid[None, :])
        best = dist.min(axis=-1, keepdims=True)
        # nearest value; among two equally near, the even code
        cand = np.where(dist == best, codes_of[None, None, :].astype(np.int32) | 0x100, 0)
        even = np.where((cand & 1) == 0, cand, 0).max(axis=-1)
        want = np.where(even > 0, even, cand.max(axis=-1)) & 0xff
        want = np.where((y < 0) & (want != 0), want | 0x80, want).astype(np.uint8)
        assert np.array_equal(codes[:, h], want), f"tensor codes h={h}"
    assert codes[250, 1, 5] == 0x7e, "the head's largest value maps to 448"


def check_attn_rows_f64(orc):
    """The fp64-input definition equals the bf16-input one on bf16 values."""
    wl = _rand_workload(1818, [37, 5], H=2, d=8, std=1.5)
    rows = inputs.all_rows(wl.cu_seqlens, wl.H)
    f = lambda a: inputs.bf16_bits_to_f64(a)
    for causal in (False, True):
        o1, l1, _ = orc.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, 0.4, causal, 1)
        o2, l2 = orc.attn_rows_f64(f(wl.q), f(wl.k), f(wl.v), wl.cu_seqlens, rows, 0.4, causal)
        _close(o2, o1, 1e-14, f"f64-input O causal={causal}")
        _close(l2, l1, 1e-14, f"f64-input LSE causal={causal}")
    # logits of several hundred: exp overflows fp64 without the true row max
    o1, l1, _ = orc.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, 400.0, False, 1)
    o2, l2 = orc.attn_rows_f64(f(wl.q), f(wl.k), f(wl.v), wl.cu_seqlens, rows, 400.0, False)
    _close(o2, o1, 1e-12, "f64-input O, large logits")
    _close(l2, l1, 1e-12, "f64-input LSE, large logits")


ALL_CHECKS = [
    check_brute_force_decimal,
    check_two_key_closed_form,
    check_probs_sum_to_one,
    check_constant_v,
    check_zero_q_or_k,
    check_one_hot_limit,
    check_torch_sdpa,
    check_merge_identity,
    check_online_loop,
    check_packing,
    check_causal_last_row,
    check_window_brute_force_decimal,
    check_window_closed_forms,
    check_window_torch_sdpa,
    check_bwd_finite_differences,
    check_bwd_torch_autograd,
    check_bwd_invariants,
    check_bwd_packing,
    check_bwd_window,
    check_e4m3_brute_force,
    check_fwht,
    check_fp8_block_quantize,
    check_fp8_tensor_quantize,
    check_attn_rows_f64,
]
