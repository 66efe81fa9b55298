"""attn_fwd_decode (one query per sequence against packed keys of different
lengths) against the fp64 oracle.

The oracle computes a decode query as the last row of a causal
self-attention problem over the same keys whose other query rows are zero:
the last position sees every key, and a zero query row changes no other row
(rows are independent in the definition).  Tolerances are the forward's."""
import numpy as np
import pytest

import oracle
from io_aware_exact_06_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    import __graft_entry__
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    __graft_entry__.build()
    return torch.device("cuda:0")


def make(seed, lens, H, d, qk_std=1.0):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    total, B = int(cu[-1]), len(lens)
    q = inputs.normal_bf16(seed * 4 + 1, B * H * d, qk_std).reshape(B, H, d)
    k = inputs.normal_bf16(seed * 4 + 2, total * H * d, qk_std).reshape(total, H, d)
    v = inputs.normal_bf16(seed * 4 + 3, total * H * d).reshape(total, H, d)
    return cu, q, k, v


def t(dev, bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def run(dev, cu, q, k, v, scale, splits, max_len=None):
    import torch
    import io_aware_exact_06_gb300 as fa
    B, H, d = q.shape
    o = torch.full((B, H, d), 7.0, dtype=torch.bfloat16, device=dev)
    lse = torch.full((B, H), 7.0, dtype=torch.float32, device=dev)
    cu_d = torch.tensor(np.asarray(cu), dtype=torch.int32, device=dev)
    ml = int(np.diff(cu).max()) if max_len is None else max_len
    fa.attn_fwd_decode(t(dev, q), t(dev, k), t(dev, v), o, lse, B, H, d, scale, cu_d, ml, splits)
    return o, lse, fa.attn_last_device_error()


def reference(cu, q, k, v, scale):
    """O [B, H, d] and LSE [B, H] of each decode query (sequences with keys)."""
    B, H, d = q.shape
    qpack = np.zeros_like(k)
    rows = []
    for b in range(B):
        L = int(cu[b + 1] - cu[b])
        if L:
            qpack[cu[b] + L - 1] = q[b]
            rows += [(b, h, L - 1) for h in range(H)]
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
    o, lse, _ = oracle.attn_rows(qpack, k, v, cu, rows, scale, True)
    return rows, o, lse


def check(dev, cu, q, k, v, scale, splits, what):
    o, lse, st = run(dev, cu, q, k, v, scale, splits)
    assert st == 0, what
    rows, ref_o, ref_lse = reference(cu, q, k, v, scale)
    got_o = o.float().cpu().numpy()[rows[:, 0], rows[:, 1]].astype(np.float64)
    got_l = lse.cpu().numpy()[rows[:, 0], rows[:, 1]].astype(np.float64)
    stats = parity.error_stats(got_o, got_l, ref_o, ref_lse)
    assert np.isfinite(got_o).all() and np.isfinite(got_l).all(), what
    assert stats["o_max_abs"] <= parity.O_MAX_ABS, (what, stats)
    assert stats["o_rel_l2"] <= parity.O_REL_L2, (what, stats)
    assert stats["lse_max_abs"] <= parity.LSE_MAX_ABS, (what, stats)
    # sequences without keys: O = 0, LSE = -inf
    empty = [b for b in range(len(cu) - 1) if cu[b + 1] == cu[b]]
    if empty:
        assert (o[empty].float() == 0).all() and (lse[empty] == -np.inf).all(), what


LENS = [0, 1, 63, 64, 65, 1000, 4097, 300]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("splits", [0, 1, 7, 256])
def test_packed_lengths(dev, d, splits):
    cu, q, k, v = make(960 + d + splits, LENS, 3, d)
    check(dev, cu, q, k, v, d ** -0.5, splits, f"d={d} splits={splits}")


def test_peaky_scores(dev):
    # Q, K ~ N(0, 3^2): the running max of a key range moves often
    cu, q, k, v = make(970, [5000, 123, 2048], 4, 128, qk_std=3.0)
    check(dev, cu, q, k, v, 128 ** -0.5, 0, "Q/K std 3")


def test_zero_scale(dev):
    cu, q, k, v = make(971, [700, 0, 31], 2, 128)
    check(dev, cu, q, k, v, 0.0, 0, "scale 0")


def test_equal_lengths_match_kvsplit(dev):
    """Equal key lengths, same range count: the same arithmetic as
    attn_fwd_kvsplit with one query row, bit for bit."""
    import torch
    import io_aware_exact_06_gb300 as fa
    B, H, Nk, d = 3, 4, 3000, 128
    cu, q, k, v = make(972, [Nk] * B, H, d)
    o1, l1, st = run(dev, cu, q, k, v, d ** -0.5, 5)
    assert st == 0
    o2 = torch.empty((B, 1, H, d), dtype=torch.bfloat16, device=dev)
    l2 = torch.empty((B, H, 1), dtype=torch.float32, device=dev)
    fa.attn_fwd_kvsplit(t(dev, q).view(B, 1, H, d), t(dev, k).view(B, Nk, H, d),
                        t(dev, v).view(B, Nk, H, d), o2, l2, B, H, 1, Nk, d, d ** -0.5, True, 5)
    assert fa.attn_last_device_error() == 0
    assert torch.equal(o1, o2.view(B, H, d)) and torch.equal(l1, l2.view(B, H))


@pytest.mark.parametrize("bad", ["decreasing", "too_long", "nonzero_start"])
def test_invalid_cu_seqlens_reported(dev, bad):
    cu, q, k, v = make(973, [100, 100, 100], 2, 128)
    cu_bad = {"decreasing": [0, 150, 120, 300], "too_long": [0, 100, 300, 300],
              "nonzero_start": [8, 100, 200, 300]}[bad]
    o, lse, st = run(dev, cu_bad, q, k, v, 0.1, 0, max_len=128)
    assert st == -8
    assert (o.float() == 7.0).all() and (lse == 7.0).all(), "nothing is written"


def test_convenience_wrapper(dev):
    import torch
    import io_aware_exact_06_gb300 as fa
    cu, q, k, v = make(974, [900, 17, 2500], 2, 128)
    o1, l1, st = run(dev, cu, q, k, v, 128 ** -0.5, 0)
    assert st == 0
    cu_d = torch.tensor(cu, dtype=torch.int32, device=dev)
    o2, l2 = fa.decode(t(dev, q), t(dev, k), t(dev, v), cu_d, 2500)
    assert fa.attn_last_device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
