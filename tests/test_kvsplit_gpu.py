"""Split-KV forward (attn_fwd_kvsplit) against the fp64 oracle.

Queries and keys have different lengths; with the causal mask the Nq queries
are the last Nq positions of the key sequence.  The oracle computes such a
row as row Nk - Nq + r of a self-attention problem whose query tensor is zero
except for those last Nq rows (a zero query row changes no other row), and a
non-causal row at any position of such a problem (every key is visible)."""
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


def make_cross(seed, B, H, Nq, Nk, d, qk_std=1.0):
    q = inputs.normal_bf16(seed * 4 + 1, B * Nq * H * d, qk_std).reshape(B, Nq, H, d)
    k = inputs.normal_bf16(seed * 4 + 2, B * Nk * H * d, qk_std).reshape(B, Nk, H, d)
    v = inputs.normal_bf16(seed * 4 + 3, B * Nk * H * d).reshape(B, Nk, H, d)
    return q, k, v


def oracle_cross(q, k, v, scale, causal, rows):
    """O, LSE of (b, h, r) rows of the cross problem via the embedding above."""
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    cu = np.arange(B + 1, dtype=np.int64) * Nk
    kk = k.reshape(B * Nk, H, d)
    vv = v.reshape(B * Nk, H, d)
    o = np.zeros((len(rows), d))
    lse = np.zeros(len(rows))
    if causal:
        qf = np.zeros((B, Nk, H, d), dtype=np.uint16)
        qf[:, Nk - Nq:] = q
        srows = rows.copy()
        srows[:, 2] += Nk - Nq
        return oracle.attn_rows(qf.reshape(B * Nk, H, d), kk, vv, cu, srows, scale, True)[:2]
    # non-causal: query rows r are placed at position r % Nk, one layer at a time
    for layer in range((Nq + Nk - 1) // Nk):
        sel = (rows[:, 2] // Nk) == layer
        if not sel.any():
            continue
        qf = np.zeros((B, Nk, H, d), dtype=np.uint16)
        lo, hi = layer * Nk, min(Nq, (layer + 1) * Nk)
        qf[:, : hi - lo] = q[:, lo:hi]
        srows = rows[sel].copy()
        srows[:, 2] -= lo
        o[sel], lse[sel], _ = oracle.attn_rows(qf.reshape(B * Nk, H, d), kk, vv, cu, srows, scale,
                                                False)
    return o, lse


def run_kvsplit(dev, q, k, v, scale, causal, splits):
    import torch
    import io_aware_exact_06_gb300 as fa
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    qt, kt, vt = t(q), t(k), t(v)
    o = torch.full_like(qt, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), device=dev)
    fa.attn_fwd_kvsplit(qt, kt, vt, o, lse, B, H, Nq, Nk, d, scale, causal, splits)
    assert fa.attn_last_device_error() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check(dev, q, k, v, causal, splits, what, scale=None):
    B, Nq, H, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    o, lse = run_kvsplit(dev, q, k, v, scale, causal, splits)
    bb, hh, rr = np.meshgrid(np.arange(B), np.arange(H), np.arange(Nq), indexing="ij")
    rows = np.stack([bb.ravel(), hh.ravel(), rr.ravel()], axis=1).astype(np.int64)
    ref_o, ref_lse = oracle_cross(q, k, v, scale, causal, rows)
    got_o = o[rows[:, 0], rows[:, 2], rows[:, 1]].astype(np.float64)
    got_l = lse[rows[:, 0], rows[:, 1], rows[:, 2]].astype(np.float64)
    stats = parity.error_stats(got_o, got_l, ref_o, ref_lse)
    assert np.isfinite(got_o).all() and np.isfinite(got_l).all(), what
    assert stats["o_max_abs"] <= parity.O_MAX_ABS, (what, stats)
    assert stats["o_rel_l2"] <= parity.O_REL_L2, (what, stats)
    assert stats["lse_max_abs"] <= parity.LSE_MAX_ABS, (what, stats)


@pytest.mark.parametrize("splits", [1, 3, 16, 0])
@pytest.mark.parametrize("causal", [False, True])
def test_decode_shapes(dev, causal, splits):
    q, k, v = make_cross(901, 2, 4, 1, 4000, 128)
    check(dev, q, k, v, causal, splits, f"decode Nq=1 Nk=4000 splits={splits}")
    q, k, v = make_cross(902, 2, 3, 64, 3000, 128, qk_std=2.0)
    check(dev, q, k, v, causal, splits, f"Nq=64 Nk=3000 splits={splits}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths_and_empty_ranges(dev, d, causal):
    # 300 queries against 1000 keys, 5 ranges; and 8 ranges over 2 KV tiles
    q, k, v = make_cross(903 + d, 2, 2, 300, 1000, d)
    check(dev, q, k, v, causal, 5, "Nq=300 Nk=1000")
    q, k, v = make_cross(905 + d, 1, 2, 100, 200, d)
    check(dev, q, k, v, causal, 8, "more ranges than tiles")


def test_noncausal_more_queries_than_keys(dev):
    q, k, v = make_cross(907, 1, 2, 700, 300, 64)
    check(dev, q, k, v, False, 3, "Nq > Nk non-causal")


def test_equal_lengths_match_attn_fwd(dev):
    import torch
    import io_aware_exact_06_gb300 as fa
    wl = inputs.config_workload("gpt2_causal")
    q, k, v, _ = parity.to_device(wl, dev)
    B, N, H, d = wl.nseq, 1024, wl.H, wl.d
    o1 = torch.empty_like(q); l1 = torch.empty((B, H, N), device=dev)
    o2 = torch.empty_like(q); l2 = torch.empty((B, H, N), device=dev)
    fa.attn_fwd(q, k, v, o1, l1, B, H, N, d, wl.scale, True)
    fa.attn_fwd_kvsplit(q, k, v, o2, l2, B, H, N, N, d, wl.scale, True, 4)
    assert (o1.float() - o2.float()).abs().max().item() <= parity.O_MAX_ABS
    assert (l1 - l2).abs().max().item() <= parity.LSE_MAX_ABS


def test_causal_needs_enough_keys(dev):
    import io_aware_exact_06_gb300 as fa
    with pytest.raises(fa.AttnError) as e:
        fa.attn_fwd_kvsplit(1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1, 1, 200, 100, 64, 0.1, True)
    assert e.value.status == -2


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_is_uniform_average(dev, causal):
    # every visible key weighs 1 in every KV range; masked keys still weigh 0
    q, k, v = make_cross(909, 2, 2, 40, 1000, 128)
    check(dev, q, k, v, causal, 5, "scale 0", scale=0.0)


# One query row takes the CUDA-core decode kernel, more take the tensor-core
# split kernel.  Ragged key counts, more ranges than keys (empty ranges), a
# single key, both head dimensions.
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq", [1, 2, 3, 4])
def test_decode_kernel_query_counts(dev, d, causal, Nq):
    q, k, v = make_cross(920 + Nq + d, 3, 2, Nq, 1999, d)
    check(dev, q, k, v, causal, 0, f"Nq={Nq} Nk=1999 d={d}")
    q, k, v = make_cross(930 + Nq + d, 1, 3, Nq, 70, d, qk_std=2.0)
    check(dev, q, k, v, causal, 200, f"Nq={Nq} Nk=70 200 ranges d={d}")


@pytest.mark.parametrize("Nq", [1, 4])
def test_decode_kernel_single_key(dev, Nq):
    q, k, v = make_cross(940 + Nq, 2, 2, Nq, Nq, 128)
    check(dev, q, k, v, True, 0, f"Nq=Nk={Nq} causal")
    check(dev, q, k, v, False, 3, f"Nq=Nk={Nq}")


def test_decode_kernel_zero_scale(dev):
    q, k, v = make_cross(950, 2, 2, 3, 777, 128)
    check(dev, q, k, v, True, 0, "Nq=3 scale 0", scale=0.0)
