"""Tensors past 4 GB against the fp64 oracle: outputs at byte offsets beyond
2^32 (the last sequences and heads of [B, N, H, d] bf16 tensors of 5.4 GB, a
key cache of 8.6 GB per tensor), where every address computation has to be
64-bit.

Each output row of the forward depends only on its own (sequence, head)
slice of Q, K and V; each gradient row of the backward only on its slice of
Q, K, V and dO (O and the LSE being computed from them); the FP8 codes of a
slice only on that slice (block scales per 128 rows of one (sequence, head),
one V scale per (sequence, head)); a decoded row only on its (sequence, head)
keys.  So the large tensors are filled on the device with seeded normals
(torch's generator), and the compared slices are overwritten with the seeded
input module's values, which the oracle then takes on their own.  Outputs
start as NaN, so a row the kernels never wrote fails.  Tolerances are those
of the forward, backward, FP8 and decode parity tests."""
import numpy as np
import pytest

import oracle
from io_aware_exact_06_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu

# dense [B, N, H, d] bf16: 256 * 1024 * 80 * 128 * 2 bytes = 5.37 GB per tensor
B, N, H, D = 256, 1024, 80, 128
# (sequence, head) slices compared; the first ends at the last byte of the tensors
PAIRS = [(B - 1, H - 1), (B // 2 + 3, 7), (0, H - 1)]


@pytest.fixture(scope="module")
def dev():
    import torch
    import __graft_entry__
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def release_memory():
    yield
    import torch
    if torch.cuda.is_available():
        torch.cuda.empty_cache()


def slice_bits(seed, n_rows):
    """Seeded bf16 bits of one (sequence, head) slice, [n_rows, 1, D]."""
    return inputs.normal_bf16(seed, n_rows * D).reshape(n_rows, 1, D)


def to_dev(dev, bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def big_tensors(dev, count, seed, shape=(B, N, H, D)):
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    return [torch.randn(shape, generator=g, dtype=torch.bfloat16, device=dev) for _ in range(count)]


def plant(dev, tensors, base_seed):
    """Overwrites each compared slice of each tensor with seeded input-module
    values; returns {pair: [host bits per tensor]}."""
    host = {}
    for s, h in PAIRS:
        vals = []
        for i, t in enumerate(tensors):
            bits = slice_bits(base_seed + 1000 * s + 10 * h + i, N)
            t[s, :, h, :].copy_(to_dev(dev, bits).reshape(N, D))
            vals.append(bits)
        host[(s, h)] = vals
    return host


def test_shapes_cross_4gb():
    assert B * N * H * D * 2 > 2 ** 32
    s, h = PAIRS[0]
    assert ((s * N + N - 1) * H + h + 1) * D * 2 == B * N * H * D * 2


def test_forward_past_4gb(dev):
    import torch
    import io_aware_exact_06_gb300 as fa
    q, k, v = big_tensors(dev, 3, 0xB16F)
    host = plant(dev, (q, k, v), 0xB16F0)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    scale = D ** -0.5
    fa.attn_fwd(q, k, v, o, lse, B, H, N, D, scale, True, None, None)
    assert fa.attn_last_device_error() == 0
    cu = np.array([0, N], dtype=np.int32)
    rows = np.stack([np.zeros(N), np.zeros(N), np.arange(N)], 1).astype(np.int64)
    for (s, h), (qb, kb, vb) in host.items():
        ref_o, ref_l, _ = oracle.attn_rows(qb, kb, vb, cu, rows, scale, True)
        got_o = o[s, :, h, :].float().cpu().numpy().astype(np.float64)
        got_l = lse[s, h, :].cpu().numpy().astype(np.float64)
        assert np.isfinite(got_o).all() and np.isfinite(got_l).all(), (s, h)
        st = parity.error_stats(got_o, got_l, ref_o, ref_l)
        assert st["o_max_abs"] <= parity.O_MAX_ABS, ((s, h), st)
        assert st["o_rel_l2"] <= parity.O_REL_L2, ((s, h), st)
        assert st["lse_max_abs"] <= parity.LSE_MAX_ABS, ((s, h), st)


# the backward parity tests' tolerances (derived in tests/test_bwd_gpu.py)
BWD_REL_L2, BWD_MAX_ABS_REL, BWD_ABS_FLOOR = 1e-2, 2.5e-2, 1e-3


def test_backward_past_4gb(dev):
    import torch
    import io_aware_exact_06_gb300 as fa
    q, k, v, do = big_tensors(dev, 4, 0xB16B)
    host = plant(dev, (q, k, v, do), 0xB16B0)
    scale = D ** -0.5
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fa.attn_fwd(q, k, v, o, lse, B, H, N, D, scale, True, None, None)
    grads = [torch.full_like(q, float("nan")) for _ in range(3)]
    fa.attn_bwd(q, k, v, o, do, lse, *grads, B, H, N, D, scale, True, None, None)
    assert fa.attn_last_device_error() == 0
    del o, lse
    cu = np.array([0, N], dtype=np.int32)
    for (s, h), (qb, kb, vb, dob) in host.items():
        ref = oracle.attn_bwd(qb, kb, vb, dob, cu, [(0, 0)], scale, True)
        for t, name in enumerate(("dq", "dk", "dv")):
            r = ref[t][0]
            g = grads[t][s, :, h, :].float().cpu().numpy().astype(np.float64)
            assert np.isfinite(g).all(), ((s, h), name)
            diff = g - r
            rel = np.linalg.norm(diff) / np.linalg.norm(r)
            assert rel <= BWD_REL_L2, ((s, h), name, rel)
            assert np.abs(diff).max() <= BWD_MAX_ABS_REL * np.abs(r).max() + BWD_ABS_FLOOR, ((s, h), name)


def test_fp8_forward_past_4gb(dev):
    import torch
    import io_aware_exact_06_gb300 as fa
    q, k, v = big_tensors(dev, 3, 0xB168)
    host = plant(dev, (q, k, v), 0xB1680)
    scale = D ** -0.5
    sg = np.where(inputs.splitmix64(0xB1681, 0, D) & np.uint64(1), -1, 1).astype(np.int8)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    fa.attn_fwd_fp8(q, k, v, o, lse, B, H, N, D, scale, True, sg)
    assert fa.attn_last_device_error() == 0
    cu = np.array([0, N], dtype=np.int64)
    rows = np.stack([np.zeros(N), np.zeros(N), np.arange(N)], 1).astype(np.int64)

    def deq(x, block_rows, rotate, signs):
        codes, scales = oracle.fp8_quantize(x, 1, N, block_rows, rotate, signs)
        vals = oracle.e4m3_decode(codes.ravel()).reshape(codes.shape)
        blk = np.zeros(N, dtype=np.int64) if block_rows == 0 else np.minimum(
            np.arange(N) // block_rows, scales.shape[2] - 1)
        return vals * scales[:, :, blk].transpose(0, 2, 1).reshape(N, 1, 1).astype(np.float64)

    for (s, h), (qb, kb, vb) in host.items():
        ref_o, ref_l = oracle.attn_rows_f64(deq(qb, 128, True, sg), deq(kb, 128, True, sg),
                                            deq(vb, 0, False, None), cu, rows, scale / D, True)
        got_o = o[s, :, h, :].float().cpu().numpy().astype(np.float64)
        got_l = lse[s, h, :].cpu().numpy().astype(np.float64)
        assert np.isfinite(got_o).all() and np.isfinite(got_l).all(), (s, h)
        # the FP8 tests' bounds against the dequantised reference
        rel = np.linalg.norm(got_o - ref_o) / np.linalg.norm(ref_o)
        assert rel <= 0.08, ((s, h), rel)
        assert np.abs(got_l - ref_l).max() <= 2e-3, (s, h)


def test_decode_key_cache_past_4gb(dev):
    """Packed key cache of 32 sequences x 2^20 keys x 8 heads x d 128 (8.6 GB
    per tensor), one query per sequence."""
    import torch
    import io_aware_exact_06_gb300 as fa
    Bd, L, Hd = 32, 1 << 20, 8
    k, v = big_tensors(dev, 2, 0xB16D, shape=(Bd * L, Hd, D))
    assert k.numel() * 2 > 2 ** 32
    q = big_tensors(dev, 1, 0xB16E, shape=(Bd, Hd, D))[0]
    pairs = [(Bd - 1, Hd - 1), (Bd // 2, 0)]
    host = {}
    for b, h in pairs:
        kb = slice_bits(0xB16D0 + 10 * b + h, L)
        vb = slice_bits(0xB16D5 + 10 * b + h, L)
        qb = slice_bits(0xB16DA + 10 * b + h, 1)
        k[b * L:(b + 1) * L, h, :].copy_(to_dev(dev, kb).reshape(L, D))
        v[b * L:(b + 1) * L, h, :].copy_(to_dev(dev, vb).reshape(L, D))
        q[b, h, :].copy_(to_dev(dev, qb).reshape(D))
        host[(b, h)] = (qb, kb, vb)
    cu = torch.arange(Bd + 1, dtype=torch.int32, device=dev) * L
    o = torch.full((Bd, Hd, D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((Bd, Hd), float("nan"), dtype=torch.float32, device=dev)
    scale = D ** -0.5
    fa.attn_fwd_decode(q, k, v, o, lse, Bd, Hd, D, scale, cu, L, 0)
    assert fa.attn_last_device_error() == 0
    cu1 = np.array([0, L], dtype=np.int64)
    for (b, h), (qb, kb, vb) in host.items():
        # the decode query is the last row of a causal problem whose other rows are zero
        qpack = np.zeros_like(kb)
        qpack[L - 1] = qb[0]
        ref_o, ref_l, _ = oracle.attn_rows(qpack, kb, vb, cu1, np.array([[0, 0, L - 1]]), scale, True)
        got_o = o[b, h].float().cpu().numpy().astype(np.float64)[None]
        got_l = lse[b, h].cpu().numpy().astype(np.float64).reshape(1)
        st = parity.error_stats(got_o, got_l, ref_o, ref_l)
        assert st["o_max_abs"] <= parity.O_MAX_ABS, ((b, h), st)
        assert st["o_rel_l2"] <= parity.O_REL_L2, ((b, h), st)
        assert st["lse_max_abs"] <= parity.LSE_MAX_ABS, ((b, h), st)
