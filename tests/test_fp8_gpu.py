"""FP8 forward (attn_fwd_fp8) against the oracle.

The quantisation step decides integers (e4m3 codes) from floating point, so
the CUDA codes and scales must equal the oracle's bit for bit (both take the
steps in fp32 in the same order).  The attention is compared with two fp64
references: the exact attention of the dequantised Q, K, V (what is left is
the quantisation of P and the fp32 / bf16 arithmetic), and the exact attention
of the original bf16 inputs (the whole FP8 error).

Tolerances, from the e4m3 format (3 mantissa bits: a rounded value is within
2^-4 of the exact one, relative, uniformly spread, rms 2^-4 / sqrt(3) ~ 0.036):
  - against the dequantised reference, only P carries that error; O is a
    P-weighted sum of V rows, so its relative L2 error is about 0.036 (the
    errors of different keys have independent signs): bound 0.08, twice that;
    the LSE comes from the unquantised fp32 row sum: bound 2e-3;
  - against the exact attention, V adds its own 0.036 to P's, in quadrature:
    O's relative L2 error is about 0.036 * sqrt(2) ~ 0.051 (measured 0.044 to
    0.055 over every case here): bound 0.11, about twice the worst measured.
    Q and K add theirs to each logit scale * sum_c q_c k_c: a standard
    deviation of about 0.036 * sqrt(2) ~ 0.05 for unit-variance inputs (the
    d products' errors add in quadrature and the scale 1/sqrt(d) divides
    them out); a row with one visible key has that whole error in its LSE,
    and the largest over the compared rows reached 0.086: bound 0.18, about
    twice that (3.5 sigma).
"""
import json
import os

import numpy as np
import pytest

import oracle
from io_aware_exact_06_gb300 import inputs

pytestmark = pytest.mark.gpu

REL_DEQ, LSE_DEQ = 0.08, 2e-3
REL_EXACT, LSE_EXACT = 0.11, 0.18


@pytest.fixture(scope="module")
def dev():
    import torch
    import __graft_entry__
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    __graft_entry__.build()
    return torch.device("cuda:0")


def signs_of(seed, d=128):
    return np.where(inputs.splitmix64(seed, 0, d) & np.uint64(1), -1, 1).astype(np.int8)


def with_outliers(bits, seed, factor=20.0, nch=3):
    """bf16 bits with a few channels scaled up (the case incoherent processing is for)."""
    x = inputs.bf16_bits_to_f64(bits).copy()
    ch = (inputs.splitmix64(seed, 0, nch) % np.uint64(x.shape[-1])).astype(np.int64)
    x[..., ch] *= factor
    return inputs.f64_to_bf16_bits(x)


def to_dev(dev, bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 300, 1024])
@pytest.mark.parametrize("rotate", [False, True])
def test_quantize_qk_bit_exact(dev, N, rotate, d):
    import torch
    import io_aware_exact_06_gb300 as fa
    B, H = 2, 3
    x = with_outliers(inputs.normal_bf16(3100 + N + d, B * N * H * d).reshape(B * N, H, d), 3101)
    sg = signs_of(3102, d) if rotate else None
    T = -(-N // 128)
    codes = torch.zeros((B * N, H, d), dtype=torch.uint8, device=dev)
    scales = torch.zeros((B, H, T), dtype=torch.float32, device=dev)
    fa.attn_fp8_quantize_qk(to_dev(dev, x), codes, scales, B, H, N, d, sg)
    assert fa.attn_last_device_error() == 0
    ref_codes, ref_scales = oracle.fp8_quantize(x, B, N, 128, rotate, sg)
    assert np.array_equal(scales.cpu().numpy(), ref_scales)
    assert np.array_equal(codes.cpu().numpy(), ref_codes)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 300, 1024])
def test_quantize_v_bit_exact(dev, N, d):
    import torch
    import io_aware_exact_06_gb300 as fa
    B, H = 2, 3
    v = inputs.normal_bf16(3200 + N + d, B * N * H * d, 1.5).reshape(B * N, H, d)
    Np = 128 * (-(-N // 128))
    codes_t = torch.full((B, H, d, Np), 0x55, dtype=torch.uint8, device=dev)
    scale = torch.zeros((B, H), dtype=torch.float32, device=dev)
    fa.attn_fp8_quantize_v(to_dev(dev, v), codes_t, scale, B, H, N, d)
    assert fa.attn_last_device_error() == 0
    ref_codes, ref_scale = oracle.fp8_quantize(v, B, N, 0, False)
    got = codes_t.cpu().numpy()
    assert np.array_equal(scale.cpu().numpy(), ref_scale[:, :, 0])
    back = got[:, :, :, :N].transpose(0, 3, 1, 2).reshape(B * N, H, d)
    assert np.array_equal(back, ref_codes)
    assert not got[:, :, :, N:].any(), "padding keys are zero"


@pytest.mark.parametrize("d", [64, 128])
def test_quantize_v_many_blocks_bit_exact(dev, d):
    """More than 256 blocks of 128 keys per sequence: the V quantiser's
    reduction of the block maxima loops over them; one outlier in the last
    block sets the scale."""
    import torch
    import io_aware_exact_06_gb300 as fa
    B, H, N = 1, 2, 33000
    v = inputs.normal_bf16(3250 + d, B * N * H * d).reshape(B * N, H, d)
    v[N - 5, 1, d - 1] = inputs.f64_to_bf16_bits(np.array([40.0]))[0]
    Np = 128 * (-(-N // 128))
    codes_t = torch.full((B, H, d, Np), 0x55, dtype=torch.uint8, device=dev)
    scale = torch.zeros((B, H), dtype=torch.float32, device=dev)
    fa.attn_fp8_quantize_v(to_dev(dev, v), codes_t, scale, B, H, N, d)
    assert fa.attn_last_device_error() == 0
    ref_codes, ref_scale = oracle.fp8_quantize(v, B, N, 0, False)
    assert ref_scale[0, 1, 0] == np.float32(40.0 / 448.0)
    got = codes_t.cpu().numpy()
    assert np.array_equal(scale.cpu().numpy(), ref_scale[:, :, 0])
    back = got[:, :, :, :N].transpose(0, 3, 1, 2).reshape(B * N, H, d)
    assert np.array_equal(back, ref_codes)
    assert not got[:, :, :, N:].any(), "padding keys are zero"


def dequantised(x, B, N, block_rows, rotate, sg):
    """fp64 values of the oracle's codes times their block scales."""
    codes, scales = oracle.fp8_quantize(x, B, N, block_rows, rotate, sg)
    H = x.shape[1]
    vals = oracle.e4m3_decode(codes.ravel()).reshape(codes.shape)
    rows = np.arange(N)
    blk = np.zeros(N, dtype=np.int64) if block_rows == 0 else np.minimum(rows // block_rows, scales.shape[2] - 1)
    s = scales[:, :, blk].transpose(0, 2, 1).reshape(B * N, H, 1).astype(np.float64)
    return vals * s


def run_fp8(dev, q, k, v, B, N, H, causal, sg, scale):
    import torch
    import io_aware_exact_06_gb300 as fa
    d = q.shape[-1]
    o = torch.empty((B * N, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fa.attn_fwd_fp8(to_dev(dev, q), to_dev(dev, k), to_dev(dev, v), o, lse, B, H, N, d, scale,
                    causal, sg)
    assert fa.attn_last_device_error() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def errors(got_o, got_lse, ref_o, ref_lse):
    rel = np.linalg.norm(got_o - ref_o) / np.linalg.norm(ref_o)
    return float(rel), float(np.abs(got_lse - ref_lse).max())


def check_case(dev, B, N, H, causal, rotate, seed, outliers, scale=None, d=128):
    if scale is None:
        scale = d ** -0.5
    q = inputs.normal_bf16(seed, B * N * H * d).reshape(B * N, H, d)
    k = inputs.normal_bf16(seed + 1, B * N * H * d).reshape(B * N, H, d)
    v = inputs.normal_bf16(seed + 2, B * N * H * d).reshape(B * N, H, d)
    if outliers:
        q, k = with_outliers(q, seed + 3), with_outliers(k, seed + 4)
    sg = signs_of(seed + 5, d) if rotate else None
    got_o, got_lse = run_fp8(dev, q, k, v, B, N, H, causal, sg, scale)
    cu = np.arange(B + 1) * N
    rows = inputs.sample_rows(cu, H, 512, seed=seed + 6)
    tok = cu[rows[:, 0]] + rows[:, 2]
    go, gl = got_o[tok, rows[:, 1]], got_lse[rows[:, 0], rows[:, 1], rows[:, 2]]
    qd = dequantised(q, B, N, 128, rotate, sg)
    kd = dequantised(k, B, N, 128, rotate, sg)
    vd = dequantised(v, B, N, 0, False, None)
    ref_o, ref_l = oracle.attn_rows_f64(qd, kd, vd, cu, rows, scale / (d if rotate else 1), causal)
    deq = errors(go, gl, ref_o, ref_l)
    ex_o, ex_l, _ = oracle.attn_rows(q, k, v, cu, rows, scale, causal)
    exact = errors(go, gl, ex_o, ex_l)
    log = os.environ.get("PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"test": "fp8", "B": B, "N": N, "H": H, "d": d, "causal": causal,
                                "rotate": rotate, "outliers": outliers, "vs_dequantised": deq,
                                "vs_exact": exact}) + "\n")
    return deq, exact


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("rotate", [False, True])
def test_fp8_attention(dev, causal, rotate, d):
    for (B, N, H) in [(1, 256, 2), (2, 1000, 3)]:
        (rel_d, lse_d), (rel_e, lse_e) = check_case(dev, B, N, H, causal, rotate, 3300 + N + d,
                                                    False, d=d)
        assert rel_d <= REL_DEQ and lse_d <= LSE_DEQ, (N, causal, rotate, rel_d, lse_d)
        assert rel_e <= REL_EXACT and lse_e <= LSE_EXACT, (N, causal, rotate, rel_e, lse_e)


def test_fp8_short_sequence(dev):
    (rel_d, lse_d), (rel_e, lse_e) = check_case(dev, 3, 77, 2, True, True, 3400, False)
    assert rel_d <= REL_DEQ and lse_d <= LSE_DEQ
    assert rel_e <= REL_EXACT and lse_e <= LSE_EXACT


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_zero_scale(dev, causal):
    # every visible key weighs 1 (256 P = 256 is exact in e4m3); masked keys 0
    (rel_d, lse_d), (rel_e, lse_e) = check_case(dev, 2, 300, 2, causal, True, 3450, False, scale=0.0)
    assert rel_d <= REL_DEQ and lse_d <= LSE_DEQ
    assert rel_e <= REL_EXACT and lse_e <= LSE_EXACT


def test_incoherent_processing_helps_with_outliers(dev):
    # channels of Q and K 20x larger than the rest: block scales are set by
    # them, the other channels lose precision; the rotation spreads them
    (_, _), (rel_plain, _) = check_case(dev, 1, 1024, 4, False, False, 3500, True)
    (_, _), (rel_rot, _) = check_case(dev, 1, 1024, 4, False, True, 3500, True)
    assert rel_rot < rel_plain, (rel_rot, rel_plain)


def sparse_outliers(bits, seed, prob=1e-3, factor=10.0):
    """bf16 bits with each entry, independently with probability prob, made
    factor times larger (rare large activations)."""
    x = inputs.bf16_bits_to_f64(bits).copy()
    u = (inputs.splitmix64(seed, 0, x.size) >> np.uint64(11)).astype(np.float64) / 2.0 ** 53
    x.reshape(-1)[u < prob] *= factor
    return inputs.f64_to_bf16_bits(x)


def per_tensor_fp8(dev, q, k, v, B, N, H, d, scale):
    """FP8 attention with per-tensor quantisation: one e4m3 scale per tensor and
    head for Q and K (oracle codes, no rotation), V per head, through the same
    attention kernel as attn_fwd_fp8 (attn_fwd_fp8_codes)."""
    import torch
    import io_aware_exact_06_gb300 as fa
    T = -(-N // 128)
    Np = 128 * T
    q8, sq = oracle.fp8_quantize_tensor(q)
    k8, sk = oracle.fp8_quantize_tensor(k)
    v8, sv = oracle.fp8_quantize(v, B, N, 0, False)
    vt = np.zeros((B, H, d, Np), dtype=np.uint8)
    vt[:, :, :, :N] = v8.reshape(B, N, H, d).transpose(0, 2, 3, 1)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    o = torch.empty((B * N, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fa.attn_fwd_fp8_codes(t(q8), t(np.broadcast_to(sq.reshape(1, H, 1), (B, H, T))), t(k8),
                          t(np.broadcast_to(sk.reshape(1, H, 1), (B, H, T))), t(vt), t(sv[:, :, 0]),
                          o, lse, B, H, N, d, scale, False, False)
    assert fa.attn_last_device_error() == 0
    return o.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("case", ["sparse_outliers", "plain"])
def test_block_and_rotation_against_per_tensor_fp8(dev, case):
    """The pages' claim for the FP8 path: block quantisation with incoherent
    processing has 2.6x lower error than FP8 attention with per-tensor
    quantisation ("flash-attention-evolution" (letsgetai), FlashAttention-3
    section, results).  The pages give no workload; this reads "outliers" as
    rare large entries: each entry of Q and K, with probability 1/1000, ten
    times larger, V unit normal (B1 N2048 H4 d128, non-causal).  Both
    quantisations run through the same attention kernel, and both errors are
    the relative L2 of O against the exact attention of the bf16 inputs.
    Measured ratios (per-tensor over block + rotation) 2.21 and 1.72 on two
    seeds; asserted > 1.5.  Without outliers the e4m3 rounding is relative
    (a floating-point format) and the rotation changes nothing: ratio 1.00,
    asserted within 5 %.  (With whole channels of Q and K 20x larger the
    rotation mixes them into every channel and is worse: ratio 0.61.)"""
    B, N, H, d, seed = 1, 2048, 4, 128, 3700
    scale = d ** -0.5
    q = inputs.normal_bf16(seed, B * N * H * d).reshape(B * N, H, d)
    k = inputs.normal_bf16(seed + 1, B * N * H * d).reshape(B * N, H, d)
    v = inputs.normal_bf16(seed + 2, B * N * H * d).reshape(B * N, H, d)
    if case == "sparse_outliers":
        q, k = sparse_outliers(q, seed + 10), sparse_outliers(k, seed + 11)
    cu = np.arange(B + 1) * N
    rows = inputs.sample_rows(cu, H, 1024, seed=seed + 6)
    tok = cu[rows[:, 0]] + rows[:, 2]
    ex_o, _, _ = oracle.attn_rows(q, k, v, cu, rows, scale, False)
    rel = lambda got: float(np.linalg.norm(got[tok, rows[:, 1]] - ex_o) / np.linalg.norm(ex_o))
    e_block = rel(run_fp8(dev, q, k, v, B, N, H, False, signs_of(seed + 5), scale)[0])
    e_tensor = rel(per_tensor_fp8(dev, q, k, v, B, N, H, d, scale))
    ratio = e_tensor / e_block
    log = os.environ.get("PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"test": "fp8_vs_per_tensor", "case": case,
                                "rel_l2_block_rotated": e_block, "rel_l2_per_tensor": e_tensor,
                                "ratio": ratio}) + "\n")
    if case == "sparse_outliers":
        assert ratio > 1.5, (e_block, e_tensor, ratio)
    else:
        assert 0.95 < ratio < 1.05, (e_block, e_tensor, ratio)


# ------------------------------------------------------------ packed batches --
# Packed variable-length batches: every per-sequence quantity is the dense one
# of that sequence alone (the oracle quantises each sequence on its own).

PACKED_LENS = [300, 0, 1, 128, 77, 513, 256]


def packed_inputs(seed, lens, H, scale_v=1.0, outliers=False, d=128):
    """Packed unit-variance Q, K, V (Q with a few 20x channels when outliers)."""
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    total = int(cu[-1])
    q = inputs.normal_bf16(seed, total * H * d).reshape(total, H, d)
    if outliers:
        q = with_outliers(q, seed + 3)
    k = inputs.normal_bf16(seed + 1, total * H * d).reshape(total, H, d)
    v = inputs.normal_bf16(seed + 2, total * H * d, scale_v).reshape(total, H, d)
    return cu, q, k, v


def cu_dev(dev, cu):
    import torch
    return torch.tensor(np.asarray(cu), dtype=torch.int32, device=dev)


@pytest.mark.parametrize("rotate", [False, True])
def test_quantize_qk_packed_bit_exact(dev, rotate):
    import torch
    import io_aware_exact_06_gb300 as fa
    H, N = 3, max(PACKED_LENS)
    cu, x, _, _ = packed_inputs(3600, PACKED_LENS, H, outliers=True)
    sg = signs_of(3601) if rotate else None
    B, T = len(PACKED_LENS), -(-N // 128)
    codes = torch.zeros((int(cu[-1]), H, 128), dtype=torch.uint8, device=dev)
    scales = torch.full((B, H, T), -1.0, dtype=torch.float32, device=dev)
    fa.attn_fp8_quantize_qk(to_dev(dev, x), codes, scales, B, H, N, 128, sg, cu_dev(dev, cu))
    assert fa.attn_last_device_error() == 0
    got_c, got_s = codes.cpu().numpy(), scales.cpu().numpy()
    for b, L in enumerate(PACKED_LENS):
        nb = -(-L // 128)
        assert (got_s[b, :, nb:] == -1.0).all(), "blocks past the sequence are not written"
        if L == 0:
            continue
        ref_c, ref_s = oracle.fp8_quantize(x[cu[b]:cu[b + 1]], 1, L, 128, rotate, sg)
        assert np.array_equal(got_s[b, :, :nb], ref_s[0]), b
        assert np.array_equal(got_c[cu[b]:cu[b + 1]], ref_c), b


@pytest.mark.parametrize("d", [64, 128])
def test_quantize_v_packed_bit_exact(dev, d):
    import torch
    import io_aware_exact_06_gb300 as fa
    H, N = 3, max(PACKED_LENS)
    cu, _, _, v = packed_inputs(3700 + d, PACKED_LENS, H, 1.5, d=d)
    B, Np = len(PACKED_LENS), 128 * -(-N // 128)
    codes_t = torch.full((B, H, d, Np), 0x55, dtype=torch.uint8, device=dev)
    scale = torch.full((B, H), -1.0, dtype=torch.float32, device=dev)
    fa.attn_fp8_quantize_v(to_dev(dev, v), codes_t, scale, B, H, N, d, cu_dev(dev, cu))
    assert fa.attn_last_device_error() == 0
    got, got_s = codes_t.cpu().numpy(), scale.cpu().numpy()
    for b, L in enumerate(PACKED_LENS):
        Lp = 128 * -(-L // 128)
        assert (got[b, :, :, Lp:] == 0x55).all(), "key tiles past the sequence are not written"
        if L == 0:
            assert (got_s[b] == -1.0).all()
            continue
        ref_c, ref_s = oracle.fp8_quantize(v[cu[b]:cu[b + 1]], 1, L, 0, False)
        assert np.array_equal(got_s[b], ref_s[0, :, 0]), b
        assert np.array_equal(got[b, :, :, :L].transpose(2, 0, 1), ref_c), b
        assert not got[b, :, :, L:Lp].any(), "padding keys of the last tile are zero"


def dequantised_packed(x, cu, block_rows, rotate, sg):
    out = np.zeros(x.shape, dtype=np.float64)
    for b in range(len(cu) - 1):
        L = int(cu[b + 1] - cu[b])
        if L:
            out[cu[b]:cu[b + 1]] = dequantised(x[cu[b]:cu[b + 1]], 1, L, block_rows, rotate, sg)
    return out


def run_fp8_packed(dev, q, k, v, cu, N, H, causal, sg, scale):
    import torch
    import io_aware_exact_06_gb300 as fa
    total, d = int(cu[-1]), q.shape[-1]
    o = torch.full((total, H, d), 7.0, dtype=torch.bfloat16, device=dev)
    lse = torch.full((H, total), 7.0, dtype=torch.float32, device=dev)
    fa.attn_fwd_fp8(to_dev(dev, q), to_dev(dev, k), to_dev(dev, v), o, lse, len(cu) - 1, H, N, d,
                    scale, causal, sg, cu_dev(dev, cu))
    assert fa.attn_last_device_error() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("rotate", [False, True])
def test_fp8_attention_packed(dev, causal, rotate, d):
    H, N = 2, max(PACKED_LENS)
    cu, q, k, v = packed_inputs(3800 + d, PACKED_LENS, H, d=d)
    sg = signs_of(3805, d) if rotate else None
    scale = d ** -0.5
    got_o, got_lse = run_fp8_packed(dev, q, k, v, cu, N, H, causal, sg, scale)
    rows = inputs.sample_rows(cu, H, 100000, seed=3806)  # every row
    tok = cu[rows[:, 0]] + rows[:, 2]
    go, gl = got_o[tok, rows[:, 1]], got_lse[rows[:, 1], tok]
    qd = dequantised_packed(q, cu, 128, rotate, sg)
    kd = dequantised_packed(k, cu, 128, rotate, sg)
    vd = dequantised_packed(v, cu, 0, False, None)
    ref_o, ref_l = oracle.attn_rows_f64(qd, kd, vd, cu, rows, scale / (d if rotate else 1), causal)
    rel_d, lse_d = errors(go, gl, ref_o, ref_l)
    ex_o, ex_l, _ = oracle.attn_rows(q, k, v, cu, rows, scale, causal)
    rel_e, lse_e = errors(go, gl, ex_o, ex_l)
    log = os.environ.get("PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"test": "fp8_packed", "lens": PACKED_LENS, "H": H, "d": d, "causal": causal,
                                "rotate": rotate, "vs_dequantised": [rel_d, lse_d],
                                "vs_exact": [rel_e, lse_e]}) + "\n")
    assert rel_d <= REL_DEQ and lse_d <= LSE_DEQ, (rel_d, lse_d)
    assert rel_e <= REL_EXACT and lse_e <= LSE_EXACT, (rel_e, lse_e)


def test_fp8_packed_equal_lengths_match_dense(dev):
    """Equal lengths: the packed call computes every unit as the dense one."""
    H, N, B = 2, 640, 3
    cu, q, k, v = packed_inputs(3900, [N] * B, H)
    sg = signs_of(3901)
    scale = 128 ** -0.5
    o_p, lse_p = run_fp8_packed(dev, q, k, v, cu, N, H, True, sg, scale)
    o_d, lse_d = run_fp8(dev, q, k, v, B, N, H, True, sg, scale)
    assert np.array_equal(o_p, o_d)
    assert np.array_equal(lse_p, lse_d.transpose(1, 0, 2).reshape(H, B * N))


@pytest.mark.parametrize("bad", ["decreasing", "too_long", "nonzero_start"])
def test_fp8_invalid_cu_seqlens_reported(dev, bad):
    import torch
    import io_aware_exact_06_gb300 as fa
    H = 2
    cu, q, k, v = packed_inputs(4000, [100, 100, 100], H)
    cu_bad = {"decreasing": [0, 150, 120, 300], "too_long": [0, 100, 300, 300],
              "nonzero_start": [8, 100, 200, 300]}[bad]
    o = torch.full((300, H, 128), 7.0, dtype=torch.bfloat16, device=dev)
    lse = torch.full((H, 300), 7.0, dtype=torch.float32, device=dev)
    fa.attn_fwd_fp8(to_dev(dev, q), to_dev(dev, k), to_dev(dev, v), o, lse, 3, H, 128, 128,
                    128 ** -0.5, True, None, cu_dev(dev, cu_bad))
    assert fa.attn_last_device_error() == -8
    assert (o.float() == 7.0).all() and (lse == 7.0).all(), "nothing is written"


# attn_fwd_fp8_codes: the attention step alone on the quantisers' outputs
# (d = 128) gives attn_fwd_fp8's O and LSE bit for bit: the quantisers are
# the same arithmetic (their codes are bit-exact against the oracle above)
# and the attention kernel is the same launch.
@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("rotate", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_codes_entry_matches_full_call(dev, packed, rotate, causal):
    import torch
    import io_aware_exact_06_gb300 as fa
    d, H = 128, 3
    lens = [300, 129, 1024, 1] if packed else [700, 700]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    B, N, total = len(lens), max(lens), int(cu[-1])
    seed = 3700 + 10 * packed + 2 * rotate + causal
    q = inputs.normal_bf16(seed, total * H * d).reshape(total, H, d)
    k = inputs.normal_bf16(seed + 1, total * H * d).reshape(total, H, d)
    v = inputs.normal_bf16(seed + 2, total * H * d).reshape(total, H, d)
    sg = signs_of(seed + 3, d) if rotate else None
    cu_d = torch.from_numpy(cu).to(dev) if packed else None
    qd, kd, vd = to_dev(dev, q), to_dev(dev, k), to_dev(dev, v)
    scale = d ** -0.5
    lse_shape = (H, total) if packed else (B, H, N)
    o1 = torch.empty((total, H, d), dtype=torch.bfloat16, device=dev)
    l1 = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    fa.attn_fwd_fp8(qd, kd, vd, o1, l1, B, H, N, d, scale, causal, sg, cu_seqlens=cu_d)
    T = -(-N // 128)
    tok_rows = total if packed else B * N
    q8 = torch.zeros((tok_rows, H, d), dtype=torch.uint8, device=dev)
    k8 = torch.zeros_like(q8)
    sq = torch.zeros((B, H, T), dtype=torch.float32, device=dev)
    sk = torch.zeros_like(sq)
    vt = torch.zeros((B, H, d, 128 * T), dtype=torch.uint8, device=dev)
    sv = torch.zeros((B, H), dtype=torch.float32, device=dev)
    fa.attn_fp8_quantize_qk(qd, q8, sq, B, H, N, d, sg, cu_seqlens=cu_d)
    fa.attn_fp8_quantize_qk(kd, k8, sk, B, H, N, d, sg, cu_seqlens=cu_d)
    fa.attn_fp8_quantize_v(vd, vt, sv, B, H, N, d, cu_seqlens=cu_d)
    o2 = torch.full((total, H, d), float("nan"), dtype=torch.bfloat16, device=dev)
    l2 = torch.full(lse_shape, float("nan"), dtype=torch.float32, device=dev)
    fa.attn_fwd_fp8_codes(q8, sq, k8, sk, vt, sv, o2, l2, B, H, N, d, scale, causal, rotate,
                          cu_seqlens=cu_d)
    assert fa.attn_last_device_error() == 0
    assert bool((o1.view(torch.int16) == o2.view(torch.int16)).all())
    assert bool((l1 == l2).all())


def test_fp8_packed_head_group_order_same_result(dev):
    """Packed FP8 calls with at least 64 units per SM (counted from the length
    bound N) take their units in head groups; the result may not depend on the
    order.  The same sequences with N = their longest length (one group) and
    with N = 8192 (16 x 20 x 32 = 10240 units on 152 SMs, one head per group)
    give bit-identical O and LSE, within the bounds against the dequantised
    reference on sampled rows."""
    H, d = 20, 128
    lens = inputs.uniform_ints(3950, 16, 1, 1500).tolist()
    cu, q, k, v = packed_inputs(3951, lens, H)
    sg = signs_of(3952)
    scale = d ** -0.5
    o1, l1 = run_fp8_packed(dev, q, k, v, cu, max(lens), H, True, sg, scale)
    o2, l2 = run_fp8_packed(dev, q, k, v, cu, 8192, H, True, sg, scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    rows = inputs.sample_rows(cu, H, 1024, seed=3953)
    tok = cu[rows[:, 0]] + rows[:, 2]
    go, gl = o2[tok, rows[:, 1]], l2[rows[:, 1], tok]
    qd = dequantised_packed(q, cu, 128, True, sg)
    kd = dequantised_packed(k, cu, 128, True, sg)
    vd = dequantised_packed(v, cu, 0, False, None)
    ref_o, ref_l = oracle.attn_rows_f64(qd, kd, vd, cu, rows, scale / d, True)
    rel_d, lse_d = errors(go, gl, ref_o, ref_l)
    assert rel_d <= REL_DEQ and lse_d <= LSE_DEQ, (rel_d, lse_d)


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_packed_outputs_stay_inside_their_rows(dev, d):
    """As for the bf16 forward: O a view at the start of a larger buffer whose
    tail holds a sentinel; the FP8 call's TMA stores and row-wise stores leave
    the tail untouched, and O matches the unguarded call bit for bit."""
    import torch
    import io_aware_exact_06_gb300 as fa
    lens = [129, 0, 256, 77, 384, 1, 200]
    H, N = 2, max(lens)
    cu, q, k, v = packed_inputs(3900 + d, lens, H, d=d)
    total = int(cu[-1])
    guard = 384
    sentinel = 0x7F81
    big = torch.full((total + guard, H, d), sentinel, dtype=torch.int16, device=dev)
    o = big[:total].view(torch.bfloat16)
    lse = torch.empty((H, total), dtype=torch.float32, device=dev)
    qd, kd, vd, cud = to_dev(dev, q), to_dev(dev, k), to_dev(dev, v), cu_dev(dev, cu)
    fa.attn_fwd_fp8(qd, kd, vd, o, lse, len(lens), H, N, d, d ** -0.5, True, None, cu_seqlens=cud)
    assert fa.attn_last_device_error() == 0
    assert bool((big[total:] == sentinel).all()), "rows past the packed tokens were written"
    o2 = torch.empty_like(o)
    lse2 = torch.empty_like(lse)
    fa.attn_fwd_fp8(qd, kd, vd, o2, lse2, len(lens), H, N, d, d ** -0.5, True, None, cu_seqlens=cud)
    assert fa.attn_last_device_error() == 0
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(lse, lse2)
