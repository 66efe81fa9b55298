"""CUDA path against the fp64 oracle, element by element, through the C ABI.

Tolerances: O max-abs <= 1.5e-2 and relative L2 <= 5e-3 (bf16 output, fp32
accumulation, bf16 P); LSE max-abs <= 2e-3.  Full-size workloads compare a
seeded sample of >= 4096 rows that always holds the first, last and
tile-edge rows of every sequence and head."""
import numpy as np
import pytest

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


_cache = {}


def workload(name):
    if name not in _cache:
        _cache[name] = inputs.config_workload(name)
    return _cache[name]


@pytest.mark.parametrize("kernel", ["one_cta", "rows"])
@pytest.mark.parametrize("name", ["tiny", "gpt2_causal"])
def test_small_configs_every_row(dev, name, kernel):
    wl = workload(name)
    o, lse, st = parity.run_cuda(wl, dev, **KERNELS[kernel])
    assert st == 0
    parity.compare(o, lse, wl, inputs.all_rows(wl.cu_seqlens, wl.H), f"{name} {kernel}")


# The forward's kernels: one CTA per unit with one softmax thread per query
# row (kernel=3, the default) or two (kernel=1), and at d = 128 without a
# window the pair of SMs (kernel=2); every one stays covered.
KERNELS = {"pair": {"kernel": 2}, "one_cta": {"kernel": 1}, "rows": {"kernel": 3}}


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("name", ["long_causal", "long_full", "stress", "varlen"])
def test_large_configs_sampled_rows(dev, name, kernel):
    wl = workload(name)
    o, lse, st = parity.run_cuda(wl, dev, **KERNELS[kernel])
    assert st == 0
    rows = inputs.sample_rows(wl.cu_seqlens, wl.H, 4096, seed=inputs.CONFIG_SEED_BASE + 7)
    assert len(rows) >= 4096
    parity.compare(o, lse, wl, rows, f"{name} {kernel}")


@pytest.mark.parametrize("causal", [False, True])
def test_pair_kernel_one_cluster_many_units(dev, causal):
    """One cluster (max_ctas = 2) walks every unit of a dense batch in turn:
    Q buffers, S buffers and ring phases carried across many units."""
    wl = inputs.make_workload("pair1", 4300 + causal, [700] * 3, 5, 128, causal)
    o, lse, st = parity.run_cuda(wl, dev, max_ctas=2, kernel=2)
    assert st == 0
    parity.compare(o, lse, wl, inputs.all_rows(wl.cu_seqlens, wl.H), "pair one cluster")


def test_pair_kernel_bounded_wait_expires(dev):
    """The test hook makes CTA 0 (the even CTA of cluster 0) skip one K copy,
    so the MMA thread's bounded wait on the pair's full barrier expires: both
    CTAs of the pair stop, the call reports ATTN_ERR_DEVICE_TIMEOUT and the
    next call is correct."""
    import io_aware_exact_06_gb300 as fa
    wl = inputs.make_workload("pairto", 4310, [512] * 2, 4, 128, True)
    _, _, st = parity.run_cuda(wl, dev, wait_timeout_ns=50_000_000, fault_inject=1, kernel=2)
    assert st == -7
    assert fa.attn_last_error_site() != 0
    o, lse, st = parity.run_cuda(wl, dev, kernel=2)
    assert st == 0
    parity.compare(o, lse, wl, inputs.all_rows(wl.cu_seqlens, wl.H), "pair after timeout")


@pytest.mark.parametrize("d,kernel", [(64, "one_cta"), (64, "rows"), (128, "pair"), (128, "one_cta"),
                                      (128, "rows")])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_packed_lengths(dev, d, causal, kernel):
    lens = [1, 127, 128, 129, 0, 255, 256, 257, 300, 2, 513]
    wl = inputs.make_workload("ragged", 4242 + d, lens, 3, d, causal, qk_std=1.5, varlen=True)
    o, lse, st = parity.run_cuda(wl, dev, packed=True, **KERNELS[kernel])
    assert st == 0
    parity.compare(o, lse, wl, inputs.all_rows(wl.cu_seqlens, wl.H), f"ragged {kernel}")


# scale 2 on unit-variance Q and K: logit standard deviation 2 sqrt(d) (16 at
# d = 64, 23 at d = 128), so row maxima move by far more than the lazy-rescale
# threshold from tile to tile, O is rescaled on most rows, and most
# probabilities underflow to 0 (P close to one-hot).  On such rows O is one or
# two rows of V, and its error is the bf16 rounding of O and of the leading
# probabilities, up to 2^-9 |v| each: V ~ N(0, 1/4) keeps that inside the O
# tolerance (with unit-variance V, whose largest entries near 5 make each
# term about 0.01, the largest of 0.8 million compared values reached
# 0.0153); the logit range is what this test stresses.
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("packed", [False, True])
def test_extreme_logit_range(dev, d, causal, packed):
    lens = [1000, 333, 777] if packed else [777, 777]
    wl = inputs.make_workload("extreme", 4500 + 4 * d + 2 * causal + packed, lens, 3, d, causal,
                              v_std=0.5, scale=2.0, varlen=packed)
    o, lse, st = parity.run_cuda(wl, dev, packed=packed)
    assert st == 0
    parity.compare(o, lse, wl, inputs.all_rows(wl.cu_seqlens, wl.H), f"extreme d={d}")


@pytest.mark.parametrize("N", [50, 200, 384, 640])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_lengths_not_multiple_of_tile(dev, N, causal):
    wl = inputs.make_workload("dense", 77 + N, [N] * 3, 2, 128, causal)
    o, lse, st = parity.run_cuda(wl, dev)
    assert st == 0
    parity.compare(o, lse, wl, inputs.all_rows(wl.cu_seqlens, wl.H), f"dense N={N}")


def test_causal_last_row_equals_full_row_at_full_size(dev):
    # row L-1 sees every key under both masks: on the long workloads (same
    # inputs, every sequence and head, full size) its causal and non-causal
    # O and LSE agree bit for bit (same tiles, same order, nothing masked)
    import torch
    wc, wf = workload("long_causal"), workload("long_full")
    assert wc.q is not None and np.array_equal(wc.q, wf.q) and np.array_equal(wc.v, wf.v)
    oc, lc, st = parity.run_cuda(wc, dev)
    assert st == 0
    of, lf, st = parity.run_cuda(wf, dev)
    assert st == 0
    N = int(wc.seqlens()[0])
    last = torch.tensor([b * N + N - 1 for b in range(wc.nseq)], device=oc.device)
    assert torch.equal(oc[last].view(torch.int16), of[last].view(torch.int16))
    assert torch.equal(lc[:, last], lf[:, last])


def _visible_means(wl, v, dev):
    """Mean of the visible V rows of every query row (fp64, [tokens, H, d])
    and the number of visible keys ([tokens]): the prefix 0..i of its
    sequence when causal, the whole sequence otherwise."""
    import torch
    cu = torch.from_numpy(wl.cu_seqlens.astype(np.int64)).to(dev)
    lens = cu[1:] - cu[:-1]
    seq = torch.repeat_interleave(torch.arange(wl.nseq, device=dev), lens)
    start = cu[:-1][seq]
    pos = torch.arange(wl.tokens, device=dev) - start
    cs = torch.cat([torch.zeros_like(v[:1]), torch.cumsum(v, dim=0)])
    if wl.causal:
        count = pos + 1
        total = cs[start + count] - cs[start]
    else:
        count = lens[seq]
        total = cs[start + count] - cs[start]
    return total / count.view(-1, 1, 1).double(), count


@pytest.mark.parametrize("name", ["long_causal", "long_full", "stress", "varlen"])
def test_zero_q_gives_mean_of_visible_v_at_full_size(dev, name):
    """Q = 0: every logit is 0, so O_i is the mean of the visible V rows and
    LSE_i = log(#visible) (closed forms of the definition, computed in fp64
    with prefix sums).  Checked on every row and head of the workload."""
    wl = workload(name)
    wl0 = inputs.Workload("zeroq", np.zeros_like(wl.q), wl.k, wl.v, wl.cu_seqlens, wl.H, wl.d,
                          wl.scale, wl.causal, wl.varlen, wl.max_seqlen)
    o, lse, st = parity.run_cuda(wl0, dev)
    assert st == 0
    v = parity.to_device(wl, dev)[2].double()
    ref, count = _visible_means(wl, v, dev)
    got = o.double()
    err = (got - ref).abs().max().item()
    rel = ((got - ref).norm() / ref.norm()).item()
    assert err <= parity.O_MAX_ABS and rel <= parity.O_REL_L2, (name, err, rel)
    lse_err = (lse.double() - count.double().log().view(1, -1)).abs().max().item()
    assert lse_err <= parity.LSE_MAX_ABS, (name, lse_err)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_is_uniform_average(dev, causal):
    """scale = 0: every visible key has weight 1, O_i is the mean of the
    visible V rows and LSE_i = log(#visible) (the masked logits must still get
    weight 0): dense with a ragged tail, packed, and a sliding window."""
    wl = inputs.make_workload("scale0", 4100 + causal, [300] * 2, 2, 128, causal, scale=0.0)
    o, lse, st = parity.run_cuda(wl, dev)
    assert st == 0
    parity.compare(o, lse, wl, inputs.all_rows(wl.cu_seqlens, wl.H), "scale 0 dense")
    wl = inputs.make_workload("scale0p", 4102 + causal, [300, 1, 77, 513], 2, 64, causal,
                              varlen=True, scale=0.0)
    o, lse, st = parity.run_cuda(wl, dev)
    assert st == 0
    parity.compare(o, lse, wl, inputs.all_rows(wl.cu_seqlens, wl.H), "scale 0 packed")
    wl = inputs.make_workload("scale0w", 4104 + causal, [400] * 2, 2, 128, causal, scale=0.0)
    o, lse, st = parity.run_cuda(wl, dev, window=(64, 32))
    assert st == 0
    parity.compare(o, lse, wl, inputs.all_rows(wl.cu_seqlens, wl.H), "scale 0 window",
                   window=(64, 32))


@pytest.mark.parametrize("name", ["long_causal", "long_full", "stress", "varlen"])
def test_constant_v_gives_constant_o(dev, name):
    """V = c on every row: O_i = c exactly in the definition (the weights of a
    row sum to 1).  The kernel's weights are bf16-rounded probabilities over
    their fp32 sum (reading 5): each rounding changes a probability by at
    most 2^-8 of itself, so the fp32 O lies within c * 2^-8 of c and rounds
    to c or a neighbouring bf16 value.  Bound: one bf16 ulp of c (2^-8 for
    c = 0.8125), on every row and head, with O = c exactly on most."""
    import torch
    wl = workload(name)
    c = 0.8125
    cb = inputs.f64_to_bf16_bits(np.array([c]))[0]
    wlc = inputs.Workload("constv", wl.q, wl.k, np.full_like(wl.v, cb), wl.cu_seqlens, wl.H, wl.d,
                          wl.scale, wl.causal, wl.varlen, wl.max_seqlen)
    o, lse, st = parity.run_cuda(wlc, dev)
    assert st == 0
    ulp = 2.0 ** -8  # bf16 spacing in [0.5, 1)
    dev_o = (o.float() - c).abs()
    assert dev_o.max().item() <= ulp, (name, dev_o.max().item())
    assert (dev_o == 0).float().mean().item() >= 0.5, name


def test_deterministic(dev):
    import torch
    wl = workload("varlen")
    o1, l1, _ = parity.run_cuda(wl, dev)
    o2, l2, _ = parity.run_cuda(wl, dev)
    assert torch.equal(o1, o2)
    assert torch.equal(l1, l2)


def test_non_default_stream(dev):
    import torch
    wl = workload("tiny")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse, st = parity.run_cuda(wl, dev, stream=s)
    assert st == 0
    parity.compare(o, lse, wl, inputs.all_rows(wl.cu_seqlens, wl.H), "stream")


def test_bounded_wait_expires_with_error_status(dev):
    """A host flag makes CTA 0 skip one copy, so its MMA warp's bounded wait
    expires: the call reports ATTN_ERR_DEVICE_TIMEOUT and the context stays
    usable for the next call."""
    import io_aware_exact_06_gb300 as fa
    wl = workload("tiny")
    _, _, st = parity.run_cuda(wl, dev, wait_timeout_ns=50_000_000, fault_inject=1)
    assert st == -7
    assert fa.attn_last_error_site() != 0
    o, lse, st = parity.run_cuda(wl, dev)
    assert st == 0
    parity.compare(o, lse, wl, inputs.all_rows(wl.cu_seqlens, wl.H), "after timeout")


@pytest.mark.parametrize("bad", ["decreasing", "too_long", "nonzero_start"])
def test_invalid_cu_seqlens_reported(dev, bad):
    import torch
    import io_aware_exact_06_gb300 as fa
    wl = inputs.make_workload("bad", 5, [100, 100, 100], 2, 64, True, varlen=True)
    q, k, v, cu = parity.to_device(wl, dev)
    cu_bad = {"decreasing": [0, 150, 120, 300], "too_long": [0, 100, 300, 300],
              "nonzero_start": [8, 100, 200, 300]}[bad]
    cu = torch.tensor(cu_bad, dtype=torch.int32, device=dev)
    o = torch.full_like(q, 7.0)
    lse = torch.full((2, 300), 7.0, device=dev)
    fa.attn_fwd(q, k, v, o, lse, 3, 2, 128, 64, wl.scale, True, cu, None)
    assert fa.attn_last_device_error() == -8
    assert (o.float() == 7.0).all() and (lse == 7.0).all(), "nothing is written"


# ---------------------------------------------------------------- windows --
# Sliding windows: key j visible to query i iff i - wl <= j <= i + wr (-1:
# unbounded), on top of the causal mask.

def test_window_long_causal_sampled(dev):
    """The long causal workload with a 1024-key window (keys i-1023 .. i)."""
    wl = workload("long_causal")
    o, lse, st = parity.run_cuda(wl, dev, window=(1023, -1))
    assert st == 0
    rows = inputs.sample_rows(wl.cu_seqlens, wl.H, 4096, seed=inputs.CONFIG_SEED_BASE + 8)
    parity.compare(o, lse, wl, rows, "window 1023 causal", window=(1023, -1))


WINDOWS = [(0, 0), (5, -1), (127, 3), (128, 128), (300, -1), (-1, 64), (0, -1), (1000, 1000)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_window_ragged_packed(dev, d, causal):
    lens = [1, 127, 128, 129, 0, 255, 256, 257, 300, 2, 513]
    wl = inputs.make_workload("ragged", 4343 + d, lens, 2, d, causal, qk_std=1.5, varlen=True)
    rows = inputs.all_rows(wl.cu_seqlens, wl.H)
    for win in WINDOWS:
        o, lse, st = parity.run_cuda(wl, dev, packed=True, window=win)
        assert st == 0
        parity.compare(o, lse, wl, rows, f"window {win} ragged", window=win)


def test_window_dense_odd_length(dev):
    wl = inputs.make_workload("dense_win", 99, [1000, 1000], 2, 128, False)
    for win in [(100, 37), (0, 200), (513, 0)]:
        o, lse, st = parity.run_cuda(wl, dev, window=win)
        assert st == 0
        parity.compare(o, lse, wl, inputs.all_rows(wl.cu_seqlens, wl.H), f"window {win} dense",
                       window=win)


def test_window_unbounded_equals_plain(dev):
    import torch
    wl = workload("gpt2_causal")
    o1, l1, _ = parity.run_cuda(wl, dev)
    o2, l2, _ = parity.run_cuda(wl, dev, window=(-1, -1))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_window_rejects_bad_values(dev):
    import io_aware_exact_06_gb300 as fa
    with pytest.raises(fa.AttnError):
        fa.attn_fwd_window(1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1, 1, 128, 64, 0.1, True,
                           -2, 0)


@pytest.mark.parametrize("d", [64, 128])
def test_grouped_causal_unit_order_every_row(dev, d):
    """A causal call with at least 64 units per SM takes the dense unit order
    with the (batch, head) pairs in groups (B16 H32 N8192: 16384 units of 256
    rows; 152 SMs take groups from 9728 units on).  With Q = 0 every logit is
    0, so O_i is the mean of V_0..V_i and LSE_i = log(i + 1) (closed forms,
    fp64 prefix sums): checked on every row and head, so a unit computed
    twice, missed, or given another (batch, head) fails.  O and LSE start as
    NaN."""
    import torch
    import io_aware_exact_06_gb300 as fa
    B, H, N = 16, 32, 8192
    g = torch.Generator(device=dev).manual_seed(0x6A0 + d)
    v = torch.randn((B, N, H, d), generator=g, device=dev).bfloat16()
    k = torch.randn((B, N, H, d), generator=g, device=dev).bfloat16()
    q = torch.zeros_like(v)
    o = torch.full_like(v, float("nan"))
    lse = torch.full((B, H, N), float("nan"), device=dev)
    fa.attn_fwd(q, k, v, o, lse, B, H, N, d, d ** -0.5, True, None, torch.cuda.current_stream())
    assert fa.attn_last_device_error(torch.cuda.current_stream()) == 0
    assert torch.isfinite(o).all().item() and torch.isfinite(lse).all().item()  # every row written
    count = torch.arange(1, N + 1, device=dev, dtype=torch.float64)
    worst = 0.0
    for b in range(B):   # one sequence at a time (fp64 prefix sums of 8192 x 32 x d)
        ref = torch.cumsum(v[b].double(), dim=0) / count.view(-1, 1, 1)
        worst = max(worst, (o[b].double() - ref).abs().max().item())
    assert worst <= parity.O_MAX_ABS, worst
    lse_err = (lse.double() - count.log().view(1, 1, -1)).abs().max().item()
    assert lse_err <= parity.LSE_MAX_ABS, lse_err


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_head_group_order_same_result(dev, d, causal):
    """Packed calls take their units in head groups (causal ones with at
    least 64 units per SM counted from the length bound N); the result may
    not depend on the order.  The same sequences with N = their longest
    length and with N = 8192 (16 sequences x 20 heads x 32 q-blocks = 10240
    units, one head per group on 152 SMs) give bit-identical O and LSE, and
    sampled rows match the oracle."""
    import io_aware_exact_06_gb300 as fa
    import torch
    lens = inputs.uniform_ints(4545 + d, 16, 1, 1500).tolist()
    wl = inputs.make_workload("packed_groups", 4546 + d, lens, 20, d, causal, varlen=True)
    q, k, v, cu = parity.to_device(wl, dev)
    outs = []
    for N in (int(max(lens)), 8192):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((wl.H, wl.tokens), float("nan"), dtype=torch.float32, device=dev)
        fa.attn_fwd(q, k, v, o, lse, wl.nseq, wl.H, N, d, wl.scale, causal, cu)
        assert fa.attn_last_device_error() == 0
        outs.append((o, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    rows = inputs.sample_rows(wl.cu_seqlens, wl.H, 2048, seed=4547 + d)
    parity.compare(outs[1][0], outs[1][1], wl, rows, "packed head groups")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_outputs_stay_inside_their_rows(dev, d, causal):
    """O goes out through whole-tile TMA stores where a query tile lies
    inside its sequence and row by row elsewhere: with O a view at the start
    of a larger buffer whose tail holds a sentinel, every row of the packed
    tokens matches the oracle and the tail is untouched (lengths whose last
    tile is pulled back, shorter than a tile, or exactly whole)."""
    import torch
    import io_aware_exact_06_gb300 as fa
    lens = [129, 0, 256, 77, 384, 1, 200]
    wl = inputs.make_workload("guard", 5151 + d, lens, 2, d, causal, varlen=True)
    q, k, v, cu = parity.to_device(wl, dev)
    guard = 384
    sentinel = 0x7F81  # a signalling-NaN bf16 bit pattern no kernel writes
    big = torch.full((wl.tokens + guard, wl.H, d), sentinel, dtype=torch.int16, device=dev)
    o = big[:wl.tokens].view(torch.bfloat16)
    lse = torch.empty((wl.H, wl.tokens), dtype=torch.float32, device=dev)
    N = max(lens)
    fa.attn_fwd(q, k, v, o, lse, wl.nseq, wl.H, N, d, wl.scale, causal, cu)
    assert fa.attn_last_device_error() == 0
    assert bool((big[wl.tokens:] == sentinel).all()), "rows past the packed tokens were written"
    parity.compare(o, lse, wl, inputs.all_rows(wl.cu_seqlens, wl.H), f"guard d={d}")
