"""attn_fwd_host (host buffers; head groups copied in, computed and copied
out on three streams) against attn_fwd on the same inputs, and against the
oracle.

Every row is computed by the same kernel with the same arithmetic whatever
the number of heads in a launch, so O and the LSE must equal attn_fwd's bit
for bit.  The cases give one group (H = 1), two groups, uneven groups (H = 7)
and more groups than the two workspace slots (H = 12: six groups of two
heads), dense and packed batches, pinned and pageable host memory, the
default and a created stream."""
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


def host_inputs(seed, B, N, H, d, pinned):
    import torch
    out = []
    for t in range(3):
        bits = inputs.normal_bf16(seed * 4 + 1 + t, B * N * H * d).reshape(B, N, H, d)
        x = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
        out.append(x.pin_memory() if pinned else x.clone())
    return out


def run_both(dev, B, N, H, d, causal, pinned, seed, stream=None):
    import torch
    import io_aware_exact_06_gb300 as fa
    q_h, k_h, v_h = host_inputs(seed, B, N, H, d, pinned)
    scale = d ** -0.5
    q, k, v = (x.to(dev) for x in (q_h, k_h, v_h))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fa.attn_fwd(q, k, v, o, lse, B, H, N, d, scale, causal)
    assert fa.attn_last_device_error() == 0
    o_h = torch.full((B, N, H, d), float("nan"), dtype=torch.bfloat16)
    lse_h = torch.full((B, H, N), float("nan"), dtype=torch.float32)
    if pinned:
        o_h, lse_h = o_h.pin_memory(), lse_h.pin_memory()
    fa.attn_fwd_host(q_h, k_h, v_h, o_h, lse_h, B, H, N, d, scale, causal, stream=stream)
    assert fa.attn_last_device_error(stream) == 0
    return o.cpu(), lse.cpu(), o_h, lse_h


CASES = [(1, 300, 1, 128, True), (2, 1000, 2, 64, False), (2, 777, 7, 128, True),
         (4, 4096, 12, 128, True), (3, 640, 16, 64, False)]


@pytest.mark.parametrize("B,N,H,d,causal", CASES)
@pytest.mark.parametrize("pinned", [True, False])
def test_bit_identical_to_attn_fwd(dev, B, N, H, d, causal, pinned):
    import torch
    o, lse, o_h, lse_h = run_both(dev, B, N, H, d, causal, pinned, seed=B * 100 + H)
    assert bool((o_h.view(torch.int16) == o.view(torch.int16)).all())
    assert bool((lse_h == lse).all())


@pytest.mark.parametrize("lens,H,d,causal", [([300, 0, 1000, 129, 640], 5, 128, True),
                                             ([64, 2048, 1], 12, 64, False)])
@pytest.mark.parametrize("pinned", [True, False])
def test_packed_bit_identical_to_attn_fwd(dev, lens, H, d, causal, pinned):
    import torch
    import io_aware_exact_06_gb300 as fa
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total, B, N = int(cu[-1]), len(lens), max(lens)
    q_h, k_h, v_h = host_inputs(len(lens) * 10 + H, 1, total, H, d, pinned)
    q_h, k_h, v_h = (x.reshape(total, H, d) for x in (q_h, k_h, v_h))
    scale = d ** -0.5
    q, k, v = (x.to(dev) for x in (q_h, k_h, v_h))
    o = torch.empty_like(q)
    lse = torch.empty((H, total), dtype=torch.float32, device=dev)
    fa.attn_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, torch.from_numpy(cu).to(dev))
    assert fa.attn_last_device_error() == 0
    o_h = torch.full((total, H, d), float("nan"), dtype=torch.bfloat16)
    lse_h = torch.full((H, total), float("nan"), dtype=torch.float32)
    cu_h = torch.from_numpy(cu)
    if pinned:
        o_h, lse_h, cu_h = o_h.pin_memory(), lse_h.pin_memory(), cu_h.pin_memory()
    fa.attn_fwd_host(q_h, k_h, v_h, o_h, lse_h, B, H, N, d, scale, causal, cu_h)
    assert fa.attn_last_device_error() == 0
    assert bool((o_h.view(torch.int16) == o.cpu().view(torch.int16)).all())
    assert bool((lse_h == lse.cpu()).all())


def test_created_stream_and_repeated_calls(dev):
    import torch
    s = torch.cuda.Stream(dev)
    # a larger problem after a smaller one grows the workspace; the same shape twice reuses it
    for shape in [(1, 512, 4, 64, True), (2, 2048, 6, 128, True), (2, 2048, 6, 128, True)]:
        B, N, H, d, causal = shape
        o, lse, o_h, lse_h = run_both(dev, B, N, H, d, causal, True, seed=7, stream=s)
        assert bool((o_h.view(torch.int16) == o.view(torch.int16)).all()), shape
        assert bool((lse_h == lse).all()), shape


def test_against_oracle(dev):
    import torch
    import io_aware_exact_06_gb300 as fa
    import oracle
    B, N, H, d = 2, 700, 3, 128
    wl = inputs.make_workload("host", 31, [N] * B, H, d, True)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
    q_h, k_h, v_h = (t(x).reshape(B, N, H, d) for x in (wl.q, wl.k, wl.v))
    o_h = torch.empty((B, N, H, d), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    fa.attn_fwd_host(q_h, k_h, v_h, o_h, lse_h, B, H, N, d, wl.scale, True)
    assert fa.attn_last_device_error() == 0
    rows = inputs.all_rows(wl.cu_seqlens, H)
    ref_o, ref_l, _ = oracle.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, wl.scale, True)
    got_o = o_h.reshape(B * N, H, d).float().numpy()[wl.cu_seqlens[rows[:, 0]] + rows[:, 2], rows[:, 1]]
    got_l = lse_h.numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    st = parity.error_stats(got_o.astype(np.float64), got_l.astype(np.float64), ref_o, ref_l)
    assert st["o_max_abs"] <= parity.O_MAX_ABS, st
    assert st["o_rel_l2"] <= parity.O_REL_L2, st
    assert st["lse_max_abs"] <= parity.LSE_MAX_ABS, st
