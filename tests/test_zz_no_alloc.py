"""attn_fwd_noalloc: the forward pass for callers that cannot allocate device
memory (their allocator belongs to another framework, or allocation is
forbidden after start-up).  It runs the same kernels with a fixed scratch
array inside the library instead of a cudaMalloc'd workspace.

The GPU tests call it through the C ABI and compare its outputs with those of
attn_fwd, on two calls in a row (the second one reuses the scratch left by the
first), within the parity tolerances of the other GPU tests.  This file is
collected last so that a run stopping at its first failure has already run
every other test."""
import numpy as np
import pytest

import io_aware_exact_06_gb300 as fa
from io_aware_exact_06_gb300 import build, inputs
from tests import parity


def _compare(o_ref, l_ref, o_new, l_new):
    d = (o_new.double() - o_ref.double())
    assert d.abs().max().item() <= parity.O_MAX_ABS
    assert (d.norm() / o_ref.double().norm()).item() <= parity.O_REL_L2
    assert (l_new - l_ref).abs().max().item() <= parity.LSE_MAX_ABS


@pytest.fixture(scope="module")
def dev():
    import torch
    import __graft_entry__
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    __graft_entry__.build()
    return torch.device("cuda:0")


CASES = {
    # dense causal, d = 128: the scratch holds only the error word
    "dense": dict(seqlens=[1024, 1024, 1024], H=4, d=128, causal=True, varlen=False),
    # packed causal, d = 64, ragged lengths: the scratch also holds the work list
    "packed": dict(seqlens=[1, 300, 129, 0, 700, 256, 1000], H=3, d=64, causal=True, varlen=True),
}


@pytest.mark.gpu
@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_attn_fwd_twice(dev, case):
    import torch
    c = CASES[case]
    wl = inputs.make_workload("noalloc", 31337, c["seqlens"], c["H"], c["d"], c["causal"],
                              varlen=c["varlen"])
    q, k, v, cu = parity.to_device(wl, dev)
    lens = wl.seqlens()
    if c["varlen"]:
        B, N, cu_arg = wl.nseq, int(lens.max()), cu
        lse_shape = (wl.H, wl.tokens)
    else:
        B, N, cu_arg = wl.nseq, int(lens[0]), None
        lse_shape = (B, wl.H, N)
    o_ref = torch.empty_like(q)
    l_ref = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    fa.attn_fwd(q, k, v, o_ref, l_ref, B, wl.H, N, wl.d, wl.scale, c["causal"], cu_arg, None)
    assert fa.attn_last_device_error() == 0
    for _ in range(2):
        o_new = torch.full_like(q, float("nan"))
        l_new = torch.full(lse_shape, float("nan"), device=dev)
        fa.attn_fwd_noalloc(q, k, v, o_new, l_new, B, wl.H, N, wl.d, wl.scale, c["causal"],
                            cu_arg, None)
        torch.cuda.synchronize()
        _compare(o_ref, l_ref, o_new, l_new)


def test_noalloc_rejects_problems_beyond_its_scratch():
    """65536 (sequence, 256-row block) pairs fit; one more is refused before
    any device work, so this runs without a GPU."""
    build.build()
    buf = 1 << 20
    lib = fa.lib()
    # B * ceil(N / 256) = 65537 > 65536
    st = lib.attn_fwd_noalloc(buf, buf, buf, buf, buf, 65537, 1, 256, 64, 0.125, 0, None, None)
    assert st == -10
    assert "scratch" in fa.attn_status_string(st)
