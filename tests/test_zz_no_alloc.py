"""attn_fwd_noalloc: the forward pass for callers that cannot allocate device
memory (their allocator belongs to another framework, or allocation is
forbidden after start-up).  It runs the same kernels with a fixed scratch
array inside the library instead of a cudaMalloc'd workspace.

The GPU tests call it through the C ABI and compare its outputs with those of
attn_fwd, on two calls in a row (the second one reuses the scratch left by the
first), within the parity tolerances of the other GPU tests; read its device
errors (invalid cu_seqlens, an expired bounded wait made to expire from the
host) through attn_fwd_noalloc_last_device_error; and check, in a fresh
process, that it leaves the library holding no device memory.  This file is
collected last so that a run stopping at its first failure has already run
every other test."""
import os
import subprocess
import sys
import textwrap

import pytest

import io_aware_exact_06_gb300 as fa
from io_aware_exact_06_gb300 import build, inputs
from tests import parity

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


def _case(dev, c):
    import torch
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
    return wl, q, k, v, cu_arg, B, N, lse_shape, o_ref, l_ref


@pytest.mark.gpu
@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_attn_fwd_twice(dev, case):
    import torch
    c = CASES[case]
    wl, q, k, v, cu_arg, B, N, lse_shape, o_ref, l_ref = _case(dev, c)
    for _ in range(2):
        o_new = torch.full_like(q, float("nan"))
        l_new = torch.full(lse_shape, float("nan"), device=dev)
        fa.attn_fwd_noalloc(q, k, v, o_new, l_new, B, wl.H, N, wl.d, wl.scale, c["causal"],
                            cu_arg, None)
        assert fa.attn_fwd_noalloc_last_device_error() == 0
        _compare(o_ref, l_ref, o_new, l_new)


@pytest.mark.gpu
def test_noalloc_reports_invalid_seqlens_then_recovers(dev):
    """Offsets that do not start at 0: the scheduler kernel rejects them on the
    device, nothing is written, the reader returns ATTN_ERR_SEQLENS (-8); the
    next valid call clears the scratch header and is correct."""
    import torch
    c = CASES["packed"]
    wl, q, k, v, cu, B, N, lse_shape, o_ref, l_ref = _case(dev, c)
    bad = cu.clone()
    bad[0] = 1
    o_new = torch.full_like(q, float("nan"))
    l_new = torch.full(lse_shape, float("nan"), device=dev)
    fa.attn_fwd_noalloc(q, k, v, o_new, l_new, B, wl.H, N, wl.d, wl.scale, True, bad, None)
    assert fa.attn_fwd_noalloc_last_device_error() == -8
    assert torch.isnan(o_new.float()).all() and torch.isnan(l_new).all()
    assert fa.attn_fwd_noalloc_last_device_error() == 0  # read and cleared
    fa.attn_fwd_noalloc(q, k, v, o_new, l_new, B, wl.H, N, wl.d, wl.scale, True, cu, None)
    assert fa.attn_fwd_noalloc_last_device_error() == 0
    _compare(o_ref, l_ref, o_new, l_new)


@pytest.mark.gpu
def test_noalloc_reports_expired_wait_then_recovers(dev):
    """The test hook makes CTA 0's producer skip one copy, so a bounded wait
    (50 ms here) expires on the device; the reader returns
    ATTN_ERR_DEVICE_TIMEOUT (-7) and the next call is correct."""
    import torch
    c = CASES["dense"]
    wl, q, k, v, cu, B, N, lse_shape, o_ref, l_ref = _case(dev, c)
    o_new = torch.empty_like(q)
    l_new = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    fa.attn_fwd_noalloc_ex(q, k, v, o_new, l_new, B, wl.H, N, wl.d, wl.scale, True, None, None,
                           wait_timeout_ns=50_000_000, fault_inject=1)
    assert fa.attn_fwd_noalloc_last_device_error() == -7
    assert fa.attn_last_error_site() != 0
    fa.attn_fwd_noalloc(q, k, v, o_new, l_new, B, wl.H, N, wl.d, wl.scale, True, None, None)
    assert fa.attn_fwd_noalloc_last_device_error() == 0
    _compare(o_ref, l_ref, o_new, l_new)


@pytest.mark.gpu
def test_noalloc_dense_batch_beyond_the_list_limit(dev):
    """A dense batch of 66000 one-token sequences (more (sequence, block) pairs
    than the scratch's list holds) runs: dense batches keep no list there."""
    import torch
    B, H, N, d = 66000, 1, 1, 64
    g = torch.Generator(device=dev).manual_seed(7)
    q, k, v = (torch.randn(B, N, H, d, device=dev, generator=g).bfloat16() for _ in range(3))
    o_ref, o_new = torch.empty_like(q), torch.empty_like(q)
    l_ref = torch.empty(B, H, N, device=dev)
    l_new = torch.empty_like(l_ref)
    fa.attn_fwd(q, k, v, o_ref, l_ref, B, H, N, d, d ** -0.5, True, None, None)
    fa.attn_fwd_noalloc(q, k, v, o_new, l_new, B, H, N, d, d ** -0.5, True, None, None)
    assert fa.attn_fwd_noalloc_last_device_error() == 0
    # one visible key: O = v (to within the exp2 approximation), LSE = its logit
    assert torch.allclose(o_new.float(), v.float(), rtol=2 ** -7, atol=0)
    assert torch.equal(o_new, o_ref) and torch.equal(l_new, l_ref)


@pytest.mark.gpu
def test_noalloc_allocates_nothing_in_a_fresh_process(dev):
    """In a new process, attn_fwd_noalloc runs first (dense and packed) and the
    library holds no device memory afterwards; attn_fwd then allocates its
    workspace (the count moves), which shows the count sees allocations."""
    script = textwrap.dedent("""
        import sys, torch
        sys.path.insert(0, %r)
        import io_aware_exact_06_gb300 as fa
        dev = torch.device("cuda:0")
        torch.cuda.init()
        B, H, N, d = 2, 2, 300, 64
        q, k, v = (torch.randn(B, N, H, d, device=dev).bfloat16() for _ in range(3))
        o = torch.empty_like(q)
        lse = torch.empty(B, H, N, device=dev)
        fa.attn_fwd_noalloc(q, k, v, o, lse, B, H, N, d, 0.125, True, None, None)
        cu = torch.tensor([0, 300, 600], dtype=torch.int32, device=dev)
        lse_p = torch.empty(H, B * N, device=dev)
        fa.attn_fwd_noalloc(q.view(B * N, H, d), k.view(B * N, H, d), v.view(B * N, H, d),
                            o.view(B * N, H, d), lse_p, B, H, N, d, 0.125, True, cu, None)
        assert fa.attn_fwd_noalloc_last_device_error() == 0
        held = fa.attn_device_bytes()
        fa.attn_fwd(q, k, v, o, lse, B, H, N, d, 0.125, True, None, None)
        torch.cuda.synchronize()
        print(held, fa.attn_device_bytes())
    """ % ROOT)
    out = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    before, after = (int(x) for x in out.stdout.split()[-2:])
    assert before == 0
    assert after > 0


def test_noalloc_rejects_packed_batches_beyond_its_scratch():
    """A packed batch of 65536 (sequence, 256-row block) pairs fits; one more
    is refused before any device work, so this runs without a GPU."""
    build.build()
    buf = 1 << 20
    lib = fa.lib()
    # B * ceil(N / 256) = 65537 > 65536; cu_seqlens (a fake address) is never read
    st = lib.attn_fwd_noalloc(buf, buf, buf, buf, buf, 65537, 1, 256, 64, 0.125, 0, buf, None)
    assert st == -10
    assert "scratch" in fa.attn_status_string(st)
    opts = fa.AttnFwdOptions(0, 0, 0, 0)
    import ctypes
    st = lib.attn_fwd_noalloc_ex(buf, buf, buf, buf, buf, 65537, 1, 256, 64, 0.125, 0, buf, None,
                                 ctypes.byref(opts))
    assert st == -10
