"""Entry points running at the same time on two streams.

The library keeps per-(device, stream) workspaces (scheduling lists, unit
counters, partial results, FP8 codes, backward row vectors).  Work issued on
two streams without synchronising between them must give, bit for bit, what
each call gives alone."""
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


def calls(dev):
    """A list of (name, run(stream) -> tuple of output tensors)."""
    import torch
    import io_aware_exact_06_gb300 as fa
    out = []
    # dense causal forward, d = 128
    wl = inputs.make_workload("s1", 0x5101, [2048] * 2, 4, 128, True)
    q, k, v, _ = parity.to_device(wl, dev)

    def fwd_dense(s, q=q, k=k, v=v):
        o = torch.empty_like(q)
        lse = torch.empty((2, 4, 2048), device=dev)
        fa.attn_fwd(q, k, v, o, lse, 2, 4, 2048, 128, wl.scale, True, None, s)
        return o, lse
    out.append(("fwd dense", fwd_dense))
    # packed forward, d = 64
    wp = inputs.make_workload("s2", 0x5102, [700, 1, 1500, 300], 3, 64, True, varlen=True)
    qp, kp, vp, cup = parity.to_device(wp, dev)

    def fwd_packed(s):
        o = torch.empty_like(qp)
        lse = torch.empty((3, wp.tokens), device=dev)
        fa.attn_fwd(qp, kp, vp, o, lse, 4, 3, 1500, 64, wp.scale, True, cup, s)
        return o, lse
    out.append(("fwd packed", fwd_packed))
    # backward of the dense case
    do = torch.randn_like(q)

    def bwd(s):
        o, lse = fwd_dense(s)
        g = [torch.empty_like(q) for _ in range(3)]
        fa.attn_bwd(q, k, v, o, do, lse, *g, 2, 4, 2048, 128, wl.scale, True, None, s)
        return tuple(g)
    out.append(("bwd", bwd))
    # decode against packed keys
    cuk = torch.tensor([0, 5000, 5001, 9000], dtype=torch.int32, device=dev)
    kd = torch.randn(9000, 4, 128, device=dev).to(torch.bfloat16)
    vd = torch.randn(9000, 4, 128, device=dev).to(torch.bfloat16)
    qd = torch.randn(3, 4, 128, device=dev).to(torch.bfloat16)

    def decode(s):
        o = torch.empty_like(qd)
        lse = torch.empty((3, 4), device=dev)
        fa.attn_fwd_decode(qd, kd, vd, o, lse, 3, 4, 128, 128 ** -0.5, cuk, 5000, 0, s)
        return o, lse
    out.append(("decode", decode))
    # FP8 forward of the dense case
    signs = np.where(inputs.splitmix64(11, 0, 128) & np.uint64(1), -1, 1).astype(np.int8)

    def fp8(s):
        o = torch.empty_like(q)
        lse = torch.empty((2, 4, 2048), device=dev)
        fa.attn_fwd_fp8(q, k, v, o, lse, 2, 4, 2048, 128, wl.scale, True, signs, stream=s)
        return o, lse
    out.append(("fp8", fp8))
    return out


def test_two_streams_match_one(dev):
    import torch
    import io_aware_exact_06_gb300 as fa
    todo = calls(dev)
    alone = {}
    for name, run in todo:
        alone[name] = [t.clone() for t in run(None)]
        torch.cuda.synchronize()
    assert fa.attn_last_device_error() == 0
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    got = {}
    # every call on both streams, interleaved, no synchronisation in between
    for rnd in range(2):
        for i, (name, run) in enumerate(todo):
            s = s1 if (i + rnd) % 2 == 0 else s2
            with torch.cuda.stream(s):
                got[(name, rnd)] = run(s)
    torch.cuda.synchronize()
    assert fa.attn_last_device_error(s1) == 0 and fa.attn_last_device_error(s2) == 0
    for (name, rnd), outs in got.items():
        for a, b in zip(alone[name], outs):
            assert torch.equal(a, b), (name, rnd)
