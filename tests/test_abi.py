"""The C-ABI library: it loads without a GPU, exports every declared symbol,
and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import io_aware_exact_06_gb300 as fa
from io_aware_exact_06_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fa.lib()


def declared_functions():
    names = []
    for f in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(fa.EXPORTED_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    assert fa.attn_status_string(0) == "ok"
    assert "timed out" in fa.attn_status_string(-7)
    assert fa.attn_status_string(12345) == "unknown status"


BUF = 1 << 20  # fake, 16-byte aligned addresses: validation fails before any use


@pytest.mark.parametrize("args,status", [
    (dict(B=-1), -2),
    (dict(H=-3), -2),
    (dict(d=96), -3),
    (dict(d=0), -3),
    (dict(scale=float("nan")), -5),
    (dict(scale=float("inf")), -5),
    (dict(scale=-0.5), -5),
    (dict(q=None), -1),
    (dict(lse=None), -1),
    (dict(q=BUF + 8), -4),
    (dict(o=BUF + 4), -4),
    (dict(lse=BUF + 2), -4),
    (dict(B=70000, N=1 << 16), -2),
    (dict(H=70000), -2),
])
def test_argument_errors(lib, args, status):
    a = dict(q=BUF, k=BUF, v=BUF, o=BUF, lse=BUF, B=2, H=4, N=256, d=128, scale=0.1,
             causal=1, cu=None, stream=None)
    a.update(args)
    st = lib.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"],
                      a["scale"], a["causal"], a["cu"], a["stream"])
    assert st == status


@pytest.mark.parametrize("zero", ["B", "H", "N"])
def test_empty_problem_is_a_noop(lib, zero):
    a = dict(B=2, H=4, N=256)
    a[zero] = 0
    # null pointers are fine when there is nothing to do
    assert lib.attn_fwd(None, None, None, None, None, a["B"], a["H"], a["N"], 64, 0.125, 0,
                        None, None) == 0


@pytest.mark.parametrize("args,status", [
    (dict(B=-1), -2),
    (dict(N=-5), -2),
    (dict(d=96), -3),
    (dict(scale=float("nan")), -5),
    (dict(scale=-0.5), -5),
    (dict(q=None), -1),
    (dict(o=None), -1),
    (dict(lse=None), -1),
    (dict(B=70000, N=1 << 16), -2),
    (dict(H=70000), -2),
])
def test_host_argument_errors(lib, args, status):
    a = dict(q=BUF, k=BUF, v=BUF, o=BUF, lse=BUF, B=2, H=4, N=256, d=128, scale=0.1,
             causal=1, cu=None, stream=None)
    a.update(args)
    st = lib.attn_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"],
                           a["d"], a["scale"], a["causal"], a["cu"], a["stream"])
    assert st == status


@pytest.mark.parametrize("zero", ["B", "H", "N"])
def test_host_empty_problem_is_a_noop(lib, zero):
    a = dict(B=2, H=4, N=256)
    a[zero] = 0
    assert lib.attn_fwd_host(None, None, None, None, None, a["B"], a["H"], a["N"], 128, 0.125, 1,
                             None, None) == 0


# host cu_seqlens is checked on the host before anything is copied
@pytest.mark.parametrize("cu,status", [
    ([1, 100, 200], -8),    # does not start at 0
    ([0, 100, 50], -8),     # decreasing
    ([0, 300, 400], -8),    # a length above N = 256
    ([0, 0, 0], 0),         # no tokens: nothing to do
])
def test_host_cu_seqlens_checked_on_the_host(lib, cu, status):
    import numpy as np
    arr = np.asarray(cu, dtype=np.int32)
    st = lib.attn_fwd_host(BUF, BUF, BUF, BUF, BUF, 2, 4, 256, 128, 0.1, 1,
                           arr.ctypes.data, None)
    assert st == status


@pytest.mark.parametrize("args,status", [
    (dict(d=64), -3),
    (dict(d=96), -3),
    (dict(B=-1), -2),
    (dict(scale=float("nan")), -5),
    (dict(q8=None), -1),
    (dict(sv=None), -1),
    (dict(vt=BUF + 8), -4),
    (dict(sk=BUF + 2), -4),
])
def test_fp8_codes_argument_errors(lib, args, status):
    a = dict(q8=BUF, sq=BUF, k8=BUF, sk=BUF, vt=BUF, sv=BUF, o=BUF, lse=BUF, B=2, H=4, N=256,
             d=128, scale=0.1, causal=1, rotated=1, cu=None, stream=None)
    a.update(args)
    st = lib.attn_fwd_fp8_codes(a["q8"], a["sq"], a["k8"], a["sk"], a["vt"], a["sv"], a["o"],
                                a["lse"], a["B"], a["H"], a["N"], a["d"], a["scale"], a["causal"],
                                a["rotated"], a["cu"], a["stream"])
    assert st == status


def test_binding_raises_on_error(lib):
    with pytest.raises(fa.AttnError) as e:
        fa.attn_fwd(BUF, BUF, BUF, BUF, BUF, 1, 1, 128, 80, 0.1, False)
    assert e.value.status == -3


@pytest.mark.parametrize("args,status", [
    (dict(B=-1), -2),
    (dict(d=96), -3),
    (dict(scale=float("nan")), -5),
    (dict(cu=BUF, N=(8193 * 128)), -2),
    (dict(dout=None), -1),
    (dict(dq=None), -1),
    (dict(lse=None), -1),
    (dict(dk=BUF + 8), -4),
    (dict(dout=BUF + 2), -4),
    (dict(lse=BUF + 2), -4),
    (dict(B=70000, N=1 << 16), -2),
])
def test_backward_argument_errors(lib, args, status):
    a = dict(q=BUF, k=BUF, v=BUF, o=BUF, dout=BUF, lse=BUF, dq=BUF, dk=BUF, dv=BUF, B=2, H=4,
             N=256, d=128, scale=0.1, causal=1, cu=None, stream=None)
    a.update(args)
    st = lib.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["dq"], a["dk"],
                      a["dv"], a["B"], a["H"], a["N"], a["d"], a["scale"], a["causal"], a["cu"],
                      a["stream"])
    assert st == status


def test_backward_empty_problem_is_a_noop(lib):
    assert lib.attn_bwd(*([None] * 9), 0, 4, 256, 64, 0.125, 0, None, None) == 0


@pytest.mark.parametrize("args,status", [
    (dict(d=96), -3),
    (dict(d=256), -3),
    (dict(B=-1), -2),
    (dict(scale=-1.0), -5),
    (dict(scale=float("nan")), -5),
    (dict(q=None), -1),
    (dict(o=BUF + 8), -4),
])
def test_fp8_argument_errors(lib, args, status):
    a = dict(q=BUF, k=BUF, v=BUF, o=BUF, lse=BUF, B=2, H=4, N=256, d=128, scale=0.1, causal=1)
    a.update(args)
    st = lib.attn_fwd_fp8(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"],
                          a["scale"], a["causal"], None, None, None)
    assert st == status
    assert lib.attn_fp8_quantize_qk(BUF, BUF, BUF, 1, 1, 128, 32, None, None, None) == -3
    assert lib.attn_fp8_quantize_v(None, BUF, BUF, 1, 1, 128, 128, None, None) == -1


def test_backward_window_below_minus_one(lib):
    assert lib.attn_bwd_window(*([BUF] * 9), 1, 1, 128, 64, 0.1, 1, -2, 0, None, None) == -2
    assert lib.attn_bwd_window(*([BUF] * 9), 1, 1, 128, 64, 0.1, 1, 0, -3, None, None) == -2


@pytest.mark.parametrize("args,status", [
    (dict(d=96), -3),
    (dict(B=-1), -2),
    (dict(max_len=-1), -2),
    (dict(splits=257), -2),
    (dict(splits=-1), -2),
    (dict(scale=-1.0), -5),
    (dict(scale=float("inf")), -5),
    (dict(cu=None), -1),
    (dict(k=None), -1),
    (dict(v=BUF + 8), -4),
    (dict(cu=BUF + 2), -4),
    (dict(B=1 << 20, max_len=1 << 12), -2),
])
def test_decode_argument_errors(lib, args, status):
    a = dict(q=BUF, k=BUF, v=BUF, o=BUF, lse=BUF, B=2, H=4, d=128, scale=0.1, cu=BUF,
             max_len=512, splits=0)
    a.update(args)
    st = lib.attn_fwd_decode(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["d"],
                             a["scale"], a["cu"], a["max_len"], a["splits"], None)
    assert st == status


def test_decode_empty_batch_is_a_noop(lib):
    assert lib.attn_fwd_decode(None, None, None, None, None, 0, 4, 128, 0.1, None, 0, 0, None) == 0


def test_pair_kernel_request_checked_before_the_device(lib):
    """Asking for the pair-of-SMs kernel with a shape it does not take (d = 64,
    or a sliding window) fails with ATTN_ERR_SHAPE before any device work."""
    opts = fa.AttnFwdOptions(0, 0, 0, 2)
    st = lib.attn_fwd_ex(BUF, BUF, BUF, BUF, BUF, 1, 1, 256, 64, 0.125, 1, None, None,
                         ctypes.byref(opts))
    assert st == -2
