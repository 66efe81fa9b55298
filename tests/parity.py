"""Shared helpers of the GPU parity tests: upload a workload, run the CUDA
path through the C ABI, compare chosen rows with the fp64 oracle."""
from __future__ import annotations

import json
import os

import numpy as np

import oracle

# Tolerances of the forward pass: O (bf16 out, fp32 accumulate) and LSE (fp32).
O_MAX_ABS = 1.5e-2
O_REL_L2 = 5e-3
LSE_MAX_ABS = 2e-3


def to_device(wl, dev):
    import torch
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    return t(wl.q), t(wl.k), t(wl.v), torch.from_numpy(wl.cu_seqlens).to(dev)


def run_cuda(wl, dev, packed: bool | None = None, stream=None, window=None, **opts):
    """Runs the CUDA path on workload wl.  Dense layout when every sequence has
    the same length and packed is not forced; returns (o [tokens,H,d] bf16,
    lse [H, tokens] fp32) on the device, plus the device error status."""
    import torch
    import io_aware_exact_06_gb300 as fa
    q, k, v, cu = to_device(wl, dev)
    lens = wl.seqlens()
    dense = (not packed) and len(set(lens.tolist())) == 1 and not wl.varlen
    o = torch.empty_like(q)
    if dense:
        B, N = wl.nseq, int(lens[0])
        lse = torch.empty((B, wl.H, N), dtype=torch.float32, device=dev)
        if window is None:
            fa.attn_fwd_ex(q, k, v, o, lse, B, wl.H, N, wl.d, wl.scale, wl.causal, None, stream, **opts)
        else:
            fa.attn_fwd_window(q, k, v, o, lse, B, wl.H, N, wl.d, wl.scale, wl.causal, window[0],
                               window[1], None, stream)
        lse_ht = lse.permute(1, 0, 2).reshape(wl.H, B * N)
    else:
        lse = torch.empty((wl.H, wl.tokens), dtype=torch.float32, device=dev)
        N = int(lens.max()) if len(lens) else 0
        if window is None:
            fa.attn_fwd_ex(q, k, v, o, lse, wl.nseq, wl.H, N, wl.d, wl.scale, wl.causal, cu, stream,
                           **opts)
        else:
            fa.attn_fwd_window(q, k, v, o, lse, wl.nseq, wl.H, N, wl.d, wl.scale, wl.causal,
                               window[0], window[1], cu, stream)
        lse_ht = lse
    status = fa.attn_last_device_error(stream)
    return o, lse_ht, status


def gather(o, lse_ht, wl, rows):
    tok = wl.cu_seqlens.astype(np.int64)[rows[:, 0]] + rows[:, 2]
    o_np = o.float().cpu().numpy()
    l_np = lse_ht.cpu().numpy()
    return o_np[tok, rows[:, 1]].astype(np.float64), l_np[rows[:, 1], tok].astype(np.float64)


def error_stats(got_o, got_lse, ref_o, ref_lse):
    d = got_o - ref_o
    return {
        "rows": int(len(ref_lse)),
        "o_max_abs": float(np.abs(d).max()) if d.size else 0.0,
        "o_rel_l2": float(np.linalg.norm(d) / max(np.linalg.norm(ref_o), 1e-300)) if d.size else 0.0,
        "lse_max_abs": float(np.abs(got_lse - ref_lse).max()) if d.size else 0.0,
    }


def compare(o, lse_ht, wl, rows, what="", window=(-1, -1)):
    ref_o, ref_lse, _ = oracle.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, wl.scale, wl.causal,
                                         window=window)
    got_o, got_lse = gather(o, lse_ht, wl, rows)
    stats = error_stats(got_o, got_lse, ref_o, ref_lse)
    log = os.environ.get("PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": what, **stats}) + "\n")
    assert np.isfinite(got_o).all() and np.isfinite(got_lse).all(), f"{what}: non-finite output"
    assert stats["o_max_abs"] <= O_MAX_ABS, f"{what}: {stats}"
    assert stats["o_rel_l2"] <= O_REL_L2, f"{what}: {stats}"
    assert stats["lse_max_abs"] <= LSE_MAX_ABS, f"{what}: {stats}"
    return stats
