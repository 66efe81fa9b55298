"""Benchmark of the GB300 fused exact attention forward.

One step = one forward pass (attn_fwd: every kernel of the path) over the
long-context causal workload B=2, H=16, N=8192, d=128 (bf16, fp32 accumulate),
with inputs resident in device memory.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  python bench.py --workload decode   # split-KV decode line (attn_fwd_kvsplit)
  python bench.py --workload bwd      # backward line (attn_bwd)
  python bench.py --workload fp8      # FP8 forward line (attn_fwd_fp8)
  python bench.py --config stress     # the forward line on another forward workload
                                      # (tiny, gpt2_causal, long_full, stress, varlen)

Metric: attention forward TFLOP/s, FLOPs = 4*B*H*N^2*d halved for causal,
whole job (all ranks) / the slowest rank's time.  N > 1 runs one independent
replica per GPU (launched by torch.distributed.run); the path needs no
exchange between GPUs.

`--impl reference` times the fp64 CPU oracle (the only other implementation
of this path) on the host cores, one bounded sample of the workload's rows
per step, and reports it in the same metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from io_aware_exact_06_gb300 import inputs  # noqa: E402

WORKLOAD = "long_causal"
METRIC = "attention fwd TFLOP/s on 1 GB300 (bf16) and fraction of dense BF16 peak"
UNIT = "TFLOP/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


def workload_config(wl, name=WORKLOAD):
    c = inputs.CONFIGS[name]
    io_bytes = 4 * wl.tokens * wl.H * wl.d * 2
    mask = "causal" if c["causal"] else "non-causal"
    std = c.get("qk_std", 1.0)
    dist = "Q,K,V iid N(0,1)" if std == 1.0 else f"Q,K iid N(0,{std:g}^2), V iid N(0,1)"
    out = {"H": c["H"], "d": c["d"], "causal": c["causal"], "scale": "1/sqrt(d)",
           "inputs": f"{dist} bf16, seeded (SplitMix64 + Box-Muller)",
           "l2": (f"Q,K,V,O = {io_bytes / 1e6:.0f} MB > 129 MB L2 (no flush between steps)"
                  if io_bytes > 129e6 else
                  f"Q,K,V,O = {io_bytes / 1e6:.1f} MB fit in the 129 MB L2: not flushed, "
                  f"steps after the first read them from L2")}
    if "nseq" in c:
        lens = wl.seqlens()
        out.update(workload=f"{name}: {c['nseq']} packed sequences, lengths {int(lens.min())}..{int(lens.max())} "
                            f"(uniform [{c['Lmin']}, {c['Lmax']}]), H={c['H']} d={c['d']} {mask}",
                   nseq=c["nseq"], tokens=int(wl.tokens))
    else:
        out.update(workload=f"{name}: B={c['B']} H={c['H']} N={c['N']} d={c['d']} {mask}",
                   B=c["B"], N=c["N"])
    return out


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), \
            float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, 1700.0, FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = ""
        self.settle_steps = 0
        self.t_start = time.perf_counter()

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        self.t_start = time.perf_counter()
        return self

    def settle(self, step, dev, seconds: float = 0.3, busy: float = 0.02):
        """Lets the sampler start (`seconds` after __enter__), the GPU idle
        but for the last `busy` seconds, which run untimed steps: a GPU left
        idle runs its next calls slower (a timed region of a few hundred µs
        would see that), and a long busy stretch can bring the power cap into
        a short timed region.  The steps' count is reported with the clocks."""
        import torch
        time.sleep(max(0.0, self.t_start + seconds - busy - time.perf_counter()))
        t0 = time.perf_counter()
        n = 0
        while n < 3 or time.perf_counter() - t0 < busy:
            step()
            n += 1
            if n % 8 == 0:
                torch.cuda.synchronize(dev)  # a bounded queue of calls
        torch.cuda.synchronize(dev)
        self.settle_steps = n

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"],
                    "settle_steps": self.settle_steps}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "settle_steps": self.settle_steps}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample(wl, budget_s: float, seed: int):
    """Rows of the workload for a bounded oracle run of about budget_s seconds
    (calibrated on a small batch of the same rows)."""
    import oracle
    rows = inputs.sample_rows(wl.cu_seqlens, wl.H, 1 << 18, seed=seed)
    rows = rows[np.argsort(inputs.splitmix64(seed + 1, 0, len(rows)))]
    calib = rows[:256]
    t0 = time.perf_counter()
    oracle.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, calib, wl.scale, wl.causal)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(min(len(rows), max(256, 256 * budget_s / dt)))
    return rows[:n]


def row_flops(wl, rows) -> float:
    """4*d FLOPs per visible key of each row (QK^T and PV), the metric's count."""
    L = (wl.cu_seqlens[rows[:, 0] + 1] - wl.cu_seqlens[rows[:, 0]]).astype(np.float64)
    vis = rows[:, 2] + 1.0 if wl.causal else L
    return float(np.sum(4.0 * wl.d * vis))


def cpu_baseline(wl, budget_s: float = 15.0, name=WORKLOAD):
    import oracle
    rows = oracle_sample(wl, budget_s, seed=0xBA5E)
    t0 = time.perf_counter()
    _, _, used = oracle.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, wl.scale, wl.causal)
    dt = time.perf_counter() - t0
    fl = row_flops(wl, rows)
    # the oracle's cost per row is proportional to its visible keys, so the
    # whole workload takes dt scaled by its FLOPs over the sample's
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": int(used),
            "kind": "oracle",
            "sample": f"{len(rows)} seeded rows of {name} (fp64, materialised score rows), "
                      f"{dt:.1f} s; FLOPs = 4*d per visible key",
            "rows_per_s": len(rows) / dt, "fp64_gflops": fl / dt / 1e9,
            "full_config_s": dt * wl.flops() / fl}


def exp_unit_bound(sm_mhz, d: int, per_gpu_tflops: float):
    """The exp-unit roofline: each score element costs 4*d flops of the metric
    and one exp2, so the bound is SMs * f_SM * (ex2 per clock per SM) * 4d.
    Also the clock-based tensor peak SMs * f_SM * (MMA flop per clock per SM);
    the probe measures every operand form the kernels issue (A and B from
    shared memory, A from TMEM, MN-major B, 256-row products of a pair of
    SMs) at that same rate.  Rates are measured on this GPU; f_SM is the
    median clock of the run."""
    try:
        from io_aware_exact_06_gb300 import unit_rates
        r = unit_rates.measure()
    except Exception as e:  # noqa: BLE001 - reported, not fatal
        return {"error": str(e)[:200]}
    f = (sm_mhz or r["max_clock_mhz"]) * 1e6
    exp_tf = r["sm_count"] * f * r["ex2_per_clk_per_sm"] * 4 * d / 1e12
    mma_tf = r["sm_count"] * f * r["mma_bf16_flop_per_clk_per_sm"] / 1e12
    out = {"ex2_per_clk_per_sm": r["ex2_per_clk_per_sm"],
           "mma_flop_per_clk_per_sm": r["mma_bf16_flop_per_clk_per_sm"],
           "sm_count": r["sm_count"], "sm_mhz": f / 1e6,
           "exp_bound_tflops": exp_tf, "frac_of_exp_bound": per_gpu_tflops / exp_tf,
           "tensor_peak_at_clock_tflops": mma_tf,
           "frac_of_tensor_peak_at_clock": per_gpu_tflops / mma_tf}
    return out


def run_reference(args, world, rank):
    """The oracle on the host cores, one bounded sample of rows per step."""
    if rank != 0:
        return
    import oracle
    wl = inputs.config_workload(WORKLOAD)
    per_step_s = args.ref_step_s or max(1.0, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    rows = oracle_sample(wl, per_step_s, seed=0x5EED)
    fl = row_flops(wl, rows)
    for _ in range(args.warmup):
        oracle.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, wl.scale, wl.causal)
    times, used = [], 1
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _, _, used = oracle.attn_rows(wl.q, wl.k, wl.v, wl.cu_seqlens, rows, wl.scale, wl.causal)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = fl * args.steps / total / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": int(used), "kind": "oracle",
                             "sample": f"{len(rows)} seeded rows of {WORKLOAD} per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_cuda(args, world, rank, local):
    import torch
    import __graft_entry__
    import io_aware_exact_06_gb300 as fa
    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    name = args.config
    wl = inputs.config_workload(name)
    B, H, N, d = wl.nseq, wl.H, int(wl.seqlens().max()), wl.d
    host = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    q_h, k_h, v_h = host(wl.q).pin_memory(), host(wl.k).pin_memory(), host(wl.v).pin_memory()
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    if wl.varlen:  # packed: lse [H, tokens], cu_seqlens on the device
        cu = torch.from_numpy(wl.cu_seqlens.astype(np.int32)).to(dev)
        lse = torch.empty((H, wl.tokens), dtype=torch.float32, device=dev)
    else:
        cu = None
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    o_h = torch.empty(o.shape, dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream(dev)
    flops_step = wl.flops()

    def step():
        fa.attn_fwd(q, k, v, o, lse, B, H, N, d, wl.scale, wl.causal, cu, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if fa.attn_last_device_error(stream) != 0:
        raise RuntimeError("device error during warm-up")

    # device-timed region: inputs resident in HBM
    with ClockSampler(local) as clk:
        clk.settle(step, dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            step()
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    status = fa.attn_last_device_error(stream)
    if status != 0:
        raise RuntimeError(f"device error status {status}")
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    # the calls run back to back (no event between them, as an application
    # issues them); one call per step, so its mean duration is total / steps
    kernel_ms = total_ms / args.steps

    # end to end through the C ABI with host buffers, every step: H2D of Q,
    # K, V from pinned memory, the forward, D2H of O and LSE, by
    # attn_fwd_host (the copies of one head group overlap the attention of
    # the next)
    cu_h = torch.from_numpy(wl.cu_seqlens.astype(np.int32)).pin_memory() if cu is not None else None
    e2e_api = "attn_fwd_host"

    def e2e_step():
        fa.attn_fwd_host(q_h, k_h, v_h, o_h, lse_h, B, H, N, d, wl.scale, wl.causal, cu_h, stream)

    e2e_steps = max(3, min(args.steps, 10))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    h2d = 3 * q.numel() * 2
    d2h = o.numel() * 2 + lse.numel() * 4

    if rank != 0:
        return
    peak, _, _, src = peaks()
    value = world * flops_step * args.steps / (total_ms * 1e-3) / 1e12
    achieved = flops_step / (kernel_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(wl, name),
        "frac_of_dense_bf16_peak": value / world / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak, "peak_source": f"{src} bf16_tflops (burst)",
                     "kernel": f"attn_fwd_row_kernel<{d}>" + (" + build_worklist_kernel" if wl.varlen else ""),
                     "traffic": args.traffic if name == WORKLOAD else CONFIG_TRAFFIC_BYTES.get(name)},
        "clocks": clk.summary(),
        "e2e": {"value": world * flops_step * e2e_steps / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "api": e2e_api},
        "gpu_launches": args.steps,
    }
    line["exp_unit_bound"] = exp_unit_bound(line["clocks"].get("sm_mhz"), d, value / world)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, name=name)
    print(json.dumps(line), flush=True)


DECODE = {"B": 8, "H": 16, "Nq": 1, "Nk": 32768, "d": 128}
# DRAM bytes (read + write) of one decode call (decode kernel + combine), from
# one ncu capture of the current kernels (None once either kernel changes).
DECODE_TRAFFIC_BYTES = 2_147_573_504 + 4_097_792 + 1_271_296  # decode kernel read + write, combine read
DECODE_METRIC = "split-KV decode: algorithmic HBM GB/s on 1 GB300 (bf16 K/V cache)"


def decode_config(S):
    c = DECODE
    return {"workload": f"decode (split-KV): B={c['B']} H={c['H']} Nq={c['Nq']} Nk={c['Nk']} "
                        f"d={c['d']} causal (bottom-right)",
            "B": c["B"], "H": c["H"], "Nq": c["Nq"], "Nk": c["Nk"], "d": c["d"], "causal": True,
            "num_splits": S, "scale": "1/sqrt(d)",
            "inputs": "Q,K,V iid N(0,1) bf16, seeded (SplitMix64 + Box-Muller)",
            "l2": "K,V = 2.1 GB > 129 MB L2 (no flush between steps)"}


def run_decode(args, world, rank, local):
    """One step = one attn_fwd_kvsplit call (decode kernel + combine kernel) of a
    batch of single-token queries against a resident 32768-token K/V cache.
    Metric: algorithmic bytes (K and V read once, Q read, O and LSE written)
    per second; the path is bound by HBM bandwidth."""
    import torch
    import __graft_entry__
    import io_aware_exact_06_gb300 as fa
    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    c = DECODE
    B, H, Nq, Nk, d = c["B"], c["H"], c["Nq"], c["Nk"], c["d"]
    seed = 0xA77E0100
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    q_h = bf(inputs.normal_bf16(4 * seed + 1, B * Nq * H * d)).reshape(B, Nq, H, d).pin_memory()
    k = bf(inputs.normal_bf16(4 * seed + 2, B * Nk * H * d)).reshape(B, Nk, H, d).to(dev)
    v = bf(inputs.normal_bf16(4 * seed + 3, B * Nk * H * d)).reshape(B, Nk, H, d).to(dev)
    q = q_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    o_h = torch.empty(o.shape, dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream(dev)
    scale = d ** -0.5
    bytes_step = 2 * B * Nk * H * d * 2 + 2 * B * Nq * H * d * 2 + B * H * Nq * 4

    def step():
        fa.attn_fwd_kvsplit(q, k, v, o, lse, B, H, Nq, Nk, d, scale, True, 0, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if fa.attn_last_device_error(stream) != 0:
        raise RuntimeError("device error during warm-up")
    with ClockSampler(local) as clk:
        clk.settle(step, dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    if fa.attn_last_device_error(stream) != 0:
        raise RuntimeError("device error in the timed region")
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    # the calls run back to back (no event between them, as an application
    # issues them); one call per step, so its mean duration is total / steps
    call_ms = total_ms / args.steps

    def e2e_step():  # a new query batch from the host, the result back
        q.copy_(q_h, non_blocking=True)
        step()
        o_h.copy_(o, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    n_e2e = max(3, min(args.steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    if rank != 0:
        return
    _, _, hbm, src = peaks()
    achieved = bytes_step / (call_ms * 1e-3) / 1e9
    line = {
        "metric": DECODE_METRIC, "value": world * bytes_step * args.steps / (total_ms * 1e-3) / 1e9,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": decode_config("auto"),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_source": f"{src} hbm_gbs",
                     "kernel": "attn_decode_kernel<128> + attn_combine_kernel<128> (one call)",
                     "traffic": DECODE_TRAFFIC_BYTES},
        "clocks": clk.summary(),
        "e2e": {"value": world * bytes_step * n_e2e / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": q.numel() * 2,
                "d2h_bytes_per_step": o.numel() * 2 + lse.numel() * 4},
        "gpu_launches": 2 * args.steps,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = decode_cpu_baseline(q_h, k, v, scale)
    print(json.dumps(line), flush=True)


def decode_cpu_baseline(q_h, k, v, scale):
    """The oracle on the decode rows of sequence 0 (every head): the query is
    the last key position of a self-attention problem whose other query rows
    are zero (they change no other row)."""
    import oracle
    B, Nq, H, d = q_h.shape
    Nk = k.shape[1]
    k0 = k[0].cpu().view(torch_int16()).numpy().view(np.uint16).reshape(Nk, H, d)
    v0 = v[0].cpu().view(torch_int16()).numpy().view(np.uint16).reshape(Nk, H, d)
    qf = np.zeros((Nk, H, d), dtype=np.uint16)
    qf[Nk - Nq:] = q_h[0].view(torch_int16()).numpy().view(np.uint16)
    cu = np.array([0, Nk], dtype=np.int64)
    rows = np.array([(0, h, Nk - Nq + r) for h in range(H) for r in range(Nq)], dtype=np.int64)
    reps, t0 = 0, time.perf_counter()
    while True:
        _, _, used = oracle.attn_rows(qf, k0, v0, cu, rows, scale, True)
        reps += 1
        dt = time.perf_counter() - t0
        if dt > 5.0:
            break
    per_row_bytes = 2 * Nk * d * 2 + 2 * d * 2 + 4
    return {"value": reps * len(rows) * per_row_bytes / dt / 1e9, "unit": "GB/s", "cores": int(used),
            "kind": "oracle",
            "sample": f"{len(rows)} decode rows (sequence 0, every head) x {reps} repetitions, "
                      f"{dt:.1f} s; bytes = K and V of the row's head once + q, o, lse"}


def torch_int16():
    import torch
    return torch.int16


BWD_METRIC = "attention bwd TFLOP/s on 1 GB300 (bf16; 2.5x the forward's FLOPs)"


def run_bwd(args, world, rank, local):
    """One step = one attn_bwd call (row prologue, dK/dV kernel, dQ kernel) on
    the long causal workload with a seeded upstream gradient dO; O and the LSE
    come from one attn_fwd call before the timed region.  FLOPs = 2.5x the
    forward's (five matrix products per visible tile pair against two)."""
    import torch
    import __graft_entry__
    import io_aware_exact_06_gb300 as fa
    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = inputs.config_workload(WORKLOAD)
    B, H, N, d = wl.nseq, wl.H, int(wl.seqlens()[0]), wl.d
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    dout_bits = inputs.normal_bf16(0xD0D0, wl.q.size).reshape(wl.q.shape)
    host = [bf(a).pin_memory() for a in (wl.q, wl.k, wl.v, dout_bits)]
    q, k, v, do = (t.to(dev) for t in host)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    fa.attn_fwd(q, k, v, o, lse, B, H, N, d, wl.scale, True, None, stream)
    o_h = o.cpu().pin_memory()
    lse_h = lse.cpu().pin_memory()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    grads_h = [torch.empty(q.shape, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    flops_step = 2.5 * wl.flops()

    def step():
        fa.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, wl.scale, True, None, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if fa.attn_last_device_error(stream) != 0:
        raise RuntimeError("device error during warm-up")
    with ClockSampler(local) as clk:
        clk.settle(step, dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    if fa.attn_last_device_error(stream) != 0:
        raise RuntimeError("device error in the timed region")
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    # the calls run back to back (no event between them, as an application
    # issues them); one call per step, so its mean duration is total / steps
    call_ms = total_ms / args.steps

    def e2e_step():  # Q, K, V, O, dO and LSE from the host, the three gradients back
        for dst, src in zip((q, k, v, do), host):
            dst.copy_(src, non_blocking=True)
        o.copy_(o_h, non_blocking=True)
        lse.copy_(lse_h, non_blocking=True)
        step()
        for dst, src in zip(grads_h, (dq, dk, dv)):
            dst.copy_(src, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    n_e2e = max(3, min(args.steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    if rank != 0:
        return
    peak, _, _, src = peaks()
    achieved = flops_step / (call_ms * 1e-3) / 1e12
    cfg = workload_config(wl)
    cfg["workload"] = cfg["workload"] + ", backward (dO ~ N(0,1) bf16, seeded)"
    line = {
        "metric": BWD_METRIC, "value": world * flops_step * args.steps / (total_ms * 1e-3) / 1e12,
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak, "peak_source": f"{src} bf16_tflops (burst)",
                     "kernel": "bwd_prep_kernel<128> + bwd_tile_kernel<128, dK/dV> + "
                               "bwd_tile_kernel<128, dQ> (one call)",
                     "tensor_work_tflops": achieved * 7.0 / 5.0,
                     "traffic": BWD_TRAFFIC_BYTES},
        "clocks": clk.summary(),
        "e2e": {"value": world * flops_step * n_e2e / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": 5 * q.numel() * 2 + lse.numel() * 4,
                "d2h_bytes_per_step": 3 * q.numel() * 2},
        "gpu_launches": 3 * args.steps,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = bwd_cpu_baseline(wl, dout_bits)
    print(json.dumps(line), flush=True)


def bwd_cpu_baseline(wl, dout_bits, budget_s: float = 10.0):
    """The oracle's gradients of whole (sequence, head) pairs of the workload,
    pair after pair until about budget_s seconds have passed."""
    import oracle
    t0 = time.perf_counter()
    done, used = 0, 1
    L = float(wl.seqlens()[0])
    pairs = [(s, h) for h in range(wl.H) for s in range(wl.nseq)]
    while done < len(pairs) and time.perf_counter() - t0 < budget_s:
        _, _, _, used = oracle.attn_bwd(wl.q, wl.k, wl.v, dout_bits, wl.cu_seqlens, [pairs[done]],
                                        wl.scale, True)
        done += 1
    dt = time.perf_counter() - t0
    flops = done * 2.5 * 4.0 * L * L * wl.d / 2
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": int(used), "kind": "oracle",
            "sample": f"{done} whole (sequence, head) pairs of {WORKLOAD} (fp64 chain rule), "
                      f"{dt:.1f} s; FLOPs = 2.5x the forward's"}


FP8_METRIC = "attention fwd TFLOP/s on 1 GB300 (FP8 e4m3 path: block quantisation + incoherent processing)"


def run_fp8(args, world, rank, local):
    """One step = one attn_fwd_fp8 call (Q and K quantisers, V max and
    quantiser, FP8 attention kernel) on the long causal workload; same FLOP
    convention as the bf16 line.  The roofline times the dominant kernel,
    the attention, alone (attn_fwd_fp8_codes on codes made once), against
    the measured bf16 burst peak times 2 (the nominal FP8 : BF16 dense
    ratio); call_frac is the whole call's."""
    import torch
    import __graft_entry__
    import io_aware_exact_06_gb300 as fa
    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = inputs.config_workload(WORKLOAD)
    B, H, N, d = wl.nseq, wl.H, int(wl.seqlens()[0]), wl.d
    signs = np.where(inputs.splitmix64(0x51635, 0, d) & np.uint64(1), -1, 1).astype(np.int8)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    host = [bf(a).pin_memory() for a in (wl.q, wl.k, wl.v)]
    q, k, v = (t.to(dev) for t in host)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    o_h = torch.empty(o.shape, dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream(dev)
    flops_step = wl.flops()

    def step():
        fa.attn_fwd_fp8(q, k, v, o, lse, B, H, N, d, wl.scale, True, signs, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if fa.attn_last_device_error(stream) != 0:
        raise RuntimeError("device error during warm-up")
    with ClockSampler(local) as clk:
        clk.settle(step, dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    if fa.attn_last_device_error(stream) != 0:
        raise RuntimeError("device error in the timed region")
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    # the calls run back to back (no event between them, as an application
    # issues them); one call per step, so its mean duration is total / steps
    call_ms = total_ms / args.steps

    # the dominant kernel alone (attn_fp8_row_kernel, about three quarters of a
    # call): the same attention launch through attn_fwd_fp8_codes, on codes
    # and scales made once by the quantiser entry points
    T = -(-N // 128)
    q8 = torch.empty((B * N, H, d), dtype=torch.uint8, device=dev)
    k8 = torch.empty_like(q8)
    sq = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    sk = torch.empty_like(sq)
    vt = torch.empty((B, H, d, 128 * T), dtype=torch.uint8, device=dev)
    sv = torch.empty((B, H), dtype=torch.float32, device=dev)
    fa.attn_fp8_quantize_qk(q, q8, sq, B, H, N, d, signs, stream=stream)
    fa.attn_fp8_quantize_qk(k, k8, sk, B, H, N, d, signs, stream=stream)
    fa.attn_fp8_quantize_v(v, vt, sv, B, H, N, d, stream=stream)

    def attention():
        fa.attn_fwd_fp8_codes(q8, sq, k8, sk, vt, sv, o, lse, B, H, N, d, wl.scale, True, True,
                              stream=stream)

    for _ in range(3):
        attention()
    torch.cuda.synchronize(dev)
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0.record(stream)
    for i in range(args.steps):
        attention()
    k1.record(stream)
    torch.cuda.synchronize(dev)
    if fa.attn_last_device_error(stream) != 0:
        raise RuntimeError("device error in the attention-kernel timing")
    kernel_ms = k0.elapsed_time(k1) / args.steps

    def e2e_step():
        for dst, src in zip((q, k, v), host):
            dst.copy_(src, non_blocking=True)
        step()
        o_h.copy_(o, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    n_e2e = max(3, min(args.steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    if rank != 0:
        return
    peak_bf16, _, _, src = peaks()
    peak = 2.0 * peak_bf16
    achieved = flops_step / (kernel_ms * 1e-3) / 1e12
    cfg = workload_config(wl)
    cfg["workload"] = cfg["workload"] + ", FP8 e4m3 (128-row blocks, Hadamard rotation)"
    line = {
        "metric": FP8_METRIC, "value": world * flops_step * args.steps / (total_ms * 1e-3) / 1e12,
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3", "data": "synthetic", "config": cfg,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak,
                     "peak_source": f"{src} bf16_tflops (burst) x 2, the nominal FP8:BF16 dense ratio",
                     "kernel": "attn_fp8_row_kernel<128> (through attn_fwd_fp8_codes)",
                     "call_tflops": flops_step / (call_ms * 1e-3) / 1e12,
                     "call_frac": flops_step / (call_ms * 1e-3) / 1e12 / peak,
                     "traffic": FP8_TRAFFIC_BYTES},
        "clocks": clk.summary(),
        "e2e": {"value": world * flops_step * n_e2e / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": 3 * q.numel() * 2,
                "d2h_bytes_per_step": o.numel() * 2 + lse.numel() * 4},
        "gpu_launches": 3 * args.steps,  # stage-1 quantiser, V codes, attention (the V max reset is a memset)
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = fp8_cpu_baseline(wl, signs)
    print(json.dumps(line), flush=True)


def fp8_cpu_baseline(wl, signs, budget_s: float = 10.0):
    """The oracle's FP8 path (quantisation of one sequence and head, then the
    fp64 attention of the dequantised values) on a bounded sample of rows."""
    import oracle
    N, H, d = int(wl.seqlens()[0]), wl.H, wl.d
    t0 = time.perf_counter()
    sl = slice(0, N)  # sequence 0
    pick = lambda a: np.ascontiguousarray(a[sl, :1])  # head 0
    qc, qs = oracle.fp8_quantize(pick(wl.q), 1, N, 128, True, signs)
    kc, ks = oracle.fp8_quantize(pick(wl.k), 1, N, 128, True, signs)
    vc, vs = oracle.fp8_quantize(pick(wl.v), 1, N, 0, False)
    blk = np.minimum(np.arange(N) // 128, qs.shape[2] - 1)
    deq = lambda c, s: oracle.e4m3_decode(c.ravel()).reshape(c.shape) * s[0, 0][blk][:, None, None]
    qd, kd = deq(qc, qs), deq(kc, ks)
    vd = oracle.e4m3_decode(vc.ravel()).reshape(vc.shape) * float(vs[0, 0, 0])
    cu = np.array([0, N])
    rows_all = np.stack([np.zeros(N, np.int64), np.zeros(N, np.int64), np.arange(N)], axis=1)
    rows_all = rows_all[np.argsort(inputs.splitmix64(0xF8, 0, N))]
    done, flops = 0, 0.0
    while done < N and time.perf_counter() - t0 < budget_s:
        batch = rows_all[done:done + 256]
        oracle.attn_rows_f64(qd, kd, vd, cu, batch, wl.scale / d, True)
        flops += float(np.sum(4.0 * d * (batch[:, 2] + 1)))
        done += len(batch)
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"quantisation of sequence 0, head 0 and the fp64 attention of {done} of its "
                      f"dequantised rows, {dt:.1f} s (single-threaded)"}


# DRAM bytes (read + write) of one attn_fp8_row_kernel<128> launch of this
# workload, from one ncu capture of the current kernel (None once it
# changes): 169.59 MB read + 33.15 MB written.
FP8_TRAFFIC_BYTES = 169_592_320 + 33_148_672

# DRAM bytes (read + write) of one backward call on this workload (all three
# kernels), from one ncu capture of the current kernels (None once one of them
# changes): prep 135.28 + 3.50 MB, dK/dV 329.99 + 101.39 MB, dQ 392.99 +
# 47.84 MB.
BWD_TRAFFIC_BYTES = 135_279_104 + 3_500_032 + 329_993_472 + 101_385_728 + 392_993_024 + 47_838_720


# DRAM bytes (read + write) of one attn_fwd_row_kernel<128> launch of this
# workload, from one ncu capture of the current kernel (None once it changes).
TRAFFIC_BYTES = 542_067_456 + 46_948_864  # 542.07 MB read + 46.95 MB written
# The same for other forward workloads: attn_fwd_row_kernel<64> on the GPT-2
# shaped one (37.82 MB read + 1.8 KB written: O, 12.6 MB, is still in L2
# when the kernel ends) and attn_fwd_row_kernel<128> on the stress and the
# packed ones.
CONFIG_TRAFFIC_BYTES = {"gpt2_causal": 37_819_648 + 1_792, "stress": 258_630_400 + 51_655_680,
                        "varlen": 2_000_659_200 + 464_386_816}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD, choices=[WORKLOAD, "decode", "bwd", "fp8"])
    ap.add_argument("--config", default=WORKLOAD, choices=sorted(inputs.CONFIGS),
                    help="forward line only: time another of the forward workloads (the default "
                         "is the one the metric is quoted on)")
    ap.add_argument("--ref-step-s", type=float, default=0.0,
                    help="reference arm: oracle seconds per step (default: fit the run in ~2.5 min)")
    args = ap.parse_args()
    args.traffic = TRAFFIC_BYTES
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.workload == "decode":
        run_decode(args, world, rank, local)
    elif args.workload == "bwd":
        run_bwd(args, world, rank, local)
    elif args.workload == "fp8":
        run_fp8(args, world, rank, local)
    else:
        run_cuda(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
