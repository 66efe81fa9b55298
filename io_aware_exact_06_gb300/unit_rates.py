"""Measures the per-SM exp-unit and tensor-core rates of the current GPU.

Builds ``csrc/unit_rates.cu`` (a standalone sm_103a program) into _build/ and
runs it; returns its JSON: SM count, ex2 results per clock per SM, bf16 MMA
flops per clock per SM at a fixed operand address and (``ksteps_*``) for
products stepping through a tile's k-slices in the attention kernels' operand
forms.  Used for the exp-unit and operand-rate rooflines of the forward pass.

    python -m io_aware_exact_06_gb300.unit_rates
"""
from __future__ import annotations

import json
import os
import subprocess

from . import build as _build

SRC = os.path.join(_build.CSRC, "unit_rates.cu")
EXE = os.path.join(_build.OUT_DIR, "unit_rates")


def build_exe() -> str:
    deps = [SRC, os.path.join(_build.CSRC, "sm100_ptx.cuh")]
    if os.path.exists(EXE) and os.path.getmtime(EXE) >= max(os.path.getmtime(p) for p in deps):
        return EXE
    os.makedirs(_build.OUT_DIR, exist_ok=True)
    tmp = EXE + f".tmp{os.getpid()}"
    subprocess.run([_build.nvcc(), *_build.ARCH, "-O3", "-std=c++17", SRC, "-o", tmp], check=True)
    os.replace(tmp, EXE)
    return EXE


def measure() -> dict:
    out = subprocess.run([build_exe()], capture_output=True, text=True, timeout=120)
    line = [l for l in out.stdout.splitlines() if l.startswith("{")]
    if out.returncode != 0 or not line:
        raise RuntimeError(f"unit_rates failed: {out.stdout[-500:]} {out.stderr[-500:]}")
    return json.loads(line[-1])


if __name__ == "__main__":
    print(json.dumps(measure()))
