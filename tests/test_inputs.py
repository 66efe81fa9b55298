"""The seeded input generators: published reference values and rounding."""
import math

import numpy as np

from io_aware_exact_06_gb300 import inputs


def test_splitmix64_reference_outputs():
    # first outputs of SplitMix64 seeded with 0 (reference implementation by Vigna)
    got = [int(x) for x in inputs.splitmix64(0, 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_splitmix64_counter_offsets():
    a = inputs.splitmix64(77, 0, 100)
    b = inputs.splitmix64(77, 40, 60)
    assert (a[40:] == b).all()


def _nearest_bf16_brute(x: float) -> int:
    """Nearest bf16 by exhaustive neighbour search in exact fp64 arithmetic."""
    f32 = np.array([x], dtype=np.float32)  # a float32 close to x (maybe off by an ulp)
    u = int(f32.view(np.uint32)[0]) >> 16
    cands = [(u + dd) & 0xFFFF for dd in (-2, -1, 0, 1, 2)]
    best = None
    for c in cands:
        val = float(np.array([c << 16], dtype=np.uint32).view(np.float32)[0])
        if not math.isfinite(val):
            continue
        err = abs(val - x)
        key = (err, c & 1)  # ties go to the even mantissa
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_bf16_rounding_matches_brute_force():
    bits = inputs.splitmix64(5, 0, 20000)
    x = ((bits >> np.uint64(11)).astype(np.float64) * 2.0 ** -53 - 0.5) * 2.0 ** ((bits & np.uint64(31)).astype(np.float64) - 12)
    # exact ties between two bf16 values, both parities
    ties = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(2.0 + 2 ** -7), 3.0 + 2 ** -7 * 1.5])
    x = np.concatenate([x, ties])
    got = inputs.f64_to_bf16_bits(x)
    for xi, gi in zip(x, got):
        assert int(gi) == _nearest_bf16_brute(float(xi)), (xi, hex(int(gi)))


def test_bf16_specials_and_widening():
    x = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e39, 3.0])
    b = inputs.f64_to_bf16_bits(x)
    assert b[0] == 0x0000 and b[1] == 0x8000
    assert b[2] == 0x7F80 and b[3] == 0xFF80 and b[5] == 0x7F80
    assert b[4] & 0x7F80 == 0x7F80 and b[4] & 0x7F
    assert b[6] == 0x4040
    assert inputs.bf16_bits_to_f64(np.array([0x4040], np.uint16))[0] == 3.0


def test_normals_moments_and_std():
    z = inputs.bf16_bits_to_f64(inputs.normal_bf16(9, 400000, std=3.0))
    assert abs(z.mean()) < 0.03
    assert abs(z.std() - 3.0) < 0.03
    # deterministic and independent of the thread count
    a = inputs.normal_bf16(9, 1 << 23, threads=1)
    b = inputs.normal_bf16(9, 1 << 23, threads=4)
    assert (a == b).all()


def test_uniform_ints_bounds():
    v = inputs.uniform_ints(3, 10000, 512, 16384)
    assert v.min() >= 512 and v.max() <= 16384
    assert v.min() < 1000 and v.max() > 15800


def test_workload_shapes_and_flops():
    w = inputs.config_workload("tiny")
    assert w.q.shape == (256, 1, 64) and w.tokens == 256 and not w.causal
    assert w.flops() == 4 * 256 * 256 * 64
    assert w.q.dtype == np.uint16
    lens = inputs.varlen_lengths(inputs.CONFIG_SEED_BASE + 4, 16, 512, 16384)
    assert len(lens) == 16 and lens.min() >= 512 and lens.max() <= 16384


def test_sample_rows_holds_tile_edges():
    cu = np.array([0, 100, 300, 301])
    rows = inputs.sample_rows(cu, 2, 500, seed=1)
    s = {tuple(r) for r in rows.tolist()}
    for h in range(2):
        assert (0, h, 0) in s and (0, h, 99) in s
        for r in (0, 127, 128, 199):
            assert (1, h, r) in s
        assert (2, h, 0) in s
    assert len(rows) >= 400
    assert (rows[:, 2] < np.diff(cu)[rows[:, 0]]).all()
