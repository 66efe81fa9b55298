"""Each planted mistake in a copy of the oracle must fail at least one pin.

The copies are built on the CPU in a temporary folder from ``oracle/oracle.c``
with one textual change each; the committed oracle is never modified.  This
shows the pins in tests/oracle_pins.py are strong enough to catch a dropped
term, a wrong sign or index, a transposed operand, a misread layout.
"""
import os
import subprocess

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "drop_scale": [("srow[j - jlo] = jb->scale * dot;", "srow[j - jlo] = dot;")],
    "no_normalise": [("const double p = exp(srow[j] - m) / l;", "const double p = exp(srow[j] - m);")],
    "lse_without_max": [("jb->lse[r] = nvis > 0 ? m + log(l)", "jb->lse[r] = nvis > 0 ? log(l)")],
    "lse_sign": [("jb->lse[r] = nvis > 0 ? m + log(l)", "jb->lse[r] = nvis > 0 ? m - log(l)")],
    "v_read_from_k": [("const uint16_t *vj = jb->v + ", "const uint16_t *vj = jb->k + ")],
    "causal_ignored": [("int64_t jlo = 0, jhi = jb->causal ? i + 1 : L;",
                        "int64_t jlo = 0, jhi = L;")],
    "causal_excludes_diagonal": [("int64_t jlo = 0, jhi = jb->causal ? i + 1 : L;",
                                  "int64_t jlo = 0, jhi = jb->causal ? (i > 0 ? i : 1) : L;")],
    "window_left_off_by_one": [("            jlo = i - jb->wl;", "            jlo = i - jb->wl + 1;")],
    "window_right_ignored": [("            jhi = i + jb->wr + 1;", "            jhi = jhi;")],
    "window_v_not_shifted": [("((base + jlo + j) * H + h)", "((base + j) * H + h)")],
    "k_wrong_head": [("const uint16_t *kj = jb->k + ((base + j) * H + h)",
                      "const uint16_t *kj = jb->k + ((base + j) * H + 0)")],
    "transposed_scores": [("const uint16_t *qi = jb->q + ((base + i) * H + h) * (int64_t)d;",
                           "const uint16_t *qi = jb->k + ((base + i) * H + h) * (int64_t)d;"),
                          ("const uint16_t *kj = jb->k + ((base + j) * H + h) * (int64_t)d;\n            double dot",
                           "const uint16_t *kj = jb->q + ((base + j) * H + h) * (int64_t)d;\n            double dot")],
    "sequence_base_ignored": [("const uint16_t *vj = jb->v + ((base + jlo + j)", "const uint16_t *vj = jb->v + ((jlo + j)")],
    "short_dot": [("for (int c = 0; c < d; ++c)\n                dot += qrow[c]",
                   "for (int c = 0; c < d - 1; ++c)\n                dot += qrow[c]")],
    "exp_sign": [("l += exp(srow[j] - m);", "l += exp(m - srow[j]);")],
    "bad_widening": [("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;")],
    "max_over_first_key_only": [("if (srow[j] > m)\n                m = srow[j];",
                                 "if (j == 0)\n                m = srow[j];")],
    # gradients
    "bwd_dq_drops_scale": [("dqi[c] += jb->scale * ds * widen_bf16(kr[c]);",
                            "dqi[c] += ds * widen_bf16(kr[c]);")],
    "bwd_no_rowsum_term": [("const double ds = p[j] * (dp[j] - D);", "const double ds = p[j] * dp[j];")],
    "bwd_dk_from_k": [("dkr[c] += jb->scale * ds * qf[c];",
                       "dkr[c] += jb->scale * ds * widen_bf16(kr[c]);")],
    "bwd_dv_from_ds": [("dvr[c] += p[j] * dorow[c];", "dvr[c] += ds * dorow[c];")],
    "bwd_causal_ignored": [("int64_t klo = 0, khi = jb->causal ? i + 1 : L;", "int64_t klo = 0, khi = L;")],
    "bwd_window_dk_not_shifted": [("double *dkr = jb->dk + (klo + j) * (int64_t)d;", "double *dkr = jb->dk + j * (int64_t)d;")],
    "bwd_window_right_ignored": [("            khi = i + jb->wr + 1;", "            khi = khi;")],
    "bwd_dp_from_k": [("acc += dorow[c] * widen_bf16(vr[c]);",
                       "acc += dorow[c] * widen_bf16(jb->k[((base + j) * H + h) * (int64_t)d + c]);")],
    "bwd_unnormalised_p": [("p[j] = exp(p[j] - m) / l;\n        /* dP_ij", "p[j] = exp(p[j] - m);\n        /* dP_ij")],
    "bwd_one_worker_summed": [("sk += jobs[t].dk[x];", "sk = jobs[t].dk[x];")],
    # FP8
    "e4m3_ties_away": [("if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) == 1.0))",
                        "if (frac >= 0.5)")],
    "e4m3_no_saturation": [("    if (a >= 448.0)\n        return sign | 0x7e;", "    if (a >= 480.0)\n        return sign | 0x7f;")],
    "e4m3_bias_off_by_one": [("double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);",
                              "double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 9);")],
    "fwht_last_stage_skipped": [("for (int h = 1; h < d; h <<= 1)", "for (int h = 1; h < d / 2; h <<= 1)")],
    "fwht_signs_ignored": [("x[c] = signs[c] < 0 ? -x[c] : x[c];", "x[c] = x[c];")],
    "quant_scale_inverted": [("const float inv = amax > 0.0f ? 448.0f / amax : 1.0f;",
                              "const float inv = amax > 0.0f ? amax / 448.0f : 1.0f;")],
    "quant_tail_overwrites_shared_rows": [("if (row < nominal || row < 0)", "if (row < 0)")],
    "tensor_scale_from_first_token": [("        for (int64_t t = 0; t < tokens; ++t)\n            for (int c = 0; c < d; ++c) {\n                const float y",
                                       "        for (int64_t t = 0; t < 1; ++t)\n            for (int c = 0; c < d; ++c) {\n                const float y")],
    "tensor_scale_inverted": [("const float inv_t = amax > 0.0f ? 448.0f / amax : 1.0f;",
                               "const float inv_t = amax > 0.0f ? amax / 448.0f : 1.0f;")],
    "tensor_reads_next_column": [("codes[at] = oracle_e4m3_encode((float)widen_bf16(x[at]) * inv_t);",
                           "codes[at] = oracle_e4m3_encode((float)widen_bf16(x[at - c + (c ^ 1)]) * inv_t);")],
    "attn_f64_no_max": [("            if (sc[j] > mx)\n                mx = sc[j];\n        }\n        double z",
                         "            if (j == 0)\n                mx = sc[j];\n        }\n        double z")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(SRC).read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation anchor not unique or missing: {old!r}"
        src = src.replace(old, new)
    path = tmp_path / "oracle_mutant.c"
    path.write_text(src)
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-pthread", str(path), "-o", str(lib), "-lm"], check=True)
    mutant = oracle.Oracle(str(lib))
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(mutant)
        except (AssertionError, ValueError) as e:
            caught.append((check.__name__, str(e)[:80]))
            break
    assert caught, f"mutant {name} passed every pin"
