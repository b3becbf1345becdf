"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of oracle.c (a transposed operand, a
wrong sign, an index shifted by one, a dropped term, a wrong tie-break),
compiles it on the CPU and runs the oracle pin suites against it in a fresh
process; the suites must fail.  The real oracle is untouched.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTATIONS = {
    "accept_test_transposed": ("if (uj * qxv[n] < pxv[n]) ++n;", "if (uj * pxv[n] < qxv[n]) ++n;"),
    "residual_sign_flipped": ("double d = p[v] - q[v];", "double d = q[v] - p[v];"),
    "bonus_uses_residual_slot": ("w[v] = p[v];\n    return gamma + 1;", "w[v] = p[v];\n    return gamma;"),
    "emitted_row_shifted": ("row_softmax(target, dtype, ((int64_t)b * G1 + n) * V, V, T, p);\n"
                            "    if (n < ell)",
                            "row_softmax(target, dtype, ((int64_t)b * G1 + (n > 0 ? n - 1 : 0)) * V, V, T, p);\n"
                            "    if (n < ell)"),
    "residual_draft_row_shifted": ("row_softmax(draft, dtype, ((int64_t)b * gamma + n) * V, V, T, q);\n"
                                   "        double W",
                                   "row_softmax(draft, dtype, ((int64_t)b * gamma + (n > 0 ? n - 1 : 0)) * V, V, T, q);\n"
                                   "        double W"),
    "draw_cdf_edge_shifted": ("lo[i] = cum[t] / W;", "lo[i] = cum[t > 0 ? t - 1 : 0] / W;"),
    "temperature_ignored": ("double y = logit_at(base, dtype, off + v) / T;",
                            "double y = logit_at(base, dtype, off + v) / 1.0;"),
    "softmax_not_normalised": ("for (int v = 0; v < V; ++v) p[v] = p[v] / S;",
                               "for (int v = 0; v < V; ++v) p[v] = p[v] / 1.0;"),
    "cdf_test_not_strict": ("if (cum > target) {", "if (cum >= target) {"),
    "cdf_target_unscaled": ("double target = u * W;", "double target = u;"),
    "greedy_ties_to_highest": ("if (!have || z > m) { m = z; a = v; have = 1; }",
                               "if (!have || z >= m) { m = z; a = v; have = 1; }"),
    "sched_ties_deep_first": ("if (a->k != c->k) return a->k < c->k ? -1 : 1;",
                              "if (a->k != c->k) return a->k > c->k ? -1 : 1;"),
    "survival_index_shifted": ("sb[k - 1] * calibrated(conf[(int64_t)b * gamma + k - 1], g_sts_T, k);",
                               "sb[k - 1] * calibrated(conf[(int64_t)b * gamma + (k > 1 ? k - 2 : 0)], g_sts_T, k);"),
    "cost_slope_sign": ("return kc[i] + ((N - kt[i]) * (kc[i + 1] - kc[i])) / (kt[i + 1] - kt[i]);",
                        "return kc[i] + ((N - kt[i]) * (kc[i + 1] + kc[i])) / (kt[i + 1] - kt[i]);"),
    "exact_last_max": ("if (obj > best) { best = obj; bestK = i + 1; }",
                       "if (obj >= best) { best = obj; bestK = i + 1; }"),
    "alg1_no_revert": ("out_len[r] = c[i].k - 1; /* early stop", "/* early stop"),
    "dcut_floor_budget": ("double K = ceil(ratios[i] * Nmax);", "double K = floor(ratios[i] * Nmax);"),
    "dcut_last_max": ("        if (obj > best) {\n            best = obj;\n            choice = i;",
                      "        if (obj >= best) {\n            best = obj;\n            choice = i;"),
    "threshold_strict": ("g_sts_T, n + 1) >= threshold) ++n;", "g_sts_T, n + 1) > threshold) ++n;"),
    "ece_no_abs": ("for (int k = 0; k < bins; ++k) e += fabs(sa[k] - sy[k]);",
                   "for (int k = 0; k < bins; ++k) e += sa[k] - sy[k];"),
    "pack_rows_inclusive": ("        target_row[b] = t;\n        draft_row[b] = d;\n        const int ell = verify_len[b];\n        if (ell >= 0 && ell <= gamma) {\n            t += ell + 1;\n            d += ell;\n        }",
                            "        const int ell = verify_len[b];\n        if (ell >= 0 && ell <= gamma) {\n            t += ell + 1;\n            d += ell;\n        }\n        target_row[b] = t;\n        draft_row[b] = d;"),
    "progress_coarse": ("#define PROG_FRAC_BITS 46", "#define PROG_FRAC_BITS 30"),
    "progress_coarser": ("#define PROG_FRAC_BITS 46", "#define PROG_FRAC_BITS 20"),
    "sts_power_inverted": ("a[i] = prefix[i] * pow((double)conf[(int64_t)i * gamma + k - 1], 1.0 / T);",
                           "a[i] = prefix[i] * pow((double)conf[(int64_t)i * gamma + k - 1], T);"),
}


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c99", "-ffp-contract=off",
                           "-o", str(lib), str(mutated), "-lm"])
    env = dict(os.environ, SPECV_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_verify.py"),
                        os.path.join(ROOT, "tests", "test_oracle_sched.py"),
                        os.path.join(ROOT, "tests", "test_oracle_sched_ext.py"),
                        os.path.join(ROOT, "tests", "test_oracle_pack.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutation {name}:\n{r.stdout[-2000:]}"
