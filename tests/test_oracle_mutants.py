"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a temporary copy of the oracle's C source
(never in the real one), builds it on the CPU, and runs the oracle pin suite
against that build in a subprocess: the suite must fail.  The mistakes are the
kinds a hand-written oracle can plausibly contain: a dropped term, a wrong
sign, a transposed operand, a wrong index, a broken tie-break or stability
rule, an off-by-one in the capacity rule, a wrong normaliser.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

MUTANTS = {
    "drop_shared_term": ("            acc[i] += y[i];\n    }\n    store_row(out_t",
                         "            acc[i] += 0.0 * y[i];\n    }\n    store_row(out_t"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "down_transposed": ("wval(Wd, dtype, i, n, F)", "wval(Wd, dtype, n, i, d)"),
    "gate_up_swapped": ("double hv = silu(g) * u;", "double hv = silu(u) * g;"),
    "wrong_slot_weight": ("acc[i] += (double)w_t[j] * y[i];", "acc[i] += (double)w_t[0] * y[i];"),
    "ties_to_higher_index": ("if (!chosen[e] && (best < 0 || sel[e] > sel[best]))",
                             "if (!chosen[e] && (best < 0 || sel[e] >= sel[best]))"),
    "no_renorm": ("w[j] = renorm ? (float)((double)probs[idx[j]] / ws) : probs[idx[j]];",
                  "w[j] = probs[idx[j]];"),
    "unstable_segments": ("perm[offsets[e] + r] = (int32_t)f;",
                          "perm[offsets[e + 1] - 1 - r] = (int32_t)f;"),
    "capacity_off_by_one": ("pos[f] = (r < kept[e]) ? kept_offsets[e] + r : -1;",
                            "pos[f] = (r <= kept[e] && r < counts[e] - 1) ? kept_offsets[e] + r : -1;"),
    "f_over_N": ("f[e] /= (double)(N * k);", "f[e] /= (double)N;"),
    "router_bias_ignored": ("double acc = (b_r && bias_mode == 1) ? (double)b_r[e] : 0.0;",
                            "double acc = 0.0;"),
    "selection_bias_ignored": ("sel[e] = (b_r && bias_mode == 2) ? (float)((double)probs[e] + (double)b_r[e]) : probs[e];",
                               "sel[e] = probs[e];"),
    "selection_bias_in_weights": ("ws += (double)probs[idx[j]];", "ws += (double)sel[idx[j]];"),
    "w4_nibble_order": ("int nib = (col & 1) ? (byte >> 4) : (byte & 15);",
                        "int nib = (col & 1) ? (byte & 15) : (byte >> 4);"),
    "w4_unsigned_codes": ("int code = nib >= 8 ? nib - 16 : nib;", "int code = nib;"),
    "w4_scale_over_8": ("float sc = mx / 7.0f;", "float sc = mx / 8.0f;"),
    "w4_round_half_away": ("float t = nearbyintf(v / sc);", "float t = roundf(v / sc);"),
    "w4_pack_swapped": ("if (col & 1)", "if (!(col & 1))"),
    "w4_first_group_scale": ("m->s[(col / ORC_W4_GROUP) * m->rows + row]", "m->s[row]"),
    "w4_scales_row_major": ("s[(int64_t)g * rows + r] = sc;", "s[r * groups + g] = sc;"),
    "z_mean_of_lse": ("z += lse[t] * lse[t];", "z += lse[t];"),
    "importance_counts": ("imp[idx[f]] += (double)w[f];", "imp[idx[f]] += 1.0;"),
    "cv2_sample_variance": ("    var /= (double)E;", "    var /= (double)(E - 1);"),
    "lse_without_max": ("*lse = mx + log(s);", "*lse = log(s);"),
    "bwd_silu_derivative": ("sg * (1.0 + g[n] * (1.0 - sg))", "sg"),
    "bwd_renorm_without_mean": ("(dw[j] - wdw) / ssel", "dw[j] / ssel"),
    "bwd_softmax_without_mean": ("(double)pt[e] * (dp[e] - pdp)", "(double)pt[e] * dp[e]"),
    "bwd_down_grad_transposed": ("dWd[(int64_t)i * F + n] += dy * h[n];",
                                 "dWd[(int64_t)n * d + i] += dy * h[n];"),
    "bwd_aux_without_E": ("aux_coef * (double)E * (counts[e] / (double)A) / (double)N",
                          "aux_coef * (counts[e] / (double)A) / (double)N"),
    "bwd_z_without_two": ("2.0 * z_coef / (double)N * lse[t]", "z_coef / (double)N * lse[t]"),
    "bwd_no_router_dx": ("                    dxt[i] += dl * (double)W_r[(int64_t)e * d + i];\n",
                         ""),
    "bwd_dropped_slots_pass": ("                if (!keep[t * k + j])\n                    continue;\n", ""),
    "logit_transposed": ("(int64_t)d + i) * (double)W_r[(int64_t)e * d + i]",
                         "(int64_t)d + i) * (double)W_r[(int64_t)i * E + e]"),
}


def _run_pins_against(source: str, tmp_path):
    mut_c = tmp_path / "copy.c"
    mut_c.write_text(source)
    so = tmp_path / "libcopy.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                           "-ffp-contract=off", "-o", str(so), str(mut_c), "-lm"])
    env = dict(os.environ, MOE_ORACLE_LIB=str(so), OMP_NUM_THREADS="2")
    tests = [os.path.join(ROOT, "tests", f) for f in
             ("test_oracle_route.py", "test_oracle_permute.py", "test_oracle_layer.py",
              "test_oracle_stats.py", "test_oracle_w4.py", "test_oracle_router_stats.py",
              "test_oracle_backward.py")]
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           *tests], env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)


def test_unmodified_copy_passes(tmp_path):
    """Control: the same harness on an unmodified copy passes, so a failure below is the
    planted mistake and not the harness."""
    r = _run_pins_against(open(SRC).read(), tmp_path)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    r = _run_pins_against(src.replace(old, new), tmp_path)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout or "error" in r.stdout.lower()
