"""The oracle's pins are strong enough to catch plausible mistakes (no GPU).

Each case plants one mistake in a private copy of the oracle's C source (a
dropped term, a flipped sign, an off-by-one index, a wrong tie rule, a
transposed operand), builds it, and runs the oracle pin suite against it in a
subprocess.  The suite must fail for every mutant.  Nothing here touches the
real oracle build or any GPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mac_oracle.c")
PINS = ["test_oracle_closed_forms.py", "test_oracle_algebra.py", "test_oracle_match.py",
        "test_oracle_bruteforce.py", "test_oracle_invariants.py"]

MUTANTS = {
    "merge_weight_sign": ("double wa = exp(la - lse), wb = exp(lb - lse);",
                          "double wa = exp(lse - la), wb = exp(lb - lse);"),
    "merge_lse_dropped_max": ("double lse = mx + log(exp(la - mx) + exp(lb - mx));",
                              "double lse = log(exp(la - mx) + exp(lb - mx));"),
    "removal_sign": ("o[i] = (oab[i] - w * ob[i]) / one_minus_w;",
                     "o[i] = (oab[i] + w * ob[i]) / one_minus_w;"),
    "removal_lse_sign": ("*l = lab + orc_log1mexp(delta);", "*l = lab - orc_log1mexp(delta);"),
    "log1mexp_branch": ("if (x > -0.6931471805599453) return log(-expm1(x));",
                        "if (x > -0.6931471805599453) return log(expm1(-x));"),
    "tie_to_oldest": ("(De == bestD && ring_pos[e] > bestPos)", "(De == bestD && ring_pos[e] < bestPos)"),
    "threshold_not_strict": ("(bestD < tau * tau * n2)", "(bestD <= tau * tau * n2)"),
    "threshold_absolute": ("(bestD < tau * tau * n2)", "(bestD < tau * tau)"),
    "band_tail_off_by_one": ("lo = p - r > 0 ? p - r : 0;", "lo = p - r + 1 > 0 ? p - r + 1 : 0;"),
    "amend_band_off_by_one": ("orc_attention_summary(q, Kh, Vh, row, m - r, m, d, s->scale, ob, &lb);",
                              "orc_attention_summary(q, Kh, Vh, row, m - r + 1, m, d, s->scale, ob, &lb);"),
    "scale_dropped": ("z[j - lo] = scale * dot;", "z[j - lo] = dot;"),
    "values_from_keys": ("const uint16_t *v = V + j * tok_stride;", "const uint16_t *v = K + j * tok_stride;"),
    "ring_slot_shift": ("const long slot_new = (long)(s->step[b] % L);",
                        "const long slot_new = (long)((s->step[b] + 1) % L);"),
    "kv_head_index": ("g = h / G;\n        if (h < h_lo", "g = h % s->Hkv;\n        if (h < h_lo"),
    "direct_miss_range_to_m": ("orc_attention_summary(q, Kh, Vh, row, 0, m - r, d, s->scale, oe, &le);",
                               "orc_attention_summary(q, Kh, Vh, row, 0, m, d, s->scale, oe, &le);"),
    "direct_hit_range_to_m": ("orc_attention_summary(q, Kh, Vh, row, lo, m - r, d, s->scale, ot, &lt);",
                              "orc_attention_summary(q, Kh, Vh, row, lo, m, d, s->scale, ot, &lt);"),
    "direct_hit_range_from_0": ("orc_attention_summary(q, Kh, Vh, row, lo, m - r, d, s->scale, ot, &lt);",
                                "orc_attention_summary(q, Kh, Vh, row, 0, m - r, d, s->scale, ot, &lt);"),
    "direct_hit_prefix_dropped": ("orc_merge(s->ring_o + (ring_base + e) * d, s->ring_lse[ring_base + e], ot, lt, d, oe, &le);",
                                  "memcpy(oe, ot, (size_t)d * sizeof(double)); le = lt;"),
    "direct_form_never_taken": ("if (cond < 0x1p-20) {", "if (cond < 0.0) {"),
    "reuse_prefix_dropped": ("orc_merge(s->ring_o + (ring_base + e) * d, s->ring_lse[ring_base + e], ot, lt, d, o, &l);",
                             "memcpy(o, ot, (size_t)d * sizeof(double)); l = lt;"),
}


def _build_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-o",
                    str(lib), str(path), "-lm"], check=True)
    return lib


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_the_mutant(name, tmp_path):
    lib = _build_mutant(name, tmp_path)
    env = dict(os.environ, MAC_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *[os.path.join(ROOT, "tests", p) for p in PINS]],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pin suite:\n{r.stdout[-2000:]}"
