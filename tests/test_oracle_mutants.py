"""Deliberately broken copies of the oracle must each fail at least one pin.

Each mutant is a plausible slip (a dropped term, a flipped sign, a wrong
index or operand) planted in a temporary copy of the oracle's C source on
the CPU; the oracle itself is never modified.  This shows the pins in
``oracle_pins.py`` are strong enough to catch such slips.
"""
import os
import shutil
import tempfile

import pytest

import oracle
from oracle import build as oracle_build
import oracle_pins

MUTANTS = [
    ("logp_sign", "logp[t] = (y >= 0) ? z[y] - L : NAN;", "logp[t] = (y >= 0) ? z[y] + L : NAN;"),
    ("entropy_sign", "*ent_out = lse - spz;", "*ent_out = spz - lse;"),
    ("max_dropped", "double lse = m + log(s);", "double lse = log(s);"),
    ("max_and_sum_swapped", "double lse = m + log(s);", "double lse = s + log(m > 0 ? m : -m);"),
    ("temperature_multiplies", "z[v] = dot_with_row(h, w, w_bf16, v, H) / tau;",
     "z[v] = dot_with_row(h, w, w_bf16, v, H) * tau;"),
    ("unnormalised_p_in_entropy", "spz += exp(z[v] - lse) * z[v];", "spz += exp(z[v] - m) * z[v];"),
    ("no_negative_wrap", "if (yy < 0) yy += V;", ""),
    ("vocab_bound_off_by_one", "(yy >= 0 && yy < V)", "(yy >= 0 && yy < V - 1)"),
    ("cotangent_sign", "double dz = gl * (onehot - p) - ge * p * (z[v] - L + E);",
     "double dz = gl * (p - onehot) - ge * p * (z[v] - L + E);"),
    ("entropy_cotangent_sign", "double dz = gl * (onehot - p) - ge * p * (z[v] - L + E);",
     "double dz = gl * (onehot - p) + ge * p * (z[v] - L + E);"),
    ("entropy_cotangent_term", "double dz = gl * (onehot - p) - ge * p * (z[v] - L + E);",
     "double dz = gl * (onehot - p) - ge * p * (z[v] - L - E);"),
    ("dweight_stats_swapped", "double p = exp(z - lse_t[t]);", "double p = exp(z - ent_t[t]);"),
    ("dhidden_tau_dropped", "dh[k] += c * wrow[k];", "dh[k] += dz * wrow[k];"),
    ("dweight_tau_dropped", "for (int32_t k = 0; k < H; ++k) dw[k] += c * h[k];",
     "for (int32_t k = 0; k < H; ++k) dw[k] += dz * h[k];"),
    ("dweight_unwrapped_target", "int64_t y = wrapped_target(targets[t], V);\n        double onehot",
     "int64_t y = targets[t];\n        double onehot"),
    ("dhidden_wrong_row", "load_row(weight, weight_bf16, v, H, wrow);",
     "load_row(weight, weight_bf16, (v + 1) % V, H, wrow);"),
    ("dweight_transposed_h", "dw[k] += c * h[k];", "dw[k] += c * hrows[k * T + t];"),
    ("mask_ignored_fwd", "if (mask && !mask[t]) {\n        logp[t] = 0.0;", "if (0) {\n        logp[t] = 0.0;"),
    ("bf16_decode_shift", "(uint32_t)bits << 16;", "(uint32_t)bits << 15;"),
    ("logits_isfinite_mask_dropped", "        if (!isfinite(z[v])) continue;          /* isfinite mask */\n", ""),
    ("logits_posinf_treated_as_finite", "if (isnan(z[v]) || (isinf(z[v]) && z[v] > 0)) return 1;",
     "if (isnan(z[v])) return 1;"),
    ("logits_neg_inf_counted_in_sum", "    if (isfinite(z[v])) s += exp(z[v] - m);",
     "    s += isfinite(z[v]) ? exp(z[v] - m) : exp(-1.0);"),
    ("logits_tau_dropped_in_grad", "        dz[v] = (gl * (onehot - p) - ge * p * (z[v] - L + E)) / tau;",
     "        dz[v] = (gl * (onehot - p) - ge * p * (z[v] - L + E));"),
    ("logits_empty_row_entropy_zero", "    *lse_out = -INFINITY;\n    *ent_out = NAN;", "    *lse_out = -INFINITY;\n    *ent_out = 0.0;"),
]


def _fails_some_pin(o):
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError, FloatingPointError, IndexError):
            return pin.__name__
    return None


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, find, repl):
    src = open(oracle_build.SOURCE).read()
    assert src.count(find) >= 1, "mutation site for %s not found" % name
    tmp = tempfile.mkdtemp(prefix="lmo_mutant_")
    try:
        path = os.path.join(tmp, "m.c")
        with open(path, "w") as f:
            f.write(src.replace(find, repl, 1))
        lib = oracle_build.build(force=True, source=path, output=os.path.join(tmp, "libm.so"))
        caught = _fails_some_pin(oracle.Oracle(lib))
        assert caught is not None, "mutant %s passed every pin" % name
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
