"""The oracle's pins must catch plausible mistakes.

Each case copies the oracle's C source, plants one mistake (a dropped term, a
wrong sign, an off-by-one index, a swapped operand...), compiles the copy with
gcc and runs the pin suite against it in a subprocess.  The pin suite must
fail for every planted mistake.  Everything here runs on the CPU.
"""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "hyb_oracle.c")

# (name, original text, mistaken text)
MUTATIONS = [
    ("stream_b_dropped", "logit[np] = load_elem(dtype, zb, off) + (double)bias[p * c + ch];", "logit[np] = -INFINITY;"),
    ("stream_b_wrong_block", "int64_t row = (lb - 1) * m + p;", "int64_t row = lb * m + p;"),
    ("stream_a_bias_position", "          int64_t pos = overlap ? m + p : p;\n          logit[np] = load_elem(dtype, za",
     "          int64_t pos = p;\n          logit[np] = load_elem(dtype, za"),
    ("softmax_denominator", "          den += e;\n", "          den += 1.0;\n"),
    ("relu_dropped", "double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    ("head_weight_dropped", "acc += (double)w[(b * n_q + j) * n_ih + h] * relu;", "acc += relu;"),
    ("query_scale_dropped", "* c_I + d) * sq;", "* c_I + d);"),
    ("key_scale_dropped", "(b * N + s) * c_I + d) * sk;", "(b * N + s) * c_I + d);"),
    ("visibility_off_by_one", "return (t + 1) / m;", "return (t + 2) / m;"),
    ("topk_ignores_visibility", "int64_t v = visible[r] < N ? visible[r] : N;", "int64_t v = N;"),
    ("tie_rule_reversed", "return (x->index < y->index) ? -1 : (x->index > y->index);",
     "return (x->index > y->index) ? -1 : (x->index < y->index);"),
    ("softmax_scale_dropped", "sc[e] = dot * scale;", "sc[e] = dot;"),
    ("lse_missing_log_term", "*lse = mx + log(den);", "*lse = mx;"),
    ("merge_weight_sign", "if (a != -INFINITY) v += exp(a - L) * o_in[qo + d];",
     "if (a != -INFINITY) v += exp(L - a) * o_in[qo + d];"),
    ("window_off_by_one", "return t + 1 < n_win ? t + 1 : n_win;", "return t + 1 < n_win ? t + 1 : n_win - 1;"),
    ("hca_visibility_shifted", "int64_t vis = orc_visible(q_pos0 + j, m);\n      if (vis > N) vis = N;",
     "int64_t vis = orc_visible(q_pos0 + j + 1, m);\n      if (vis > N) vis = N;"),
    ("e4m3_exponent_bias", "mag = ldexp(1.0 + (double)mant / 8.0, e - 7);", "mag = ldexp(1.0 + (double)mant / 8.0, e - 8);"),
    ("quantiser_range", "amax / 448.0f", "amax / 240.0f"),
    ("bf16_rounding_width", "int q = e - 8; ", "int q = e - 9; "),
    ("key_value_swapped", "o_h[d] += p * load_elem(kv_dtype, v,", "o_h[d] += p * load_elem(kv_dtype, k,"),
    ("rmsnorm_sum_not_mean", "double inv = 1.0 / sqrt(ss / (double)c + eps);", "double inv = 1.0 / sqrt(ss + eps);"),
    ("rmsnorm_eps_outside_root", "double inv = 1.0 / sqrt(ss / (double)c + eps);",
     "double inv = 1.0 / (sqrt(ss / (double)c) + eps);"),
    ("rmsnorm_gain_dropped", "y[r * c + d] = x[r * c + d] * inv * (gamma ? gamma[d] : 1.0);",
     "y[r * c + d] = x[r * c + d] * inv;"),
    ("rope_frequency_exponent", "double freq = pow(theta, -(double)(2 * i) / (double)rope_dims);",
     "double freq = pow(theta, -(double)i / (double)rope_dims);"),
    ("rope_rotation_sign", "y[r * c + d0 + 2 * i + 1] = re * sin(ang) + im * cos(ang);",
     "y[r * c + d0 + 2 * i + 1] = -re * sin(ang) + im * cos(ang);"),
    ("rope_whole_row", "int64_t d0 = c - rope_dims;", "int64_t d0 = 0;"),
    ("sink_weight_inverted", "double w = (a == -INFINITY) ? 0.0 : exp(a - L);",
     "double w = (a == -INFINITY) ? 0.0 : exp(L - a);"),
    ("sink_ignored_in_lse", "        L = mx + log(exp(a - mx) + exp(s - mx));\n      }\n      double w",
     "        L = a;\n      }\n      double w"),
    ("grouped_proj_wrong_group_input", "o[r * n_h * c + j * in_g + d]", "o[r * n_h * c + d]"),
    ("grouped_proj_transposed_weight", "W[(j * d_g + e) * in_g + d]", "W[(j * in_g + d) * d_g + e]"),
    ("e2m1_exponent_bias", "ldexp(1.0 + 0.5 * (double)mant, e - 1)", "ldexp(1.0 + 0.5 * (double)mant, e - 2)"),
    ("mxfp4_shared_exponent_offset", "E = (e - 1) - 2;", "E = (e - 1) - 1;"),
    ("e2m1_ties_to_odd", "if (err < best_err || (err == best_err && (code & 1) == 0)) {\n      best = code;\n      best_err = err;\n    }\n  }\n  if (ax > 6.0)",
     "if (err < best_err || (err == best_err && (code & 1) == 1)) {\n      best = code;\n      best_err = err;\n    }\n  }\n  if (ax > 6.0)"),
]


def _run_mutant(name, old, new, workdir):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"{name}: pattern not found in the oracle source"
    mutant_src = os.path.join(workdir, f"{name}.c")
    with open(mutant_src, "w") as f:
        f.write(src.replace(old, new, 1))
    lib = os.path.join(workdir, f"lib{name}.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o", lib, mutant_src, "-lm"],
                   check=True, capture_output=True)
    env = dict(os.environ, HYB_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-W", "ignore",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    return name, r.returncode


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as d:
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            results = list(ex.map(lambda m: _run_mutant(*m, d), MUTATIONS))
    survivors = [name for name, rc in results if rc == 0]
    assert not survivors, f"planted mistakes not caught by any pin: {survivors}"
