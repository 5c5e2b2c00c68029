"""Planted mistakes in a copy of the oracle must each fail the pin suite.

Each mutant rewrites one spot of oracle.cpp in a temporary copy (never the tracked file),
builds it with the same flags, and runs tests/test_oracle_pins.py against it in a fresh
process.  A mutant that passes every pin would mean the pins cannot see that mistake.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

MUTANTS = {
    "adagrad_sign": ("(double)w[c] - m->lr * g[c] / denom", "(double)w[c] + m->lr * g[c] / denom"),
    "eps_inside_sqrt": ("const double denom = std::sqrt(acc_new) + m->eps;\n        const double w_new",
                        "const double denom = std::sqrt(acc_new + m->eps);\n        const double w_new"),
    "old_accumulator": ("const double denom = std::sqrt(acc_new) + m->eps;\n        const double w_new",
                        "const double denom = std::sqrt((double)a[c]) + m->eps;\n        const double w_new"),
    "mean_scale_dropped": ("(m->mean && L > 0) ? 1.0 / (double)L : 1.0", "1.0"),
    "rowwise_sum_not_mean": ("sq / (double)D", "sq"),
    "last_vector_dropped": ("for (int i = 1; i < F; ++i) {\n      for (int j = 0; j < i; ++j) {\n        double s = 0.0, a = 0.0;",
                            "for (int i = 1; i < F - 1; ++i) {\n      for (int j = 0; j < i; ++j) {\n        double s = 0.0, a = 0.0;"),
    "pair_order_column_major": ("out[b * W + D + p] = s;", "out[b * W + D + (i * (i - 1) / 2 + j == p ? (p % 2 ? p - 1 : p + 1 < P ? p + 1 : p) : p)] = s;"),
    "backward_one_triangle": ("        G[(size_t)j * F + i] = dout[b * W + D + p];\n", ""),
    "passthrough_dropped": ("d_dense[b * D + k] = s + (double)dout[b * W + k];", "d_dense[b * D + k] = s;"),
    "bf16_round_half_up": ("b += 0x7FFFu + lsb;", "b += 0x8000u;"),
    "splitmix_constant": ("0xBF58476D1CE4E5B9ull", "0xBF58476D1CE4E5B7ull"),
    "init_shift": ("(uint32_t)(z >> 40)", "(uint32_t)(z >> 41)"),
    "hash_init_value": ("float v = hashed ? hash_init :", "float v = hashed ? hash_init + 1.0f :"),
    "id_range_off_by_one": ("id >= m->rows[t]", "id > m->rows[t]"),
    "admission_strict": ("m->freq[r] < m->admit_min", "m->freq[r] <= m->admit_min"),
    "admission_counts_steps": ("m->freq[r] += lookups[kv.first];", "m->freq[r] += 1;"),
    "decay_after_gradient": ("(double)a[c] * f + g[c] * g[c]", "((double)a[c] + g[c] * g[c]) * f"),
    "decay_period_off_by_one": ("(m->step - 1) / m->decay_period", "m->step / m->decay_period"),
    "cross_dxl_without_dout": ("dxl[r * K + k] = g + (double)w[k] * t;", "dxl[r * K + k] = (double)w[k] * t;"),
    "cross_scalar_from_x0": ("s += (double)xl[r * K + k] * w[k];", "s += (double)x0[r * K + k] * w[k];"),
    "codec_levels": ("const float s = amax / 127.0f;", "const float s = amax / 128.0f;"),
    "codec_round_half_away": ("std::nearbyint(row[c] / s)", "std::round(row[c] / s)"),
    "eviction_idle_inclusive": ("m->step - m->last_step[r] > (int64_t)max_idle",
                                "m->step - m->last_step[r] >= (int64_t)max_idle"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    if shutil.which("g++") is None:
        pytest.skip("g++ not available")
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site of {name} not found"
    mutated = src.replace(old, new, 1)
    cpp = tmp_path / "oracle_mutant.cpp"
    so = tmp_path / "liboracle_mutant.so"
    cpp.write_text(mutated)
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-ffp-contract=off",
                           "-o", str(so), str(cpp)])
    env = dict(os.environ, ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
