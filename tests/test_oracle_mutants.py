"""Plant plausible mistakes in copies of the oracle source and check that the pins catch
every one of them (CPU only). Each planted copy is built in a temporary directory and its
pins run in a separate process, so a copy that corrupts memory cannot harm the test run."""
import json
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, original text, replacement, occurrences expected)
MUTANTS = [
    ("bias_on_C", "num += e * bf16_to_double(C[at]);",
     "num += e * (bf16_to_double(C[at]) + bias[static_cast<size_t>(t) * d + c]);", 1),
    ("rope_inverse_direction", "x[d0] = e * cs - o * sn;", "x[d0] = e * cs + o * sn;", 1),
    ("rope_frequency_exponent", "std::pow(theta, -2.0 * j / rope_dim)", "std::pow(theta, -1.0 * j / rope_dim)", 1),
    ("rope_pairs_split_halves", "const int d0 = d - rope_dim + 2 * j;",
     "const int d0 = d - rope_dim + j;", 1),
    ("rmsnorm_eps_outside_sqrt", "1.0 / std::sqrt(ms + eps)", "1.0 / (std::sqrt(ms) + eps)", 1),
    ("rmsnorm_sum_not_mean", "ms /= d;", "ms /= 1;", 1),
    ("bias_rows_reversed", "bias[static_cast<size_t>(t) * d + c]", "bias[static_cast<size_t>(ratio - 1 - t) * d + c]", 2),
    ("entry_position_unscaled", "pos0[s] + static_cast<int64_t>(b) * ratio", "pos0[s] + static_cast<int64_t>(b)", 1),
    ("score_no_relu", "std::max(0.0, dot)", "dot", 1),
    ("score_per_head_key", "bf16_to_double(k[i])", "bf16_to_double(k[(i + h) % Di])", 1),
    ("score_weight_dropped", "static_cast<double>(w[row * H + h]) * std::max(0.0, dot)", "std::max(0.0, dot)", 1),
    ("topk_ties_higher_index", "return a < b;", "return a > b;", 1),
    ("visibility_strict", "int64_t by_pos = (p + 1) / ratio;", "int64_t by_pos = p / ratio;", 1),
    ("sink_dropped", "double den = std::exp(sk - m);", "double den = 0.0;", 1),
    ("scale_dropped", "sc[r] = scale * dot;", "sc[r] = dot;", 1),
    ("window_off_by_one", "int64_t lo = hi - window + 1;", "int64_t lo = hi - window;", 1),
    ("window_wrong_end", "const int64_t hi = qa + win_len[b] - n_q_total;",
     "const int64_t hi = qa + win_len[b] - n_q_total - 1;", 1),
    ("bf16_truncates", "double r = std::nearbyint(scaled);", "double r = std::trunc(scaled);", 1),
    ("max_comp_floor", "return (max_context + ratio - 1) / ratio;", "return max_context / ratio;", 1),
    ("e4m3_round_half_up", "double q = std::nearbyint(std::ldexp(a, 3 - e));",
     "double q = std::floor(std::ldexp(a, 3 - e) + 0.5);", 1),
    ("e4m3_bias_6", "((e + 7) << 3)", "((e + 6) << 3)", 1),
    ("e4m3_no_saturation", "if (e > 8 || (e == 8 && q > 14.0))", "if (e > 8)", 1),
    ("e4m3_subnormal_spacing", "if (e < -6) e = -6;", "if (e < -7) e = -7;", 1),
    ("quant_scale_max_code", "amax / 448.0f", "amax / 240.0f", 1),
    ("kv_mixed_scale_max_code", "amax / 448.f", "amax / 240.f", 1),
    ("fp8_score_key_scale_dropped", "static_cast<double>(k_scale[kr]) * e4m3_to_double(keys[kr * Di + i])",
     "e4m3_to_double(keys[kr * Di + i])", 1),
    ("fp8_score_no_relu", "(dot > 0.0 ? dot : 0.0);   // ReLU", "dot;   // ReLU", 1),
    ("fp8_score_query_scale_dropped",
     "static_cast<double>(q_scale[row * H + h]) * e4m3_to_double(q[(row * H + h) * Di + i]);",
     "e4m3_to_double(q[(row * H + h) * Di + i]);", 1),
    ("kv_mixed_amax_includes_rope", "for (int i = 0; i < nd; ++i) amax = std::max(amax, std::fabs(xr[i]));",
     "for (int i = 0; i < dim; ++i) amax = std::max(amax, std::fabs(xr[i]));", 1),
    ("kv_mixed_dequant_scale_dropped",
     "static_cast<float>(e4m3_to_double(nope[static_cast<size_t>(r) * nd + i])) * scale[r];",
     "static_cast<float>(e4m3_to_double(nope[static_cast<size_t>(r) * nd + i]));", 1),
    ("kv_mixed_rope_from_first_dims", "double_to_bf16(static_cast<double>(xr[nd + i]))",
     "double_to_bf16(static_cast<double>(xr[i]))", 1),
    ("inverse_rope_forward_direction", "v[e0] = ev * cs + ov * sn;", "v[e0] = ev * cs - ov * sn;", 1),
    ("inverse_rope_odd_sign", "v[e0 + 1] = -ev * sn + ov * cs;", "v[e0 + 1] = ev * sn + ov * cs;", 1),
    ("inverse_rope_frequency", "std::pow(theta, -(2.0 * j) / rope_dim)", "std::pow(theta, -(1.0 * j) / rope_dim)", 1),
    ("inverse_rope_first_dims", "const int e0 = D - rope_dim + 2 * j;", "const int e0 = 2 * j;", 1),
    ("overlap_a_from_own_block", "static_cast<size_t>(i - 1) * ratio + t) * w + c",
     "static_cast<size_t>(i) * ratio + t) * w + c", 1),
    ("overlap_bias_halves_swapped", "bias[static_cast<size_t>(t) * w + c]",
     "bias[static_cast<size_t>(t) * w + d + c]", 1),
    ("overlap_bias_on_C", "val[n] = bf16_to_double(cb);",
     "val[n] = bf16_to_double(cb) + static_cast<double>(bias[static_cast<size_t>(t) * w + c]);", 1),
    ("overlap_ignores_previous_block", "if (i > 0 || prev_C) {", "if (i > 0) {", 1),
    ("overlap_position_unscaled", "static_cast<double>(i) * ratio", "static_cast<double>(i)", 1),
    ("overlap_b_reads_stream_a", "static_cast<size_t>(i) * ratio + t) * w + d + c;",
     "static_cast<size_t>(i) * ratio + t) * w + c;", 1),
]

RUNNER = r"""
import json, sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
oracle.use_library({lib!r})
caught = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin()
    except (AssertionError, ValueError):
        caught.append(pin.__name__)
print(json.dumps(caught))
"""


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as fh:
        return fh.read()


@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(source, name, old, new, count):
    assert source.count(old) == count, f"mutation site for {name} not found as expected"
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "mutant.cpp")
        with open(src, "w") as fh:
            fh.write(source.replace(old, new))
        lib = oracle.compile_oracle(src, os.path.join(tmp, "libmutant.so"))
        code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, f"mutant {name} crashed the pin run:\n{r.stderr[-2000:]}"
    caught = json.loads(r.stdout.strip().splitlines()[-1])
    assert caught, f"no pin caught the planted mistake '{name}'"
