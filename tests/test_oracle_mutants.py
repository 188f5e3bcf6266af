"""The oracle's pins catch plausible mistakes.

Each mutant is a copy of the oracle with one planted mistake (a wrong constant, rounding
rule, sign, index, operand or dropped term). It is built on the CPU into a temporary
directory and the pin suite (test_oracle_pins.py) runs against it in a subprocess; every
mutant must make at least one pin fail. Nothing here touches a GPU or the library.
"""
import importlib
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

oracle_build = importlib.import_module("oracle.build")  # the module (the package re-exports its function)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, original text, planted mistake); the original occurs exactly once in the source.
MUTANTS = [
    ("quant_scale_128", "const float s = amax / 127.0f;", "const float s = amax / 128.0f;"),
    ("quant_ties_away", "std::nearbyint(v[i] / s)", "std::round(v[i] / s)"),
    ("quant_amax_no_abs", "amax = std::max(amax, std::fabs(v[i]));", "amax = std::max(amax, v[i]);"),
    ("quant_clamp_126", "if (r > 127.0f) r = 127.0f;", "if (r > 126.0f) r = 126.0f;"),
    ("route_ties_to_highest_id", "(best < 0 || l[e] > l[best])", "(best < 0 || l[e] >= l[best])"),
    ("route_unnormalised", "static_cast<float>(ex[j] / z)", "static_cast<float>(ex[j])"),
    ("gate_without_token_scale", "const float g = (static_cast<float>(ag) * sx) * sg[i];",
     "const float g = static_cast<float>(ag) * sg[i];"),
    ("up_with_gate_scale", "const float u = (static_cast<float>(au) * sx) * su[i];",
     "const float u = (static_cast<float>(au) * sx) * sg[i];"),
    ("silu_sign", "g / (1.0f + std::exp(-g))", "g / (1.0f + std::exp(g))"),
    ("gate_up_swapped", "const float silu = g / (1.0f + std::exp(-g));\n    h[i] = silu * u;",
     "const float silu = u / (1.0f + std::exp(-u));\n    h[i] = silu * g;"),
    ("gate_weight_transposed", "Wg[(size_t)i * H + c]", "Wg[(size_t)c * I + i]"),
    ("down_weight_transposed", "Wd[(size_t)o * I + i]", "Wd[(size_t)i * H + o]"),
    ("down_without_h_scale", "d[o] = (static_cast<float>(ad) * sh) * sd[o];",
     "d[o] = static_cast<float>(ad) * sd[o];"),
    ("combine_ignores_route_weights",
     "const double wt = shared ? 1.0 : static_cast<double>(w[(size_t)t * k + s]);",
     "const double wt = 1.0;"),
    ("shared_expert_dropped", "const int S = k + (Is > 0 ? 1 : 0);", "const int S = k;"),
    ("permute_unstable_within_expert",
     "for (long r = 0; r < R; ++r)\n      if (idx[r] == e) perm[pos++] = (int32_t)r;",
     "for (long r = R - 1; r >= 0; --r)\n      if (idx[r] == e) perm[pos++] = (int32_t)r;"),
    ("rmsnorm_sample_variance", "std::sqrt(ss / H + 1e-6)", "std::sqrt(ss / (H - 1) + 1e-6)"),
    ("residual_ignored",
     "bf16_to_float(xr[h]) + static_cast<float>(y[(size_t)t * H + h])", "bf16_to_float(xr[h])"),
    ("bf16_ties_away", "u += 0x7fffu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    ("router_weight_transposed", "Wr[(size_t)h * E + e]", "Wr[(size_t)e * H + h]"),
    ("quant_scale_by_reciprocal", "const float s = amax / 127.0f;",
     "const float s = amax * (1.0f / 127.0f);"),
    ("quant_multiply_by_reciprocal", "std::nearbyint(v[i] / s)", "std::nearbyint(v[i] * (1.0f / s))"),
    ("route_repeats_best", "taken[best] = 1;", "taken[best] = 0;"),
    ("route_skips_last_expert", "for (int e = 0; e < E; ++e)\n        if (!taken[e]",
     "for (int e = 0; e < E - 1; ++e)\n        if (!taken[e]"),
    ("gate_drops_last_term", "for (int c = 0; c < H; ++c) {\n      ag +=",
     "for (int c = 0; c < H - 1; ++c) {\n      ag +="),
    ("down_drops_last_term", "for (int i = 0; i < I; ++i)\n      ad +=",
     "for (int i = 1; i < I; ++i)\n      ad +="),
    ("rmsnorm_without_eps", "std::sqrt(ss / H + 1e-6)", "std::sqrt(ss / H)"),
    ("router_float_accumulation", "double acc = 0.0;\n      for (int h = 0; h < H; ++h)",
     "float acc = 0.0f;\n      for (int h = 0; h < H; ++h)"),
    ("dense_drops_shared_expert", "if (Is > 0) {\n      expert_ffn", "if (Is < 0) {\n      expert_ffn"),
    # NVFP4 expert weights
    ("fp4_nibbles_swapped", "(codes[j / 2] >> (4 * (j % 2)))", "(codes[j / 2] >> (4 * (1 - j % 2)))"),
    ("fp4_block_of_8", "e4m3_value(bscale[j / 16])", "e4m3_value(bscale[j / 8])"),
    ("e2m1_bias_2", "std::ldexp(1.0 + 0.5 * man, (int)ex - 1)", "std::ldexp(1.0 + 0.5 * man, (int)ex - 2)"),
    ("e2m1_subnormal_1", "ex == 0 ? 0.5 * man :", "ex == 0 ? 1.0 * man :"),
    ("e2m1_sign_bit_2", "const unsigned sgn = (code >> 3) & 1u", "const unsigned sgn = (code >> 2) & 1u"),
    ("e4m3_bias_8", "std::ldexp(1.0 + man / 8.0, (int)ex - 7)", "std::ldexp(1.0 + man / 8.0, (int)ex - 8)"),
    ("e4m3_subnormal_exp", "std::ldexp(man / 8.0, -6)", "std::ldexp(man / 8.0, -7)"),
    ("e4m3_implicit_one_dropped", "std::ldexp(1.0 + man / 8.0,", "std::ldexp(man / 8.0,"),
    ("fp4_up_with_gate_scale", "L->g_gate[e], L->g_up[e]", "L->g_gate[e], L->g_gate[e]"),
    ("fp4_shared_up_scale", "L->sh_g[0], L->sh_g[1], L->sh_g[2]", "L->sh_g[0], L->sh_g[0], L->sh_g[2]"),
    ("fp4_down_scale_row", "Bd + (size_t)o * (I / 16)", "Bd + (size_t)(o / 2) * (I / 16)"),
    ("fp4_nan_scale_accepted", "if (b[i] >= 0x7f) return false;", "if (b[i] > 0x7f) return false;"),
    ("fp4_gate_without_token_scale", "const float g4 = (static_cast<float>(ag) * sx) * gg;",
     "const float g4 = static_cast<float>(ag) * gg;"),
]


def _run_mutant(tmp, name, old, new):
    src = open(oracle_build.SRC).read()
    assert src.count(old) == 1, (name, src.count(old))
    d = os.path.join(tmp, name)
    os.makedirs(d, exist_ok=True)
    cpp = os.path.join(d, "moe_oracle.cpp")
    so = os.path.join(d, "libmoe_oracle.so")
    with open(cpp, "w") as f:
        f.write(src.replace(old, new))
    subprocess.run(["g++", *oracle_build.FLAGS, cpp, "-o", so], check=True)
    env = dict(os.environ, MOE_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-600:]


def test_every_mutant_fails_a_pin(tmp_path):
    workers = max(1, min(8, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else 4))
    with ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda m: _run_mutant(str(tmp_path), *m), MUTANTS))
    survivors = [(n, out) for n, rc, out in results if rc == 0]
    assert not survivors, "mutants not caught by any pin: " + ", ".join(n for n, _ in survivors)
    # a caught mutant fails a test (rc 1) or crashes the run; it must not break collection
    for n, rc, out in results:
        assert rc == 1 or rc < 0, (n, rc, out)


def test_unmutated_oracle_passes_the_pins():
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-600:]
