"""The oracle's pins catch plausible mistakes planted in the oracle.

Each mutant below is one small, plausible slip in a copy of the oracle (a
swapped nibble, a tie rounded the wrong way, a dropped global scale, a
transposed operand, a sign flipped in the rotation, ...). The copy is built
in a temporary folder and the oracle pin tests (``test_oracle_*.py``, which
check the oracle against the pages' worked values, closed forms, library
routines and brute force, never against itself) are run on it in a child
process. Every mutant must make at least one pin fail, and the unmutated
copy must pass them all.

Planting happens only in the temporary copy on the CPU; the committed oracle
is untouched.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIN_TESTS = ["test_oracle_formats.py", "test_oracle_quant.py", "test_oracle_moe.py",
             "test_oracle_norm_rope.py"]
CPP = "oracle/nvfp4_oracle.cpp"
PY = "oracle/__init__.py"

# (name, file, text in the oracle, planted replacement)
MUTANTS = [
    # E2M1 (README "What We Have": 4-bit E2M1 codes)
    ("e2m1_nibble_order_swapped", CPP,
     "out8[j] = (uint8_t)(c[0] | (c[1] << 4));", "out8[j] = (uint8_t)(c[1] | (c[0] << 4));"),
    ("e2m1_ties_to_odd", CPP, "(err == best_err && (i % 2) == 0)", "(err == best_err && (i % 2) == 1)"),
    ("e2m1_ties_upward", CPP, "if (err < best_err || (err == best_err && (i % 2) == 0))",
     "if (err <= best_err)"),
    ("e2m1_value_3_as_2_5", CPP, "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}",
     "{0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 4.0, 6.0}"),
    ("e2m1_negative_zero_loses_sign", CPP, "uint8_t sign = std::signbit(v) ? 8 : 0;",
     "uint8_t sign = (v < 0.0f) ? 8 : 0;"),
    ("e2m1_saturates_to_4", CPP, "if (a >= 6.0) return sign | 7;", "if (a >= 6.0) return sign | 6;"),
    # E4M3 block scale
    ("e4m3_decode_bias_8", CPP, "else v = std::ldexp(1.0 + m / 8.0, e - 7);",
     "else v = std::ldexp(1.0 + m / 8.0, e - 8);"),
    ("e4m3_encode_truncates", CPP, "double m = std::nearbyint((2.0 * fr - 1.0) * 8.0);",
     "double m = std::floor((2.0 * fr - 1.0) * 8.0);"),
    ("e4m3_subnormal_truncates", CPP, "double m = std::nearbyint(std::ldexp(a, 9));",
     "double m = std::floor(std::ldexp(a, 9));"),
    ("e4m3_overflow_to_nan", CPP, "if (a >= 448.0) return sign | 0x7E;", "if (a >= 448.0) return sign | 0x7F;"),
    # global scale and block rule (README "Correctness Bugs Fixed" 3 and 4)
    ("global_scale_448_not_2688", CPP, "volatile float num = 2688.0f;", "volatile float num = 448.0f;"),
    ("global_scale_zero_amax_gives_inf", CPP, "if (amax == 0.0f) return 1.0f;", "if (amax < 0.0f) return 1.0f;"),
    ("underflow_tested_before_global_scale", CPP, "if (amax == 0.0f || p < underflow)",
     "if (amax == 0.0f || amax < underflow)"),
    ("underflow_inclusive", CPP, "if (amax == 0.0f || p < underflow)", "if (amax == 0.0f || p <= underflow)"),
    ("underflow_rule_dropped", CPP, "if (amax == 0.0f || p < underflow)", "if (amax == 0.0f)"),
    ("scale_ignores_global_scale", CPP, "volatile float ps = p / 6.0f;", "volatile float ps = amax / 6.0f;"),
    ("scale_divides_by_4", CPP, "volatile float ps = p / 6.0f;", "volatile float ps = p / 4.0f;"),
    ("codes_ignore_global_scale", CPP, "volatile float scaled = v[2 * j + h] * gs;",
     "volatile float scaled = v[2 * j + h];"),
    ("amax_signed", CPP, "float a = std::fabs(bf16_to_f32(x[r * ldx + c]));", "float a = bf16_to_f32(x[r * ldx + c]);"),
    ("dequant_f64_drops_global_scale", CPP, "out[r * cols + c] = orc_e2m1_decode(code) * s / (double)gs;",
     "out[r * cols + c] = orc_e2m1_decode(code) * s;"),
    ("dequant_f32_high_nibble_first", CPP,
     "uint8_t code = (c & 1) ? (byte >> 4) : (byte & 15);\n      float s",
     "uint8_t code = (c & 1) ? (byte & 15) : (byte >> 4);\n      float s"),
    # gate/up interleave (README "Fused SwiGLU - How It Works")
    ("interleave_gate_up_swapped", CPP,
     "    std::memcpy(dst + base * row_bytes, src + n * row_bytes, row_bytes);\n"
     "    std::memcpy(dst + (base + g) * row_bytes, src + (inter + n) * row_bytes, row_bytes);",
     "    std::memcpy(dst + base * row_bytes, src + (inter + n) * row_bytes, row_bytes);\n"
     "    std::memcpy(dst + (base + g) * row_bytes, src + n * row_bytes, row_bytes);"),
    ("interleave_granularity_4", PY, "def interleave_rows(a: np.ndarray, g: int = 8)",
     "def interleave_rows(a: np.ndarray, g: int = 4)"),
    # routing and permutation
    ("softmax_over_all_experts", CPP, "for (int j = 0; j < k; ++j) den += std::exp",
     "for (int j = 0; j < E; ++j) den += std::exp"),
    ("topk_ties_to_higher_index", CPP, "std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return key[a] > key[b]; });",
     "std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return key[a] > key[b] || (key[a] == key[b] && a > b); });"),
    ("topk_nan_not_ranked_as_minus_inf", CPP,
     "key[e] = std::isnan(l[e]) ? -INFINITY : (double)l[e];", "key[e] = (double)l[e];"),
    ("permutation_not_stable", CPP,
     "  for (int64_t f = 0; f < T * k; ++f) {\n    int64_t pos = next[ids[f]]++;",
     "  for (int64_t f = T * k - 1; f >= 0; --f) {\n    int64_t pos = next[ids[f]]++;"),
    # GEMM, SwiGLU, combine (README "MoE Runner" steps 2-6)
    ("matmul_b_transposed", CPP, "for (int64_t kk = 0; kk < K; ++kk) acc += a[kk] * b[kk];",
     "for (int64_t kk = 0; kk < K; ++kk) acc += a[kk] * B[kk * N + n];"),
    ("matmul_drops_last_k", CPP, "for (int64_t kk = 0; kk < K; ++kk) acc += a[kk] * b[kk];",
     "for (int64_t kk = 0; kk + 1 < K; ++kk) acc += a[kk] * b[kk];"),
    ("grouped_gemm_first_expert_scale", CPP, "gs_b[e], B.data());", "gs_b[0], B.data());"),
    ("grouped_gemm_a_global_scale_ignored", CPP,
     "orc_dequantize_f64(a_codes + r0 * (K / 2), a_sf + r0 * (K / 16), r1 - r0, K, gs_a, A.data());",
     "orc_dequantize_f64(a_codes + r0 * (K / 2), a_sf + r0 * (K / 16), r1 - r0, K, 1.0f, A.data());"),
    ("swiglu_silu_on_up", CPP,
     "double silu = g / (1.0 + std::exp(-g));\n      h[r * I + i] = (float)(silu * u);",
     "double silu = u / (1.0 + std::exp(-u));\n      h[r * I + i] = (float)(silu * g);"),
    ("swiglu_sigmoid_not_silu", CPP, "double silu = g / (1.0 + std::exp(-g));", "double silu = 1.0 / (1.0 + std::exp(-g));"),
    ("combine_first_weight_only", CPP, "acc += w[t * k + j] * out[", "acc += w[t * k] * out["),
    ("combine_flat_index", CPP, "out[(int64_t)flat_to_perm[t * k + j] * K + c]", "out[(int64_t)(t * k + j) * K + c]"),
    # norm and rotation (README "THE PLAN" item 3)
    ("rmsnorm_sum_not_mean", CPP, "std::sqrt(ss / (double)D + eps)", "std::sqrt(ss + eps)"),
    ("rmsnorm_gamma_dropped", CPP, "* inv * gamma[i];", "* inv;"),
    ("rope_rotation_sign", CPP, "yr[s0 + 2 * j] = a * c - b * s;", "yr[s0 + 2 * j] = a * c + b * s;"),
    ("rope_half_split_pairs", CPP, "const double a = yr[s0 + 2 * j], b = yr[s0 + 2 * j + 1];",
     "const double a = yr[s0 + j], b = yr[s0 + j + R / 2];"),
    ("rope_on_first_elements", CPP, "const int64_t s0 = D - R;", "const int64_t s0 = 0;"),
    # the forward's composition (oracle/__init__.py)
    ("forward_h_dequantized_with_gs_x", PY, "o = matmul_nt(dequantize_f64(hc, hs, gs_h)",
     "o = matmul_nt(dequantize_f64(hc, hs, gs_x)"),
    ("forward_unweighted_sum", PY, "y = combine(outs.reshape(n * k, K), w[tokens],",
     "y = combine(outs.reshape(n * k, K), np.ones_like(w[tokens]),"),
    ("forward_w1_with_w2_scale", PY, "v = matmul_nt(a, dequantize_f64(c1, s1, g1))",
     "v = matmul_nt(a, dequantize_f64(c1, s1, g2))"),
    ("forward_gs_x_ignored_when_given", PY,
     "gs_x = global_scale(amax_x) if gs_x is None else np.float32(gs_x)", "gs_x = global_scale(amax_x)"),
    ("forward_h_requantized_with_gs_x", PY, "hc, hs = quantize_f32(h, gs_h)", "hc, hs = quantize_f32(h, gs_x)"),
]


def _stage(dest):
    """Copy what the pin tests need (oracle sources, tests, goldens, the seeded
    input generators) into ``dest``; nothing built is copied."""
    ign = shutil.ignore_patterns("*.so", "*.tmp*", "__pycache__")
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dest, "oracle"), ignore=ign)
    os.makedirs(os.path.join(dest, "tests"))
    for f in PIN_TESTS + ["conftest.py", "helpers.py"]:
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dest, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dest, "tests", "golden"))
    pkg = os.path.join(dest, "nvfp4_block_scaled_05_gb300")
    os.makedirs(pkg)
    open(os.path.join(pkg, "__init__.py"), "w").close()
    shutil.copy(os.path.join(ROOT, "nvfp4_block_scaled_05_gb300", "workloads.py"), pkg)


def _plant(dest, rel, old, new):
    path = os.path.join(dest, rel)
    src = open(path).read()
    assert src.count(old) == 1, "mutation site not unique in %s: %r" % (rel, old)
    open(path, "w").write(src.replace(old, new))


def _run_pins(dest):
    """Build the copy's oracle and run the pin tests there; returns (rc, tail)."""
    env = dict(os.environ, PYTHONPATH=dest)
    env.pop("PYTHONSTARTUP", None)
    b = subprocess.run([sys.executable, "-c", "import oracle.build as b; b.build(force=True)"],
                       cwd=dest, env=env, capture_output=True, text=True, timeout=300)
    if b.returncode != 0:
        return "build", b.stderr[-400:]
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu"] + ["tests/" + f for f in PIN_TESTS],
                       cwd=dest, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-600:]


def _check_copy_is_used(dest):
    env = dict(os.environ, PYTHONPATH=dest)
    r = subprocess.run([sys.executable, "-c", "import oracle; print(oracle.__file__)"], cwd=dest,
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().startswith(dest), r.stdout + r.stderr


def test_every_planted_mistake_is_caught(tmp_path):
    names = [m[0] for m in MUTANTS]
    assert len(set(names)) == len(names)

    def one(mut):
        name, rel, old, new = mut
        dest = str(tmp_path / name)
        if rel is not None:
            _stage(dest)
            _plant(dest, rel, old, new)
        return name, _run_pins(dest)

    control = str(tmp_path / "control")
    _stage(control)
    _check_copy_is_used(control)
    jobs = [("control", None, None, None)] + MUTANTS
    with ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
        results = dict(ex.map(one, jobs))

    rc, out = results.pop("control")
    assert rc == 0, "the unmutated copy must pass its pins:\n" + str(out)
    for name, (rc, out) in results.items():
        assert rc != "build", "mutant %s did not compile: %s" % (name, out)
    survivors = [name for name, (rc, _) in results.items() if rc == 0]
    assert not survivors, "planted mistakes no pin caught: %s" % survivors
