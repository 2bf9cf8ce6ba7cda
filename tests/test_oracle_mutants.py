"""The pins catch plausible mistakes: each mutant below is hc_oracle.c with
one planted slip (a dropped term, a wrong sign or index, a transposed
operand, an extra or missing round, a misplaced eps, a wrong rounding
rule).  Each mutant is compiled on the CPU and run against the pin tests of
test_oracle_pins.py; every mutant must fail at least one of them.  The real
oracle is untouched (the mutants live in a temporary directory)."""
import ctypes
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "hc_oracle.c")

MUTANTS = {
    "sum_sq_one_stream": ("for (int64_t k = 0; k < K; ++k) {\n            double v = hco_bf16_to_double(xt[k]);\n            ss += v * v;",
                          "for (int64_t k = 0; k < d; ++k) {\n            double v = hco_bf16_to_double(xt[k]);\n            ss += v * v;"),
    "rsqrt_divides": ("mixes[t * mix + i] = acc * r;", "mixes[t * mix + i] = acc / r;"),
    "pre_no_eps": ("sigmoid(m[j] * s0 + (double)hc_base[j]) + eps;", "sigmoid(m[j] * s0 + (double)hc_base[j]);"),
    "post_not_doubled": ("post[t * hc + j] = 2.0 * sigmoid(m[hc + j] * s1", "post[t * hc + j] = sigmoid(m[hc + j] * s1"),
    "post_wrong_scale": ("2.0 * sigmoid(m[hc + j] * s1", "2.0 * sigmoid(m[hc + j] * s0"),
    "comb_transposed_read": ("int i = 2 * hc + j * hc + k;", "int i = 2 * hc + k * hc + j;"),
    "softmax_eps_inside": ("c[j * hc + k] = c[j * hc + k] / s + eps;", "c[j * hc + k] = c[j * hc + k] / (s + eps);"),
    "softmax_no_max_shift_sign": ("exp(c[j * hc + k] - mx)", "exp(mx - c[j * hc + k])"),
    "no_first_column_step": ("c[j * hc + k] = c[j * hc + k] / (sum[k] + eps);\n        /* the later rounds",
                             "c[j * hc + k] = c[j * hc + k];\n        /* the later rounds"),
    "one_extra_round": ("for (int it = 1; it < iters; ++it)", "for (int it = 0; it < iters; ++it)"),
    "columns_before_rows": (
        "            for (int j = 0; j < hc; ++j) {\n                sum[j] = 0.0;\n                for (int k = 0; k < hc; ++k)\n                    sum[j] += c[j * hc + k];\n            }\n            for (int j = 0; j < hc; ++j)\n                for (int k = 0; k < hc; ++k)\n                    c[j * hc + k] = c[j * hc + k] / (sum[j] + eps);\n            for (int k = 0; k < hc; ++k) {\n                sum[k] = 0.0;\n                for (int j = 0; j < hc; ++j)\n                    sum[k] += c[j * hc + k];\n            }\n            for (int j = 0; j < hc; ++j)\n                for (int k = 0; k < hc; ++k)\n                    c[j * hc + k] = c[j * hc + k] / (sum[k] + eps);\n        }",
        "            for (int k = 0; k < hc; ++k) {\n                sum[k] = 0.0;\n                for (int j = 0; j < hc; ++j)\n                    sum[k] += c[j * hc + k];\n            }\n            for (int j = 0; j < hc; ++j)\n                for (int k = 0; k < hc; ++k)\n                    c[j * hc + k] = c[j * hc + k] / (sum[k] + eps);\n            for (int j = 0; j < hc; ++j) {\n                sum[j] = 0.0;\n                for (int k = 0; k < hc; ++k)\n                    sum[j] += c[j * hc + k];\n            }\n            for (int j = 0; j < hc; ++j)\n                for (int k = 0; k < hc; ++k)\n                    c[j * hc + k] = c[j * hc + k] / (sum[j] + eps);\n        }"),
    "row_sum_transposed": ("                for (int k = 0; k < hc; ++k)\n                    sum[j] += c[j * hc + k];\n            }\n            for (int j = 0; j < hc; ++j)\n                for (int k = 0; k < hc; ++k)\n                    c[j * hc + k] = c[j * hc + k] / (sum[j] + eps);",
                           "                for (int k = 0; k < hc; ++k)\n                    sum[j] += c[k * hc + j];\n            }\n            for (int j = 0; j < hc; ++j)\n                for (int k = 0; k < hc; ++k)\n                    c[j * hc + k] = c[j * hc + k] / (sum[j] + eps);"),
    "pre_mix_one_weight": ("acc += pre_mix[t * hc + s] * hco_bf16_to_double", "acc += pre_mix[t * hc + 0] * hco_bf16_to_double"),
    "rms_mean_off_by_one": ("double rs = 1.0 / sqrt(ss / (double)d + eps);", "double rs = 1.0 / sqrt(ss / (double)(d - 1) + eps);"),
    "rms_no_gain": ("hco_bf16_from_double((v * rs) * (double)w[c]);", "hco_bf16_from_double(v * rs);"),
    "post_comb_transposed": ("acc += comb[(t * hc + j) * hc + k] *", "acc += comb[(t * hc + k) * hc + j] *"),
    "post_wrong_stream_weight": ("double acc = post[t * hc + k] * hco_bf16_to_double(f[t * d + c]);",
                                 "double acc = post[t * hc + 0] * hco_bf16_to_double(f[t * d + c]);"),
    "round_ties_away": ("    return (fmod(r, 2.0) == 0.0) ? r : r + 1.0;", "    return r + 1.0;"),
    "round_truncate": ("    if (frac > 0.5)\n        return r + 1.0;", "    if (frac > 2.0)\n        return r + 1.0;"),
    "block_reads_with_own_pre": ("rc = hco_pre(x, pre_mix, n, hc, d, h);", "rc = hco_pre(x, pre, n, hc, d, h);"),
    "mx_scale_rounded_down": ("int ex = (m == 0.5f) ? e - 1 : e;", "int ex = e - 1;"),
    "mx_no_1e4_floor": ("            if (amax < 1e-4f)\n                amax = 1e-4f;\n", ""),
    "mx_scale_bias": ("scales[t * groups + g] = (uint8_t)(ex + 127);", "scales[t * groups + g] = (uint8_t)(ex + 128);"),
    "e4m3_two_mantissa_bits": ("double ulp = ldexp(1.0, ex - 3); /* 3 mantissa bits */",
                               "double ulp = ldexp(1.0, ex - 2); /* 3 mantissa bits */"),
    "bwd_no_rs3_term": ("gh[c] = rs * gh[c] - rs * rs * rs / (double)d * h[c] * T;", "gh[c] = rs * gh[c];"),
    "bwd_sigmoid_derivative": ("const double gq = gpost[j] * 2.0 * sq * (1.0 - sq);",
                               "const double gq = gpost[j] * 2.0 * sq;"),
    "bwd_sinkhorn_step_no_projection": ("g[idx] = (g[idx] - dot) / (s + eps);", "g[idx] = g[idx] / (s + eps);"),
    "bwd_no_statistic_term": ("const double cr = -gr * r * r * r / (double)K;", "const double cr = 0.0;"),
    "bwd_softmax_not_centred": ("gL[j * hc + k] = S[j * hc + k] * (g[j * hc + k] - dot);",
                                "gL[j * hc + k] = S[j * hc + k] * g[j * hc + k];"),
    "bwd_norm_w_unnormalised": ("g_w[c] += (h[c] * rs) * g_hn[t * d + c];", "g_w[c] += h[c] * g_hn[t * d + c];"),
    "e4m3_subnormal_threshold": ("    if (ex < -6)\n        ex = -6; /* subnormals share",
                                 "    if (ex < -7)\n        ex = -7; /* subnormals share"),
}

# the pin tests run against each mutant (all take no fixtures except golden_constants)
PIN_TESTS = [getattr(pins, name) for name in dir(pins) if name.startswith("test_")]


def _golden():
    import json
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "tests",
                        "golden", "v41_hc_constants.json")
    with open(path) as fh:
        return {k: v["value"] for k, v in json.load(fh).items() if not k.startswith("_")}


def _run_pins():
    """Return the names of pin tests that fail against the currently loaded library."""
    import inspect
    failed = []
    golden = _golden()
    for fn in PIN_TESTS:
        sig = inspect.signature(fn)
        params = list(sig.parameters)
        marks = getattr(fn, "pytestmark", [])
        cases = [dict()]
        for m in marks:
            if m.name == "parametrize":
                names = [s.strip() for s in m.args[0].split(",")]
                new = []
                for c in cases:
                    for v in m.args[1]:
                        vals = v if len(names) > 1 else (v,)
                        new.append({**c, **dict(zip(names, vals))})
                cases = new
        for c in cases:
            kwargs = dict(c)
            if "golden_constants" in params:
                kwargs["golden_constants"] = golden
            try:
                fn(**kwargs)
            except Exception:
                failed.append(fn.__name__)
                break
    return failed


@pytest.fixture(scope="module")
def tmpdir_mut():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmpdir_mut):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, "mutation anchor for %s must occur exactly once in the oracle" % name
    mutated = src.replace(old, new, 1)
    c_path = os.path.join(tmpdir_mut, name + ".c")
    so_path = os.path.join(tmpdir_mut, name + ".so")
    with open(c_path, "w") as fh:
        fh.write(mutated)
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-std=c99", "-shared", "-fPIC", "-o", so_path,
                    c_path, "-lm"], check=True)
    real = oracle._load()
    try:
        lib = ctypes.CDLL(so_path)
        for attr in ("hco_bf16_to_double", "hco_bf16_from_double", "hco_mixes", "hco_split_sinkhorn",
                     "hco_pre", "hco_rmsnorm", "hco_post", "hco_block_step", "hco_e4m3_from_double",
                     "hco_mxfp8", "hco_side_f64", "hco_side_backward_f64"):
            f, g = getattr(lib, attr), getattr(real, attr)
            f.argtypes, f.restype = g.argtypes, g.restype
        oracle._lib = lib
        failed = _run_pins()
    finally:
        oracle._lib = real
    assert failed, "mutant %s passed every pin" % name


def test_real_oracle_passes_the_same_harness():
    assert _run_pins() == []
