"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
the pins in test_oracle.py catch every one of them.

Each mutant is a one-line textual change of oracle.c compiled to a temporary
library; the pin suite runs against it in a child process through the
ORACLE_LIB override and must fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "drops_last_rank": ("for (int p = 1; p < n; ++p)\n        acc = acc + widen",
                        "for (int p = 1; p < n - 1; ++p)\n        acc = acc + widen"),
    "starts_from_zero": ("float acc = widen(in[0], src_i, dtype);\n    for (int p = 1;",
                         "float acc = 0.0f;\n    for (int p = 0;"),
    "reversed_rank_order": ("float acc = widen(in[0], src_i, dtype);\n    for (int p = 1; p < n; ++p)\n"
                            "        acc = acc + widen(in[p], src_i, dtype);",
                            "float acc = widen(in[n - 1], src_i, dtype);\n    for (int p = n - 2; p >= 0; --p)\n"
                            "        acc = acc + widen(in[p], src_i, dtype);"),
    "wrong_sign": ("acc = acc + widen(in[p]", "acc = acc - widen(in[p]"),
    "bf16_half_up": ("(dropped == 0x8000u && (hi & 1u))", "(dropped == 0x8000u)"),
    "bf16_truncates": ("        hi += 1u;\n", "        hi += 0u;\n"),
    "f16_subnormal_binade": ("if (e < -14) e = -14;", "if (e < -15) e = -15;"),
    "f16_overflow_threshold": ("if (a >= 65520.0)", "if (a >= 65504.0)"),
    "f16_subnormal_widen": ("ldexp((double)m, -24)", "ldexp((double)m, -25)"),
    "rs_shard_index": ("(size_t)rank * recv_count + j", "(size_t)rank + j"),
    "ag_offset_elements_not_bytes": ("(size_t)q * send_count * es", "(size_t)q * send_count"),
    "int32_subtracts": ("acc += (uint32_t)((const int32_t*)in[p])[src_i];",
                        "acc -= (uint32_t)((const int32_t*)in[p])[src_i];"),
    "accumulates_in_output_precision": (
        "acc = acc + widen(in[p], src_i, dtype);",
        "{ float t = acc + widen(in[p], src_i, dtype); uint16_t h = dtype == ORC_FP16 ? "
        "orc_f32_to_f16(t) : orc_f32_to_bf16(t); acc = dtype == ORC_FP32 ? t : (dtype == ORC_FP16 ? "
        "orc_f16_to_f32(h) : orc_bf16_to_f32(h)); }"),
    "ring_wrong_neighbour": ("(s == (d + n - 1) % n)", "(s == (d + 1) % n)"),
    "linear_drops_rank_weight": ("acc += (double)widen(w[p], i * kp + k, dtype) * (double)widen(x[p], k, dtype);",
                                 "acc += (double)widen(w[p], i * kp + k, dtype) * (double)widen(x[p ? p - 1 : 0], k, dtype);"),
    "linear_rounds_through_fp32": ("((uint16_t*)out)[i] = f64_to_half_once(acc, dtype);",
                                   "((uint16_t*)out)[i] = f64_to_half_once((double)(float)acc, dtype);"),
    "half_once_ties_up": ("if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;\n    long k = (long)fl;               /* quanta, <= 2^p */",
                          "if (r >= 0.5) fl += 1.0;\n    long k = (long)fl;               /* quanta, <= 2^p */"),
    "max_drops_nan": ("if (isnan(a) || isnan(b)) return NAN;\n    if (a == b) return signbit(a) ? b : a;",
                      "if (isnan(a)) return b;\n    if (isnan(b)) return a;\n    if (a == b) return signbit(a) ? b : a;"),
    "max_signed_zero_first_wins": ("if (a == b) return signbit(a) ? b : a;", "if (a == b) return a;"),
    "min_signed_zero_wrong": ("if (a == b) return signbit(a) ? a : b;", "if (a == b) return signbit(a) ? b : a;"),
    "op_max_min_swapped": ("acc = op == ORC_OP_MAX ? max_ieee(acc, widen(in[p], i, dtype)) : min_ieee(acc, widen(in[p], i, dtype));",
                           "acc = op == ORC_OP_MAX ? min_ieee(acc, widen(in[p], i, dtype)) : max_ieee(acc, widen(in[p], i, dtype));"),
    "op_int_drops_last_rank": ("for (int p = 1; p < n; ++p) {\n                const int32_t v",
                               "for (int p = 1; p < n - 1; ++p) {\n                const int32_t v"),
    "op_skips_rank_0": ("float acc = widen(in[0], i, dtype);\n        for (int p = 1; p < n; ++p)\n            acc = op",
                        "float acc = widen(in[n - 1], i, dtype);\n        for (int p = 1; p < n; ++p)\n            acc = op"),
    "op_nan_not_canonical_at_one_rank": ("if (isnan(acc)) acc = NAN;   /* canonical", "if (0) acc = NAN;   /* canonical"),
    "residual_of_rank_0": ("const double y = acc + (double)widen(res[q], i, dtype);",
                           "const double y = acc + (double)widen(res[0], i, dtype);"),
    "residual_dropped": ("const double y = acc + (double)widen(res[q], i, dtype);",
                         "const double y = acc + 0.0 * (double)widen(res[q], i, dtype);"),
    "residual_after_rounding_the_layer": (
        "const double y = acc + (double)widen(res[q], i, dtype);",
        "const double y = (double)(dtype == ORC_FP16 ? orc_f16_to_f32(f64_to_half_once(acc, dtype))"
        " : orc_bf16_to_f32(f64_to_half_once(acc, dtype))) + (double)widen(res[q], i, dtype);"),
    "tokens_ignore_token_offset": ("acc += (double)widen(w[p], i * kp + k, dtype) * (double)widen(x[p], t * kp + k, dtype);",
                                   "acc += (double)widen(w[p], i * kp + k, dtype) * (double)widen(x[p], k, dtype);"),
    "tokens_output_transposed": ("((uint16_t*)out)[t * rows + i] = f64_to_half_once(acc, dtype);",
                                 "((uint16_t*)out)[i * tokens + t] = f64_to_half_once(acc, dtype);"),
    "tokens_drop_last_rank": ("            for (int p = 0; p < n; ++p)\n                for (size_t k = 0; k < kp; ++k)\n                    acc += (double)widen(w[p], i * kp + k, dtype) * (double)widen(x[p], t * kp + k, dtype);",
                              "            for (int p = 0; p < n - 1; ++p)\n                for (size_t k = 0; k < kp; ++k)\n                    acc += (double)widen(w[p], i * kp + k, dtype) * (double)widen(x[p], t * kp + k, dtype);"),
    "tokens_residual_of_rank_0": ("const double y = dot + (double)widen(res[q], t * rows + i, dtype);",
                                  "const double y = dot + (double)widen(res[0], t * rows + i, dtype);"),
    "tokens_residual_wrong_token": ("const double y = dot + (double)widen(res[q], t * rows + i, dtype);",
                                    "const double y = dot + (double)widen(res[q], i, dtype);"),
    "tokens_residual_product_of_rank_0": ("dot += (double)widen(w[p], i * kp + k, dtype) * (double)widen(x[p],",
                                          "dot += (double)widen(w[0], i * kp + k, dtype) * (double)widen(x[p],"),
    "allreduce_at_wrong_slot": ("reduce_one(n, in, (size_t)idx[k], out, k, dtype);",
                                "reduce_one(n, in, (size_t)idx[k], out, (size_t)idx[k] % (nidx ? nidx : 1), dtype);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor not found once: " + name
    mutant_c = tmp_path / ("oracle_%s.c" % name)
    mutant_c.write_text(src.replace(old, new))
    lib = tmp_path / ("liboracle_%s.so" % name)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
                    "-shared", "-pthread", "-w", "-o", str(lib), str(mutant_c), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "pins did not catch mutant %s:\n%s" % (name, r.stdout[-2000:])
