"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of oracle/nvfp4_oracle.c (a dropped term,
a wrong sign, an inverted comparison, a transposed operand, a wrong packing or
operation order), compiles it, and runs the oracle pin tests against it in a
subprocess: they must fail.  CPU only.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "nvfp4_oracle.c")

MUTANTS = {
    "block scale with T=4 for the T=6 candidate":
        ("encode_candidate(v, n, b, 6.0f, S, c6, &s6);", "encode_candidate(v, n, b, 4.0f, S, c6, &s6);"),
    "global scale dropped from the block scale": ("float s32 = q * S;", "float s32 = q;"),
    "E2M1 sign dropped": ("uint8_t sign = signbit(y) ? 8u : 0u;", "uint8_t sign = 0u;"),
    "E2M1 ties to odd": ("if (dist < best_dist || (dist == best_dist && (k & 1) == 0)) {\n            best = k;\n            best_dist = dist;\n        }\n    }\n    return (uint8_t)(sign | (uint8_t)best);\n}\n\n/* E4M3",
                         "if (dist < best_dist || (dist == best_dist && (k & 1) == 1)) {\n            best = k;\n            best_dist = dist;\n        }\n    }\n    return (uint8_t)(sign | (uint8_t)best);\n}\n\n/* E4M3"),
    "encode factor inverted": ("float e = (sd == 0.0f) ? 0.0f : S / sd;", "float e = (sd == 0.0f) ? 0.0f : sd / S;"),
    "four-over-six comparison inverted": ("if (err4 < err6) {", "if (err4 > err6) {"),
    "error uses |d| instead of d^2": ("float d2 = d * d;", "float d2 = fabsf(d);"),
    "columnwise reads the wrong operand layout":
        ("oracle_quantize_line(x + c, rows, cols, a,", "oracle_quantize_line(x + c * rows, rows, 1, a,"),
    "nibble order swapped": ("if (idx & 1) packed", "if (!(idx & 1)) packed"),
    "dequantize factor grouped differently": ("float t = sd * amax;\n    return t * F_inv;",
                                              "float t = amax * F_inv;\n    return sd * t;"),
    "amax of x instead of |x|": ("float a = fabsf(x[r * cols + c]);", "float a = x[r * cols + c];"),
    "E4M3 saturates to NaN": ("if (!(m < 448.0f)) return (uint8_t)(sign | 0x7Eu);",
                              "if (!(m < 448.0f)) return (uint8_t)(sign | 0x7Fu);"),
    "F uses 4 instead of the E2M1 max 6": ("float F = bound * 6.0f; /* exact: 2688 or 1536 */",
                                           "float F = bound * 4.0f;"),
    "group amax drops the last row of each group":
        ("if (end > start) oracle_amax(x + start * cols, end - start, cols, NULL, NULL, &t);",
         "if (end > start + 1) oracle_amax(x + start * cols, end - start - 1, cols, NULL, NULL, &t);"),
    "noop ignored": ("    if (noop_set(noop)) return 0;\n    int do_row", "    int do_row"),
    "16x16 error summed in column-major order":
        ("for (int j = 0; j < w; ++j) v[i * w + j] = x[(ti * 16 + i) * cols + tj * 16 + j];",
         "for (int j = 0; j < w; ++j) v[j * h + i] = x[(ti * 16 + i) * cols + tj * 16 + j];"),
    "GEMM uses the first amax for every line":
        ("double a = (double)amax[row_scaled ? r : 0];", "double a = (double)amax[0];"),
    "GEMM drops the code sign":
        ("return (double)oracle_e2m1_decode(code) * sd", "return (double)oracle_e2m1_decode(code & 7u) * sd"),
    "GEMM scale index per 32 columns":
        ("scales[r * (k / 16) + c / 16]", "scales[r * (k / 16) + c / 32]"),
    "GEMM reads B with A's row index":
        ("element_value(b_codes, b_scales, b_amax, b_row_scaled, b_bound, k, j, c)",
         "element_value(b_codes, b_scales, b_amax, b_row_scaled, b_bound, k, i % n, c)"),
    "GEMM divides by bound * 4": ("a / ((double)bound * 6.0)", "a / ((double)bound * 4.0)"),
    "RHT sign mask read in reverse bit order":
        ("v[j] = ((sign_mask >> j) & 1u) ? -t : t;", "v[j] = ((sign_mask >> (15 - j)) & 1u) ? -t : t;"),
    "RHT normalised by 1/2": ("y[(r0 + j) * cols + c] = v[j] * 0.25f;",
                              "y[(r0 + j) * cols + c] = v[j] * 0.5f;"),
    "RHT butterfly difference reversed": ("v[i + h] = u - w;", "v[i + h] = w - u;"),
    "RHT skips the last butterfly stage": ("for (int h = 1; h < 16; h *= 2) {",
                                           "for (int h = 1; h < 8; h *= 2) {"),
    "RHT reads the block along a row": ("float t = x[(r0 + j) * cols + c];",
                                        "float t = x[r0 * cols + (c + j) % cols];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    from oracle import build
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not found once: {old!r}"
    lib = build.build_variant(text.replace(old, new), str(tmp_path / "liboracle_mutant.so"))
    env = dict(os.environ, NVFP4_ORACLE_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_formats.py"),
                        os.path.join(ROOT, "tests", "test_oracle_recipe.py"),
                        os.path.join(ROOT, "tests", "test_oracle_gemm.py"),
                        os.path.join(ROOT, "tests", "test_oracle_rht.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch: {name}\n{r.stdout[-2000:]}"
