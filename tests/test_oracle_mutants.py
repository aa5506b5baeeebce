"""The pins must catch plausible mistakes in the oracle.

Each case compiles a copy of ``oracle/oracle.c`` with one planted slip (on the
CPU, into a temporary directory), points the pin tests at it and requires at
least one of the named pins to fail.  The real oracle stays untouched.
"""
import os
import subprocess
import sys

import pytest

from oracle import build as obuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, exact source text, replacement, pytest -k expression expected to fail)
MUTANTS = [
    ("add_wrong_sign", "double s = (double)a[i] + (double)b[i];",
     "double s = (double)a[i] - (double)b[i];", "add_f32_matches_numpy"),
    ("add_rounds_twice_via_half", "c[i] = (float)s; /* one rounding, to nearest even */",
     "c[i] = (float)(double)(float)(s * 1.0000001);", "add_f32"),
    ("ties_away_from_zero", "} else if (frac == 0.5) {\n        if (fmod(r, 2.0) != 0.0) r += 1.0;",
     "} else if (frac == 0.5) {\n        r += 1.0;", "midpoints or thresholds or exact_rounding"),
    ("bf16_wrong_field_width", "return decode_bits(h, 8, 7); }",
     "return decode_bits(h, 7, 8); }", "bf16_decode"),
    ("subnormal_threshold_off_by_one", "if (a < ldexp(1.0, emin)) {",
     "if (a < ldexp(1.0, emin - 1)) {", "roundtrips or thresholds"),
    ("overflow_one_binade_late", "if (E > bias) return", "if (E > bias + 1) return",
     "thresholds or roundtrips"),
    ("saxpy_unfused", "for (int64_t i = 0; i < n; ++i) y[i] = fmaf(alpha, x[i], y[i]);",
     "for (int64_t i = 0; i < n; ++i) y[i] = alpha * x[i] + y[i];", "saxpy_f32_equals_exact"),
    ("saxpy16_transposed_operands", "float r = fmaf(alpha, xf, yf);\n        y[i] = orc_f64_to_f16((double)r);",
     "float r = fmaf(alpha, yf, xf);\n        y[i] = orc_f64_to_f16((double)r);", "saxpy_16bit"),
    ("relu_keeps_negative_zero", "if (isnan(v) || v > 0.0) {\n            y[i] = x[i];",
     "if (isnan(v) || v >= 0.0) {\n            y[i] = x[i];", "relu_f32 or signed_zero"),
    ("relu_zeroes_nan", "y[i] = (isnan(v) || v > 0.0) ? x[i] : (uint16_t)0;\n    }\n}\n\nORC_API void orc_relu_bf16",
     "y[i] = (v > 0.0) ? x[i] : (uint16_t)0;\n    }\n}\n\nORC_API void orc_relu_bf16", "relu_16bit"),
    ("gather_64bit_overflow", "unsigned __int128 p = (unsigned __int128)(uint64_t)s * (uint64_t)i;",
     "uint64_t p = (uint64_t)s * (uint64_t)i;", "gather_index or gather_brute"),
    ("gather_wrong_modulus", "return (int64_t)(p % (uint64_t)n);",
     "return (int64_t)(p % (uint64_t)(n > 2 ? n - 1 : n));", "gather"),
    ("ceil_div_floor", "return (n + t - 1) / t;", "return n / t;", "ceil_div"),
    ("select_swapped_branches", "if (x[i] % 2 == 0) {\n            y[i] = (int32_t)(u * 2u);",
     "if (x[i] % 2 != 0) {\n            y[i] = (int32_t)(u * 2u);", "select"),
]


@pytest.fixture(scope="module")
def source():
    with open(os.path.join(ROOT, "oracle", "oracle.c"), encoding="utf-8") as f:
        return f.read()


@pytest.mark.parametrize("name,old,new,kexpr", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, source, name, old, new, kexpr):
    assert source.count(old) == 1, "mutation anchor not found exactly once: %s" % name
    src = tmp_path / "oracle_mut.c"
    src.write_text(source.replace(old, new), encoding="utf-8")
    lib = tmp_path / "liboracle_mut.so"
    subprocess.run(["cc", *obuild.CFLAGS, str(src), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, EW_ORACLE_LIB=str(lib))
    tests = [os.path.join(ROOT, "tests", "test_oracle_pins.py"),
             os.path.join(ROOT, "tests", "test_golden.py")]
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-k", kexpr, *tests], cwd=ROOT, env=env,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    assert r.returncode == 1, "mutant %s survived the pins:\n%s" % (name, r.stdout[-2000:])
