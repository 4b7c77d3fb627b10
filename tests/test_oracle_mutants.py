"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C sources (on the
CPU), builds it, and runs the CPU pin suite against that build: at least one
pin must fail.  The unmodified sources must pass the same suite."""
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

from conftest import ROOT

ORACLE = os.path.join(ROOT, "oracle")
PINS = ["tests/test_oracle_formats.py", "tests/test_oracle_scaler.py", "tests/test_oracle_quant.py",
        "tests/test_oracle_mx.py", "tests/test_oracle_delayed.py", "tests/test_oracle_master.py",
        "tests/test_oracle_gemm.py"]

MUTANTS = {
    "ties round up instead of to even": (
        "fp_formats.c", "(frac == 0.5 && fmod(lo, 2.0) != 0.0)", "(frac == 0.5)"),
    "subnormal quantum dropped": (
        "fp_formats.c", "if (e < emin) e = emin;", ""),
    "E4M3 treated as IEEE-style (Inf, 7 NaNs)": (
        "fp_formats.c", "FMT_E4M3 = {4, 3, 7, 0}", "FMT_E4M3 = {4, 3, 7, 1}"),
    "E5M2 bias off by one": (
        "fp_formats.c", "FMT_E5M2 = {5, 2, 15, 1}", "FMT_E5M2 = {5, 2, 16, 1}"),
    "saturation code is the NaN pattern": (
        "fp_formats.c", "return (emask << f->mbits) | (mmask - 1);", "return (emask << f->mbits) | mmask;"),
    "growth test strict": (
        "gradscaler.c", "if (*growth_tracker >= growth_interval)", "if (*growth_tracker > growth_interval)"),
    "tracker not reset on overflow": (
        "gradscaler.c", "*scale = *scale * backoff_factor;\n    *growth_tracker = 0;",
        "*scale = *scale * backoff_factor;"),
    "inf check misses NaN": (
        "gradscaler.c", "if (isinf(v) || isnan(v)) found = 1;", "if (isinf(v)) found = 1;"),
    "amax floor dropped": (
        "fp8_quant.c", "if (!isnan(a) && a < floor_amax) a = floor_amax;", ""),
    "quotient by reciprocal": (
        "fp8_quant.c", "float v = x / s;", "float v = x * (1.0f / s);"),
    "block scales transposed": (
        "fp8_quant.c", "scales[bi * nbc + bj] = s;", "scales[bj * (R / br) + bi] = s;"),
    "amax skips NaN": (
        "fp8_quant.c", "if (isnan(v)) return NAN;", "if (isnan(v)) continue;"),
    "MX emax of E4M3 off by one": (
        "mx_quant.c", "return fmt == ORC_E5M2 ? 15 : 8;", "return fmt == ORC_E5M2 ? 15 : 7;"),
    "MX scale applied the wrong way": (
        "mx_quant.c", "ldexp(orc__load_elem(x, dtype, base + i), 127 - code)",
        "ldexp(orc__load_elem(x, dtype, base + i), code - 127)"),
    "delayed scale from the current amax": (
        "delayed.c", "float s = orc_scale_from_amax(hnan ? NAN : hmax, fmt);",
        "float s = orc_scale_from_amax(orc_amax(x, dtype, n), fmt);"),
    "history position not advanced": (
        "delayed.c", "*pos = (*pos + 1) % hist_len;", ""),
    "hysteresis not restored on growth": (
        "delayed.c", "    if (!consecutive) *hyst = hysteresis;\n", ""),
    "min loss scale ignored": (
        "delayed.c", "*scale = s < min_scale ? min_scale : s;", "*scale = s;"),
    "skipped step applied": (
        "master.c", "if (found_inf) return;", ""),
    "clip coefficient inverted": (
        "master.c", "return max_norm / norm;", "return norm / max_norm;"),
    "update by the fused form": (
        "master.c", "float t1 = coef * g[i];\n    float t2 = lr * t1;\n    w[i] = w[i] - t2;",
        "w[i] = fmaf(-lr, coef * g[i], w[i]);"),
    "GEMM weight scale indexed by row instead of block": (
        "gemm.c", "(double)sb[(n / 128) * nkb + kb]", "(double)sb[n * nkb + kb]"),
    "GEMM decodes B in A's format": (
        "gemm.c", "orc_fp8_decode(qb[n * K + k], fmt_b)", "orc_fp8_decode(qb[n * K + k], fmt_a)"),
    "GEMM promotion with one block's scale for all": (
        "gemm.c", "(double)sa[m * nkb + kb]", "(double)sa[m * nkb]"),
    "MX all-zero block scaled by 2^0": (
        "mx_quant.c", "    e = -127;\n  } else {", "    e = 0;\n  } else {"),
    "bf16 master copy truncated": (
        "master.c", "w_bf16[i] = orc_bf16_encode(w[i]);",
        "w_bf16[i] = (uint16_t)(*(const uint32_t*)&w[i] >> 16);"),
    "GEMM activation scale of the next K-block": (
        "gemm.c", "(double)sa[m * nkb + kb]", "(double)sa[m * nkb + (kb + 1) % nkb]"),
    "unscale by S instead of 1/S": (
        "gradscaler.c", "out[i] = (float)v * inv_scale;", "out[i] = (float)v * scale;"),
    "backoff by the growth factor": (
        "gradscaler.c", "*scale = *scale * backoff_factor;", "*scale = *scale * growth_factor;"),
    "delayed history max ignores NaN": (
        "delayed.c", "if (isnan(history[j])) hnan = 1;", "if (0) hnan = 1;"),
    "delayed amax recorded before the step's cast reads it": (
        "delayed.c", "*pos = (*pos + 1) % hist_len;", "*pos = (*pos + 2) % hist_len;"),
    "MX exponent from the rounded-up log2": (
        "mx_quant.c", "e = (k - 1) - emax_elem(fmt);", "e = k - emax_elem(fmt);"),
    "bf16 quiet NaN pattern of f16": (
        "fp_formats.c", "orc_bf16_encode(float f) { return (uint16_t)encode_ieee(f, &FMT_BF16, 0x7FC0u); }",
        "orc_bf16_encode(float f) { return (uint16_t)encode_ieee(f, &FMT_BF16, 0x7E00u); }"),
    "dequant scale index transposed": (
        "fp8_quant.c", "float s = scales[(r / br) * nbc + c / bc];", "float s = scales[(c / bc) * (R / br) + r / br];"),
}


def _build_variant(tmp, name, patch):
    d = os.path.join(tmp, name.replace(" ", "_").replace("(", "").replace(")", "").replace(",", ""))
    os.makedirs(d)
    for f in ["oracle.h", "fp_formats.c", "gradscaler.c", "fp8_quant.c", "mx_quant.c", "delayed.c",
              "master.c", "gemm.c"]:
        shutil.copy(os.path.join(ORACLE, f), d)
    if patch is not None:
        fname, old, new = patch
        path = os.path.join(d, fname)
        with open(path) as f:
            src = f.read()
        assert src.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
        with open(path, "w") as f:
            f.write(src.replace(old, new))
    lib = os.path.join(d, "liboracle.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-o", lib, *[os.path.join(d, f) for f in
                                            ["fp_formats.c", "gradscaler.c", "fp8_quant.c",
                                             "mx_quant.c", "delayed.c", "master.c", "gemm.c"]],
                   "-lm"],
                   check=True)
    return lib


# The pin files that exercise each source file (a planted mistake runs only
# these; the unmodified build runs them all).
PINS_FOR = {
    "fp_formats.c": ["tests/test_oracle_formats.py", "tests/test_oracle_quant.py", "tests/test_oracle_mx.py"],
    "gradscaler.c": ["tests/test_oracle_scaler.py", "tests/test_oracle_formats.py"],
    "fp8_quant.c": ["tests/test_oracle_quant.py", "tests/test_oracle_delayed.py"],
    "mx_quant.c": ["tests/test_oracle_mx.py"],
    "delayed.c": ["tests/test_oracle_delayed.py"],
    "master.c": ["tests/test_oracle_master.py"],
    "gemm.c": ["tests/test_oracle_gemm.py"],
}


def _run_pins(lib, pins):
    env = dict(os.environ, GS_ORACLE_LIB=lib)
    # the exhaustive 2^32 encoder sweep runs once in the main suite, not per mistake
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu", "-k", "not exhaustive_over_every", *pins], cwd=ROOT,
                       env=env, capture_output=True, text=True)
    return r.returncode


def test_pins_catch_every_planted_mistake():
    with tempfile.TemporaryDirectory() as tmp:
        cases = {"unmodified": None, **MUTANTS}
        libs = {name: _build_variant(tmp, name, patch) for name, patch in cases.items()}
        pins = {name: PINS if patch is None else PINS_FOR[patch[0]] for name, patch in cases.items()}
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
            rc = dict(zip(libs, ex.map(_run_pins, libs.values(), [pins[n] for n in libs])))
    assert rc.pop("unmodified") == 0, "the pins must pass on the unmodified oracle"
    survived = [name for name, code in rc.items() if code == 0]
    assert not survived, f"mistakes no pin caught: {survived}"
