"""The oracle's pins must catch plausible mistakes.

Each case below plants one mistake in a copy of ``oracle/oracle.c`` (on the
CPU, in a temporary directory), builds it, and runs the pin suite against the
mutant; the suite must fail.  The real oracle is untouched.
"""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "flipped_kernel": ("w[ohwi(co, r, s, j, KH, KW, cin_g)]",
                       "w[ohwi(co, KH - 1 - r, KW - 1 - s, j, KH, KW, cin_g)]"),
    "pad_axes_swapped": ("int ih = oh * stride - pad_h + r;", "int ih = oh * stride - pad_w + r;"),
    "bias_dropped": ("if (b) v += b[co];", "(void)b;"),
    "group_offset_zero": ("int g0 = (co / cout_g) * cin_g;", "int g0 = 0;"),
    "weight_transposed": ("return (((size_t)co * KH + r) * KW + s) * CPG + j;",
                          "return (((size_t)co * KW + s) * KH + r) * CPG + j;"),
    "requant_truncates": ("float r = nearbyintf(p);", "float r = truncf(p);"),
    "requant_rounds_half_away": ("float r = nearbyintf(p);", "float r = roundf(p);"),
    "no_saturation": ("if (r > 127.0f) r = 127.0f;", ""),
    "requant_scale_w_only": ("M[co] = (float)((double)in_scale * (double)w_scales[co] /\n"
                             "                        (double)out_scale);",
                             "M[co] = (float)(double)w_scales[co];"),
    "requant_scale_ratio_inverted": ("M[co] = (float)((double)in_scale * (double)w_scales[co] /\n"
                                     "                        (double)out_scale);",
                                     "M[co] = (float)((double)out_scale * (double)w_scales[co] /\n"
                                     "                        (double)in_scale);"),
    "requant_scale_first_channel_full": ("(int8_t)oracle_requant_one(v, M[co], relu);",
                                         "(int8_t)oracle_requant_one(v, M[0], relu);"),
    "requant_scale_first_channel": ("vals[i] = (int8_t)oracle_requant_one(v, M[p[3]], relu);",
                                    "vals[i] = (int8_t)oracle_requant_one(v, M[0], relu);"),
    "ceil_output_dim": ("return span / stride + 1;", "return (span + stride - 1) / stride + 1;"),
    "hardmish": ("return v * tanh(softplus(v));",
                 "return v * fmin(fmax(v + 2.0, 0.0), 2.0) / 2.0;"),
    "relu_as_abs": ("return v > 0.0 ? v : 0.0;", "return fabs(v);"),
    "stride_ignored_w": ("int iw = ow * stride - pad_w + s;", "int iw = ow - pad_w + s;"),
    "maxpool_zero_padding": ("double m = -INFINITY;", "double m = 0.0;"),
    "maxpool_window_short": ("for (int j = w - r; j <= w + r; ++j) {", "for (int j = w - r; j < w + r; ++j) {"),
}


def _run_mutant(name, tmp):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"pattern of mutant {name} not found in oracle.c"
    mutated = src.replace(old, new)
    c = os.path.join(tmp, f"{name}.c")
    so = os.path.join(tmp, f"{name}.so")
    with open(c, "w") as f:
        f.write(mutated)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-shared",
                    "-fPIC", c, "-o", so, "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=so, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-400:]


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            results = list(ex.map(lambda n: _run_mutant(n, tmp), MUTANTS))
    survivors = [(n, out) for n, rc, out in results if rc == 0]
    assert not survivors, f"mutants not caught by any pin: {survivors}"
    # rc 1 = tests failed; anything else (2 = collection error ...) is not a catch
    bad = [(n, rc, out) for n, rc, out in results if rc != 1]
    assert not bad, bad
