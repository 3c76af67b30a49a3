"""The oracle's pins must catch plausible mistakes.

Each case below plants one slip into a copy of the oracle's C source (a dropped
term, a wrong sign or index, a transposed operand, a wrong rounding rule),
compiles it on the CPU into a temporary directory, swaps it in, and runs the
pin suite of tests/test_oracle_pins.py against it.  At least one pin must fail
for every mutant; the real oracle passes them all (that file's own run).
"""
import inspect
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

# (name, original text, replacement) -- every occurrence of the original is replaced.
MUTANTS = [
    ("dropped alpha in the correction", "beta * (v[a] - alpha * work[a])", "beta * (v[a] - work[a])"),
    ("sign of the correction", "beta * (v[a] - alpha * work[a])", "beta * (v[a] + alpha * work[a])"),
    ("transposed state in S k", "acc += S[(int64_t)a * d + b] * k[b];", "acc += S[(int64_t)b * d + a] * k[b];"),
    ("outer product k v^T", "alpha * S[(int64_t)a * d + b] + r * k[b];",
     "alpha * S[(int64_t)a * d + b] + beta * (v[b] - alpha * work[b]) * k[a];"),
    ("repeat-interleaved key heads", "int g = h % nk;", "int g = h / (nv / nk);"),
    ("missing 1/sqrt(D)", "o[a] = acc * scale;", "o[a] = acc;"),
    ("read-out with k instead of q", "acc += S[(int64_t)a * d + b] * q[b];", "acc += S[(int64_t)a * d + b] * k[b];"),
    ("decay not applied", "S[(int64_t)a * d + b] = alpha * S[(int64_t)a * d + b] + r * k[b];",
     "S[(int64_t)a * d + b] = S[(int64_t)a * d + b] + r * k[b];"),
    ("norm without the mean", "sqrt(ss / (double)d + eps)", "sqrt(ss + eps)"),
    ("eps outside the root", "sqrt(ss / (double)d + eps)", "(sqrt(ss / (double)d) + eps)"),
    ("sigmoid gate instead of silu", "double silu = zz / (1.0 + exp(-zz));", "double silu = 1.0 / (1.0 + exp(-zz));"),
    ("no norm weight", "out[h * d + a] = (double)gn[a] * oh[a] / den * silu;", "out[h * d + a] = oh[a] / den * silu;"),
    ("prefill reuses token 0 gates", "alpha + bt * nv, beta + bt * nv", "alpha + (int64_t)b * T * nv, beta + (int64_t)b * T * nv"),
    ("round half up", "(rem == half && (n & 1u))", "(rem == half)"),
    ("truncating rounding", "if (rem > half || (rem == half && (n & 1u))) n += 1;", "(void)half;"),
    ("overflow saturates", "if (E > 15) return (uint16_t)(sign | 0x7c00u);", "if (E > 15) return (uint16_t)(sign | 0x7bffu);"),
    ("widened subnormal exponent off by one", "int32_t E = -14;\n        while", "int32_t E = -15;\n        while"),
    ("conv ring not shifted", "ring[(int64_t)t * channels + c] = ring[(int64_t)(t + 1) * channels + c];",
     "ring[(int64_t)t * channels + c] = ring[(int64_t)t * channels + c];"),
    ("conv newest tap at the front", "ring[(int64_t)(taps - 1) * channels + c] = x[c];", "ring[c] = x[c];"),
    ("conv without silu", "y[c] = acc / (1.0 + exp(-acc));", "y[c] = acc;"),
    ("l2 eps on the mean", "double den = sqrt(ss + eps);", "double den = sqrt(ss / d + eps);"),
    ("gate rate applied twice", "pow(1.0 + exp((double)ar[i] + (double)dt[i]), (double)rate[i])",
     "pow(1.0 + exp((double)ar[i] + (double)dt[i]), -exp((double)rate[i]))"),
    ("beta not a sigmoid", "beta[i] = 1.0 / (1.0 + exp(-(double)br[i]));", "beta[i] = (double)br[i];"),
    ("q8 scale over 128", "am > 0.0f ? am / 127.0f : 1.0f", "am > 0.0f ? am / 128.0f : 1.0f"),
    ("q8 ties rounded away from zero", "(frac > 0.5 || (frac == 0.5 && fmod(f, 2.0) != 0.0))", "(frac >= 0.5)"),
    ("q8 truncation", "if (frac > 0.5 || (frac == 0.5 && fmod(f, 2.0) != 0.0)) f += 1.0;", "(void)frac;"),
    ("q8 group max over half the group", "for (int i = 0; i < 32; ++i) {\n            float m = fabsf",
     "for (int i = 0; i < 16; ++i) {\n            float m = fabsf"),
    ("q8 zero group scale 0", "am > 0.0f ? am / 127.0f : 1.0f", "am / 127.0f"),
    ("widening drops the sign", "return sign | (ex - 15u + 127u) << 23 | (fr << 13);", "return (ex - 15u + 127u) << 23 | (fr << 13);"),
]


def _pin_calls():
    """Every pin function with each of its parametrisations."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            calls.append((name, fn, {}))
            continue
        m = marks[0]
        argnames = [a.strip() for a in m.args[0].split(",")] if isinstance(m.args[0], str) else list(m.args[0])
        for vals in m.args[1]:
            vals = vals if isinstance(vals, (tuple, list)) else (vals,)
            calls.append((name, fn, dict(zip(argnames, vals))))
    return calls


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor absent: {old!r}"
    mut = tmp_path / "mut.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "mut.so"
    subprocess.check_call(["gcc", *oracle.CFLAGS, "-o", str(so), str(mut), "-lm"])
    saved = oracle._load()
    oracle._lib = oracle.bind(str(so))
    failed = []
    try:
        for pname, fn, kw in _pin_calls():
            try:
                fn(**kw)
            except AssertionError:
                failed.append(pname)
    finally:
        oracle._lib = saved
    assert failed, f"no pin caught the mutant '{name}'"
