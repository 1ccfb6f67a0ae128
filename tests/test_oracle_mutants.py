"""Planted mistakes: each one, compiled into a copy of the oracle, must fail a pin.

The mistakes are edits of the oracle's C source of the kinds a reader would
worry about (a wrong offset or sign, a dropped term or weight, a swapped
operand, a wrong index or bit position, an unstable order).  None of them
reads or writes out of bounds.  Each mutant is built in a temporary
directory; the committed oracle is never touched.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

MUTANTS = [
    ("2-bit level offset", "double mid = (bits == 3) ? 3.5 : 1.5;", "double mid = (bits == 3) ? 3.5 : 1.0;"),
    ("3-bit level offset", "double mid = (bits == 3) ? 3.5 : 1.5;", "double mid = (bits == 3) ? 4.0 : 1.5;"),
    ("fp16 subnormal exponent", "v = ldexp((double)man, -24);", "v = ldexp((double)man, -25);"),
    ("fp16 bias", "exp - 25); /* (1", "exp - 24); /* (1"),
    ("scale block index", "scales[(int64_t)o * (cols / 32) + i / 32]", "scales[(int64_t)o * (cols / 32) + i / 64]"),
    ("silu sign", "return g / (1.0 + exp(-g));", "return g / (1.0 + exp(g));"),
    ("gate and up swapped", "g[r] = silu(g[r]) * u[r];", "g[r] = silu(u[r]) * g[r];"),
    ("tie goes to higher id", "return a < b;", "return a > b;"),
    ("ties ignored", "if (la > lb) return 1;", "if (la >= lb) return 1;"),
    ("no renormalisation", "w[(int64_t)t * k + j] = (p[ids[(int64_t)t * k + j]] / z) / zs;",
     "w[(int64_t)t * k + j] = (p[ids[(int64_t)t * k + j]] / z);"),
    ("softmax without max shift in the infinite case", "if (isinf(m)) p[e] = ((double)l[e] == m) ? 1.0 : 0.0;",
     "if (0) p[e] = 0.0;"),
    ("routing weight dropped", "routed[i] += w[(int64_t)t * k + j] * y[i];", "routed[i] += y[i];"),
    ("shared expert dropped", "if (swg) oracle_shared_expert", "if (0) oracle_shared_expert"),
    ("router bias dropped", "double acc = bias ? (double)bias[e] : 0.0;", "double acc = 0.0;"),
    ("shared down transposed", "oracle_bf16_to_double(wd[(int64_t)o * I + r])",
     "oracle_bf16_to_double(wd[(int64_t)(r % (H < I ? H : I)) * I + (o % I)])"),
    ("high-bit position", "return (i & 7) | ((i & 8) << 1) | ((i & 16) >> 1);", "return (i & 7) | (i & 8) | (i & 16);"),
    ("most-significant-first codes", "(uint8_t)((c & 3) << (2 * (i % 4)))", "(uint8_t)((c & 3) << (6 - 2 * (i % 4)))"),
    ("permutation unstable", "int32_t pos = fill[ids[f]]++;", "int32_t pos = offsets[ids[f] + 1] - 1 - (fill[ids[f]]++ - offsets[ids[f]]);"),
    ("offsets shifted", "for (int64_t f = 0; f < n; f++) offsets[ids[f] + 1]++;", "for (int64_t f = 0; f < n; f++) offsets[ids[f]]++;"),
    ("bf16 read as the low half", "uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    ("rms norm without the mean", "double r = sqrt(ss / (double)H + eps);", "double r = sqrt(ss + eps);"),
    ("rms norm eps outside the root", "double r = sqrt(ss / (double)H + eps);", "double r = sqrt(ss / (double)H) + eps;"),
    ("e4m3 subnormal spacing", "int E = e - 1 < -6 ? -6 : e - 1;", "int E = e - 1 < -7 ? -7 : e - 1;"),
    ("e4m3 mantissa width", "double q = ldexp(1.0, E - 3);", "double q = ldexp(1.0, E - 4);"),
    ("e4m3 without saturation", "if (r > 448.0) r = 448.0;", "if (r > 480.0) r = 480.0;"),
    ("e4m3 exponent bias", "ldexp((double)(8 + man), exp - 10)", "ldexp((double)(8 + man), exp - 9)"),
    ("fp16 rounding width", "double q = ldexp(1.0, E - 10);", "double q = ldexp(1.0, E - 9);"),
    ("fp8 scaling exponent off by one", "int k = 7 - (e - 1);", "int k = 8 - (e - 1);"),
    ("fp8 input scaling not undone", "y[o] = ldexp(acc, -(kw[o] + ex));", "y[o] = ldexp(acc, -kw[o]);"),
    ("fp8 h not held in fp16", "g[r] = oracle_fp16_round(silu(g[r]) * u[r]);", "g[r] = silu(g[r]) * u[r];"),
    ("fp8 gate and up swapped", "g[r] = oracle_fp16_round(silu(g[r]) * u[r]);",
     "g[r] = oracle_fp16_round(silu(u[r]) * g[r]);"),
    ("fp8 row exponent from the first block", "for (int b = 0; b < cols / 32; b++) {", "for (int b = 0; b < 1; b++) {"),
    ("fp8 row exponent from the 2-bit levels for 3 bits", "double maxc = (bits == 3) ? 3.5 : 1.5;",
     "double maxc = 1.5;"),
]

PIN_TESTS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]


def _run_pins():
    failed = []
    for fn in PIN_TESTS:
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        calls = [()]
        if params:
            argnames = params[0].args[0]
            calls = [v if isinstance(v, tuple) else (v,) for v in params[0].args[1]]
        for args in calls:
            try:
                fn(*args)
            except Exception:  # noqa: BLE001 - any failure counts as "caught"
                failed.append(fn.__name__)
                break
        if failed:
            return failed
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation anchor missing: {old!r}"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-shared", "-fPIC", "-o", so,
                    str(mutant_src), "-lm"], check=True)
    prev = oracle.use_library(so)
    try:
        failed = _run_pins()
    finally:
        oracle.use_library(prev)
    assert failed, f"no pin caught the planted mistake: {name}"
