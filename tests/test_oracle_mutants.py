"""The oracle's pins are strong enough: each plausible mistake planted in a copy of the oracle's C
source (a dropped term, a wrong sign or index, a transposed operand, a wrong rounding, a swapped
order) makes at least one pin in tests/test_oracle_pins.py fail.

Every mutant is built on the CPU from a temporary copy of oracle.c with the oracle's own compiler
flags and loaded in place of the real oracle for the duration of its check; the real oracle is
restored afterwards.  A control build of the unmodified source must pass every pin, so a mutant is
caught by its mistake and not by the harness.
"""
import itertools
import os
import subprocess

import numpy as np
import pytest

import oracle
import oracle.build as obuild
import test_oracle_pins as pins

# (name, snippet of oracle.c that occurs exactly once, replacement, test-name filters)
MUTANTS = [
    ("bf16 ties away from zero", "(lower == 0x8000u && (upper & 1u))", "(lower == 0x8000u)", ["bf16", "epilogue"]),
    ("bf16 truncates", "upper += 1u;", "upper += 0u;", ["bf16", "epilogue"]),
    ("f16 subnormal scale", "ldexp((double)frac, -24)", "ldexp((double)frac, -25)", ["f16", "dequant"]),
    ("f16 exponent bias", "ldexp((double)(1024 + frac), e - 25)", "ldexp((double)(1024 + frac), e - 24)",
     ["f16", "dequant", "q8_0"]),
    ("acc drops the last k", "for (int k = 0; k < K; ++k) {\n            int64_t xv",
     "for (int k = 0; k < K - 1; ++k) {\n            int64_t xv", ["w8a8_acc", "w8a8_closed", "w8a8_gemm"]),
    ("acc reads W transposed", "row[n] += xv * (int64_t)wk[n];",
     "row[n] += xv * (int64_t)W[((size_t)n * K + k) % ((size_t)K * N)]; (void)wk;",
     ["w8a8_acc", "w8a8_closed", "w8a8_gemm"]),
    ("acc without the overflow check", "if (row[n] > INT32_MAX || row[n] < INT32_MIN) rc = -1;", "",
     ["overflow"]),
    ("split drops a slice", "for (int p = 0; p < parts; ++p) {\n                int32_t slice",
     "for (int p = 0; p + 1 < parts; ++p) {\n                int32_t slice", ["split"]),
    ("epilogue scales w first", "volatile float a = f * x_scale[m];", "volatile float a = f * w_scale[n];",
     ["epilogue"]),
    ("epilogue rounds once", "volatile float b = a * w_scale[n];",
     "volatile float b = (float)((double)f * (double)x_scale[m] * (double)w_scale[n]); (void)a;", ["epilogue"]),
    ("q8_0 scale index along the block",
     "d[(size_t)n * nb + k / 32]) * (double)q[(size_t)n * K + k];\n                s += oracle_bf16_to_f64",
     "d[(size_t)n * nb + k % nb]) * (double)q[(size_t)n * K + k];\n                s += oracle_bf16_to_f64", ["q8_0"]),
    ("q8_0 sign", "s += oracle_bf16_to_f64(x[(size_t)t * K + k]) * w;", "s -= oracle_bf16_to_f64(x[(size_t)t * K + k]) * w;",
     ["q8_0"]),
    ("q8_0 weight norm without the scale", "s += w * w;", "s += (double)q[(size_t)n * K + k] * q[(size_t)n * K + k];",
     ["q8_0_norms", "q8_0"]),
    ("rms eps outside the root", "1.0 / sqrt(ss / (double)K + eps)", "1.0 / (sqrt(ss / (double)K) + eps)", ["rms"]),
    ("rms sum instead of mean", "1.0 / sqrt(ss / (double)K + eps)", "1.0 / sqrt(ss + eps)", ["rms"]),
    ("rms drops gamma", "* oracle_bf16_to_f64(g[k]);\n                double w", ";\n                double w", ["rms"]),
    ("ggml scale big-endian", "(uint16_t)(blk[0] | (blk[1] << 8))", "(uint16_t)((blk[0] << 8) | blk[1])",
     ["ggml", "blocks", "split_layout"]),
    ("pack without offset binary", "^ 0x80u) : 0x80u", ") : 0x80u", ["pack"]),
    ("pack swaps the row and k halves", "int n = 64 * t + 16 * s + g + 8 * (w % 2);\n                        int k = 32 * kb + 8 * c + 4 * (w / 2) + b;",
     "int n = 64 * t + 16 * s + g + 8 * (w / 2);\n                        int k = 32 * kb + 8 * c + 4 * (w % 2) + b;",
     ["pack"]),
    ("f16 ties away from zero", "(rem == 0x1000u && (r & 1u))", "(rem == 0x1000u)", ["f16_from", "quantize"]),
    ("q8_0 quantize rounds half to even", "(int8_t)roundf(bf16_to_f32(blk[j]) / dd)", "(int8_t)rintf(bf16_to_f32(blk[j]) / dd)",
     ["quantize"]),
    ("q8_0 quantize divides by the fp16 scale", "(int8_t)roundf(bf16_to_f32(blk[j]) / dd)",
     "(int8_t)roundf(bf16_to_f32(blk[j]) / (float)oracle_f16_to_f64(d[(size_t)n * nb + b]))", ["quantize"]),
    ("q8_0 quantize amax without the absolute value",
     "const float a = fabsf(bf16_to_f32(blk[j]));", "const float a = bf16_to_f32(blk[j]);", ["quantize"]),
    ("rms squares x * gamma", "double v = oracle_bf16_to_f64(x[(size_t)t * K + k]);\n            ss += v * v;",
     "double v = oracle_bf16_to_f64(x[(size_t)t * K + k]) * oracle_bf16_to_f64(g[k]);\n            ss += v * v;",
     ["rms"]),
    ("f16 subnormal cut-off", "if (e < 102) return sign;", "if (e < 103) return sign;", ["f16_from", "quantize"]),
    ("activation scale over 128", "const float s = amax / 127.0f;", "const float s = amax / 128.0f;", ["quantize_rows"]),
    ("blocks scale byte order", "blk[0] = (uint8_t)(s & 0xFFu);\n            blk[1] = (uint8_t)(s >> 8);",
     "blk[1] = (uint8_t)(s & 0xFFu);\n            blk[0] = (uint8_t)(s >> 8);", ["inverse", "blocks"]),
]


def _cases(fn):
    """Keyword arguments for every case of a (possibly parametrized) pin."""
    grids = []
    for mark in getattr(fn, "pytestmark", []):
        if mark.name != "parametrize":
            continue
        names = [n.strip() for n in mark.args[0].split(",")]
        grids.append([dict(zip(names, v if len(names) > 1 else (v,))) for v in mark.args[1]])
    for combo in itertools.product(*grids):
        kw = {}
        for d in combo:
            kw.update(d)
        yield kw


def _first_failing_pin(filters):
    """Name of the first pin (among those whose name contains a filter) that fails, else None."""
    for name in sorted(n for n in dir(pins) if n.startswith("test_")):
        if filters and not any(f in name for f in filters):
            continue
        fn = getattr(pins, name)
        for kw in _cases(fn):
            try:
                fn(**kw)
            except (Exception, pytest.fail.Exception):   # an assertion, a pytest.raises that saw
                return name                               # nothing, or an error the mistake causes
    return None


def _build(src_text, out_dir, tag):
    src = os.path.join(out_dir, f"oracle_{tag}.c")
    lib = os.path.join(out_dir, f"liboracle_{tag}.so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *obuild.CFLAGS, src, "-o", lib, "-lm"], check=True)
    return lib


@pytest.fixture(scope="module")
def source():
    with open(obuild.SRC) as f:
        return f.read()


def _use(monkeypatch, lib_path):
    monkeypatch.setattr(obuild, "build", lambda force=False: lib_path)
    monkeypatch.setattr(oracle, "_lib", None)


def test_control_build_passes_every_pin(source, tmp_path, monkeypatch):
    _use(monkeypatch, _build(source, str(tmp_path), "control"))
    assert _first_failing_pin([]) is None


@pytest.mark.parametrize("name,old,new,filters", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(name, old, new, filters, source, tmp_path, monkeypatch):
    assert source.count(old) == 1, f"snippet for '{name}' must occur exactly once"
    _use(monkeypatch, _build(source.replace(old, new), str(tmp_path), "mutant"))
    assert _first_failing_pin(filters) is not None, f"no pin catches: {name}"


def _bound_without_weight_norm(x_bits, q, d_bits, rel=2e-3):
    xn, wn = oracle.q8_0_norms(x_bits, q, d_bits)
    return rel * xn[:, None] * np.ones_like(wn)[None, :]


def _bound_rows_reversed(x_bits, q, d_bits, rel=2e-3):
    xn, wn = oracle.q8_0_norms(x_bits, q, d_bits)
    return rel * np.outer(xn[::-1], wn)


def _rms_bound_without_rs(x_bits, g_bits, eps, q, d_bits, rel=8e-3):
    T, K = x_bits.shape
    xg = np.zeros(T, dtype=np.float64)
    oracle.lib().oracle_q8_0_rms_xg_norms(oracle._ptr(np.ascontiguousarray(x_bits, np.uint16)),
                                          oracle._ptr(np.ascontiguousarray(g_bits, np.uint16)), T, K,
                                          oracle._ptr(xg))
    _, wn = oracle.q8_0_norms(x_bits, q, d_bits)
    return rel * xg[:, None] * wn[None, :]


# Mistakes in the oracle's Python-level tolerance functions: (name, attribute, replacement, filters)
PY_MUTANTS = [
    ("bound without the weight norm", "q8_0_bound", _bound_without_weight_norm, ["bound"]),
    ("bound pairs the wrong activation row", "q8_0_bound", _bound_rows_reversed, ["bound"]),
    ("rms bound without rs", "q8_0_rms_bound", _rms_bound_without_rs, ["bound"]),
]


@pytest.mark.parametrize("name,attr,fn,filters", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_planted_tolerance_mistake_fails_a_pin(name, attr, fn, filters, monkeypatch):
    monkeypatch.setattr(oracle, attr, fn)
    assert _first_failing_pin(filters) is not None, f"no pin catches: {name}"
