"""The oracle's pins are discriminating: each plausible mistake, planted in a
temporary copy of the oracle's C source on the CPU, makes at least one pin
fail. The oracle file itself is never modified."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "cachegen_oracle.c")

# (id, text to replace, replacement, pytest -k selection)
MUTANTS = [
    ("quant-drop-offset", "    y = y + (float)M;\n", "    y = y + 0.0f;\n", "quantize"),
    ("quant-max-bins-half", "int orc_quantize_row(const uint16_t *x, int32_t C, int32_t bins, float *amax_out, uint8_t *q)\n{\n    int32_t M = bins / 2 - 1;",
     "int orc_quantize_row(const uint16_t *x, int32_t C, int32_t bins, float *amax_out, uint8_t *q)\n{\n    int32_t M = bins / 2;", "quantize"),
    ("quant-truncate", "float r = rintf(y);", "float r = floorf(y);", "quantize"),
    ("quant-round-half-away", "float r = rintf(y);", "float r = roundf(y);", "quantize"),
    ("quant-fused-muladd", "        float y = bf16_to_float(x[c]) * f;\n        y = y + (float)M;",
     "        double yd = (double)bf16_to_float(x[c]) * (double)f + (double)M;\n        float y = (float)yd;", "quantize"),
    ("dequant-sign", "float t = (float)((int32_t)q[c] - M);", "float t = (float)(M - (int32_t)q[c]);", "dequant or idempotent"),
    ("dequant-order", "        t = t / fm;\n        t = t * a;", "        t = t * a;\n        t = t / fm;", "idempotent or dequant"),
    ("cdf-no-ramp", "cdf[i] = (uint32_t)((cum * scale) / n) + (uint32_t)i;", "cdf[i] = (uint32_t)((cum * scale) / n);", "int_cdf"),
    ("cdf-full-scale", "uint64_t scale = (uint64_t)ORC_CDF_TOTAL - (uint64_t)N;", "uint64_t scale = (uint64_t)ORC_CDF_TOTAL - (uint64_t)N + 1;", "int_cdf"),
    ("cdf-round-not-floor", "cdf[i] = (uint32_t)((cum * scale) / n) + (uint32_t)i;", "cdf[i] = (uint32_t)((cum * scale + n / 2) / n) + (uint32_t)i;", "int_cdf"),
    ("wnc-pending-same-bit", "        put_bit(w, !b);", "        put_bit(w, b);", "wnc"),
    ("wnc-no-final-pending", "    pending++;\n    if (low < WNC_QUARTER)", "    if (low < WNC_QUARTER)", "wnc"),
    ("wnc-high-no-minus-one", "        high = low + ((r * row[s + 1]) >> 16) - 1;\n        low = low + ((r * row[s]) >> 16);\n        for (;;) {\n            if (high < WNC_HALF) {\n                put_bit_and_pending",
     "        high = low + ((r * row[s + 1]) >> 16);\n        low = low + ((r * row[s]) >> 16);\n        for (;;) {\n            if (high < WNC_HALF) {\n                put_bit_and_pending", "wnc or brute"),
    ("wnc-e3-inclusive", "            } else if (low >= WNC_QUARTER && high < WNC_3QUARTER) {\n                pending++;",
     "            } else if (low >= WNC_QUARTER && high <= WNC_3QUARTER) {\n                pending++;", "wnc or brute"),
    ("wnc-flush-threshold-half", "    if (low < WNC_QUARTER)\n        put_bit_and_pending(&w, 0, &pending);",
     "    if (low < WNC_HALF)\n        put_bit_and_pending(&w, 0, &pending);", "wnc or brute"),
    ("dec-no-shift-in", "            value = 2 * value + get_bit(&br);", "            value = 2 * value;", "wnc or brute"),
    ("groups-255", "#define ORC_GROUP_TOKENS 256", "#define ORC_GROUP_TOKENS 255", "groups"),
    ("bins-allow-odd", "if (b < 4 || b > 64 || (b % 2) != 0)", "if (b < 4 || b > 64)", "layer_bins"),
    ("int8-divide-form", "    float f = (a == 0.0f) ? 0.0f : 127.0f / a;\n    if (!isfinite(f)) /* as in orc_quantize_row */\n        return ORC_ERR_NONFINITE;\n    for (int32_t c = 0; c < C; ++c) {\n        float y = bf16_to_float(x[c]) * f;",
     "    float f = (a == 0.0f) ? 0.0f : a / 127.0f;\n    if (!isfinite(f)) /* as in orc_quantize_row */\n        return ORC_ERR_NONFINITE;\n    for (int32_t c = 0; c < C; ++c) {\n        float y = (f == 0.0f) ? 0.0f : bf16_to_float(x[c]) / f;", "int8"),
    ("int8-scale-128", "float f = (a == 0.0f) ? 0.0f : 127.0f / a;", "float f = (a == 0.0f) ? 0.0f : 128.0f / a;", "int8"),
    ("int8-round-away", "        int32_t iq = (int32_t)rintf(y);\n        if (iq < -127", "        int32_t iq = (int32_t)roundf(y);\n        if (iq < -127", "int8"),
    ("int8-dequant-order", "        float t = (float)q[c] / 127.0f;\n        t = t * a;", "        float t = (float)q[c] * a;\n        t = t / 127.0f;", "int8"),
]


@pytest.mark.parametrize("mid,old,new,sel", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, mid, old, new, sel):
    from oracle import oracle
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor missing for {mid}"
    mut = src.replace(old, new, 1)
    assert mut != src
    csrc = tmp_path / "mutant.c"
    csrc.write_text(mut)
    so = tmp_path / "libmutant.so"
    oracle.compile_source(str(csrc), str(so))
    env = dict(os.environ, CG_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_int8.py"), "-k", sel],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"mutant {mid} survived:\n{r.stdout[-2000:]}"
