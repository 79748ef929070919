"""Pins of the oracle's int8 baseline codec: hand-derived fixture, closed
forms, quantise/dequantise idempotence, the error bound, and exact-rational
emulation of the fp32 operation order where another order gives another
result."""
import os
from fractions import Fraction

import numpy as np
import pytest

from test_oracle_pins import _rint_even, _rn32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int8_hand.txt")


def _f(bits):
    return float(np.array([int(bits) << 16], np.uint32).view(np.float32)[0])


def test_int8_golden(orc):
    n = 0
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        xs, a, qs = [p.strip() for p in line.split("|")]
        x = np.array([int(h, 16) for h in xs.split()], dtype=np.uint16)
        amax, q = orc.int8_quantize_row(x)
        assert amax == float(a)
        assert q.tolist() == [int(v) for v in qs.split()]
        n += 1
    assert n == 3


def test_int8_extremes_and_dequant_closed_forms(orc):
    rng = np.random.default_rng(8)
    for _ in range(50):
        ab = int(rng.integers(0x3000, 0x5000))
        a = _f(ab)
        amax, q = orc.int8_quantize_row(np.array([ab, ab | 0x8000, 0], np.uint16))
        assert amax == a and q.tolist() == [127, -127, 0]
        y = orc.int8_dequant_row(np.array([127, -127, 0], np.int8), a)
        assert y.tolist() == [ab, ab | 0x8000, 0]


def test_int8_roundtrip_bound_and_idempotence(orc):
    rng = np.random.default_rng(9)
    for _ in range(40):
        x = (rng.standard_normal(300) * rng.lognormal(0, 2)).astype(np.float32)
        xb = (x.view(np.uint32) >> 16).astype(np.uint16)
        a, q = orc.int8_quantize_row(xb)
        y = orc.int8_dequant_row(q, a)
        a2, q2 = orc.int8_quantize_row(y)
        assert a2 == a and np.array_equal(q, q2)
        xf = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        yf = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert np.all(np.abs(xf - yf) <= 0.5 * a / 127 * (1 + 2.0 ** -20) + np.abs(yf) * 2.0 ** -8)


def test_int8_operation_order(orc):
    """q uses the product x * fp32(127 / a), not x / fp32(a / 127); y uses
    fp32(q / 127) * a. Find inputs where the other forms differ and check
    the oracle against exact-rational emulation there. For the quantiser
    they are the exact ties x = a / 2; for the dequantiser, where the
    result is rounded to bf16, only a scale that is not itself a bf16 value
    separates the two orders, so it is driven with fp32 scales."""
    m = np.arange(128, dtype=np.uint32)
    qcases = 0
    for ea in range(112, 144):
        a_bits = ((ea << 7) | m).astype(np.uint32) << 16
        a = a_bits.view(np.float32)
        f = (np.float32(127) / a).astype(np.float32)
        g = (a / np.float32(127)).astype(np.float32)
        for ex in range(ea - 12, ea + 1):
            xb = ((ex << 7) | m).astype(np.uint32) << 16
            x = xb.view(np.float32)
            mul = np.rint((x[None, :] * f[:, None]).astype(np.float32))
            div = np.rint((x[None, :] / g[:, None]).astype(np.float32))
            for i, j in np.argwhere((mul != div) & (x[None, :] <= a[:, None]))[:2]:
                av, xv = Fraction(float(a[i])), Fraction(float(x[j]))
                want = _rint_even(_rn32(xv * _rn32(Fraction(127) / av)))
                _, q = orc.int8_quantize_row(
                    np.array([a_bits[i] >> 16, xb[j] >> 16], np.uint16))
                assert int(q[1]) == want
                qcases += 1
    assert qcases >= 20

    def to_bf16(v):
        u = np.asarray(v, np.float32).view(np.uint32)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    rng = np.random.default_rng(10)
    a = (rng.uniform(0.5, 8.0, 32768)).astype(np.float32)
    ycases = 0
    for q in range(-127, 128):
        y_def = to_bf16((np.float32(q) / np.float32(127)).astype(np.float32) * a)
        y_alt = to_bf16((np.float32(q) * a).astype(np.float32) / np.float32(127))
        for i in np.nonzero(y_def != y_alt)[0][:2]:
            got = orc.int8_dequant_row(np.array([q], np.int8), float(a[i]))
            t = _rn32(_rn32(Fraction(q, 127)) * Fraction(float(a[i])))
            assert int(got[0]) == int(to_bf16(float(t)))
            ycases += 1
    assert ycases >= 5


def test_int8_whole_blob_matches_rows(orc):
    from kv_cache_compression_03_gb300 import synthetic
    kv = synthetic.generate("opt125m_t256", num_tokens=40)
    q, sc = orc.int8_encode(kv)
    C = kv.shape[-1]
    flat = kv.reshape(-1, C)
    for r in (0, 7, flat.shape[0] - 1):
        a, qr = orc.int8_quantize_row(flat[r])
        assert a == sc[r] and np.array_equal(qr, q.reshape(-1, C)[r])
    y = orc.int8_decode(q, sc)
    assert np.array_equal(y.reshape(-1, C)[5], orc.int8_dequant_row(q.reshape(-1, C)[5], sc[5]))


def test_overflowing_scale_factor_rejected(orc):
    """A row so small that MAX / a rounds to inf in fp32 has no scale
    factor; both quantisers reject it (status 4, non-finite). The boundary
    is where the exact quotient reaches 2^128 - 2^103, the point from which
    round-to-nearest gives inf."""
    limit = Fraction(2 ** 128 - 2 ** 103)
    seen = {True: 0, False: 0}
    for bits in list(range(1, 0x0400, 3)) + [0x0080, 0x0100, 0x0180]:
        a = Fraction(_f(bits))
        row = np.array([bits, 0, bits | 0x8000], np.uint16)
        for M, call in ((127, lambda: orc.int8_quantize_row(row)),
                        (7, lambda: orc.quantize_row(row, 16)),
                        (15, lambda: orc.quantize_row(row, 32)),
                        (31, lambda: orc.quantize_row(row, 64))):
            overflow = Fraction(M) / a >= limit
            seen[overflow] += 1
            if overflow:
                with pytest.raises(orc.OracleError) as e:
                    call()
                assert e.value.status == 4
            else:
                amax, q = call()
                assert amax == float(a)
                off = 0 if M == 127 else M
                assert q.astype(int).tolist() == [off + M, off, off - M]
    assert seen[True] > 20 and seen[False] > 20
