"""Pins of the CPU oracle against facts fixed outside the oracle itself:
hand-derived fixtures (tests/golden), closed forms, invariants, an
exact-rational model of the coder, and brute force on tiny inputs."""
import itertools
import os

import numpy as np
import pytest

from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(fname):
    with open(os.path.join(GOLDEN, fname)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [p.strip() for p in line.split("|")]


def _f32_bits(x: float) -> int:
    return int(np.array([x], dtype=np.float32).view(np.uint32)[0])


# ------------------------------------------------------------------ config

def test_layer_bins_presets(orc):
    # 7B/8B preset: 32 layers, K's first 10 layers 32 bins, V's first 2.
    k = orc.layer_bins(32, [(0, 10, 32), (10, 32, 16)])
    v = orc.layer_bins(32, [(0, 2, 32), (2, 32, 16)])
    assert k.tolist() == [32] * 10 + [16] * 22
    assert v.tolist() == [32] * 2 + [16] * 30
    # specs may come in any order
    assert orc.layer_bins(5, [(3, 5, 8), (0, 3, 4)]).tolist() == [4, 4, 4, 8, 8]


@pytest.mark.parametrize("specs", [
    [(0, 10, 32), (9, 32, 16)],       # overlap
    [(0, 10, 32), (11, 32, 16)],      # gap
    [(0, 32, 17)],                    # odd bins
    [(0, 32, 2)],                     # too few bins
    [(0, 32, 66)],                    # too many bins
    [(0, 33, 16)],                    # past the last layer
    [(-1, 32, 16)],                   # negative start
    [(4, 4, 16), (0, 32, 16)],        # empty range
])
def test_layer_bins_rejects(orc, specs):
    with pytest.raises(orc.OracleError) as e:
        orc.layer_bins(32, specs)
    assert e.value.status == orc.ERR_SPEC


@pytest.mark.parametrize("T,chunk,starts,counts", [
    (256, 256, [0], [256]),
    (600, 256, [0, 256, 512], [256, 256, 88]),
    (768, 768, [0, 256, 512], [256, 256, 256]),
    (768, 64, list(range(0, 768, 64)), [64] * 12),
    (700, 300, [0, 256, 300, 556, 600], [256, 44, 256, 44, 100]),
    (1, 256, [0], [1]),
    (257, 1000, [0, 256], [256, 1]),
])
def test_groups(orc, T, chunk, starts, counts):
    s, c = orc.groups(T, chunk)
    assert s.tolist() == starts and c.tolist() == counts


# ---------------------------------------------------------------- quantise

def test_quantize_golden(orc):
    n = 0
    for bins, xs, a, qs in _rows("quantize_hand.txt"):
        x = np.array([int(h, 16) for h in xs.split()], dtype=np.uint16)
        amax, q = orc.quantize_row(x, int(bins))
        assert amax == float(a)
        assert q.tolist() == [int(v) for v in qs.split()]
        n += 1
    assert n == 4


@pytest.mark.parametrize("bins", [4, 6, 16, 32, 64])
def test_quantize_extremes(orc, bins):
    M = bins // 2 - 1
    rng = np.random.default_rng(bins)
    for _ in range(50):
        a = np.float32(rng.uniform(0.01, 100.0))
        a_bits = np.array([a], dtype=np.float32).view(np.uint32)[0] >> 16
        a_val = float(np.array([a_bits << 16], dtype=np.uint32).view(np.float32)[0])
        row = np.array([a_bits, a_bits | 0x8000, 0, 0x8000], dtype=np.uint16)
        amax, q = orc.quantize_row(row, bins)
        assert amax == a_val
        assert q.tolist() == [2 * M, 0, M, M]


def test_quantize_nonfinite(orc):
    for bad in (0x7F80, 0xFF80, 0x7FC0):
        with pytest.raises(orc.OracleError) as e:
            orc.quantize_row(np.array([0x3F80, bad], dtype=np.uint16), 16)
        assert e.value.status == orc.ERR_NONFINITE


@pytest.mark.parametrize("bins", [4, 16, 32, 64])
def test_quantize_dequantize_idempotent(orc, bins):
    """dequantise(q) quantises back to q, and the reconstruction error stays
    within half a quantisation step plus the bf16 rounding of the output."""
    M = bins // 2 - 1
    rng = np.random.default_rng(100 + bins)
    for trial in range(40):
        x = (rng.standard_normal(257) * rng.lognormal(0, 2)).astype(np.float32)
        xb = (x.view(np.uint32) >> 16).astype(np.uint16)
        a, q = orc.quantize_row(xb, bins)
        assert q.min() >= 0 and q.max() <= 2 * M
        assert (q == 0).any() or (q == 2 * M).any()
        y = orc.dequant_row(q, bins, a)
        a2, q2 = orc.quantize_row(y, bins)
        assert a2 == a
        assert np.array_equal(q2, q)
        xf = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        yf = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        bound = 0.5 * a / M * (1 + 2.0 ** -20) + np.abs(yf) * 2.0 ** -8
        assert np.all(np.abs(xf - yf) <= bound + 1e-30)


@pytest.mark.parametrize("bins", [4, 16, 32])
def test_dequant_closed_forms(orc, bins):
    M = bins // 2 - 1
    for a in (1.0, 0.375, 1234.0, 3.0e-5):
        ab = _f32_bits(a) >> 16
        a = float(np.array([ab << 16], dtype=np.uint32).view(np.float32)[0])
        y = orc.dequant_row(np.array([2 * M, 0, M], dtype=np.uint8), bins, a)
        assert y.tolist() == [ab, ab | 0x8000, 0]


# ------------------------------------------------------------- integer CDF

def test_int_cdf_golden(orc):
    n = 0
    for N, cnt, counts, cdf in _rows("int_cdf_hand.txt"):
        got = orc.int_cdf(np.array([int(v) for v in counts.split()]), int(cnt))
        assert got.tolist() == [int(v) for v in cdf.split()]
        assert len(got) == int(N) + 1
        n += 1
    assert n == 5


@pytest.mark.parametrize("N", [4, 16, 32, 64])
def test_int_cdf_single_symbol(orc, N):
    for n in (1, 7, 256):
        for s0 in range(N - 1):
            counts = np.zeros(N, dtype=np.uint32)
            counts[s0] = n
            cdf = orc.int_cdf(counts, n)
            freq = np.diff(cdf.astype(np.int64))
            assert freq[s0] == 65536 - N + 1
            assert np.all(np.delete(freq, s0) == 1)


@pytest.mark.parametrize("N", [4, 16, 32, 64])
def test_int_cdf_invariants(orc, N):
    rng = np.random.default_rng(N)
    for _ in range(200):
        n = int(rng.integers(1, 257))
        counts = np.bincount(rng.integers(0, N - 1, n), minlength=N).astype(np.uint32)
        cdf = orc.int_cdf(counts, n).astype(np.int64)
        freq = np.diff(cdf)
        assert cdf[0] == 0 and cdf[-1] == 65536
        assert np.all(freq >= 1) and freq.sum() == 65536
        # a symbol is given frequency 1 exactly when it never occurs
        assert np.array_equal(freq == 1, counts == 0)
        # the scaled count is within one of its share of 2^16 - N
        share = counts * (65536 - N) / n
        assert np.all(np.abs((freq - 1) - share) < 1.0)


# ---------------------------------------------------------------- the coder

def _trace_rows():
    for cdf, syms, hexbytes in _rows("wnc_hand_trace.txt"):
        yield (np.array([int(v) for v in cdf.split()], dtype=np.uint32),
               np.array([int(v) for v in syms.split()], dtype=np.uint8), bytes.fromhex(hexbytes))


def test_wnc_hand_traces(orc):
    n = 0
    for cdf, syms, want in _trace_rows():
        assert orc.wnc_encode(syms, cdf) == want
        assert orc.wnc_decode(want, len(syms), cdf).tolist() == syms.tolist()
        n += 1
    assert n == 4


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5, 6])
def test_wnc_uniform_power_of_two(orc, k):
    """With 2^k equally likely symbols the stream is the symbols' k-bit
    codes, then the termination bits 01, then zero padding."""
    rng = np.random.default_rng(k)
    cdf = (np.arange(2 ** k + 1) * (65536 >> k)).astype(np.uint32)
    for length in (0, 1, 5, 100, 1023):
        syms = rng.integers(0, 2 ** k, length).astype(np.uint8)
        bits = "".join(format(int(s), f"0{k}b") for s in syms) + "01"
        bits += "0" * (-len(bits) % 8)
        want = bytes(int(bits[i:i + 8], 2) for i in range(0, len(bits), 8))
        assert orc.wnc_encode(syms, cdf) == want


def _random_table(rng, N, extreme=False):
    if extreme:
        # one dominant symbol, the rest at the minimum frequency 1
        freq = np.ones(N, dtype=np.int64)
        freq[rng.integers(0, N)] += 65536 - N
    else:
        w = rng.dirichlet(np.full(N, 0.3))
        freq = 1 + np.floor(w * (65536 - N)).astype(np.int64)
        freq[np.argmax(freq)] += 65536 - freq.sum()
    return np.concatenate([[0], np.cumsum(freq)]).astype(np.uint32)


def test_brute_force_exact_model(orc):
    """Every sequence of length <= 6 over alphabets of 2..4 symbols, for
    several tables (including frequency-1 neighbours of 65533): the stream's
    dyadic interval lies inside the exact interval (so any continuation
    decodes), the stream decodes back with trailing 0s, 1s and random
    bits, and its length is within two bits (plus padding) of
    -log2(interval width)."""
    rng = np.random.default_rng(7)
    tables = []
    for N in (2, 3, 4):
        tables.append(_random_table(rng, N))
        tables.append(_random_table(rng, N, extreme=True))
        tables.append(np.array([0] + [1 + i for i in range(N - 1)] + [65536], dtype=np.uint32))
    tables.append(np.array([0, 1, 2, 65535, 65536], dtype=np.uint32))
    tables.append(np.array([0, 65533, 65534, 65535, 65536], dtype=np.uint32))
    checked = 0
    for cdf in tables:
        N = len(cdf) - 1
        for length in range(0, 7):
            for syms in itertools.product(range(N), repeat=length):
                syms = np.array(syms, dtype=np.uint8)
                data = orc.wnc_encode(syms, cdf)
                lo, hi, _ = brute.final_interval(syms.tolist(), [cdf] * length)
                assert brute.dyadic_inside(data, lo, hi), (cdf, syms, data.hex())
                # length: never shorter than the information, at most 2 bits + pad over it
                fl, ce = brute.neg_log2_bounds(hi - lo)
                assert 8 * len(data) >= fl
                assert 8 * len(data) - 7 <= ce + 2
                for tail in (b"\x00" * 8, b"\xff" * 8, bytes(rng.integers(0, 256, 8).tolist())):
                    got = orc.wnc_decode(data + tail, length, cdf)
                    assert got.tolist() == syms.tolist()
                checked += 1
    assert checked > 10000


def test_wnc_roundtrip_long_random(orc):
    rng = np.random.default_rng(11)
    for trial in range(60):
        N = int(rng.choice([2, 4, 16, 17, 32, 33, 64]))
        C = int(rng.integers(1, 2000))
        rows = np.stack([_random_table(rng, N, extreme=bool(rng.integers(0, 4) == 0))
                         for _ in range(C)])
        syms = np.array([rng.choice(N, p=np.diff(r.astype(np.float64)) / 65536) for r in rows],
                        dtype=np.uint8)
        data = orc.wnc_encode(syms, rows)
        assert orc.wnc_decode(data, C, rows).tolist() == syms.tolist()
        assert orc.wnc_decode(data + b"\xff" * 8, C, rows).tolist() == syms.tolist()
        # information content bounds (P_int = prod freq / 2^16)
        freq = np.diff(rows.astype(np.int64), axis=1)[np.arange(C), syms]
        info = float(np.sum(16 - np.log2(freq)))
        assert 8 * len(data) >= info - C * 2.0 ** -13 - 1e-9
        assert 8 * len(data) <= info + 2 + 7 + C * 2.0 ** -13


def test_wnc_exact_interval_long(orc):
    """Longer sequences against the exact-rational model (fewer of them)."""
    rng = np.random.default_rng(12)
    for trial in range(30):
        N = int(rng.choice([2, 5, 16, 32]))
        n = int(rng.integers(20, 120))
        rows = [_random_table(rng, N, extreme=bool(trial % 3 == 0)) for _ in range(n)]
        syms = [int(rng.choice(N, p=np.diff(r.astype(np.float64)) / 65536)) for r in rows]
        data = orc.wnc_encode(np.array(syms, dtype=np.uint8), np.stack(rows))
        lo, hi, _ = brute.final_interval(syms, rows)
        assert brute.dyadic_inside(data, lo, hi)


# ------------------------------------------- fp32 evaluation order of §2

def _rn32(v):
    """Round a Fraction to the nearest fp32 value, ties to even (normal range)."""
    from fractions import Fraction
    if v == 0:
        return Fraction(0)
    s = -1 if v < 0 else 1
    m = abs(v)
    e = m.numerator.bit_length() - m.denominator.bit_length()
    if Fraction(2) ** e > m:
        e -= 1
    ulp = Fraction(2) ** (e - 23)
    k = m / ulp
    fl = k.numerator // k.denominator
    rem = k - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return s * fl * ulp


def _rint_even(v):
    from fractions import Fraction
    fl = v.numerator // v.denominator
    rem = v - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def test_quantize_two_roundings(orc):
    """The quantiser evaluates x*factor and +MAX as two separately rounded
    fp32 operations. Over every bf16 mantissa pair (a in [1,2), x = +-m*2^-e)
    find the inputs where a fused multiply-add would give another symbol,
    and check the oracle against an exact-rational emulation of the
    two-rounding definition there."""
    from fractions import Fraction
    am = np.arange(128, dtype=np.uint32)
    a_bits = ((127 << 7) | am).astype(np.uint32) << 16
    a = a_bits.view(np.float32)
    cases = []
    for bins in (16, 32):
        M = np.float32(bins // 2 - 1)
        f = (M / a).astype(np.float32)
        for e in range(0, 12):
            xb = (((127 - e) << 7) | am).astype(np.uint32) << 16
            for sgn in (0, 0x80000000):
                x = (xb | np.uint32(sgn)).view(np.float32)
                X, F, A = x[None, :], f[:, None], a[:, None]
                fused = np.rint((X.astype(np.float64) * F.astype(np.float64)
                                 + np.float64(M)).astype(np.float32))
                split = np.rint((X * F).astype(np.float32) + M)
                for i, j in np.argwhere((fused != split) & (np.abs(X) <= A)):
                    cases.append((bins, int(a_bits[i] >> 16), int((xb[j] | sgn) >> 16),
                                  int(fused[i, j])))
    assert len(cases) >= 6
    for bins, ab, xb, q_fused in cases:
        M = bins // 2 - 1
        av = Fraction(int(np.array([ab << 16], np.uint32).view(np.float32)[0] * 2 ** 20), 2 ** 20)
        xv = np.array([xb << 16], np.uint32).view(np.float32)[0]
        xv = Fraction(float(xv))
        f = _rn32(Fraction(M) / av)
        want = _rint_even(_rn32(_rn32(xv * f) + M))
        assert want != q_fused
        _, q = orc.quantize_row(np.array([ab, xb], dtype=np.uint16), bins)
        assert int(q[1]) == want, (bins, hex(ab), hex(xb))


def test_dequant_operation_order(orc):
    """Dequantisation is t = (q - MAX) / MAX, then t * a, each an fp32
    rounding, then a round-to-nearest-even cast to bf16. Over every bf16
    mantissa of a and every symbol of every even bin count, find where the
    other order (t * a) / MAX gives another bf16, and check the oracle
    against an exact-rational emulation of the definition there."""
    from fractions import Fraction
    am = np.arange(128, dtype=np.uint32)
    a_bits = (((127 << 7) | am).astype(np.uint32) << 16)
    a = a_bits.view(np.float32)

    def to_bf16(x):
        u = x.astype(np.float32).view(np.uint32)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)

    def bf16_rne_exact(v):
        # nearest bf16 (8 significant bits), ties to even, from an exact value
        if v == 0:
            return 0
        s = 0x8000 if v < 0 else 0
        m = abs(v)
        e = m.numerator.bit_length() - m.denominator.bit_length()
        if Fraction(2) ** e > m:
            e -= 1
        k = m / Fraction(2) ** (e - 7)
        fl = k.numerator // k.denominator
        rem = k - fl
        if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
            fl += 1
        val = Fraction(fl) * Fraction(2) ** (e - 7)
        bits = int(np.array([float(val)], np.float32).view(np.uint32)[0] >> 16)
        return bits | s

    cases = 0
    for bins in range(4, 66, 2):
        M = bins // 2 - 1
        for q in range(0, 2 * M + 1):
            t = np.float32(q - M)
            y_def = to_bf16((t / np.float32(M)).astype(np.float32) * a)
            y_alt = to_bf16((t * a).astype(np.float32) / np.float32(M))
            for i in np.nonzero(y_def != y_alt)[0]:
                av = Fraction(float(a[i]))
                want = bf16_rne_exact(_rn32(_rn32(Fraction(q - M) / M) * av))
                assert want != int(y_alt[i])
                got = orc.dequant_row(np.array([q], dtype=np.uint8), bins, float(a[i]))
                assert int(got[0]) == want, (bins, q, hex(int(a_bits[i] >> 16)))
                cases += 1
    assert cases >= 10


def test_wnc_middle_half_boundary(orc):
    """A constructed state where, right after an update, high is exactly
    3/4 of the window (0xC0000000) while low lies in [1/4, 1/2): the
    interval does not fit in the middle half (whose last code value is
    0xBFFFFFFF), so no underflow step may be taken. First symbol: table
    0 23407 65536, symbol 1 -> low = 23407 * 2^16, high = 2^32 - 1;
    second: table 0 40049 65536, symbol 0 -> high = low + floor(r * 40049
    / 2^16) - 1 = 0xC0000000."""
    rows = [np.array([0, 23407, 65536], np.uint32), np.array([0, 40049, 65536], np.uint32)]
    r = (1 << 32) - 23407 * 65536
    assert 23407 * 65536 + ((r * 40049) >> 16) - 1 == 0xC0000000
    # By hand: no renormalisation after either symbol; termination adds one
    # pending bit and, with low = 0x5B6F0000 >= 1/4, emits 1 then 0 -> 0x80.
    assert orc.wnc_encode(np.array([1, 0], np.uint8), np.stack(rows)) == bytes([0x80])
    rng = np.random.default_rng(3)
    uni = np.array([0, 16384, 32768, 49152, 65536], np.uint32)
    for tail_len in (0, 1, 3, 17):
        tail = rng.integers(0, 4, tail_len).tolist()
        syms = [1, 0] + tail
        tabs = rows + [uni] * tail_len
        width = max(len(t) for t in tabs)
        padded = np.stack([np.concatenate([t, np.full(width - len(t), 65536, np.uint32)])
                           for t in tabs])
        data = b"".join([orc.wnc_encode(np.array(syms, np.uint8), padded)])
        lo, hi, _ = brute.final_interval(syms, tabs)
        assert brute.dyadic_inside(data, lo, hi)
        got = orc.wnc_decode(data, len(syms), padded)
        assert got.tolist() == syms
