"""Exact-rational model of the arithmetic coder, for brute-force checks.

TEST INFRASTRUCTURE (imported by the tests only).

The 32-bit low/high coder of Witten, Neal & Cleary ("Arithmetic coding for
data compression", CACM 30(6), 1987) keeps a 32-bit window onto an interval
of [0, 1). Here the same interval is tracked in absolute terms with
``fractions.Fraction``: a frame [F, F + W) (the part of [0, 1) that the
window spans, W a power of two) and the coding interval [lo, hi) inside it.
The partition of each step uses the same integer floors as the coder
(unit u = W / 2^32, r = (hi - lo) / u), and the frame halves whenever the
interval lies in its lower, upper or middle half. There is no bit output,
no pending-bit bookkeeping and no 32-bit state: what a correct coder must
produce is any codeword whose dyadic interval lies inside the final
[lo, hi).
"""
from __future__ import annotations

from fractions import Fraction

TOTAL = 1 << 16


def final_interval(symbols, cdf_rows):
    """Return (lo, hi, frame_width) after coding ``symbols``; ``cdf_rows[i]``
    is the CDF (0 .. 65536) used for symbol i."""
    F = Fraction(0)
    W = Fraction(1)
    lo = Fraction(0)
    hi = Fraction(1)
    for s, row in zip(symbols, cdf_rows):
        u = W / (1 << 32)
        rr = (hi - lo) / u
        assert rr.denominator == 1
        r = rr.numerator
        lo, hi = lo + (r * int(row[s]) // TOTAL) * u, lo + (r * int(row[s + 1]) // TOTAL) * u
        assert hi > lo
        while True:
            if hi <= F + W / 2:
                W = W / 2
            elif lo >= F + W / 2:
                F = F + W / 2
                W = W / 2
            elif lo >= F + W / 4 and hi <= F + 3 * W / 4:
                F = F + W / 4
                W = W / 2
            else:
                break
    return lo, hi, W


def codeword_value(data: bytes) -> Fraction:
    """The binary fraction 0.b1 b2 ... of a byte string read MSB-first."""
    v = 0
    for b in data:
        v = (v << 8) | b
    return Fraction(v, 1 << (8 * len(data)))


def dyadic_inside(data: bytes, lo: Fraction, hi: Fraction) -> bool:
    """True when every continuation of ``data`` lies in [lo, hi)."""
    v = codeword_value(data)
    return lo <= v and v + Fraction(1, 1 << (8 * len(data))) <= hi


def neg_log2_bounds(width: Fraction):
    """Integers (a, b) with 2^-b <= width < 2^-a... returned as the exact
    floor and ceil of -log2(width)."""
    # find k with 2^-k <= width < 2^-(k-1)
    k = 0
    while Fraction(1, 1 << k) > width:
        k += 1
    # now 2^-k <= width; -log2(width) in (k-1, k]
    exact = Fraction(1, 1 << k) == width
    return (k if exact else k - 1), k
