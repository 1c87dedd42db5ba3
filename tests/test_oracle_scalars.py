"""Pins of the oracle's scalar rules against closed forms and exact arithmetic.

Rules ("Integer On-Device Training: Overview", section 3, NITI Steps 2-5):
bits_needed = ceil(log2(max_val + 1)), shift = max(0, bits_needed - target_bits),
round-half-up shift, weight_shift = max(0, shift - mu_weight), sat_int8.
"""
from fractions import Fraction
import math

import pytest

import oracle as O


def exact_ceil_log2_plus1(m: int) -> int:
    # smallest k with 2^k >= m + 1, by integer comparison only
    k = 0
    while (1 << k) < m + 1:
        k += 1
    return k


def test_bitlen_small_exhaustive_vs_bit_length():
    # int.bit_length is the number of binary digits: equal to ceil(log2(m+1))
    for m in range(0, 1 << 20, 1):
        if m < 4096 or m % 97 == 0:
            assert O.bitlen(m) == m.bit_length()


def test_bitlen_powers_of_two_neighbourhood():
    for k in range(0, 33):
        for m in (max(0, (1 << k) - 1), 1 << k, (1 << k) + 1):
            if m < (1 << 32):
                assert O.bitlen(m) == exact_ceil_log2_plus1(m), m


def test_bitlen_matches_log2_where_float_is_safe():
    # away from exact powers of two, float log2 agrees with the exact value
    for m in range(1, 5000):
        if (m + 1) & m:  # m + 1 not a power of two
            assert O.bitlen(m) == math.ceil(math.log2(m + 1))


@pytest.mark.parametrize("m,bits,s,ws", [
    (0, 0, 0, 0), (1, 1, 0, 0), (127, 7, 0, 0), (128, 8, 1, 0), (255, 8, 1, 0),
    (256, 9, 2, 0), (511, 9, 2, 0), (512, 10, 3, 1), (65535, 16, 9, 7),
    (65536, 17, 10, 8), (1 << 31, 32, 25, 23),
])
def test_shift_table(m, bits, s, ws):
    assert O.bitlen(m) == bits
    assert O.shift_from_max(m, 7) == s
    assert max(0, O.shift_from_max(m, 7) - 2) == ws


def rhu_exact(x: int, s: int) -> int:
    return math.floor(Fraction(x, 1 << s) + Fraction(1, 2))


def test_rhu_exhaustive_exact_rational():
    for s in range(0, 13):
        for x in range(-4096, 4097):
            assert O.rhu(x, s) == rhu_exact(x, s), (x, s)


@pytest.mark.parametrize("x,s,want", [
    (3, 1, 2), (-3, 1, -1), (1, 1, 1), (-1, 1, 0), (128, 1, 64), (-128, 1, -64),
    (255, 1, 128), (-255, 1, -127), (-511, 2, -128), (511, 2, 128), (5, 0, 5),
    (-7, 0, -7), (-2, 2, 0), (-6, 2, -1), (6, 2, 2), (2, 2, 1),
])
def test_rhu_hand_cases(x, s, want):
    assert O.rhu(x, s) == want


def test_rhu_large_operands():
    for x in (2**31 - 1, -2**31, 2**40 + 12345, -(2**41) - 7):
        for s in (1, 5, 17, 30, 45):
            assert O.rhu(x, s) == rhu_exact(x, s)
    assert O.rhu(-(2**40), 63) == 0 and O.rhu(2**40, 70) == 0


@pytest.mark.parametrize("v,want", [(-129, -128), (-128, -128), (0, 0), (127, 127), (128, 127),
                                    (10**9, 127), (-10**9, -128)])
def test_sat8(v, want):
    assert O.sat8(v) == want


@pytest.mark.parametrize("v,want", [(-32768, -32767), (-32767, -32767), (32767, 32767),
                                    (32768, 32767), (5, 5)])
def test_sat16(v, want):
    assert O.sat16(v) == want
