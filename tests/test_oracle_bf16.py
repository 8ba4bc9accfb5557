"""Pins of the oracle's bfloat16 routines and of its BF16-activation
projection, each against something other than the oracle itself:

- decoding: every one of the 65,536 patterns against numpy's IEEE 754 binary32
  decoding of the pattern shifted into the upper half (bfloat16 is, by
  definition, the upper 16 bits of a binary32);
- rounding: round trip of every finite pattern, and random and adversarial
  doubles (exact midpoints, both sides of them, the overflow threshold, the
  subnormal range) against a nearest-value search over the sorted table of
  all finite bfloat16 values with ties to the even pattern;
- the projection with bfloat16 x and y: exact rational brute force and the
  closed form y = bf16(s * sum x) for q = 1.

The BF16-activation variant is the pages' W4A16 projection ("Building a
Custom LLM Inference Runtime ...", "Technical Specifications and Hardware
Alignment") with bfloat16 x and y in place of binary16."""
import bisect
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle

ALL = np.arange(0, 1 << 16, dtype=np.uint32)
with np.errstate(invalid="ignore"):  # NaN patterns
    AS_F32 = (ALL << 16).astype(np.uint32).view(np.float32).astype(np.float64)
_POS = [b for b in range(0, 0x7F80)]                   # +0 .. largest finite
_POS_VALS = [float(AS_F32[b]) for b in _POS]


def nearest_bf16_by_search(v: float) -> int:
    sign = 0x8000 if math.copysign(1.0, v) < 0 else 0
    a = Fraction(abs(v))
    top = Fraction(255) * 2 ** 120
    if a >= top + Fraction(2 ** 119):                  # the midpoint to 2^128
        return sign | 0x7F80
    i = bisect.bisect_right(_POS_VALS, float(a)) - 1
    while Fraction(_POS_VALS[i]) > a:
        i -= 1
    while i + 1 < len(_POS_VALS) and Fraction(_POS_VALS[i + 1]) <= a:
        i += 1
    if i == len(_POS_VALS) - 1:
        return sign | _POS[i]
    lo, hi = Fraction(_POS_VALS[i]), Fraction(_POS_VALS[i + 1])
    dl, dh = a - lo, hi - a
    if dl < dh or (dl == dh and _POS[i] % 2 == 0):
        return sign | _POS[i]
    return sign | _POS[i + 1]


def test_decode_every_pattern_matches_binary32():
    for b in range(1 << 16):
        got = oracle.double_from_bf16(b)
        want = AS_F32[b]
        if math.isnan(want):
            assert math.isnan(got), hex(b)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), hex(b)


def test_round_trip_of_every_finite_pattern():
    for b in range(1 << 16):
        v = AS_F32[b]
        if math.isnan(v):
            r = oracle.bf16_from_double(v)
            assert (r & 0x7FFF) == 0x7FC0 and (r & 0x8000) == (b & 0x8000)
        elif math.isinf(v):
            assert oracle.bf16_from_double(v) == b
        else:
            assert oracle.bf16_from_double(v) == b, hex(b)


def test_rounding_against_table_search():
    rng = np.random.default_rng(1)
    vals = list(rng.standard_normal(3000) * 10.0 ** rng.integers(-45, 39, 3000))
    # exact midpoints between neighbours, and one double either side
    for b in list(rng.integers(1, 0x7F7F, 400)) + [0x0000, 0x007F, 0x0080, 0x3F80, 0x7F7E]:
        lo, hi = Fraction(_POS_VALS[b]), Fraction(_POS_VALS[b + 1])
        mid = float((lo + hi) / 2)
        vals += [mid, math.nextafter(mid, 0.0), math.nextafter(mid, math.inf), -mid]
    top = 255.0 * 2.0 ** 120
    vals += [top, 255.5 * 2.0 ** 120, math.nextafter(255.5 * 2.0 ** 120, 0.0), 1e39, 2.0 ** -140,
             2.0 ** -134, 3 * 2.0 ** -134, 2.0 ** -133 * 0.5, 5e-324]
    for v in vals:
        assert oracle.bf16_from_double(v) == nearest_bf16_by_search(v), v


def bf16_x(rng, M, K):
    xs = rng.standard_normal((M, K))
    return np.array([[oracle.bf16_from_double(v) for v in row] for row in xs], dtype=np.uint16)


@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (2, 5, 256)])
def test_bruteforce_exact_rationals_bf16(M, N, K):
    rng = np.random.default_rng(M * 100 + N + K)
    x = bf16_x(rng, M, K)
    q = rng.integers(-8, 8, (N, K)).astype(np.int8)
    s = (0.005 + 0.015 * rng.random((N, K // 128))).astype(np.float16).view(np.uint16)
    y, acc = oracle.linear(x, q, s, want_acc=True, act="bf16")
    sf = s.view(np.float16).astype(np.float64)
    for m in range(M):
        xv = [Fraction(AS_F32[int(b)]) for b in x[m]]
        for n in range(N):
            exact = sum(xv[k] * int(q[n, k]) * Fraction(float(sf[n, k // 128])) for k in range(K))
            assert abs(Fraction(acc[m, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 80)
            assert y[m, n] == nearest_bf16_by_search(float(exact))


def test_closed_form_all_ones_bf16():
    rng = np.random.default_rng(5)
    M, N, K = 3, 4, 384
    x = bf16_x(rng, M, K)
    q = np.ones((N, K), dtype=np.int8)
    sv = np.float16(0.0137)
    s = np.full((N, K // 128), sv, dtype=np.float16).view(np.uint16)
    y = oracle.linear(x, q, s, act="bf16")
    for m in range(M):
        total = sum(Fraction(AS_F32[int(b)]) for b in x[m]) * Fraction(float(sv))
        assert all(int(y[m, n]) == nearest_bf16_by_search(float(total)) for n in range(N))
