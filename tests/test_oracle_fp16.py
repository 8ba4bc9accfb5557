"""Pins of the oracle's IEEE-754 binary16 conversions.

The oracle's rounding is arithmetic (binade, quantum, floor, tie test).  It is
checked here against (a) a textbook table of binary16 encodings, (b) exhaustive
enumeration of every half value and every midpoint between neighbours, and
(c) numpy's float64 -> float16 conversion, a library routine that rounds
directly from double."""
import math

import numpy as np
import pytest

import oracle
from conftest import golden_lines

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _all_finite_positive_halves():
    pats = np.arange(0x0000, 0x7C00, dtype=np.uint16)  # +0 .. 65504
    return pats, pats.view(np.float16).astype(np.float64)


def test_golden_table():
    for text, bits in golden_lines("fp16_binary16.txt"):
        v = float.fromhex(text) if "0x" in text.lower() else float(text)
        assert oracle.half_from_double(v) == int(bits, 16), (text, bits)


def test_decode_all_patterns_match_numpy():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    for p, r in zip(pats.tolist(), ref.tolist()):
        d = oracle.double_from_half(p)
        if math.isnan(r):
            assert math.isnan(d)
        else:
            assert d == r and math.copysign(1, d) == math.copysign(1, r), hex(p)


def test_roundtrip_every_finite_half():
    for sign in (0, 0x8000):
        for p in range(0, 0x7C00):
            h = p | sign
            assert oracle.half_from_double(oracle.double_from_half(h)) == h


def test_every_midpoint_ties_to_even_and_neighbours_round_away():
    pats, vals = _all_finite_positive_halves()
    for i in range(len(vals) - 1):
        a, b = vals[i], vals[i + 1]
        mid = (a + b) / 2.0  # exact in double
        even = int(pats[i]) if pats[i] % 2 == 0 else int(pats[i + 1])
        assert oracle.half_from_double(mid) == even
        assert oracle.half_from_double(-mid) == even | 0x8000
        assert oracle.half_from_double(np.nextafter(mid, -np.inf)) == int(pats[i])
        assert oracle.half_from_double(np.nextafter(mid, np.inf)) == int(pats[i + 1])


def test_random_doubles_match_numpy():
    rng = np.random.default_rng(7)
    v = rng.standard_normal(100_000) * np.exp2(rng.integers(-30, 17, 100_000))
    ref = v.astype(np.float16).view(np.uint16)
    got = np.array([oracle.half_from_double(t) for t in v.tolist()], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_special_values():
    assert oracle.half_from_double(float("inf")) == 0x7C00
    assert oracle.half_from_double(float("-inf")) == 0xFC00
    assert (oracle.half_from_double(float("nan")) & 0x7FFF) == 0x7E00
    assert oracle.half_from_double(1e300) == 0x7C00
    assert oracle.half_from_double(-1e-300) == 0x8000
