"""Pins of the oracle's Path A (INT8 activations; "Building a Custom LLM
Inference Runtime ...", "3. The INT8 vs. FP16 Activation Trade-off"): the
per-token quantisation against numpy's IEEE binary32 arithmetic (division
and round-half-even done independently), its defining properties, and the
projection against exact rational brute force and a closed form."""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def h2f(b):
    return np.asarray(b, dtype=np.uint16).view(np.float16)


def rand_x(rng, M, K, scale=1.0):
    return (rng.standard_normal((M, K)) * scale).astype(np.float16).view(np.uint16)


@pytest.mark.parametrize("scale", [1.0, 1e-3, 300.0])
def test_quantisation_matches_numpy_binary32(scale):
    rng = np.random.default_rng(int(scale * 10) + 1)
    M, K = 6, 1024
    x = rand_x(rng, M, K, scale)
    xq, sx = oracle.quantize_x8(x)
    xf = h2f(x).astype(np.float32)
    amax = np.max(np.abs(xf), axis=1)
    want_s = (amax / np.float32(127.0)).astype(np.float32)
    assert np.array_equal(sx, want_s)
    t = (xf / want_s[:, None]).astype(np.float32)
    want_q = np.clip(np.rint(t), -127, 127).astype(np.int8)  # np.rint: half to even
    assert np.array_equal(xq, want_q)
    # defining properties: range, the absmax element maps to +-127, error <= sx/2 (+ binary32 rounding)
    assert np.all(np.abs(xq.astype(int)) <= 127)
    for m in range(M):
        i = int(np.argmax(np.abs(xf[m])))
        assert abs(int(xq[m, i])) == 127
        err = np.abs(xq[m].astype(np.float64) * float(sx[m]) - xf[m].astype(np.float64))
        # half a step, plus the binary32 roundings of sx and x / sx (~127 ulps of sx)
        assert np.all(err <= 0.5 * float(sx[m]) + 1e-4 * float(sx[m]) + 1e-30)


def test_quantisation_ties_go_to_even():
    """With max|x| = 127 the step sx is exactly 1, so x / sx = x and every
    half-integer x is a tie: round half to even, as the reading of the
    quantisation states (not half away from zero)."""
    vals = [127.0, 0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 126.5, -125.5, 4.0, -7.25]
    want = [127, 0, 2, 2, 4, 0, -2, -2, 126, -126, 4, -7]
    x = np.array([vals], dtype=np.float16).view(np.uint16)
    xq, sx = oracle.quantize_x8(x)
    assert float(sx[0]) == 1.0
    assert xq[0].tolist() == want


def test_zero_row_quantises_to_zero():
    x = np.zeros((2, 256), dtype=np.uint16)
    xq, sx = oracle.quantize_x8(x)
    assert not xq.any() and not sx.any()


@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (3, 5, 256)])
def test_bruteforce_exact_rationals_q8(M, N, K):
    rng = np.random.default_rng(M + N + K)
    x = rand_x(rng, M, K)
    q = rng.integers(-8, 8, (N, K)).astype(np.int8)
    s = (0.005 + 0.015 * rng.random((N, K // 128))).astype(np.float16).view(np.uint16)
    xq, sx = oracle.quantize_x8(x)
    y, acc = oracle.linear_q8(x, q, s, want_acc=True)
    sf = h2f(s).astype(np.float64)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(sf[n, g])) * Fraction(float(sx[m])) *
                        sum(int(xq[m, k]) * int(q[n, k]) for k in range(128 * g, 128 * g + 128))
                        for g in range(K // 128))
            assert abs(Fraction(acc[m, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 48) + Fraction(1, 2 ** 90)
            assert int(y[m, n]) == oracle.half_from_double(float(exact))


def test_closed_form_all_ones_q8():
    rng = np.random.default_rng(11)
    M, N, K = 2, 4, 384
    x = rand_x(rng, M, K)
    q = np.ones((N, K), dtype=np.int8)
    sv = np.float16(0.0125)
    s = np.full((N, K // 128), sv, dtype=np.float16).view(np.uint16)
    xq, sx = oracle.quantize_x8(x)
    y = oracle.linear_q8(x, q, s)
    for m in range(M):
        want = Fraction(float(sv)) * Fraction(float(sx[m])) * int(xq[m].astype(np.int64).sum())
        assert all(int(y[m, n]) == oracle.half_from_double(float(want)) for n in range(N))
