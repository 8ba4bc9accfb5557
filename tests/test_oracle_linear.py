"""Pins of the oracle's projection y = fp16(x . (q*s)^T).

Each test checks the oracle against something other than itself: exact
rational arithmetic on small inputs (brute force), a closed form, group
isolation, linearity in one group's scale, sign symmetry, and numpy's float64
matmul of the dequantised weights (a library routine).  The quantisation
scheme is the pages' symmetric group-wise INT4 with group 128 and one FP16
scale per group ("Building a Custom LLM Inference Runtime ...", "Technical
Specifications and Hardware Alignment")."""
import bisect
from fractions import Fraction

import numpy as np
import pytest

import oracle

U = 2.0 ** -53
_POS = np.arange(0, 0x7C00, dtype=np.uint16)
_POS_VALS = _POS.view(np.float16).astype(np.float64).tolist()


def h2f(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def nearest_half_by_search(e: Fraction) -> int:
    """binary16 RNE of an exact rational by searching the sorted table of
    all finite halves (independent of the oracle's arithmetic rounding)."""
    sign = 0x8000 if e < 0 else 0
    a = abs(e)
    if a >= Fraction(65520):
        return sign | 0x7C00
    i = bisect.bisect_right(_POS_VALS, a) - 1      # _POS_VALS[i] <= a
    if i == len(_POS_VALS) - 1:                     # between 65504 and 65520
        return sign | int(_POS[i])
    lo, hi = Fraction(_POS_VALS[i]), Fraction(_POS_VALS[i + 1])
    dl, dh = a - lo, hi - a
    if dl < dh or (dl == dh and int(_POS[i]) % 2 == 0):
        return sign | int(_POS[i])
    return sign | int(_POS[i + 1])


def rand_inputs(rng, M, N, K, qlo=-8, qhi=7):
    x = rng.standard_normal((M, K)).astype(np.float16).view(np.uint16)
    q = rng.integers(qlo, qhi + 1, (N, K)).astype(np.int8)
    s = (0.005 + 0.015 * rng.random((N, K // 128))).astype(np.float16).view(np.uint16)
    return x, q, s


def exact_terms(x, q, s, m, n):
    K = x.shape[1]
    xf, sf = h2f(x[m]), h2f(s[n])
    return [Fraction(float(xf[k])) * int(q[n, k]) * Fraction(float(sf[k // 128]))
            for k in range(K)]


@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (3, 5, 256), (2, 17, 384)])
def test_bruteforce_exact_rationals(M, N, K):
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    x, q, s = rand_inputs(rng, M, N, K)
    y, acc = oracle.linear(x, q, s, want_acc=True)
    gamma = K * U / (1 - K * U)
    near_tie = 0
    for m in range(M):
        for n in range(N):
            t = exact_terms(x, q, s, m, n)
            e = sum(t, Fraction(0))
            bound = gamma * float(sum(abs(v) for v in t))
            assert abs(Fraction(float(acc[m, n])) - e) <= Fraction(bound) + Fraction(1, 2 ** 1074)
            want = nearest_half_by_search(e)
            if int(y[m, n]) != want:
                # allowed only if the exact value sits within the FP64 error of a tie
                near_tie += 1
                assert abs(float(e) - float(acc[m, n])) <= bound
    assert near_tie == 0


def test_closed_form_all_q_one_uniform_scale():
    rng = np.random.default_rng(11)
    M, N, K = 3, 7, 512
    x = rng.standard_normal((M, K)).astype(np.float16).view(np.uint16)
    q = np.ones((N, K), dtype=np.int8)
    s0 = np.float16(0.0123)
    s = np.full((N, K // 128), s0).view(np.uint16)
    y = oracle.linear(x, q, s)
    for m in range(M):
        e = Fraction(float(s0)) * sum((Fraction(float(v)) for v in h2f(x[m])), Fraction(0))
        want = nearest_half_by_search(e)
        assert all(int(v) == want for v in y[m])


@pytest.mark.parametrize("g_star", [0, 1, 3])
def test_group_isolation(g_star):
    rng = np.random.default_rng(20 + g_star)
    M, N, K = 2, 9, 512
    x, q, s = rand_inputs(rng, M, N, K)
    s_only = np.zeros_like(s)
    s_only[:, g_star] = s[:, g_star]
    inside = np.zeros_like(x)
    inside[:, 128 * g_star:128 * (g_star + 1)] = x[:, 128 * g_star:128 * (g_star + 1)]
    outside = x.copy()
    outside[:, 128 * g_star:128 * (g_star + 1)] = 0
    y_full = oracle.linear(x, q, s_only)
    assert np.array_equal(y_full, oracle.linear(inside, q, s_only))
    assert not np.any(oracle.linear(outside, q, s_only) & 0x7FFF)
    assert np.any(y_full & 0x7FFF)


def test_linearity_in_one_group_scale():
    rng = np.random.default_rng(31)
    M, N, K = 2, 6, 640
    x, q, s = rand_inputs(rng, M, N, K)
    for n, g in [(0, 0), (3, 2), (5, 4)]:
        s2 = s.copy()
        s2[n, g] = (h2f(s[n, g]) * 2).astype(np.float16).view(np.uint16)  # exact doubling
        only = np.zeros_like(s)
        only[n, g] = s[n, g]
        _, a1 = oracle.linear(x, q, s, want_acc=True)
        _, a2 = oracle.linear(x, q, s2, want_acc=True)
        _, a3 = oracle.linear(x, q, only, want_acc=True)
        tol = 4 * K * U * np.abs(a1).max() + 4 * K * U * np.abs(a3).max()
        assert np.all(np.abs((a2 - a1) - a3) <= tol + 1e-300)
        other = np.ones(N, bool)
        other[n] = False
        assert np.array_equal(a1[:, other], a2[:, other])


def test_sign_symmetry():
    rng = np.random.default_rng(41)
    x, q, s = rand_inputs(rng, 4, 33, 384, qlo=-7, qhi=7)
    y1, a1 = oracle.linear(x, q, s, want_acc=True)
    y2, a2 = oracle.linear(x, (-q).astype(np.int8), s, want_acc=True)
    assert np.array_equal(a2, -a1)
    nz = (y1 & 0x7FFF) != 0
    assert np.array_equal(y2[nz], y1[nz] ^ 0x8000)


def test_matches_float64_library_matmul():
    rng = np.random.default_rng(51)
    M, N, K = 4, 64, 1024
    x, q, s = rand_inputs(rng, M, N, K)
    w = q.astype(np.float64) * np.repeat(h2f(s), 128, axis=1)
    ref = h2f(x) @ w.T
    y, acc = oracle.linear(x, q, s, want_acc=True)
    bound = 2 * K * U * (np.abs(h2f(x)) @ np.abs(w).T)
    assert np.all(np.abs(acc - ref) <= bound)
    assert np.array_equal(y, ref.astype(np.float16).view(np.uint16))


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(61)
    x, q, s = rand_inputs(rng, 3, 101, 256)
    y1, a1 = oracle.linear(x, q, s, threads=1, want_acc=True)
    y8, a8 = oracle.linear(x, q, s, threads=8, want_acc=True)
    assert np.array_equal(y1, y8) and np.array_equal(a1, a8)


def test_rejects_bad_arguments():
    rng = np.random.default_rng(71)
    x, q, s = rand_inputs(rng, 1, 4, 128)
    bad = q.copy()
    bad[0, 0] = 8
    with pytest.raises(ValueError):
        oracle.linear(x, bad, s)
    x2 = np.zeros((1, 100), np.uint16)
    with pytest.raises(ValueError):
        oracle.linear(x2, np.zeros((4, 100), np.int8), np.zeros((4, 0), np.uint16))


def test_empty_shapes():
    y = oracle.linear(np.zeros((0, 128), np.uint16), np.zeros((4, 128), np.int8),
                      np.zeros((4, 1), np.uint16))
    assert y.shape == (0, 4)
