"""Pins of the oracle's gated MLP output h = rne(silu(g) * u) (SwiGLU, the
MLP activation of the pages' model, Qwen2.5; the pages do not name it), each
against something other than the oracle's own formula: a closed form whose
sigmoid is evaluated through tanh (1 + tanh(z/2)) / 2 with exact rational
sums, zero up rows, and the identity of g and u with the two halves of the
plain projection's FP64 sums."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle


def bits_f16(v):
    return np.asarray(v, dtype=np.uint16).view(np.float16).astype(np.float64)


def rand_x(rng, M, K):
    return rng.standard_normal((M, K)).astype(np.float16).view(np.uint16)


@pytest.mark.parametrize("act", ["fp16", "bf16"])
def test_closed_form_through_tanh(act):
    rng = np.random.default_rng(3)
    M, I, K = 4, 8, 256
    if act == "bf16":
        xs = rng.standard_normal((M, K))
        x = np.array([[oracle.bf16_from_double(v) for v in r] for r in xs], dtype=np.uint16)
        xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        x = rand_x(rng, M, K)
        xv = bits_f16(x)
    sg, su = np.float16(0.0125), np.float16(0.0073)
    q = np.ones((2 * I, K), dtype=np.int8)
    s = np.concatenate([np.full((I, K // 128), sg), np.full((I, K // 128), su)]).astype(np.float16).view(np.uint16)
    h, hf = oracle.swiglu(x, q, s, want_acc=True, act=act)
    enc = oracle.bf16_from_double if act == "bf16" else oracle.half_from_double
    for m in range(M):
        tot = sum(Fraction(float(v)) for v in xv[m])
        g, u = float(tot * Fraction(float(sg))), float(tot * Fraction(float(su)))
        want = g * (1.0 + math.tanh(g / 2.0)) / 2.0 * u
        for n in range(I):
            assert abs(hf[m, n] - want) <= 1e-13 * abs(want) + 1e-300
            assert int(h[m, n]) == enc(want)


def test_zero_up_rows_give_zero():
    rng = np.random.default_rng(4)
    M, I, K = 2, 16, 384
    x = rand_x(rng, M, K)
    q = rng.integers(-8, 8, (2 * I, K)).astype(np.int8)
    q[I:] = 0
    s = (0.005 + 0.015 * rng.random((2 * I, K // 128))).astype(np.float16).view(np.uint16)
    h = oracle.swiglu(x, q, s)
    assert np.all((h & 0x7FFF) == 0)


def test_gate_and_up_are_the_plain_projection_halves():
    rng = np.random.default_rng(5)
    M, I, K = 3, 24, 256
    x = rand_x(rng, M, K)
    q = rng.integers(-8, 8, (2 * I, K)).astype(np.int8)
    s = (0.005 + 0.015 * rng.random((2 * I, K // 128))).astype(np.float16).view(np.uint16)
    _, acc = oracle.linear(x, q, s, want_acc=True)
    _, hf = oracle.swiglu(x, q, s, want_acc=True)
    g, u = acc[:, :I], acc[:, I:]
    sig = 0.5 * (1.0 + np.tanh(g / 2.0))
    assert np.allclose(hf, g * sig * u, rtol=1e-13, atol=1e-300)
