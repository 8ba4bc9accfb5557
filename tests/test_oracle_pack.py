"""Pins of the oracle's packed-layout writer.

The layout is this library's design (the pages fix only that the nibbles are
shuffled for the byte-permute datapath: "The .nanoqwen File Format and Safety
Protocols", ValueShuffle).  The oracle writes it from its definition; it is
pinned by hand-derived positions (tests/golden/pack_layout_positions.txt), by
a bijection check (every element of a tile owns exactly one nibble), and by
the padding rule."""
import numpy as np
import pytest

import oracle
from conftest import golden_lines


def test_hand_derived_positions():
    N, K = 32, 256
    q0 = np.zeros((N, K), np.int8)
    s0 = np.zeros((N, K // 128), np.uint16)
    base = oracle.pack_layout(q0, s0)
    assert base.size == 2 * 2 * 1056
    for row in golden_lines("pack_layout_positions.txt"):
        if row[0] == "q":
            n, k, byte, half = int(row[1]), int(row[2]), int(row[3]), row[4]
            q = q0.copy()
            q[n, k] = 7  # u = 15 against a background of u = 8
            out = oracle.pack_layout(q, s0)
            diff = np.nonzero(out != base)[0]
            assert diff.tolist() == [byte], (row, diff[:5])
            nib = (out[byte] & 0xF) if half == "lo" else (out[byte] >> 4)
            assert nib == 0xF
        else:
            n, g, byte = int(row[1]), int(row[2]), int(row[3])
            s = s0.copy()
            s[n, g] = 0x3C01
            out = oracle.pack_layout(q0, s)
            diff = np.nonzero(out != base)[0]
            assert diff.tolist() == [byte, byte + 1]
            assert out[byte] == 0x01 and out[byte + 1] == 0x3C


def test_every_element_owns_one_nibble():
    N, K = 16, 128
    q0 = np.zeros((N, K), np.int8)
    s0 = np.zeros((N, 1), np.uint16)
    base = oracle.pack_layout(q0, s0)
    seen = set()
    for n in range(N):
        for k in range(K):
            q = q0.copy()
            q[n, k] = -8  # u = 0
            out = oracle.pack_layout(q, s0)
            d = np.nonzero(out != base)[0]
            assert len(d) == 1 and d[0] < 1024
            b = int(d[0])
            half = 0 if (out[b] & 0xF) == 0 else 1
            assert (out[b] >> (4 * half)) & 0xF == 0
            seen.add((b, half))
    assert len(seen) == 2048


def test_offset_binary_and_padding_rows():
    N, K = 20, 256
    rng = np.random.default_rng(3)
    q = rng.integers(-8, 8, (N, K)).astype(np.int8)
    s = rng.integers(1, 0x7BFF, (N, 2)).astype(np.uint16)
    out = oracle.pack_layout(q, s)
    assert out.size == 2 * 2 * 1056
    # nibble histogram of band 0 equals the histogram of u = q + 8 over rows 0..15
    band0 = out[:2 * 1056].reshape(2, 1056)[:, :1024]
    nibs = np.concatenate([band0 & 0xF, band0 >> 4]).ravel()
    assert np.array_equal(np.bincount(nibs, minlength=16),
                          np.bincount((q[:16] + 8).ravel(), minlength=16))
    # band 1 holds rows 16..19; rows 20..31 are padding u = 8 with scale 0
    band1 = out[2 * 1056:].reshape(2, 1056)
    nibs1 = np.concatenate([band1[:, :1024] & 0xF, band1[:, :1024] >> 4]).ravel()
    expect = np.bincount((q[16:] + 8).ravel(), minlength=16)
    expect[8] += 12 * 256
    assert np.array_equal(np.bincount(nibs1, minlength=16), expect)
    sc = band1[:, 1024:].copy().view(np.uint16).reshape(2, 8, 2)  # [group, p, (row p, row p+8)]
    for g in range(2):
        for p in range(8):
            assert sc[g, p, 0] == (s[16 + p, g] if 16 + p < N else 0)
            assert sc[g, p, 1] == 0  # rows 24..31 do not exist


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.pack_layout(np.zeros((4, 100), np.int8), np.zeros((4, 1), np.uint16))
    q = np.zeros((4, 128), np.int8)
    q[1, 1] = -9
    with pytest.raises(ValueError):
        oracle.pack_layout(q, np.zeros((4, 1), np.uint16))
