"""Seeded synthetic inputs for the W4A16 projection path (host side).

This module is the only code shared by the oracle's callers and the CUDA
path's callers.  It draws random numbers; it contains none of the
projection's arithmetic (no dequantisation, no dot products, no packing).

Generator: splitmix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014).  A stream started at state
``seed`` yields, as its i-th output (i = 0, 1, ...),

    r_i = mix64(seed + (i + 1) * 0x9E3779B97F4A7C15)   (mod 2**64)

with the published finaliser

    z ^= z >> 30; z *= 0xBF58476D1CE4E5B9
    z ^= z >> 27; z *= 0x94D049BB133111EB
    z ^= z >> 31

Because every element is a function of (seed, index) alone, any row or any
sample of a tensor can be drawn without drawing the rest, and the device
generator (``synth/gen.cu``) produces the same bits.

Distributions (the workloads of the Qwen2.5-7B projection shapes):
  q  int8   uniform over the 16 values [-8, 7]:  q_i = (r_i >> 60) - 8
  s  fp16   uniform in [0.005, 0.02]:            U = (r_i >> 11) * 2**-53,
            v = 0.005 + (0.015 * U)  (a product and a sum, each rounded once
            in float64, never fused), s = binary16 round-to-nearest-even(v)
  x  fp16   N(0, 1) by Box-Muller in float64, rounded to binary16 (RNE):
            U1 = ((r_i >> 32) + 1) * 2**-32 in (0, 1],
            U2 = (r_i & 0xFFFFFFFF) * 2**-32 in [0, 1),
            x_i = sqrt(-2 ln U1) * cos(2 pi U2)
x is drawn on the host only (it is small), so its transcendental functions
never need to agree between two implementations.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1

# tensor ids inside one projection's seed family
T_Q, T_SCALE, T_X = 0, 1, 2
# projection ids in the order a decoder layer runs them
PROJ_NAMES = ("qkv", "o", "gate_up", "down")


def _mix64_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def seed_of(config: int, layer: int, proj: int, tensor: int) -> int:
    """Seed of one tensor: the first splitmix64 output of a stream whose
    state is a tag built from (config, layer, projection, tensor)."""
    tag = (0x57344131 ^ (config << 48) ^ (layer << 40) ^ (proj << 32) ^ tensor) & _MASK64
    return _mix64_int(tag + 0x9E3779B97F4A7C15)


def draws(seed: int, index: np.ndarray) -> np.ndarray:
    """r_i for the element indices ``index`` (any shape, int64/uint64)."""
    idx = np.asarray(index, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & _MASK64) + (idx + np.uint64(1)) * GOLDEN
    return mix64(z)


def _row_index(rows: np.ndarray, width: int) -> np.ndarray:
    rows = np.asarray(rows, dtype=np.uint64).reshape(-1, 1)
    return rows * np.uint64(width) + np.arange(width, dtype=np.uint64).reshape(1, -1)


def q_rows(seed: int, K: int, rows) -> np.ndarray:
    """int8 q[rows, K] of the [N, K] tensor with this seed (row-major index n*K+k)."""
    r = draws(seed, _row_index(rows, K))
    return ((r >> np.uint64(60)).astype(np.int16) - 8).astype(np.int8)


def q_full(seed: int, N: int, K: int) -> np.ndarray:
    return q_rows(seed, K, np.arange(N))


def scale_rows(seed: int, G: int, rows) -> np.ndarray:
    """fp16 bit patterns (uint16) of s[rows, G] of the [N, G] scale tensor."""
    r = draws(seed, _row_index(rows, G))
    u = (r >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    prod = np.float64(0.015) * u          # rounded once
    v = np.float64(0.005) + prod          # rounded once
    return v.astype(np.float16).view(np.uint16)


def scale_full(seed: int, N: int, G: int) -> np.ndarray:
    return scale_rows(seed, G, np.arange(N))


def x_full(seed: int, M: int, K: int) -> np.ndarray:
    """fp16 bit patterns (uint16) of x[M, K] ~ N(0, 1)."""
    r = draws(seed, np.arange(M * K, dtype=np.uint64)).reshape(M, K)
    u1 = ((r >> np.uint64(32)).astype(np.float64) + 1.0) * (2.0 ** -32)
    u2 = (r & np.uint64(0xFFFFFFFF)).astype(np.float64) * (2.0 ** -32)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return z.astype(np.float16).view(np.uint16)


def x_full_bf16(seed: int, M: int, K: int) -> np.ndarray:
    """bfloat16 bit patterns (uint16) of the same N(0, 1) draws as x_full:
    the draws go to binary32, then to the nearest bfloat16 (ties to even on
    the binary32 pattern).  An input recipe only: any fixed rounding would do,
    as both sides read the same bits."""
    r = draws(seed, np.arange(M * K, dtype=np.uint64)).reshape(M, K)
    u1 = ((r >> np.uint64(32)).astype(np.float64) + 1.0) * (2.0 ** -32)
    u2 = (r & np.uint64(0xFFFFFFFF)).astype(np.float64) * (2.0 ** -32)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    b = z.astype(np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def projection_inputs(config: int, layer: int, proj: int, M: int, N: int, K: int,
                      rows=None):
    """(q, s, x) of one projection; ``rows`` limits q and s to a sample of rows."""
    G = K // 128
    sq = seed_of(config, layer, proj, T_Q)
    ss = seed_of(config, layer, proj, T_SCALE)
    sx = seed_of(config, layer, proj, T_X)
    if rows is None:
        rows = np.arange(N)
    return q_rows(sq, K, rows), scale_rows(ss, G, rows), x_full(sx, M, K)


# ---- device generator (synth/gen.cu) ------------------------------------
_HERE = os.path.dirname(os.path.abspath(__file__))
_GEN_SRC = os.path.join(_HERE, "gen.cu")
_GEN_LIB = os.path.join(_HERE, "libsynth.so")
_gen = None


def build_device(force: bool = False) -> str:
    """Compile the device generator for sm_103a (nvcc)."""
    if force or not os.path.exists(_GEN_LIB) or os.path.getmtime(_GEN_LIB) < os.path.getmtime(_GEN_SRC):
        nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
        tmp = _GEN_LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                               "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared", "-o", tmp, _GEN_SRC])
        os.replace(tmp, _GEN_LIB)
    return _GEN_LIB


def _device_lib():
    global _gen
    if _gen is None:
        build_device()
        L = ctypes.CDLL(_GEN_LIB)
        for name in ("synth_q_device", "synth_scale_device"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
        _gen = L
    return _gen


def q_device(seed: int, N: int, K: int, out, stream=None):
    """Fill the int8 device tensor ``out`` ([N, K]) with q of this seed."""
    import torch
    st = (stream or torch.cuda.current_stream()).cuda_stream
    rc = _device_lib().synth_q_device(seed & _MASK64, 0, N * K, out.data_ptr(), st)
    if rc != 0:
        raise RuntimeError("synth_q_device failed: cuda error %d" % rc)


def scale_device(seed: int, N: int, G: int, out, stream=None):
    """Fill the int16/uint16 device tensor ``out`` ([N, G]) with fp16 scale bits."""
    import torch
    st = (stream or torch.cuda.current_stream()).cuda_stream
    rc = _device_lib().synth_scale_device(seed & _MASK64, 0, N * G, out.data_ptr(), st)
    if rc != 0:
        raise RuntimeError("synth_scale_device failed: cuda error %d" % rc)
