"""ctypes front of the CPU oracle (``oracle/w4_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  Nothing in the product
package imports this module.

The oracle is plain C, FP64, k ascending, one binary16 rounding at the end;
it reads the unpacked int8 q, never the packed layout.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4_oracle.c")
_HDR = os.path.join(_HERE, "w4_oracle.h")
_LIB = os.path.join(_HERE, "libw4oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable C11, no target-specific flags)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = load(_LIB)
    return _lib


def load(path: str) -> ctypes.CDLL:
    """The oracle library at `path` with its entry points typed (a test may
    load a copy built from a modified source)."""
    L = ctypes.CDLL(path)
    L.w4o_double_from_half.restype = ctypes.c_double
    L.w4o_double_from_half.argtypes = [ctypes.c_uint16]
    L.w4o_half_from_double.restype = ctypes.c_uint16
    L.w4o_half_from_double.argtypes = [ctypes.c_double]
    L.w4o_double_from_bf16.restype = ctypes.c_double
    L.w4o_double_from_bf16.argtypes = [ctypes.c_uint16]
    L.w4o_bf16_from_double.restype = ctypes.c_uint16
    L.w4o_bf16_from_double.argtypes = [ctypes.c_double]
    L.w4o_linear_act.restype = ctypes.c_int
    L.w4o_linear_act.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                 ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    L.w4o_quantize_x8.restype = None
    L.w4o_quantize_x8.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                  ctypes.c_void_p]
    L.w4o_linear_q8.restype = ctypes.c_int
    L.w4o_linear_q8.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                ctypes.c_void_p, ctypes.c_void_p]
    L.w4o_linear.restype = ctypes.c_int
    L.w4o_linear.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                             ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    L.w4o_pack_layout.restype = ctypes.c_int
    L.w4o_pack_layout.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    return L


def double_from_half(h: int) -> float:
    return lib().w4o_double_from_half(int(h) & 0xFFFF)


def half_from_double(v: float) -> int:
    return int(lib().w4o_half_from_double(float(v)))


def double_from_bf16(b: int) -> float:
    return lib().w4o_double_from_bf16(int(b) & 0xFFFF)


def bf16_from_double(v: float) -> int:
    return int(lib().w4o_bf16_from_double(float(v)))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def linear(x: np.ndarray, q: np.ndarray, s: np.ndarray, threads: int = 0,
           want_acc: bool = False, act: str = "fp16"):
    """y = rne(x . (q*s)^T) in FP64.  x: uint16 [M,K] activation bits
    (binary16, or bfloat16 with ``act="bf16"``), q: int8 [N,K], s: uint16
    [N,K/128] fp16 bits.  Returns y as uint16 [M,N] bits of the activation
    type (and the FP64 sums if ``want_acc``)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    q = np.ascontiguousarray(q, dtype=np.int8)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    M, K = x.shape
    N = q.shape[0]
    if q.shape != (N, K) or s.shape != (N, K // 128):
        raise ValueError("shape mismatch: x %s q %s s %s" % (x.shape, q.shape, s.shape))
    y = np.zeros((M, N), dtype=np.uint16)
    acc = np.zeros((M, N), dtype=np.float64) if want_acc else None
    if threads <= 0:
        threads = os.cpu_count() or 1
    if act not in ("fp16", "bf16"):
        raise ValueError("act must be fp16 or bf16")
    rc = lib().w4o_linear_act(_ptr(x), 1 if act == "bf16" else 0, _ptr(q), _ptr(s), M, N, K, _ptr(y),
                              _ptr(acc) if acc is not None else None, threads)
    if rc != 0:
        raise ValueError("w4o_linear failed: %d" % rc)
    return (y, acc) if want_acc else y


def quantize_x8(x: np.ndarray):
    """Path A's per-token INT8 quantisation of fp16 x [M, K]: (xq int8, sx float32)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    M, K = x.shape
    xq = np.zeros((M, K), dtype=np.int8)
    sx = np.zeros(M, dtype=np.float32)
    lib().w4o_quantize_x8(_ptr(x), M, K, _ptr(xq), _ptr(sx))
    return xq, sx


def linear_q8(x: np.ndarray, q: np.ndarray, s: np.ndarray, want_acc: bool = False):
    """Path A: y = fp16_rne(sum_g s * sx * sum_k xq * q) (uint16 [M, N])."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    q = np.ascontiguousarray(q, dtype=np.int8)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    M, K = x.shape
    N = q.shape[0]
    y = np.zeros((M, N), dtype=np.uint16)
    acc = np.zeros((M, N), dtype=np.float64) if want_acc else None
    rc = lib().w4o_linear_q8(_ptr(x), _ptr(q), _ptr(s), M, N, K, _ptr(y), _ptr(acc) if acc is not None else None)
    if rc != 0:
        raise ValueError("w4o_linear_q8 failed: %d" % rc)
    return (y, acc) if want_acc else y


def swiglu(x: np.ndarray, q: np.ndarray, s: np.ndarray, threads: int = 0, want_acc: bool = False,
           act: str = "fp16"):
    """Gated MLP output h = rne(silu(g) * u) of a stacked [gate; up] weight
    (q [2I, K], s [2I, K/128]): g and u are the FP64 sums of gate row n and up
    row n (no intermediate rounding), silu(g) = g / (1 + exp(-g)) in FP64.
    SwiGLU is Qwen2.5's MLP activation; the pages do not name it.  Returns h
    as uint16 [M, I] bits of the activation type (and the FP64 h)."""
    _, acc = linear(x, q, s, threads=threads, want_acc=True, act=act)
    I = q.shape[0] // 2
    g, u = acc[:, :I], acc[:, I:]
    with np.errstate(over="ignore"):
        h = g / (1.0 + np.exp(-g)) * u
    enc = bf16_from_double if act == "bf16" else half_from_double
    bits = np.array([enc(v) for v in h.ravel()], dtype=np.uint16).reshape(h.shape)
    return (bits, h) if want_acc else bits


def pack_layout(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """The packed layout of (q, s), written from its definition (uint8)."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    N, K = q.shape
    out = np.zeros(((N + 15) // 16) * (K // 128) * 1056, dtype=np.uint8)
    rc = lib().w4o_pack_layout(_ptr(q), _ptr(s), N, K, _ptr(out))
    if rc != 0:
        raise ValueError("w4o_pack_layout failed: %d" % rc)
    return out
