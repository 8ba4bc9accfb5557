"""Python binding of libw4.so (W4A16 projections for GB300, sm_103a).

Argument marshalling only: every step of the projection runs in the CUDA
library; PyTorch supplies device memory and streams.  The names follow the C
ABI in include/w4.h.  There is no fallback: if libw4.so is missing, every
call raises.

Tensors may be passed as torch tensors (their data_ptr() is used) or as raw
integer addresses; NumPy arrays are accepted where the C entry point takes
host memory.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libw4.so")

W4_OK = 0
W4_PACK_MAGIC = 0x4B503457
W4_PACK_VERSION = 1
STATUS_NAMES = {0: "W4_OK", 1: "W4_ERR_ARG", 2: "W4_ERR_SHAPE", 3: "W4_ERR_RANGE", 4: "W4_ERR_ALIGN",
                5: "W4_ERR_WORKSPACE", 6: "W4_ERR_CUDA", 7: "W4_ERR_UNSUPPORTED"}


class W4Error(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), detail))


class Weight(ctypes.Structure):
    """w4_weight: descriptor of a packed weight in device memory."""
    _fields_ = [("data", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("magic", ctypes.c_uint32), ("version", ctypes.c_uint32)]


class GemvConfig(ctypes.Structure):
    """w4_gemv_config: launch shape of the decode kernel."""
    _fields_ = [("bands_per_cta", ctypes.c_int), ("splits", ctypes.c_int), ("depth", ctypes.c_int),
                ("pdl", ctypes.c_int), ("ctas_per_sm", ctypes.c_int)]


_vp, _i64, _sz, _int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
_SIGNATURES = {
    "w4_strerror": (ctypes.c_char_p, [_int]),
    "w4_last_error": (ctypes.c_char_p, []),
    "w4_version": (_int, []),
    "w4_packed_bytes": (_sz, [_i64, _i64]),
    "w4_weight_view": (_int, [_vp, _i64, _i64, ctypes.POINTER(Weight)]),
    "w4_pack_host": (_int, [_vp, _vp, _i64, _i64, _vp, _sz]),
    "w4_unpack_host": (_int, [_vp, _i64, _i64, _vp, _vp]),
    "w4_pack": (_int, [_vp, _vp, _i64, _i64, _vp, _sz, _int, _vp, ctypes.POINTER(Weight)]),
    "w4_unpack": (_int, [ctypes.POINTER(Weight), _vp, _vp, _int, _vp]),
    "w4_workspace_bytes": (_sz, [_int, _i64, _i64]),
    "w4a16_gemv": (_int, [_vp, ctypes.POINTER(Weight), _vp, _int, _vp, _sz, _vp]),
    "w4a16_gemv_config": (_int, [_vp, ctypes.POINTER(Weight), _vp, _int, ctypes.POINTER(GemvConfig), _vp]),
    "w4a16_gemv_default_config": (_int, [_int, _i64, _i64, ctypes.POINTER(GemvConfig)]),
    "w4a16_gemm": (_int, [_vp, ctypes.POINTER(Weight), _vp, _int, _vp, _sz, _vp]),
    "w4a16_gemm_static_scratch": (_int, [_vp, ctypes.POINTER(Weight), _vp, _int, _vp]),
    "w4a16_gemm_static_scratch_status": (_int, []),
    "w4_decode_seq_create": (_int, [ctypes.POINTER(Weight), ctypes.POINTER(_vp), ctypes.POINTER(_vp), _int, _int,
                                    _int, _vp, ctypes.POINTER(_vp)]),
    "w4_decode_seq_replay": (_int, [_vp, _vp]),
    "w4_decode_seq_eager": (_int, [_vp, _vp]),
    "w4_decode_seq_run_host": (_int, [_vp, _vp, _vp, _sz, _vp, _vp, _sz, _vp]),
    "w4_decode_seq_kernels": (_int, [_vp]),
    "w4_decode_seq_workspace_bytes": (_sz, [ctypes.POINTER(Weight), _int, _int]),
    "w4_decode_seq_create_persistent": (_int, [ctypes.POINTER(Weight), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                               _int, _int, _vp, _sz, _vp, ctypes.POINTER(_vp)]),
    "w4_decode_seq_create_persistent_act": (_int, [ctypes.POINTER(Weight), ctypes.POINTER(_vp),
                                                   ctypes.POINTER(_vp), _int, _int, _int, _vp, _sz, _vp,
                                                   ctypes.POINTER(_vp)]),
    "w4_decode_seq_create_persistent_ex": (_int, [ctypes.POINTER(Weight), ctypes.POINTER(_vp),
                                                  ctypes.POINTER(_vp), ctypes.POINTER(ctypes.c_uint32), _int, _int,
                                                  _int, _vp, _sz, _vp, ctypes.POINTER(_vp)]),
    "w4_pack_glu": (_int, [_vp, _vp, _i64, _i64, _vp, _sz, _int, _vp, ctypes.POINTER(Weight)]),
    "w4_decode_seq_status": (_int, [_vp]),
    "w4_decode_seq_splits": (_int, [ctypes.POINTER(Weight), _int, _int, _int, ctypes.POINTER(ctypes.c_uint32),
                                     ctypes.POINTER(_int)]),
    "w4_decode_seq_destroy": (None, [_vp]),
    "w4_file_write": (_int, [ctypes.c_char_p, ctypes.POINTER(Weight), _int, _vp]),
    "w4_file_info": (_int, [ctypes.c_char_p, ctypes.POINTER(_i64), ctypes.POINTER(_i64), ctypes.POINTER(_sz)]),
    "w4_file_read": (_int, [ctypes.c_char_p, _vp, _sz, _int, _vp, ctypes.POINTER(Weight)]),
}
EXPORTED = tuple(_SIGNATURES)
_lib = None


def lib():
    """The loaded libw4.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libw4.so is not built (%s): run int4_weight_only_pack_gb300.build.build()"
                               % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int):
    if status != W4_OK:
        raise W4Error(status, lib().w4_last_error().decode())


def _addr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def w4_strerror(status: int) -> str:
    return lib().w4_strerror(status).decode()


def w4_packed_bytes(N: int, K: int) -> int:
    return lib().w4_packed_bytes(N, K)


def w4_workspace_bytes(M: int, N: int, K: int) -> int:
    return lib().w4_workspace_bytes(M, N, K)


def w4_weight_view(packed, N: int, K: int) -> Weight:
    w = Weight()
    _check(lib().w4_weight_view(_addr(packed), N, K, ctypes.byref(w)))
    return w


def _on_device(t) -> bool:
    return not isinstance(t, np.ndarray) and getattr(t, "is_cuda", False)


def w4_file_write(path: str, w: Weight, src_on_device: bool, stream=None):
    """Write one packed weight (w.data on the device or the host) to a packed-weight file."""
    _check(lib().w4_file_write(path.encode(), ctypes.byref(w), int(src_on_device),
                               _stream(stream) if src_on_device else None))


def w4_file_info(path: str):
    """(N, K, payload bytes) from a validated packed-weight file header."""
    N, K, nb = _i64(), _i64(), _sz()
    _check(lib().w4_file_info(path.encode(), ctypes.byref(N), ctypes.byref(K), ctypes.byref(nb)))
    return N.value, K.value, nb.value


def w4_file_read(path: str, dst, dst_bytes: int | None = None, stream=None) -> Weight:
    """Validate a packed-weight file and copy its payload into dst (a CUDA
    tensor or a host numpy array); returns the descriptor of dst."""
    dev = _on_device(dst)
    nb = dst_bytes if dst_bytes is not None else (dst.nbytes if isinstance(dst, np.ndarray)
                                                  else dst.numel() * dst.element_size())
    w = Weight()
    _check(lib().w4_file_read(path.encode(), _addr(dst), nb, int(dev), _stream(stream) if dev else None,
                              ctypes.byref(w)))
    return w


def w4_pack_host(q: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Host repack: q int8 [N, K], scales fp16 bits uint16 [N, K/128] -> uint8 bytes."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    N, K = q.shape
    out = np.empty(max(lib().w4_packed_bytes(N, K), 1), dtype=np.uint8)
    _check(lib().w4_pack_host(q.ctypes.data, scales.ctypes.data, N, K, out.ctypes.data, out.size))
    return out


def w4_unpack_host(packed: np.ndarray, N: int, K: int):
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    q = np.empty((N, K), dtype=np.int8)
    s = np.empty((N, K // 128 if K >= 128 else 1), dtype=np.uint16)
    _check(lib().w4_unpack_host(packed.ctypes.data, N, K, q.ctypes.data, s.ctypes.data))
    return q, s


def w4_pack(q, scales, N: int, K: int, dst, dst_bytes: int | None = None, src_on_device: bool | None = None,
            stream=None) -> Weight:
    """Repack into the device buffer ``dst`` (synchronous).  ``q``/``scales``
    are device tensors (src_on_device) or host arrays/tensors."""
    if src_on_device is None:
        src_on_device = not isinstance(q, np.ndarray) and getattr(q, "is_cuda", False)
    if dst_bytes is None:
        dst_bytes = dst.numel() * dst.element_size()
    w = Weight()
    _check(lib().w4_pack(_addr(q), _addr(scales), N, K, _addr(dst), dst_bytes, int(bool(src_on_device)),
                         _stream(stream), ctypes.byref(w)))
    return w


W4_OP_SWIGLU = 1


def w4_pack_glu(q, scales, I: int, K: int, dst, dst_bytes: int | None = None, src_on_device: bool | None = None,
                stream=None) -> Weight:
    """Pack a stacked [gate; up] weight (2I rows) with gate and up rows
    interleaved per band, for a W4_OP_SWIGLU projection."""
    if src_on_device is None:
        src_on_device = _on_device(q)
    if dst_bytes is None:
        dst_bytes = dst.numel() * dst.element_size()
    w = Weight()
    _check(lib().w4_pack_glu(_addr(q), _addr(scales), I, K, _addr(dst), dst_bytes, int(src_on_device),
                             _stream(stream) if src_on_device else None, ctypes.byref(w)))
    return w


def w4_unpack(w: Weight, q_out, s_out, dst_on_device: bool | None = None, stream=None):
    if dst_on_device is None:
        dst_on_device = not isinstance(q_out, np.ndarray) and getattr(q_out, "is_cuda", False)
    _check(lib().w4_unpack(ctypes.byref(w), _addr(q_out), _addr(s_out), int(bool(dst_on_device)), _stream(stream)))


def w4a16_gemv(x, w: Weight, y, M: int, workspace=None, workspace_bytes: int = 0, stream=None):
    _check(lib().w4a16_gemv(_addr(x), ctypes.byref(w), _addr(y), M, _addr(workspace), workspace_bytes,
                            _stream(stream)))


def w4a16_gemv_config(x, w: Weight, y, M: int, cfg: GemvConfig | None, stream=None):
    _check(lib().w4a16_gemv_config(_addr(x), ctypes.byref(w), _addr(y), M,
                                   ctypes.byref(cfg) if cfg is not None else None, _stream(stream)))


def w4a16_gemv_default_config(M: int, N: int, K: int) -> GemvConfig:
    c = GemvConfig()
    _check(lib().w4a16_gemv_default_config(M, N, K, ctypes.byref(c)))
    return c


def w4a16_gemm(x, w: Weight, y, M: int, workspace=None, workspace_bytes: int = 0, stream=None):
    _check(lib().w4a16_gemm(_addr(x), ctypes.byref(w), _addr(y), M, _addr(workspace), workspace_bytes,
                            _stream(stream)))


W4_STATIC_SCRATCH_BYTES = 4 << 20


def w4a16_gemm_static_scratch(x, w: Weight, y, M: int, stream=None):
    """w4a16_gemm without a workspace: the library's static device scratch."""
    _check(lib().w4a16_gemm_static_scratch(_addr(x), ctypes.byref(w), _addr(y), M, _stream(stream)))


def w4a16_gemm_static_scratch_status() -> int:
    """Status word the last static-scratch prefill left on the current device
    (0 = every pipeline wait completed; synchronise its stream first)."""
    return lib().w4a16_gemm_static_scratch_status()


def w4_decode_seq_splits(weights, M: int, act: str = "fp16", op_flags=None):
    """K split per projection of the persistent sequence's plan."""
    n = len(weights)
    flags = (ctypes.c_uint32 * n)(*op_flags) if op_flags is not None else None
    out = (_int * n)()
    _check(lib().w4_decode_seq_splits((Weight * n)(*weights), n, M, DecodeSeq.ACT[act], flags, out))
    return list(out)


def w4_decode_seq_workspace_bytes(weights, M: int) -> int:
    n = len(weights)
    return lib().w4_decode_seq_workspace_bytes((Weight * n)(*weights), n, M)


class DecodeSeq:
    """w4_decode_seq_*: a captured chain of decode projections.  With
    ``workspace`` (a 256-byte-aligned device buffer of
    w4_decode_seq_workspace_bytes), the chain runs as one persistent kernel
    (w4_decode_seq_create_persistent); otherwise as a graph of one kernel per
    projection (w4_decode_seq_create)."""

    ACT = {"fp16": 0, "bf16": 1, "int8": 2}

    def __init__(self, weights, xs, ys, M: int, use_pdl: bool = True, stream=None, workspace=None,
                 workspace_bytes: int | None = None, act: str = "fp16", op_flags=None):
        n = len(weights)
        self._w = (Weight * n)(*weights)
        self._x = (ctypes.c_void_p * n)(*[_addr(t) for t in xs])
        self._y = (ctypes.c_void_p * n)(*[_addr(t) for t in ys])
        self._h = ctypes.c_void_p()
        self.n, self.M = n, M
        self.persistent = workspace is not None
        if self.persistent:
            if workspace_bytes is None:
                workspace_bytes = workspace.numel() * workspace.element_size()
            self._ws = workspace
            flags = None
            if op_flags is not None:
                self._flags = (ctypes.c_uint32 * n)(*op_flags)
                flags = self._flags
            _check(lib().w4_decode_seq_create_persistent_ex(self._w, self._x, self._y, flags, n, M, self.ACT[act],
                                                            _addr(workspace), workspace_bytes, _stream(stream),
                                                            ctypes.byref(self._h)))
        else:
            if act != "fp16" or op_flags is not None:
                raise ValueError("bfloat16 or INT8 activations and projection options need the persistent "
                                 "sequence (pass a workspace)")
            _check(lib().w4_decode_seq_create(self._w, self._x, self._y, n, M, int(use_pdl), _stream(stream),
                                              ctypes.byref(self._h)))

    def status(self) -> int:
        return lib().w4_decode_seq_status(self._h)

    def replay(self, stream=None):
        _check(lib().w4_decode_seq_replay(self._h, _stream(stream)))

    def eager(self, stream=None):
        _check(lib().w4_decode_seq_eager(self._h, _stream(stream)))

    def run_host(self, x_host, x_dev, x_bytes, y_dev, y_host, y_bytes, stream=None):
        _check(lib().w4_decode_seq_run_host(self._h, _addr(x_host), _addr(x_dev), x_bytes, _addr(y_dev),
                                            _addr(y_host), y_bytes, _stream(stream)))

    def kernels(self) -> int:
        return lib().w4_decode_seq_kernels(self._h)

    def close(self):
        if self._h:
            lib().w4_decode_seq_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
