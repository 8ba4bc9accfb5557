"""Packed-weight file (no GPU): the bytes the library writes are the header
spelled out field by field from the format's definition (built here with
struct, independently of the library) followed by the packed layout, which is
itself checked bit-exactly against the oracle's writer; reading validates
every field and both checksums, and refuses, with W4_ERR_ARG, a file that is
wrong in any of them."""
import struct

import numpy as np
import pytest

import oracle

w4 = pytest.importorskip("int4_weight_only_pack_gb300")

W4_ERR_ARG, W4_ERR_ALIGN, W4_ERR_WORKSPACE = 1, 4, 5


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_weight_only_pack_gb300 import build
    build.build()
    oracle.build()


def fnv1a64(data: bytes) -> int:
    """FNV-1a 64 over little-endian 64-bit words, as the format defines it."""
    assert len(data) % 8 == 0
    h = 0xcbf29ce484222325
    for (w,) in struct.iter_unpack("<Q", data):
        h ^= w
        h = (h * 0x100000001b3) & 0xFFFFFFFFFFFFFFFF
    return h


def expected_header(N, K, payload: bytes) -> bytes:
    head = struct.pack("<8sIIqqIIQQQ", b"W4A16PK1", 1, 256, N, K, 128, 1056, len(payload), 256, fnv1a64(payload))
    assert len(head) == 64
    head += struct.pack("<Q", fnv1a64(head))
    return head + bytes(256 - len(head))


def problem(N, K, seed):
    rng = np.random.default_rng(seed)
    q = rng.integers(-8, 8, size=(N, K), dtype=np.int8)
    s = rng.uniform(0.005, 0.02, size=(N, K // 128)).astype(np.float16).view(np.uint16)
    return q, s


def aligned(nbytes):
    buf = np.zeros(nbytes + 64, dtype=np.uint8)
    off = (-buf.ctypes.data) % 16
    return buf[off:off + nbytes]


@pytest.mark.parametrize("N,K", [(40, 256), (16, 128), (3, 1152)])
def test_write_matches_the_format_and_reads_back(tmp_path, N, K):
    q, s = problem(N, K, N + K)
    packed = w4.w4_pack_host(q, s)
    assert np.array_equal(packed, oracle.pack_layout(q, s))  # the payload is the pinned layout
    path = str(tmp_path / "w.pk")
    w4.w4_file_write(path, w4.w4_weight_view(packed, N, K), src_on_device=False)
    raw = open(path, "rb").read()
    assert raw == expected_header(N, K, packed.tobytes()) + packed.tobytes()
    assert w4.w4_file_info(path) == (N, K, packed.nbytes)
    dst = aligned(packed.nbytes + 32)
    w = w4.w4_file_read(path, dst)
    assert (w.N, w.K, w.data) == (N, K, dst.ctypes.data)
    assert np.array_equal(dst[:packed.nbytes], packed)
    assert np.array_equal(dst[packed.nbytes:], np.zeros(32, np.uint8))


@pytest.mark.parametrize("what", ["magic", "version", "reserved", "header_sum", "payload", "truncated",
                                  "extended", "shape"])
def test_every_corruption_is_refused(tmp_path, what):
    N, K = 40, 256
    q, s = problem(N, K, 7)
    packed = w4.w4_pack_host(q, s)
    path = str(tmp_path / "w.pk")
    w4.w4_file_write(path, w4.w4_weight_view(packed, N, K), src_on_device=False)
    raw = bytearray(open(path, "rb").read())
    if what == "magic":
        raw[0] ^= 0x20
    elif what == "version":
        raw[8] = 2
    elif what == "reserved":
        raw[200] = 1
    elif what == "header_sum":
        raw[64] ^= 1
    elif what == "payload":
        raw[256 + 777] ^= 0x10
    elif what == "truncated":
        raw = raw[:-1]
    elif what == "extended":
        raw += b"\0"
    elif what == "shape":  # a consistent header whose payload size does not fit N x K
        head = bytearray(expected_header(N + 16, K, bytes(packed)))
        raw[:256] = head
    open(path, "wb").write(bytes(raw))
    dst = aligned(packed.nbytes * 2)
    before = dst.copy()
    with pytest.raises(w4.W4Error) as e:
        w4.w4_file_read(path, dst)
    assert e.value.status == W4_ERR_ARG
    assert np.array_equal(dst, before)  # nothing copied
    if what not in ("payload",):
        with pytest.raises(w4.W4Error):
            w4.w4_file_info(path)


def test_destination_checks(tmp_path):
    N, K = 40, 256
    q, s = problem(N, K, 9)
    packed = w4.w4_pack_host(q, s)
    path = str(tmp_path / "w.pk")
    w4.w4_file_write(path, w4.w4_weight_view(packed, N, K), src_on_device=False)
    small = aligned(packed.nbytes - 16)
    with pytest.raises(w4.W4Error) as e:
        w4.w4_file_read(path, small)
    assert e.value.status == W4_ERR_WORKSPACE
    buf = aligned(packed.nbytes + 16)
    with pytest.raises(w4.W4Error) as e:
        w4.w4_file_read(path, buf[4:], packed.nbytes)
    assert e.value.status == W4_ERR_ALIGN
    with pytest.raises(w4.W4Error) as e:
        w4.w4_file_info(str(tmp_path / "missing.pk"))
    assert e.value.status == W4_ERR_ARG
