"""The C-ABI library without a GPU: it loads, exports every entry point that
include/w4.h declares, and its host-side pack/unpack is bit-exact against the
oracle's writer of the layout.  No device compute is called here."""
import os
import re

import numpy as np
import pytest

import oracle
from conftest import ROOT

w4 = pytest.importorskip("int4_weight_only_pack_gb300")


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_weight_only_pack_gb300 import build
    build.build()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "w4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    names = re.findall(r"\b(w4\w*)\s*\([^;{}]*\)\s*;", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 20
    L = w4.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(w4.EXPORTED)


def test_strerror_and_version():
    assert w4.w4_strerror(0) == "ok"
    assert "[-8, 7]" in w4.w4_strerror(3)
    assert w4.lib().w4_version() >= 10000


@pytest.mark.parametrize("N,K", [(16, 128), (4608 // 64, 3584 // 4), (37, 256), (1, 128), (100, 384)])
def test_packed_bytes(N, K):
    assert w4.w4_packed_bytes(N, K) == ((N + 15) // 16) * (K // 128) * 1056


def test_packed_bytes_of_the_layer_shapes():
    total = sum(w4.w4_packed_bytes(N, K) for N, K in
                [(4608, 3584), (3584, 3584), (37888, 3584), (3584, 18944)])
    assert total == 120_164_352
    assert w4.w4_packed_bytes(4608, 3584) == 8_515_584


@pytest.mark.parametrize("N,K,seed", [(16, 128, 0), (37, 384, 1), (100, 256, 2), (5, 1280, 3)])
def test_host_pack_matches_oracle_layout_bit_exact(N, K, seed):
    rng = np.random.default_rng(seed)
    q = rng.integers(-8, 8, (N, K)).astype(np.int8)
    s = rng.integers(0, 0x7C00, (N, K // 128)).astype(np.uint16)
    got = w4.w4_pack_host(q, s)
    want = oracle.pack_layout(q, s)
    assert np.array_equal(got, want)
    q2, s2 = w4.w4_unpack_host(got, N, K)
    assert np.array_equal(q2, q) and np.array_equal(s2, s)


def test_host_pack_every_nibble_value_in_every_position():
    N, K = 16, 128
    base = np.arange(N * K).reshape(N, K)
    for shift in range(16):
        q = (((base + shift) % 16) - 8).astype(np.int8)
        s = np.full((N, 1), 0x3C00, np.uint16)
        p = w4.w4_pack_host(q, s)
        assert np.array_equal(p, oracle.pack_layout(q, s))
        assert np.array_equal(w4.w4_unpack_host(p, N, K)[0], q)


def test_host_pack_rejects_out_of_range_and_bad_shapes():
    q = np.zeros((4, 128), np.int8)
    s = np.zeros((4, 1), np.uint16)
    q[2, 5] = 8
    with pytest.raises(w4.W4Error) as e:
        w4.w4_pack_host(q, s)
    assert e.value.status == 3
    with pytest.raises(w4.W4Error) as e:
        w4.w4_pack_host(np.zeros((4, 100), np.int8), np.zeros((4, 1), np.uint16))
    assert e.value.status == 2
    assert w4.w4_packed_bytes(0, 128) == 0 and w4.w4_packed_bytes(4, 100) == 0


def test_weight_view_checks():
    w = w4.w4_weight_view(0x1000, 16, 128)
    assert w.magic == w4.W4_PACK_MAGIC and w.version == w4.W4_PACK_VERSION
    with pytest.raises(w4.W4Error) as e:
        w4.w4_weight_view(0x1008, 16, 128)
    assert e.value.status == 4
    with pytest.raises(w4.W4Error) as e:
        w4.w4_weight_view(0x1000, 16, 200)
    assert e.value.status == 2


def test_projection_argument_checks_need_no_gpu():
    """Bad arguments are rejected before anything is launched."""
    w = w4.w4_weight_view(0x1000, 64, 256)
    for M, x, y, code in [(0, 0x2000, 0x3000, 2), (17, 0x2000, 0x3000, 2), (1, 0x2004, 0x3000, 4),
                          (1, 0, 0x3000, 1)]:
        with pytest.raises(w4.W4Error) as e:
            w4.w4a16_gemv(x, w, y, M, stream=0)
        assert e.value.status == code
    bad = w4.Weight(0x1000, 64, 256, 0x12345678, 1)
    with pytest.raises(w4.W4Error) as e:
        w4.w4a16_gemv(0x2000, bad, 0x3000, 1, stream=0)
    assert e.value.status == 1


def test_default_configs_of_the_layer_shapes():
    for M in (1, 2, 4, 8, 16):
        for N, K in [(4608, 3584), (3584, 3584), (37888, 3584), (3584, 18944)]:
            c = w4.w4a16_gemv_default_config(M, N, K)
            assert c.bands_per_cta in (1, 2, 4) and 1 <= c.splits <= 8 and 8 <= c.depth <= 96 and c.depth % 8 == 0
            assert c.ctas_per_sm in (1, 2)


def _sm_count_is_152_or_no_gpu():
    try:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.get_device_properties(0).multi_processor_count == 152
    except ImportError:
        pass
    return True  # no device: the planner assumes 152 SMs


@pytest.mark.skipif(not _sm_count_is_152_or_no_gpu(), reason="the plan below is GB300's (152 SMs)")
def test_step_plan_of_the_benchmarked_step():
    """The persistent step's planner on the benchmarked 28-layer sequence
    (qkv, o, gate_up, down per layer).  At one token only down's K is split,
    four ways (its x slice then fits beside three ring slots per warp), at two
    tokens eight ways, the same for bfloat16 and INT8 activations.  The
    workspace holds the completion counters and status word (768 bytes for
    112 projections) plus, per split projection, an arrival counter per band
    and FP32 partials [bands][S][16 M] (each 256-byte aligned)."""
    layer = [(4608, 3584), (3584, 3584), (37888, 3584), (3584, 18944)]
    ws = [w4.w4_weight_view(0x100000, N, K) for _ in range(28) for N, K in layer]
    for act in ("fp16", "bf16", "int8"):
        assert w4.w4_decode_seq_splits(ws, 1, act) == [1, 1, 1, 4] * 28
        assert w4.w4_decode_seq_splits(ws, 2, act) == [1, 1, 1, 8] * 28
    gated = [0, 0, w4.W4_OP_SWIGLU, 0] * 28
    assert w4.w4_decode_seq_splits(ws, 1, "fp16", gated) == [1, 1, 1, 4] * 28

    def align(v):
        return (v + 255) // 256 * 256

    def down_split(S, M):
        bands = 3584 // 16
        return align(4 * bands) + align(4 * bands * S * 16 * M)

    assert w4.w4_decode_seq_workspace_bytes(ws, 1) == 768 + 28 * down_split(4, 1)
    assert w4.w4_decode_seq_workspace_bytes(ws, 2) == 768 + 28 * down_split(8, 2)
    sizes = [w4.w4_decode_seq_workspace_bytes(ws, M) for M in range(1, 17)]
    assert all(a <= b for a, b in zip(sizes, sizes[1:]))  # partials grow with the tokens


def test_step_splits_argument_checks():
    w = w4.w4_weight_view(0x1000, 16, 128)
    assert w4.w4_decode_seq_splits([w], 1) == [1]  # one tile is never split
    for bad in (0, 17):
        with pytest.raises(w4.W4Error):
            w4.w4_decode_seq_splits([w], bad)
    with pytest.raises(w4.W4Error):
        w4.w4_decode_seq_splits([w4.Weight(0x1000, 16, 128, 0x12345678, 1)], 1)


def test_step_workspace_argument_checks():
    w = w4.w4_weight_view(0x1000, 16, 128)
    assert w4.w4_decode_seq_workspace_bytes([w], 1) == 512  # counters only: one tile is never split
    for M in (0, 17):
        assert w4.w4_decode_seq_workspace_bytes([w], M) == 0
    assert w4.w4_decode_seq_workspace_bytes([w4.Weight(0x1000, 16, 128, 0x12345678, 1)], 1) == 0


@pytest.mark.skipif(not _sm_count_is_152_or_no_gpu(), reason="the plan below is GB300's (152 SMs)")
def test_prefill_plan_of_a_512_token_prompt():
    """The prefill workspace pins the GEMM planner's K splits: a 256-byte head
    (status word) plus FP32 partials [splits][M][N] when K is split.  At 512
    tokens qkv, o and gate_up are not split and down is split 5 ways."""
    head = 256
    for N, K, splits in [(4608, 3584, 1), (3584, 3584, 1), (37888, 3584, 1), (3584, 18944, 5)]:
        want = head + (splits * 512 * N * 4 if splits > 1 else 0)
        assert w4.w4_workspace_bytes(512, N, K) == want, (N, K)
    assert w4.w4_workspace_bytes(16, 3584, 18944) == 0  # the decode kernel needs none
