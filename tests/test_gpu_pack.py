"""Device pack/unpack through the C ABI: bit-exact against the oracle's
writer of the layout, round trips, and the device input generator."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import dev, host, pack_on_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
w4 = pytest.importorskip("int4_weight_only_pack_gb300")


@pytest.fixture(scope="module", autouse=True)
def ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_weight_only_pack_gb300 import build
    build.build()


@pytest.mark.parametrize("N,K", [(300, 384), (4608, 3584)])
def test_device_generator_matches_host_generator(N, K):
    G = K // 128
    sq, ss = synth.seed_of(9, 3, 1, synth.T_Q), synth.seed_of(9, 3, 1, synth.T_SCALE)
    q = torch.empty((N, K), dtype=torch.int8, device="cuda")
    s = torch.empty((N, G), dtype=torch.int16, device="cuda")
    synth.q_device(sq, N, K, q)
    synth.scale_device(ss, N, G, s)
    torch.cuda.synchronize()
    assert np.array_equal(host(q), synth.q_full(sq, N, K))
    assert np.array_equal(host(s), synth.scale_full(ss, N, G))


@pytest.mark.parametrize("N,K,seed", [(16, 128, 0), (37, 384, 1), (1000, 1280, 2), (3584, 2432, 3)])
def test_device_pack_is_bit_exact(N, K, seed):
    rng = np.random.default_rng(seed)
    q = rng.integers(-8, 8, (N, K)).astype(np.int8)
    s = rng.integers(0, 0x7C00, (N, K // 128)).astype(np.uint16)
    packed, w = pack_on_device(q, s)
    assert w.N == N and w.K == K and w.magic == w4.W4_PACK_MAGIC
    assert np.array_equal(host(packed), oracle.pack_layout(q, s))


def test_host_source_pack_to_device_is_bit_exact():
    rng = np.random.default_rng(5)
    N, K = 45, 640
    q = rng.integers(-8, 8, (N, K)).astype(np.int8)
    s = rng.integers(0, 0x7C00, (N, K // 128)).astype(np.uint16)
    packed = torch.empty(w4.w4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    w4.w4_pack(q, s, N, K, packed, src_on_device=False)
    assert np.array_equal(host(packed), oracle.pack_layout(q, s))


@pytest.mark.parametrize("on_device", [True, False])
def test_unpack_round_trip(on_device):
    rng = np.random.default_rng(6)
    N, K = 77, 512
    q = rng.integers(-8, 8, (N, K)).astype(np.int8)
    s = rng.integers(0, 0x7C00, (N, K // 128)).astype(np.uint16)
    packed, w = pack_on_device(q, s)
    if on_device:
        q2 = torch.empty((N, K), dtype=torch.int8, device="cuda")
        s2 = torch.empty((N, K // 128), dtype=torch.int16, device="cuda")
        w4.w4_unpack(w, q2, s2)
        q2, s2 = host(q2), host(s2)
    else:
        q2 = np.empty((N, K), np.int8)
        s2 = np.empty((N, K // 128), np.uint16)
        w4.w4_unpack(w, q2, s2, dst_on_device=False)
    assert np.array_equal(q2, q) and np.array_equal(s2, s)


def test_device_pack_rejects_out_of_range_q():
    q = np.zeros((32, 256), np.int8)
    q[17, 3] = -9
    s = np.zeros((32, 2), np.uint16)
    packed = torch.empty(w4.w4_packed_bytes(32, 256), dtype=torch.uint8, device="cuda")
    with pytest.raises(w4.W4Error) as e:
        w4.w4_pack(dev(q), dev(s), 32, 256, packed)
    assert e.value.status == 3
    with pytest.raises(w4.W4Error) as e:
        w4.w4_pack(q, s, 32, 256, packed, src_on_device=False)
    assert e.value.status == 3
    with pytest.raises(w4.W4Error) as e:
        w4.w4_pack(dev(q), dev(s), 32, 256, packed, dst_bytes=100)
    assert e.value.status == 1


@pytest.mark.parametrize("I,K", [(8, 128), (320, 256), (72, 1152)])
def test_pack_glu_is_the_layout_of_interleaved_rows(I, K):
    """w4_pack_glu equals the oracle's layout writer applied to the stacked
    [gate; up] rows permuted (in numpy) so that band b holds gate rows
    8b..8b+7 then up rows 8b..8b+7."""
    rng = np.random.default_rng(I + K)
    q = rng.integers(-8, 8, (2 * I, K)).astype(np.int8)
    s = (0.005 + 0.015 * rng.random((2 * I, K // 128))).astype(np.float16).view(np.uint16)
    order = np.concatenate([np.concatenate([np.arange(8 * b, 8 * b + 8), I + np.arange(8 * b, 8 * b + 8)])
                            for b in range(I // 8)])
    want = oracle.pack_layout(q[order], s[order])
    dst = torch.zeros(w4.w4_packed_bytes(2 * I, K), dtype=torch.uint8, device="cuda")
    w = w4.w4_pack_glu(dev(q), dev(s), I, K, dst)
    torch.cuda.synchronize()
    assert (w.N, w.K) == (2 * I, K)
    assert np.array_equal(dst.cpu().numpy(), want)
