"""Packed-weight file on the GPU: a weight packed on the device, written from
device memory, read back into a fresh device buffer through the C ABI, gives
the same bytes and, through the decode kernel, outputs within tolerance of
the oracle."""
import numpy as np
import pytest

import oracle
from gpu_helpers import assert_close, dev, host, pack_on_device, rand_problem

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
w4 = pytest.importorskip("int4_weight_only_pack_gb300")


@pytest.fixture(scope="module", autouse=True)
def ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_weight_only_pack_gb300 import build
    build.build()


@pytest.mark.parametrize("M,N,K", [(1, 4608, 3584), (3, 200, 1280)])
def test_device_round_trip_and_gemv(tmp_path, M, N, K):
    rng = np.random.default_rng(N)
    x, q, s = rand_problem(rng, M, N, K)
    packed, w = pack_on_device(q, s)
    path = str(tmp_path / "w.pk")
    w4.w4_file_write(path, w, src_on_device=True)
    assert w4.w4_file_info(path) == (N, K, w4.w4_packed_bytes(N, K))
    dst = torch.zeros(w4.w4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    w2 = w4.w4_file_read(path, dst)
    torch.cuda.synchronize()
    assert torch.equal(dst, packed[:dst.numel()])
    y = torch.zeros((M, N), dtype=torch.int16, device="cuda")
    w4.w4a16_gemv(dev(x), w2, y, M)
    torch.cuda.synchronize()
    assert_close(host(y), oracle.linear(x, q, s))
