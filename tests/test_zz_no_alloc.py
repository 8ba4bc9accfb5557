"""The prefill entry point that allocates nothing (w4a16_gemm_static_scratch).

It serves callers that cannot allocate device memory themselves and so cannot
hand w4a16_gemm a workspace; its scratch is a static device array inside the
library.  Called through the C ABI, it must give the workspace entry point's
results (within the tolerance of the other parity tests) on two calls in a
row, since the second call finds the first call's leftovers in the array.
This file is collected last so that a first-failure run has already run every
other test; it also passes on its own in a fresh process."""
import numpy as np
import pytest

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


def with_workspace(xd, w, N, M):
    y = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    nbytes = w4.w4_workspace_bytes(M, N, w.K)
    ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    w4.w4a16_gemm(xd, w, y, M, ws if nbytes else None, nbytes)
    torch.cuda.synchronize()
    return host(y)


# (M, N, K): one tile, several tiles with a ragged token block, and a long-K
# shape that splits K across CTAs (its FP32 partials live in the scratch too)
@pytest.mark.parametrize("M,N,K", [(40, 136, 384), (512, 256, 1024), (40, 136, 8192)])
def test_matches_the_workspace_entry_point_twice(M, N, K):
    rng = np.random.default_rng(M * 31 + N + K)
    x, q, s = rand_problem(rng, M, N, K)
    packed, w = pack_on_device(q, s)
    xd = dev(x)
    want = with_workspace(xd, w, N, M)
    assert w4.w4_workspace_bytes(M, N, K) <= w4.W4_STATIC_SCRATCH_BYTES
    for _ in range(2):
        y = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
        w4.w4a16_gemm_static_scratch(xd, w, y, M)
        torch.cuda.synchronize()
        assert_close(host(y), want, "static scratch M=%d N=%d K=%d" % (M, N, K))


def test_rejects_shapes_beyond_the_scratch():
    M, N, K = 512, 3584, 18944  # split-K partials need ~37 MB
    need = w4.w4_workspace_bytes(M, N, K)
    assert need > w4.W4_STATIC_SCRATCH_BYTES
    w = w4.w4_weight_view(0x100000, N, K)
    with pytest.raises(w4.W4Error) as e:
        w4.w4a16_gemm_static_scratch(0x200000, w, 0x300000, M)
    assert e.value.status == 5
