"""The prefill entry point that allocates nothing (w4a16_gemm_static_scratch).

Some callers cannot allocate device memory: a plugin whose host framework
owns every device allocation, or code that must not call cudaMalloc because
it can synchronise the device or fail at a memory cap.  They cannot hand
w4a16_gemm a workspace, so this entry point takes its scratch from a static
device array inside the library.  Called through the C ABI, it must agree
with the oracle within the tolerance of the other parity tests and give the
same bits as the workspace entry point, call after call, although every call
finds the previous call's leftovers in the shared array: here a shape whose
split-K partials cover the same bytes runs in between.  This file is
collected last so that a first-failure run has already run every other test;
it also passes on its own in a fresh process."""
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


def with_workspace(xd, w, N, M):
    y = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    nbytes = w4.w4_workspace_bytes(M, N, w.K)
    ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    w4.w4a16_gemm(xd, w, y, M, ws if nbytes else None, nbytes)
    torch.cuda.synchronize()
    return host(y)


def static_scratch(xd, w, N, M):
    y = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    w4.w4a16_gemm_static_scratch(xd, w, y, M)
    torch.cuda.synchronize()
    assert w4.w4a16_gemm_static_scratch_status() == 0
    return host(y)


class Problem:
    def __init__(self, M, N, K):
        rng = np.random.default_rng(M * 31 + N + K)
        self.M, self.N, self.K = M, N, K
        self.x, self.q, self.s = rand_problem(rng, M, N, K)
        self.packed, self.w = pack_on_device(self.q, self.s)
        self.xd = dev(self.x)
        self.ref = oracle.linear(self.x, self.q, self.s)
        self.want = with_workspace(self.xd, self.w, N, M)
        assert_close(self.want, self.ref, "workspace entry point M=%d N=%d K=%d" % (M, N, K))

    def check(self, what):
        y = static_scratch(self.xd, self.w, self.N, self.M)
        assert_close(y, self.ref, "%s, static scratch against the oracle" % what)
        assert np.array_equal(y, self.want), "%s: static scratch differs from the workspace entry point" % what


# (M, N, K): one tile, several tiles with a ragged token block, and two
# long-K shapes that split K across CTAs (their FP32 partials live in the
# scratch from byte 256 on, the second's over more bytes than the first's)
@pytest.mark.parametrize("M,N,K", [(40, 136, 384), (512, 256, 1024), (40, 136, 8192)])
def test_matches_the_oracle_and_the_workspace_entry_point_twice(M, N, K):
    p = Problem(M, N, K)
    assert w4.w4_workspace_bytes(M, N, K) <= w4.W4_STATIC_SCRATCH_BYTES
    p.check("first call")
    p.check("second call")


def test_leftovers_of_another_shape_do_not_leak():
    a, b = Problem(40, 136, 8192), Problem(64, 200, 8192)
    need_a, need_b = w4.w4_workspace_bytes(a.M, a.N, a.K), w4.w4_workspace_bytes(b.M, b.N, b.K)
    assert 256 < need_a < need_b <= w4.W4_STATIC_SCRATCH_BYTES  # both split K; b's partials cover a's
    a.check("first shape")
    b.check("second shape over the first's partials")
    a.check("first shape again over the second's partials")


def test_rejects_shapes_beyond_the_scratch():
    M, N, K = 512, 3584, 18944  # split-K partials need ~37 MB
    need = w4.w4_workspace_bytes(M, N, K)
    assert need > w4.W4_STATIC_SCRATCH_BYTES
    w = w4.w4_weight_view(0x100000, N, K)
    with pytest.raises(w4.W4Error) as e:
        w4.w4a16_gemm_static_scratch(0x200000, w, 0x300000, M)
    assert e.value.status == 5
