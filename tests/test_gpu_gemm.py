"""Prefill projection (M > 16) through the C ABI against the oracle."""
import numpy as np
import pytest

import oracle
from gpu_helpers import LAYER, assert_close, dev, host, oracle_rows, pack_on_device, rand_problem, synth_weight

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
w4 = pytest.importorskip("int4_weight_only_pack_gb300")


@pytest.fixture(scope="module", autouse=True)
def ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_weight_only_pack_gb300 import build
    build.build()


def run(x, w, N, M):
    y = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    ws = w4.w4_workspace_bytes(M, N, w.K)
    buf = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    w4.w4a16_gemm(dev(x), w, y, M, buf if ws else None, ws)
    torch.cuda.synchronize()
    return host(y)


# Token tiles are 128 or 192 wide and weight tiles 128 rows (8 bands): the
# cases straddle both boundaries (M = 128, 191, 192, 193, 385, 576; N with a
# partial band and a partial 8-band tile) and include a call that splits K.
@pytest.mark.parametrize("M,N,K", [(17, 64, 256), (40, 136, 384), (128, 256, 512), (512, 256, 1024),
                                   (512, 200, 1280), (300, 128, 2048), (1, 64, 256), (16, 64, 256),
                                   (191, 200, 1024), (192, 128, 512), (193, 136, 4096), (385, 264, 768),
                                   (576, 72, 384)])
def test_parity(M, N, K):
    rng = np.random.default_rng(M + N + K)
    x, q, s = rand_problem(rng, M, N, K)
    packed, w = pack_on_device(q, s)
    assert_close(run(x, w, N, M), oracle.linear(x, q, s), "M=%d N=%d K=%d" % (M, N, K))


# More tiles than SMs: each persistent CTA walks several tiles (token blocks and
# row blocks change between them; (800, 4000, 2560) also splits K), checked on
# sampled rows against the oracle (rows are independent outputs).  y leaves
# through the x stage of each tile's last group and TMA stores where N is a
# multiple of 8 (tile ends exactly 4 groups apart at K = 512: the stage cycle),
# else through plain stores (N = 5002 at 128 tokens, N = 3002 at 192); 2048
# tokens give 16 token blocks.
@pytest.mark.parametrize("M,N,K", [(600, 5000, 512), (800, 4000, 2560), (2048, 2000, 512), (600, 5002, 512),
                                   (1000, 3002, 768)])
def test_parity_several_tiles_per_cta(M, N, K):
    rng = np.random.default_rng(M * 7 + N + K)
    x, q, s = rand_problem(rng, M, N, K)
    packed, w = pack_on_device(q, s)
    y = run(x, w, N, M)
    rows = np.unique(np.concatenate([[0, 15, 127, 128, 1023, 1024, N - 16, N - 1],
                                     rng.integers(0, N, 56)]))
    assert_close(y[:, rows], oracle.linear(x, q[rows], s[rows]), "M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("proj", list(LAYER))
def test_full_layer_shapes_m512_sampled(proj):
    M = 512
    N, K = LAYER[proj]
    pid = list(LAYER).index(proj)
    packed, w = synth_weight(5, 0, pid, N, K)
    rows = np.unique(np.concatenate([[0, 1, N - 1], np.random.default_rng(pid).integers(0, N, 13)]))
    ref, x = oracle_rows(5, 0, pid, M, N, K, rows)
    assert_close(run(x, w, N, M)[:, rows], ref, "%s M=512" % proj)


# 128-token tiles leave y through shared memory and one TMA store per promote
# warp (32 rows x 64 tokens, clipped at M and N) when N is a multiple of 8,
# else through plain stores: a ragged last row block (1000 = 7 x 128 + 104)
# and token block (300 = 2 x 128 + 44, 193 = 128 + 65), and N = 130 (no
# tensor map for y).
# Nothing is written past y.
@pytest.mark.parametrize("M,N,K", [(300, 1000, 512), (193, 1000, 768), (100, 130, 512)])
def test_parity_y_epilogues(M, N, K):
    rng = np.random.default_rng(M + 3 * N + K)
    x, q, s = rand_problem(rng, M, N, K)
    packed, w = pack_on_device(q, s)
    buf = torch.full((M * N + 64,), -1, dtype=torch.int16, device="cuda")
    ws = w4.w4_workspace_bytes(M, N, w.K)
    wsb = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")
    w4.w4a16_gemm(dev(x), w, buf[:M * N], M, wsb if ws else None, ws)
    torch.cuda.synchronize()
    got = host(buf)
    assert_close(got[:M * N].reshape(M, N), oracle.linear(x, q, s), "M=%d N=%d K=%d" % (M, N, K))
    assert np.all(got[M * N:] == 0xFFFF)


# K split: the FP32 partials leave through TMA stores when N is a multiple of
# 4 (300 x 132: 8 splits of 4 groups, the smallest the stage cycle allows),
# else through the promote warps' own stores (301 x 130, 33 x 130); the reduce
# then adds four outputs per thread when M * N is a multiple of 4 (300 x 132),
# else one (301 x 130 and 33 x 130: 39130 and 4290 outputs).
@pytest.mark.parametrize("M,N,K", [(300, 132, 4096), (301, 130, 4096), (33, 130, 8192)])
def test_parity_split_epilogues(M, N, K):
    rng = np.random.default_rng(M * 5 + N + K)
    x, q, s = rand_problem(rng, M, N, K)
    packed, w = pack_on_device(q, s)
    assert w4.w4_workspace_bytes(M, N, K) > 256  # K is split: the partials follow the status word
    assert_close(run(x, w, N, M), oracle.linear(x, q, s), "M=%d N=%d K=%d" % (M, N, K))


def test_deterministic():
    rng = np.random.default_rng(4)
    x, q, s = rand_problem(rng, 256, 512, 1024)
    packed, w = pack_on_device(q, s)
    a, b = run(x, w, 512, 256), run(x, w, 512, 256)
    assert np.array_equal(a, b)
