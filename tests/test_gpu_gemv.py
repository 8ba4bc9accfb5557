"""Decode projection (1 <= M <= 16) through the C ABI against the oracle:
small shapes spanning several tiles with ragged tails, every kernel
instantiation and cluster split, determinism, and the full layer shapes at
the launch configuration the benchmark uses (sampled rows)."""
import numpy as np
import pytest

import oracle
from gpu_helpers import (LAYER, assert_close, dev, host, oracle_rows, pack_on_device, rand_problem,
                         sample_rows, synth_weight)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
w4 = pytest.importorskip("int4_weight_only_pack_gb300")


@pytest.fixture(scope="module", autouse=True)
def ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_weight_only_pack_gb300 import build
    build.build()


def run(x, w, N, M, cfg=None):
    y = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    xd = dev(x)
    if cfg is None:
        w4.w4a16_gemv(xd, w, y, M)
    else:
        w4.w4a16_gemv_config(xd, w, y, M, cfg)
    torch.cuda.synchronize()
    return host(y)


SHAPES = [(1, 16, 128), (1, 100, 384), (1, 4608, 3584), (2, 257, 1280), (3, 200, 2560), (4, 64, 18944),
          (5, 40, 18944), (7, 130, 640), (8, 96, 1024), (9, 33, 640), (12, 300, 1152), (13, 100, 2432),
          (16, 512, 3584), (16, 31, 128)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_parity_default_config(M, N, K):
    rng = np.random.default_rng(M * 7919 + N * 31 + K)
    x, q, s = rand_problem(rng, M, N, K)
    _, w = packed_w = pack_on_device(q, s)
    y = run(x, w, N, M)
    assert_close(y, oracle.linear(x, q, s), "M=%d N=%d K=%d" % (M, N, K))


CONFIGS = [(bb, sp, d) for bb, d in [(1, 8), (1, 48), (2, 16), (2, 96), (4, 8), (4, 48)]
           for sp in (1, 2, 3, 5, 8)]


@pytest.mark.parametrize("bb,splits,depth", CONFIGS)
def test_every_instantiation_and_split_nt1(bb, splits, depth):
    M, N, K = 3, 200, 2560  # 20 groups: ragged splits, 13 bands: ragged band blocks
    rng = np.random.default_rng(bb * 100 + splits * 10 + depth)
    x, q, s = rand_problem(rng, M, N, K)
    packed, w = pack_on_device(q, s)
    cfg = w4.GemvConfig(bb, splits, depth, 1)
    assert_close(run(x, w, N, M, cfg), oracle.linear(x, q, s), "cfg %s" % ((bb, splits, depth),))


def test_unsupported_launch_shapes_are_rejected():
    rng = np.random.default_rng(1)
    x, q, s = rand_problem(rng, 1, 32, 256)
    packed, w = pack_on_device(q, s)
    for cfg in [w4.GemvConfig(3, 1, 8, 1), w4.GemvConfig(1, 3, 8, 1), w4.GemvConfig(1, 1, 4, 1),
                w4.GemvConfig(1, 9, 8, 1), w4.GemvConfig(1, 1, 200, 1), w4.GemvConfig(1, 1, 12, 1),
                w4.GemvConfig(1, 1, 8, 1, 3)]:
        with pytest.raises(w4.W4Error) as e:
            run(x, w, 32, 1, cfg)
        assert e.value.status == 7


@pytest.mark.parametrize("bb,splits,depth", [(1, 1, 8), (1, 2, 48), (1, 8, 24), (2, 1, 48), (2, 3, 16),
                                             (4, 1, 48), (4, 5, 8), (4, 8, 48)])
def test_every_instantiation_and_split_nt2(bb, splits, depth):
    M, N, K = 14, 72, 2304
    rng = np.random.default_rng(bb * 100 + splits * 10 + depth + 5000)
    x, q, s = rand_problem(rng, M, N, K)
    packed, w = pack_on_device(q, s)
    cfg = w4.GemvConfig(bb, splits, depth, 0)
    assert_close(run(x, w, N, M, cfg), oracle.linear(x, q, s), "cfg %s" % ((bb, splits, depth),))


@pytest.mark.parametrize("ctas,pdl", [(1, 1), (2, 0), (1, 0)])
def test_launch_variants(ctas, pdl):
    M, N, K = 5, 300, 1536
    rng = np.random.default_rng(ctas * 10 + pdl)
    x, q, s = rand_problem(rng, M, N, K)
    packed, w = pack_on_device(q, s)
    cfg = w4.GemvConfig(0, 0, 0, pdl, ctas)
    assert_close(run(x, w, N, M, cfg), oracle.linear(x, q, s), "ctas %d pdl %d" % (ctas, pdl))


def test_runs_are_bit_identical():
    rng = np.random.default_rng(77)
    M, N, K = 16, 3584, 18944 // 4
    x, q, s = rand_problem(rng, M, N, K)
    packed, w = pack_on_device(q, s)
    ys = [run(x, w, N, M) for _ in range(5)]
    for y in ys[1:]:
        assert np.array_equal(y, ys[0])


def test_extreme_values_stay_within_tolerance():
    """All q = -8 or 7 with the largest scales: the accumulators' widest case."""
    rng = np.random.default_rng(88)
    M, N, K = 4, 48, 3584
    x = (rng.choice([-1, 1], (M, K)) * 2.0).astype(np.float16).view(np.uint16)
    q = rng.choice(np.array([-8, 7], np.int8), (N, K))
    s = np.full((N, K // 128), np.float16(0.02)).view(np.uint16)
    packed, w = pack_on_device(q, s)
    assert_close(run(x, w, N, M), oracle.linear(x, q, s), "extremes")


def test_zero_scales_give_exact_zeros():
    rng = np.random.default_rng(89)
    M, N, K = 2, 40, 512
    x, q, _ = rand_problem(rng, M, N, K)
    s = np.zeros((N, K // 128), np.uint16)
    packed, w = pack_on_device(q, s)
    assert not np.any(run(x, w, N, M) & 0x7FFF)


@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("proj", list(LAYER))
def test_full_layer_shapes_sampled_rows(M, proj):
    """The benchmark's shapes, inputs and launch configuration; the oracle
    computes a sample of rows (all M tokens)."""
    N, K = LAYER[proj]
    pid = list(LAYER).index(proj)
    packed, w = synth_weight(2, 0, pid, N, K)
    rows = sample_rows(np.random.default_rng(pid * 10 + M), N)
    ref, x = oracle_rows(2, 0, pid, M, N, K, rows)
    y = run(x, w, N, M)
    assert_close(y[:, rows], ref, "%s M=%d" % (proj, M))
