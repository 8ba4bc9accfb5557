"""The captured decode-step sequence through the C ABI: graph replay, eager
launches and the host-buffer entry point agree bit for bit with one-off
projection calls, and with the oracle; the full 28-layer step (the
benchmark's configuration) is checked on sampled rows of every layer."""
import numpy as np
import pytest

import oracle
import synth
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


MINI = [(160, 256), (128, 256), (640, 256), (128, 1280)]  # a scaled-down layer


def build_chain(M, layers, rng):
    probs, keep, ws, xs, ys = [], [], [], [], []
    for _ in range(layers):
        for N, K in MINI:
            x, q, s = rand_problem(rng, M, N, K)
            packed, w = pack_on_device(q, s)
            keep.append(packed)
            ws.append(w)
            xs.append(dev(x))
            ys.append(torch.zeros((M, N), dtype=torch.int16, device="cuda"))
            probs.append((x, q, s))
    return probs, keep, ws, xs, ys


def make_seq(ws, xs, ys, M, mode):
    """mode: 'pdl' / 'nopdl' graph of kernels, or 'persistent' step kernel."""
    if mode == "persistent":
        nb = w4.w4_decode_seq_workspace_bytes(ws, M)
        buf = torch.zeros(nb + 256, dtype=torch.uint8, device="cuda")
        off = (-buf.data_ptr()) % 256
        wsbuf = buf[off:off + nb]
        seq = w4.DecodeSeq(ws, xs, ys, M, workspace=wsbuf)
        seq._keep = buf
        return seq
    return w4.DecodeSeq(ws, xs, ys, M, use_pdl=(mode == "pdl"))


@pytest.mark.parametrize("M,mode", [(1, "pdl"), (1, "nopdl"), (5, "pdl"), (16, "pdl"), (1, "persistent"),
                                    (3, "persistent"), (8, "persistent"), (16, "persistent")])
def test_replay_matches_oracle_and_single_calls(M, mode):
    rng = np.random.default_rng(M * 10 + len(mode))
    probs, keep, ws, xs, ys = build_chain(M, 3, rng)
    seq = make_seq(ws, xs, ys, M, mode)
    assert seq.kernels() == (1 if mode == "persistent" else len(ws))
    for y in ys:
        y.fill_(0)
    seq.replay()
    torch.cuda.synchronize()
    got = [host(y).copy() for y in ys]
    for i, (x, q, s) in enumerate(probs):
        assert_close(got[i], oracle.linear(x, q, s), "projection %d" % i)
        if mode != "persistent":
            # same kernel and launch shape as a single call: same bits.  (The
            # persistent kernel may split K differently, so only the oracle
            # tolerance and its own run-to-run identity apply to it.)
            single = torch.zeros_like(ys[i])
            w4.w4a16_gemv(xs[i], ws[i], single, M)
            torch.cuda.synchronize()
            assert np.array_equal(host(single), got[i])
    for y in ys:
        y.fill_(0)
    seq.eager()
    torch.cuda.synchronize()
    for i in range(len(ys)):
        assert np.array_equal(host(ys[i]), got[i])
    for _ in range(3):
        seq.replay()
    torch.cuda.synchronize()
    for i in range(len(ys)):
        assert np.array_equal(host(ys[i]), got[i])
    assert seq.status() == 0
    seq.close()


@pytest.mark.parametrize("mode", ["pdl", "persistent"])
def test_run_host_copies_in_replays_and_copies_out(mode):
    M = 2
    rng = np.random.default_rng(3)
    shapes = MINI * 2
    xsz = [M * K for _, K in shapes]
    ysz = [M * N for N, _ in shapes]
    x_arena = torch.zeros(sum(xsz), dtype=torch.int16, device="cuda")
    y_arena = torch.zeros(sum(ysz), dtype=torch.int16, device="cuda")
    keep, ws, xs, ys, probs = [], [], [], [], []
    xo = yo = 0
    for (N, K), nx, ny in zip(shapes, xsz, ysz):
        x, q, s = rand_problem(rng, M, N, K)
        packed, w = pack_on_device(q, s)
        keep.append(packed)
        ws.append(w)
        xs.append(x_arena[xo:xo + nx])
        ys.append(y_arena[yo:yo + ny])
        probs.append((x, q, s))
        xo += nx
        yo += ny
    seq = make_seq(ws, xs, ys, M, mode)
    x_host = torch.from_numpy(np.concatenate([p[0].ravel() for p in probs]).view(np.int16)).pin_memory()
    y_host = torch.zeros(sum(ysz), dtype=torch.int16).pin_memory()
    stream = torch.cuda.current_stream()
    seq.run_host(x_host, x_arena, x_arena.numel() * 2, y_arena, y_host, y_arena.numel() * 2, stream)

    def check(yh, probs):
        yo = 0
        for (x, q, s), (N, _), ny in zip(probs, shapes, ysz):
            assert_close(yh[yo:yo + ny].reshape(M, N), oracle.linear(x, q, s))
            yo += ny

    check(y_host.numpy().view(np.uint16), probs)
    # the same buffers again with new x in the pinned buffer: the graph kept from the first
    # call copies the new values in
    probs2 = [(rand_problem(rng, M, N, K)[0], q, s) for (N, K), (_, q, s) in zip(shapes, probs)]
    x_host.copy_(torch.from_numpy(np.concatenate([p[0].ravel() for p in probs2]).view(np.int16)))
    seq.run_host(x_host, x_arena, x_arena.numel() * 2, y_arena, y_host, y_arena.numel() * 2, stream)
    first = y_host.numpy().view(np.uint16).copy()
    check(first, probs2)
    # another host output buffer: the graph is built again for it, same bits
    y_host2 = torch.full((sum(ysz),), -1, dtype=torch.int16).pin_memory()
    seq.run_host(x_host, x_arena, x_arena.numel() * 2, y_arena, y_host2, y_arena.numel() * 2, stream)
    assert np.array_equal(y_host2.numpy().view(np.uint16), first)
    seq.close()


def test_full_decode_step_sampled():
    """28 layers x 4 projections at M = 1 with distinct seeded weights (the
    benchmark's workload), as a graph of per-projection kernels and as the
    persistent step kernel (the benchmark's launch configuration), each
    replayed twice; every projection of layers 0 and 27 and one projection of
    every other layer is checked on sampled rows."""
    M, CONFIG = 1, 3
    keep, ws, xs, ys, meta = [], [], [], [], []
    for layer in range(28):
        for pid, proj in enumerate(LAYER):
            N, K = LAYER[proj]
            packed, w = synth_weight(CONFIG, layer, pid, N, K)
            x = synth.x_full(synth.seed_of(CONFIG, layer, pid, synth.T_X), M, K)
            keep.append(packed)
            ws.append(w)
            xs.append(dev(x))
            ys.append(torch.zeros((M, N), dtype=torch.int16, device="cuda"))
            meta.append((layer, pid, N, K, x))
    for mode in ("pdl", "persistent"):
        for y in ys:
            y.zero_()
        seq = make_seq(ws, xs, ys, M, mode)
        seq.replay()
        seq.replay()
        torch.cuda.synchronize()
        assert seq.status() == 0
        check_step(meta, ys, CONFIG, M)
        seq.close()


RAGGED = [(200, 1024), (37, 384), (16, 128), (1000, 2432), (3584, 18944), (4608, 3584)]


@pytest.mark.parametrize("M", [1, 2, 3, 4, 6, 7, 9, 12, 13, 15, 16])
def test_persistent_step_ragged_shapes_every_token_count(M):
    """The persistent step kernel on row counts that are not a multiple of 16
    (a padded last band), a one-band one-group projection, a group count with
    no small divisor, the down shape (K split across CTAs; at 16 tokens also
    the smaller x slice) and token counts that pad to 2, 4, 8 and 16: against
    the oracle, and the same bits on a second replay."""
    rng = np.random.default_rng(400 + M)
    probs, keep, ws, xs, ys = [], [], [], [], []
    for N, K in RAGGED:
        x, q, s = rand_problem(rng, M, N, K)
        packed, w = pack_on_device(q, s)
        keep.append(packed)
        ws.append(w)
        xs.append(dev(x))
        ys.append(torch.zeros((M, N), dtype=torch.int16, device="cuda"))
        probs.append((x, q, s))
    seq = make_seq(ws, xs, ys, M, "persistent")
    seq.replay()
    torch.cuda.synchronize()
    assert seq.status() == 0
    got = [host(y).copy() for y in ys]
    for i, (x, q, s) in enumerate(probs):
        assert_close(got[i], oracle.linear(x, q, s), "N=%d K=%d" % RAGGED[i])
    for y in ys:
        y.fill_(0)
    seq.replay()
    torch.cuda.synchronize()
    for i in range(len(ys)):
        assert np.array_equal(host(ys[i]), got[i])
    seq.close()


@pytest.mark.parametrize("M", [4, 16])
def test_full_layer_shapes_step_small_batch_sampled(M):
    """Four layers of the real projection shapes at M tokens through the
    persistent step kernel (the launch configuration the small-batch step is
    timed in: K splits on every projection at 16 tokens), every projection
    checked against the oracle on sampled rows."""
    CONFIG = 3
    keep, ws, xs, ys, meta = [], [], [], [], []
    for layer in range(4):
        for pid, proj in enumerate(LAYER):
            N, K = LAYER[proj]
            packed, w = synth_weight(CONFIG, layer, pid, N, K)
            x = synth.x_full(synth.seed_of(CONFIG, layer, pid, synth.T_X), M, K)
            keep.append(packed)
            ws.append(w)
            xs.append(dev(x))
            ys.append(torch.zeros((M, N), dtype=torch.int16, device="cuda"))
            meta.append((layer, pid, N, K, x))
    seq = make_seq(ws, xs, ys, M, "persistent")
    seq.replay()
    seq.replay()
    torch.cuda.synchronize()
    assert seq.status() == 0
    rng = np.random.default_rng(12)
    for i, (layer, pid, N, K, x) in enumerate(meta):
        rows = np.unique(np.concatenate([[0, 15, 16, N - 1], rng.integers(0, N, 20)]))
        ref, _ = oracle_rows(CONFIG, layer, pid, M, N, K, rows, x_bits=x)
        assert_close(host(ys[i])[:, rows], ref, "layer %d proj %d" % (layer, pid))
    seq.close()


def check_step(meta, ys, CONFIG, M):
    rng = np.random.default_rng(11)
    for i, (layer, pid, N, K, x) in enumerate(meta):
        if layer not in (0, 27) and pid != layer % 4:
            continue
        rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 24)]))
        ref, _ = oracle_rows(CONFIG, layer, pid, M, N, K, rows, x_bits=x)
        assert_close(host(ys[i])[:, rows], ref, "layer %d proj %d" % (layer, pid))


def bf16_problem(rng, M, N, K):
    x = synth.x_full_bf16(int(rng.integers(1 << 62)), M, K)
    q = rng.integers(-8, 8, (N, K)).astype(np.int8)
    s = (0.005 + 0.015 * rng.random((N, K // 128))).astype(np.float16).view(np.uint16)
    return x, q, s


@pytest.mark.parametrize("M", [1, 3, 8, 16])
def test_bf16_sequence_matches_oracle(M):
    """bfloat16 activations through the persistent sequence (scaled-down
    layers plus the K-split down shape), against the oracle's bfloat16
    projection; replays are bit-identical."""
    rng = np.random.default_rng(100 + M)
    shapes = MINI * 2 + [(3584, 18944)]
    probs, keep, ws, xs, ys = [], [], [], [], []
    for N, K in shapes:
        x, q, s = bf16_problem(rng, M, N, K)
        packed, w = pack_on_device(q, s)
        keep.append(packed)
        ws.append(w)
        xs.append(dev(x))
        ys.append(torch.zeros((M, N), dtype=torch.int16, device="cuda"))
        probs.append((x, q, s))
    nb = w4.w4_decode_seq_workspace_bytes(ws, M)
    buf = torch.zeros(nb + 256, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    seq = w4.DecodeSeq(ws, xs, ys, M, workspace=buf[off:off + nb], act="bf16")
    seq.replay()
    torch.cuda.synchronize()
    got = [host(y).copy() for y in ys]
    for i, (x, q, s) in enumerate(probs):
        assert_close(got[i], oracle.linear(x, q, s, act="bf16"), "projection %d" % i, act="bf16")
    seq.replay()
    seq.eager()
    torch.cuda.synchronize()
    for i in range(len(ys)):
        assert np.array_equal(host(ys[i]), got[i])
    assert seq.status() == 0
    seq.close()


def to_bf16_bits(a):
    """float32 values -> bfloat16 bits, round to nearest even (finite values)."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def extreme_bf16_tokens(rng, K):
    """Five tokens of bfloat16 x whose groups of 128 span what binary16 cannot
    hold as they are: ~1e30 (above binary16's range), ~1e-30 (below it),
    all zero, per-group alternation of those with N(0,1), and groups with one
    element of 1e4 among elements of ~1e-6 (a range of 2^33 inside a group,
    wider than the 2^28 the rescale keeps exact)."""
    G = K // 128
    z = rng.standard_normal((5, K)).astype(np.float32)
    x = np.empty_like(z)
    x[0] = z[0] * 1e30
    x[1] = z[1] * 1e-30
    x[2] = 0.0
    scale = np.array([1e30, 1e-30, 0.0, 1.0])[np.arange(G) % 4]
    x[3] = (z[3].reshape(G, 128) * scale[:, None]).ravel()
    x[4] = z[4] * 1e-6
    x[4].reshape(G, 128)[:, 7] = 1e4
    return to_bf16_bits(x)


@pytest.mark.parametrize("M", [1, 2, 5])
def test_bf16_rescale_extreme_ranges(M):
    """The bfloat16 path stages x as binary16 after a power-of-two rescale per
    (group, token): x far above and below binary16's range, zero groups, and a
    group range wider than the rescale keeps exact all come out within the
    bfloat16 tolerance of the oracle, token by token (one- and two-token
    fragment staging, five tokens in natural order; the down shape splits K)."""
    rng = np.random.default_rng(700 + M)
    shapes = [(64, 768), (48, 1280), (3584, 18944)]
    for N, K in shapes:
        xall = extreme_bf16_tokens(rng, K)
        for first in range(0, 5, M):
            x = xall[first:first + M]
            if x.shape[0] < M:
                x = np.concatenate([x, xall[:M - x.shape[0]]])
            q = rng.integers(-8, 8, (N, K)).astype(np.int8)
            s = (0.005 + 0.015 * rng.random((N, K // 128))).astype(np.float16).view(np.uint16)
            packed, w = pack_on_device(q, s)
            y = torch.zeros((M, N), dtype=torch.int16, device="cuda")
            nb = w4.w4_decode_seq_workspace_bytes([w], M)
            buf = torch.zeros(nb + 256, dtype=torch.uint8, device="cuda")
            off = (-buf.data_ptr()) % 256
            seq = w4.DecodeSeq([w], [dev(x)], [y], M, workspace=buf[off:off + nb], act="bf16")
            seq.replay()
            torch.cuda.synchronize()
            assert seq.status() == 0
            got = host(y)
            ref = oracle.linear(x, q, s, act="bf16")
            for m in range(M):
                assert_close(got[m:m + 1], ref[m:m + 1], "N=%d K=%d token %d of %d" % (N, K, first + m, M),
                             act="bf16")
            seq.close()
            del packed


def test_bf16_activation_type_is_checked():
    rng = np.random.default_rng(1)
    x, q, s = rand_problem(rng, 1, 128, 256)
    packed, w = pack_on_device(q, s)
    y = torch.zeros((1, 128), dtype=torch.int16, device="cuda")
    nb = w4.w4_decode_seq_workspace_bytes([w], 1)
    buf = torch.zeros(nb + 256, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    with pytest.raises(KeyError):
        w4.DecodeSeq([w], [dev(x)], [y], 1, workspace=buf[off:off + nb], act="fp8")
    with pytest.raises(ValueError):
        w4.DecodeSeq([w], [dev(x)], [y], 1, act="bf16")  # graph mode is binary16 only
    import ctypes
    warr = (w4.Weight * 1)(w)
    xa = (ctypes.c_void_p * 1)(dev(x).data_ptr())
    ya = (ctypes.c_void_p * 1)(y.data_ptr())
    h = ctypes.c_void_p()
    rc = w4.lib().w4_decode_seq_create_persistent_act(warr, xa, ya, 1, 1, 7, buf[off:].data_ptr(), nb, None,
                                                      ctypes.byref(h))
    assert rc == 1 and not h.value  # W4_ERR_ARG, nothing created


@pytest.mark.parametrize("M,act", [(1, "fp16"), (5, "fp16"), (11, "fp16"), (16, "fp16"), (1, "bf16"), (3, "bf16"),
                                   (8, "bf16")])
def test_swiglu_projection_in_sequence(M, act):
    """Gated MLP projections (W4_OP_SWIGLU, weights from w4_pack_glu) mixed
    with plain ones in one persistent sequence, against the oracle's
    h = rne(silu(g) * u); includes the real gate_up shape (I = 18944)."""
    rng = np.random.default_rng(200 + M)
    plan = [("plain", 160, 256), ("glu", 320, 256), ("plain", 640, 1280), ("glu", 18944, 3584)]
    keep, ws, xs, ys, flags, probs = [], [], [], [], [], []
    for kind, n, K in plan:
        rows = 2 * n if kind == "glu" else n
        if act == "bf16":
            x, q, s = bf16_problem(rng, M, rows, K)
        else:
            x, q, s = rand_problem(rng, M, rows, K)
        packed = torch.empty(w4.w4_packed_bytes(rows, K), dtype=torch.uint8, device="cuda")
        if kind == "glu":
            w = w4.w4_pack_glu(dev(q), dev(s), n, K, packed)
        else:
            w = w4.w4_pack(dev(q), dev(s), rows, K, packed)
        keep.append(packed)
        ws.append(w)
        xs.append(dev(x))
        ys.append(torch.zeros((M, n), dtype=torch.int16, device="cuda"))
        flags.append(w4.W4_OP_SWIGLU if kind == "glu" else 0)
        probs.append((kind, x, q, s))
    nb = w4.w4_decode_seq_workspace_bytes(ws, M)
    buf = torch.zeros(nb + 256, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    seq = w4.DecodeSeq(ws, xs, ys, M, workspace=buf[off:off + nb], act=act, op_flags=flags)
    seq.replay()
    torch.cuda.synchronize()
    assert seq.status() == 0
    for i, (kind, x, q, s) in enumerate(probs):
        ref = oracle.swiglu(x, q, s, act=act) if kind == "glu" else oracle.linear(x, q, s, act=act)
        assert_close(host(ys[i]), ref, "%s projection %d" % (kind, i), act=act)
    seq.close()


def test_swiglu_flag_checks():
    rng = np.random.default_rng(9)
    x, q, s = rand_problem(rng, 1, 40, 256)  # N = 40 is not a gated weight
    packed, w = pack_on_device(q, s)
    y = torch.zeros((1, 20), dtype=torch.int16, device="cuda")
    nb = w4.w4_decode_seq_workspace_bytes([w], 1)
    buf = torch.zeros(nb + 256, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    with pytest.raises(w4.W4Error) as e:
        w4.DecodeSeq([w], [dev(x)], [y], 1, workspace=buf[off:off + nb], op_flags=[w4.W4_OP_SWIGLU])
    assert e.value.status == 2
    with pytest.raises(w4.W4Error) as e:
        w4.DecodeSeq([w], [dev(x)], [y], 1, workspace=buf[off:off + nb], op_flags=[4])
    assert e.value.status == 1
    q2 = rng.integers(-8, 8, (24, 256)).astype(np.int8)  # I = 12: not a multiple of 8
    s2 = (0.005 + 0.015 * rng.random((24, 2))).astype(np.float16).view(np.uint16)
    dst = torch.empty(w4.w4_packed_bytes(24, 256), dtype=torch.uint8, device="cuda")
    with pytest.raises(w4.W4Error) as e:
        w4.w4_pack_glu(dev(q2), dev(s2), 12, 256, dst)
    assert e.value.status == 2


@pytest.mark.parametrize("M", [1, 2, 8, 16])
def test_int8_path_matches_oracle(M):
    """Path A (W4_ACT_I8): x quantised per token to INT8 inside the kernel,
    exact integer group sums, against the oracle's Path A (same binary32
    quantisation decisions, exact integer sums, FP64 scaling).  Includes the
    K-split down shape and an all-zero token."""
    rng = np.random.default_rng(300 + M)
    shapes = MINI + [(3584, 18944), (4608, 3584)]
    probs, keep, ws, xs, ys = [], [], [], [], []
    for N, K in shapes:
        x, q, s = rand_problem(rng, M, N, K)
        if M > 1:
            x[M - 1] = 0  # sx = 0: xq = 0, y = 0
        packed, w = pack_on_device(q, s)
        keep.append(packed)
        ws.append(w)
        xs.append(dev(x))
        ys.append(torch.zeros((M, N), dtype=torch.int16, device="cuda"))
        probs.append((x, q, s))
    nb = w4.w4_decode_seq_workspace_bytes(ws, M)
    buf = torch.zeros(nb + 256, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    seq = w4.DecodeSeq(ws, xs, ys, M, workspace=buf[off:off + nb], act="int8")
    seq.replay()
    torch.cuda.synchronize()
    assert seq.status() == 0
    for i, (x, q, s) in enumerate(probs):
        got = host(ys[i])
        assert_close(got, oracle.linear_q8(x, q, s), "projection %d" % i)
        if M > 1:
            assert np.all((got[M - 1] & 0x7FFF) == 0)
    seq.close()


def test_int8_path_accuracy_against_fp16_activations():
    """What INT8 activations cost in accuracy (the trade-off the pages weigh):
    Path A's y against the unquantised W4A16 oracle, rms error relative to
    rms(y), on the four layer shapes at M = 1 (per-token absmax INT8 keeps it
    near 1%)."""
    rng = np.random.default_rng(7)
    for name, (N, K) in LAYER.items():
        x, q, s = rand_problem(rng, 1, N, K)
        packed, w = pack_on_device(q, s)
        y = torch.zeros((1, N), dtype=torch.int16, device="cuda")
        nb = w4.w4_decode_seq_workspace_bytes([w], 1)
        buf = torch.zeros(nb + 256, dtype=torch.uint8, device="cuda")
        off = (-buf.data_ptr()) % 256
        seq = w4.DecodeSeq([w], [dev(x)], [y], 1, workspace=buf[off:off + nb], act="int8")
        seq.replay()
        torch.cuda.synchronize()
        ya = host(y).view(np.float16).astype(np.float64)
        yb = oracle.linear(x, q, s).view(np.float16).astype(np.float64)
        rel = np.sqrt(np.mean((ya - yb) ** 2)) / np.sqrt(np.mean(yb ** 2))
        assert 1e-4 < rel < 0.03, (name, rel)
        seq.close()
