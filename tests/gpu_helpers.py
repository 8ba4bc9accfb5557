"""Helpers of the GPU parity tests: seeded inputs, device buffers, the
tolerance check.  The expected values always come from the oracle."""
import numpy as np

import oracle
import synth

# (N, K) of one decoder layer's projections (Qwen2.5-7B: hidden 3584,
# intermediate 18944; qkv and gate_up fused)
LAYER = {"qkv": (4608, 3584), "o": (3584, 3584), "gate_up": (37888, 3584), "down": (3584, 18944)}
REL_TOL = 1e-3   # |y - y_ref| <= 1e-3 |y_ref| + 1e-3 rms(y_ref), per element
RMS_TOL = 1e-3


def torch_mod():
    import torch
    return torch


def h2f(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf2f(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_close(y_bits, ref_bits, what="", act="fp16"):
    dec = bf2f if act == "bf16" else h2f
    y, r = dec(y_bits), dec(ref_bits)
    assert y.shape == r.shape, (y.shape, r.shape)
    assert np.all(np.isfinite(y)), what + ": non-finite output"
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    err = np.abs(y - r)
    if act == "bf16":
        # bfloat16 output: one unit in the last place of the reference (the
        # FP32 sum lies within ~1e-5 relative of the exact one, so only the
        # final rounding can differ, by at most one step of 2^-8..2^-7
        # relative, which is wider than the binary16 bound) plus the same
        # rms term
        e = np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -126)))
        bound = 2.0 ** (e - 7) + RMS_TOL * rms
    else:
        bound = REL_TOL * np.abs(r) + RMS_TOL * rms
    bad = err > bound
    if np.any(bad):
        i = np.argwhere(bad)[0]
        raise AssertionError("%s: %d/%d outside tolerance; first at %s: got %r want %r (bound %r)" % (
            what, int(bad.sum()), bad.size, tuple(i), y[tuple(i)], r[tuple(i)], bound[tuple(i)]))


def rand_problem(rng, M, N, K):
    x = rng.standard_normal((M, K)).astype(np.float16).view(np.uint16)
    q = rng.integers(-8, 8, (N, K)).astype(np.int8)
    s = (0.005 + 0.015 * rng.random((N, K // 128))).astype(np.float16).view(np.uint16)
    return x, q, s


def dev(a: np.ndarray):
    torch = torch_mod()
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t) -> np.ndarray:
    a = t.cpu().numpy()
    return a.view(np.uint16) if a.dtype == np.int16 else a


def pack_on_device(q: np.ndarray, s: np.ndarray):
    import int4_weight_only_pack_gb300 as w4
    torch = torch_mod()
    N, K = q.shape
    packed = torch.empty(w4.w4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    w = w4.w4_pack(dev(q), dev(s), N, K, packed)
    return packed, w


def synth_weight(config, layer, proj, N, K):
    """Packed weight of one seeded projection, generated and packed on the
    device (the benchmark's way).  Returns (packed tensor, descriptor)."""
    import int4_weight_only_pack_gb300 as w4
    torch = torch_mod()
    G = K // 128
    q = torch.empty((N, K), dtype=torch.int8, device="cuda")
    s = torch.empty((N, G), dtype=torch.int16, device="cuda")
    synth.q_device(synth.seed_of(config, layer, proj, synth.T_Q), N, K, q)
    synth.scale_device(synth.seed_of(config, layer, proj, synth.T_SCALE), N, G, s)
    packed = torch.empty(w4.w4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    w = w4.w4_pack(q, s, N, K, packed)
    del q, s
    return packed, w


def oracle_rows(config, layer, proj, M, N, K, rows, x_bits=None, act="fp16"):
    """Oracle y[:, rows] of one seeded projection, from host-drawn q and s rows."""
    q, s, x = synth.projection_inputs(config, layer, proj, M, N, K, rows=rows)
    if x_bits is not None:
        x = x_bits
    return oracle.linear(x, q, s, act=act), x


def sample_rows(rng, N, count=48):
    rows = {0, 1, 15, 16, N - 1, N - 16, N // 2}
    rows |= set(rng.integers(0, N, count).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < N))
