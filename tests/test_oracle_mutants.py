"""The oracle's pins catch plausible mistakes.  Each case plants one mistake
in a copy of the oracle's C source (a wrong group index, a dropped term, a
tie rounded the wrong way, a transposed layout offset, a wrong sign or
stride; for the gated MLP output, which the oracle forms in Python, a copy
of that function), builds the copy with gcc and runs every oracle pin of the
`test_oracle_*` files against it: at least one pin must fail.  An unmodified
copy built the same way passes them all, so a failure comes from the planted
mistake, not from the harness.  Nothing here touches a GPU."""
import importlib
import inspect
import itertools
import os
import shutil
import subprocess
import warnings

import pytest

import oracle

PIN_MODULES = ["test_oracle_fp16", "test_oracle_bf16", "test_oracle_linear", "test_oracle_pack", "test_oracle_q8",
               "test_oracle_swiglu"]

# name -> [(text in w4_oracle.c, replacement, which occurrence)]
MUTANTS = {
    "group index transposed": [("sn[k / 128]", "sn[k % G]", 0)],
    "last k term dropped": [("for (int64_t k = 0; k < K; ++k) {\n                /* w[n,k]",
                             "for (int64_t k = 0; k < K - 1; ++k) {\n                /* w[n,k]", 0)],
    "weight sign flipped": [("double w = (double)qn[k] *", "double w = -(double)qn[k] *", 0)],
    "x row stride dropped": [("const uint16_t* xm = jb->x + m * K;", "const uint16_t* xm = jb->x + m;", 0)],
    "binary16 ties rounded away": [("if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0))",
                                    "if (frac >= 0.5)", 0)],
    "bfloat16 ties rounded away": [("if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0))",
                                    "if (frac >= 0.5)", 1)],
    "binary16 subnormal scale off by one": [("mag = ldexp((double)f, -24);", "mag = ldexp((double)f, -25);", 0)],
    "layout k offsets 1 and 2 swapped": [
        ("16 * j + 4 * c + 2, 16 * j + 4 * c + 2,\n                                       "
         "16 * j + 4 * c + 1, 16 * j + 4 * c + 1,",
         "16 * j + 4 * c + 1, 16 * j + 4 * c + 1,\n                                       "
         "16 * j + 4 * c + 2, 16 * j + 4 * c + 2,", 0)],
    "layout rows r and r + 8 swapped": [("const int row[8] = {r, r + 8, r, r + 8, r, r + 8, r, r + 8};",
                                         "const int row[8] = {r + 8, r, r + 8, r, r + 8, r, r + 8, r};", 0)],
    "layout two's complement nibbles": [("u = (uint32_t)(q[n * K + k] + 8);", "u = (uint32_t)(q[n * K + k] & 15);", 0)],
    "layout scale halves swapped": [("uint16_t s0 = n0 < N ? s[n0 * G + g] : 0;", "uint16_t s0 = n1 < N ? s[n1 * G + g] : 0;", 0),
                                    ("uint16_t s1 = n1 < N ? s[n1 * G + g] : 0;", "uint16_t s1 = n0 < N ? s[n0 * G + g] : 0;", 0)],
    "Path A ties rounded away": [("r = lrintf(t);", "r = lroundf(t);", 0)],
    "Path A scale of token 0 for every token": [("(double)sx[m] * (double)isum", "(double)sx[0] * (double)isum", 0)],
    "Path A step from 128 instead of 127": [("const float scale = amax / 127.0f;", "const float scale = amax / 128.0f;", 0)],
}

# The gated MLP output is formed in Python (oracle.swiglu): its mistakes are
# planted in a copy of that function.  name -> (text, replacement)
PY_MUTANTS = {
    "SwiGLU sigmoid sign": ("h = g / (1.0 + np.exp(-g)) * u", "h = g / (1.0 + np.exp(g)) * u"),
    "SwiGLU gate and up swapped": ("g, u = acc[:, :I], acc[:, I:]", "u, g = acc[:, :I], acc[:, I:]"),
    "SwiGLU gate rounded to binary16 first": ("g, u = acc[:, :I], acc[:, I:]",
                                              "g, u = acc[:, :I].astype(np.float16).astype(np.float64), acc[:, I:]"),
}


def _replace_nth(src, old, new, nth):
    at = -1
    for _ in range(nth + 1):
        at = src.find(old, at + 1)
        assert at >= 0, "mutation target not found: %r" % old[:60]
    return src[:at] + new + src[at + len(old):]


def _build(tmp_path, edits):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "w4_oracle.c")).read()
    for old, new, nth in edits:
        src = _replace_nth(src, old, new, nth)
    d = tmp_path / "oracle_copy"
    d.mkdir()
    shutil.copy(os.path.join(os.path.dirname(oracle.__file__), "w4_oracle.h"), d / "w4_oracle.h")
    (d / "w4_oracle.c").write_text(src)
    so = str(d / "libw4oracle_copy.so")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", so, str(d / "w4_oracle.c"),
                           "-lm", "-lpthread"])
    return oracle.load(so)


def _pins():
    """Every test function of the oracle pin files, with each parameter set
    its parametrize marks give (functions that need fixtures are left out)."""
    out = []
    for name in PIN_MODULES:
        mod = importlib.import_module(name)
        for fname, fn in sorted(vars(mod).items()):
            if not fname.startswith("test_") or not callable(fn):
                continue
            marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
            params = set(inspect.signature(fn).parameters)
            axes = []
            for m in marks:
                names = [a.strip() for a in m.args[0].split(",")] if isinstance(m.args[0], str) else list(m.args[0])
                vals = [v if len(names) > 1 else (v,) for v in m.args[1]]
                axes.append([dict(zip(names, v)) for v in vals])
            covered = set().union(*[set(a[0]) for a in axes]) if axes else set()
            if params - covered:
                continue
            for combo in itertools.product(*axes) if axes else [()]:
                kw = {}
                for part in combo:
                    kw.update(part)
                out.append(("%s.%s%s" % (name, fname, kw if kw else ""), fn, kw))
    return out


def _failing_pins(monkeypatch, lib):
    monkeypatch.setattr(oracle, "_lib", lib)
    failed = []
    with warnings.catch_warnings():
        warnings.simplefilter("ignore", RuntimeWarning)  # numpy's own overflow notes in the reference casts
        for label, fn, kw in _pins():
            try:
                fn(**kw)
            except Exception as e:  # an assertion, or a return code the wrapper turns into an error
                failed.append("%s: %s" % (label, type(e).__name__))
    return failed


def test_pins_are_collected():
    labels = [p[0] for p in _pins()]
    assert len(labels) >= 30
    assert any("test_bruteforce_exact_rationals" in x for x in labels)
    assert any("test_hand_derived_positions" in x for x in labels)


def test_unmodified_copy_passes_every_pin(tmp_path, monkeypatch):
    assert _failing_pins(monkeypatch, _build(tmp_path, [])) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(tmp_path, monkeypatch, name):
    failed = _failing_pins(monkeypatch, _build(tmp_path, MUTANTS[name]))
    assert failed, "no pin catches: " + name


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_planted_swiglu_mistake_fails_a_pin(monkeypatch, name):
    old, new = PY_MUTANTS[name]
    src = inspect.getsource(oracle.swiglu)
    assert old in src, "mutation target not found: %r" % old
    ns = dict(vars(oracle))
    exec(src.replace(old, new), ns)
    monkeypatch.setattr(oracle, "swiglu", ns["swiglu"])
    failed = _failing_pins(monkeypatch, oracle.lib())
    assert failed, "no pin catches: " + name
