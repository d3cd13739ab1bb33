"""CPU checks of two floating-point procedures of the CUDA kernels, emulated
operation for operation in tests/fp_emulation.c (no GPU needed):

* the FP8 quantiser divides by the block scale with one Markstein FMA
  correction of x * RN(1/s) instead of an IEEE division, and takes each
  code's sign from x; swept over every bf16 amax >= 2^-64 and every bf16
  |x| <= amax, its quotient must equal RN(x / s) except where both are so
  small that the e4m3 code is a signed zero (the codes, which the pages fix
  -- "[Infra-10] All-to-All Optimization", 4.1, FP8 on the wire; pplx blog,
  "Dispatch", block scale factors -- are then identical);
* the router's softmax weights are evaluated in float-float arithmetic; on
  millions of top-8 weights they must be within one fp32 ulp of the oracle's
  double softmax rounded to fp32, and the float-float exp itself must carry
  about 42 correct bits over the range the kernel uses.
"""
import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fp_emulation.c")
LIB = os.path.join(HERE, "_build", "libfp_emulation.so")

_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


@pytest.fixture(scope="module")
def emu():
    if not (os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        os.makedirs(os.path.dirname(LIB), exist_ok=True)
        tmp = LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-Wall", "-o", tmp, SRC, "-lm"])
        os.replace(tmp, LIB)
    lib = ctypes.CDLL(LIB)
    lib.emu_fmaf.restype = ctypes.c_float
    lib.emu_fmaf.argtypes = [ctypes.c_float] * 3
    p64 = ctypes.POINTER(ctypes.c_int64)
    lib.markstein_sweep.restype = None
    lib.markstein_sweep.argtypes = [ctypes.c_uint32, ctypes.c_uint32, p64, p64, p64,
                                    ctypes.POINTER(ctypes.c_double)]
    lib.markstein_many.restype = None
    lib.markstein_many.argtypes = [ctypes.c_int64, _f32p, _f32p, _f32p]
    lib.ff_exp_many.restype = None
    lib.ff_exp_many.argtypes = [ctypes.c_int64, _f32p, _f64p]
    lib.ff_softmax_many.restype = None
    lib.ff_softmax_many.argtypes = [ctypes.c_int64, ctypes.c_int, _f32p, _f32p]
    return lib


def _threads():
    return max(1, min(16, os.cpu_count() or 1))


def test_emulated_fma_is_the_correctly_rounded_fma(emu):
    """The emulated fmaf against exact rational arithmetic (Python fractions)."""
    from fractions import Fraction
    rng = np.random.default_rng(21)
    a = (rng.standard_normal(3000) * 2.0 ** rng.integers(-30, 30, 3000)).astype(np.float32)
    b = (rng.standard_normal(3000) * 2.0 ** rng.integers(-30, 30, 3000)).astype(np.float32)
    c = (-(a.astype(np.float64) * b) * (1 + rng.standard_normal(3000) * 2.0 ** -20)).astype(
        np.float32)  # near-cancellation: the cases a separate multiply gets wrong
    for x, y, z in zip(a, b, c):
        exact = Fraction(float(x)) * Fraction(float(y)) + Fraction(float(z))
        got = emu.emu_fmaf(float(x), float(y), float(z))
        # the float nearest the exact value (ties to even), by comparing neighbours
        g = np.float32(got)
        lo, hi = np.nextafter(g, np.float32(-np.inf)), np.nextafter(g, np.float32(np.inf))
        d = abs(Fraction(float(g)) - exact)
        assert d <= abs(Fraction(float(lo)) - exact) and d <= abs(Fraction(float(hi)) - exact)


def test_markstein_quotient_gives_the_ieee_codes_exhaustively(emu):
    """Every positive finite bf16 amax >= 2^-64 (encodings 0x1F80..0x7F7F) and
    every non-negative bf16 x <= amax: about 5.0e8 pairs. The steps are odd in
    x (round to nearest is symmetric and the sign is carried over), so the
    negative half follows; a sampled check below covers it too."""
    lo, hi = 0x1F80, 0x7F80
    n = _threads() * 4
    # the inner loop length grows with amax: cut the range into pieces of
    # about equal work (work ~ amax encoding)
    enc = np.arange(lo, hi, dtype=np.float64)
    cum = np.cumsum(enc)
    cuts = [lo] + [lo + int(np.searchsorted(cum, cum[-1] * i / n)) for i in range(1, n)] + [hi]
    cuts = sorted(set(cuts))

    def run(a, b):
        r = [ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_double()]
        emu.markstein_sweep(a, b, *[ctypes.byref(v) for v in r])
        return r[0].value, r[1].value, r[2].value, r[3].value

    with ThreadPoolExecutor(_threads()) as ex:
        parts = list(ex.map(lambda ab: run(*ab), zip(cuts[:-1], cuts[1:])))
    pairs = sum(p[0] for p in parts)
    n_diff = sum(p[1] for p in parts)
    n_code_diff = sum(p[2] for p in parts)
    max_ref = max(p[3] for p in parts)
    print(f"markstein: {pairs} pairs, {n_diff} quotients differ, max |x/s| there {max_ref}")
    assert pairs > 4.9e8
    assert n_code_diff == 0
    # the differences that exist are far below the smallest e4m3 step (2^-9)
    assert n_diff == 0 or max_ref < 2.0 ** -40, (n_diff, max_ref)


def test_markstein_quotient_sampled_with_signs(emu):
    """Negative and positive x with random block maxima: codes of the kernel's
    quotient equal those of RN(x / s) (torch's e4m3 cast of both, saturated)."""
    import torch
    rng = np.random.default_rng(22)
    n = 2_000_000
    amax = np.abs(rng.standard_normal(n) * 2.0 ** rng.integers(-60, 100, n)).astype(np.float32)
    amax = np.maximum(amax, np.float32(2.0 ** -64))
    amax = (amax.view(np.uint32) & 0xFFFF0000).view(np.float32)  # bf16 values
    frac = rng.random(n) * np.where(rng.random(n) < 0.5, -1.0, 1.0)
    x = (amax * frac).astype(np.float32)
    x = (x.view(np.uint32) & 0xFFFF0000).view(np.float32)
    s = (amax / np.float32(448.0)).astype(np.float32)
    q = np.empty(n, np.float32)
    emu.markstein_many(n, x, s, q)
    ref = (x / s).astype(np.float32)

    def codes(v):
        v = np.clip(v, -448, 448)
        return torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()

    # the kernel's code: the quotient's e4m3 magnitude, the sign of x
    x[:1000] = np.float32(-0.0)  # negative zeros, whose quotient may lose the sign
    q = np.empty(n, np.float32)
    emu.markstein_many(n, x, s, q)
    ref = (x / s).astype(np.float32)
    kernel = (codes(np.abs(q)) | (np.signbit(x).astype(np.uint8) << 7)).astype(np.uint8)
    assert np.array_equal(kernel, codes(ref))
    same = np.abs(q).view(np.uint32) == np.abs(ref).view(np.uint32)
    assert np.all(same | (np.abs(ref) < 2.0 ** -40))


def test_float_float_exp_relative_error(emu):
    """exp(d) over the kernel's range d in [-80, 0]: relative error below 2^-42
    against the host's double exp (itself within an ulp of 2^-53)."""
    rng = np.random.default_rng(23)
    d = np.concatenate([-rng.random(1_000_000) * 80.0, -rng.random(200_000) * 2.0 ** -10,
                        [0.0, -80.0, -0.3465735902799727, -0.6931471805599453]]).astype(np.float32)
    got = np.empty(d.size, np.float64)
    emu.ff_exp_many(d.size, d, got)
    want = np.exp(d.astype(np.float64))
    rel = np.abs(got - want) / want
    assert rel.max() < 2.0 ** -42, rel.max()


def _top_logits(rng, T, E, k):
    """The k largest of E N(0,1) logits per token, in descending order: the
    chosen logits the kernel's softmax sees."""
    z = rng.standard_normal((T, E), dtype=np.float32)
    part = -np.partition(-z, k - 1, axis=1)[:, :k]
    return -np.sort(-part, axis=1)


def test_float_float_softmax_matches_the_double_softmax(emu):
    """6.4 million top-8 weights (800,000 tokens of 256 N(0,1) logits) plus
    top-2 weights and edge cases (equal logits, gaps beyond 80 that take the
    double path, large logits): every weight within one fp32 ulp of the
    oracle's softmax in double rounded to fp32, and all but a handful equal."""
    rng = np.random.default_rng(24)
    cases = []
    for _ in range(8):
        cases.append(_top_logits(rng, 100_000, 256, 8))
    z2 = _top_logits(rng, 200_000, 64, 2)
    edge = np.zeros((6, 8), np.float32)
    edge[1] = [3, 3, 3, 3, 3, 3, 3, 3]
    edge[2] = [0, -1, -85, -90, -100, -120, -200, -300]
    edge[3] = [1e4, 1e4 - 1, 1e4 - 2, 1e4 - 3, 1e4 - 40, 1e4 - 79.5, 1e4 - 80.5, 1e4 - 81]
    edge[4] = [-5, -5.5, -6, -7, -9, -12, -20, -60]
    edge[5] = [2.0 ** -20, 0, -1e-7, -(2.0 ** -20), -0.5, -0.5, -0.75, -1]
    cases.append(edge)
    total = exact = 0
    for z, k in [(c, 8) for c in cases] + [(z2, 2)]:
        z = np.ascontiguousarray(z, np.float32)
        T = z.shape[0]
        w = np.empty((T, k), np.float32)
        parts = oracle._ranges(T, _threads())
        with ThreadPoolExecutor(len(parts)) as ex:
            list(ex.map(lambda ab: emu.ff_softmax_many(ab[1] - ab[0], k, z[ab[0]:ab[1]],
                                                       w[ab[0]:ab[1]]), parts))
        ids, w_ref = oracle.route_topk(z, k, threads=_threads())
        assert np.array_equal(ids, np.tile(np.arange(k, dtype=np.int32), (T, 1)))
        a = w.view(np.int32).astype(np.int64)
        b = w_ref.view(np.int32).astype(np.int64)
        d = np.abs(a - b)  # weights are positive: ulp distance = encoding distance
        assert d.max() <= 1, int(d.max())
        total += d.size
        exact += int((d == 0).sum())
    assert total >= 6_400_000
    print(f"softmax weights: {total}, equal: {exact}")
    assert total - exact <= 10, total - exact
