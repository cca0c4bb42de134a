"""The RoPE angle reduction of the CUDA kernels, modelled on the CPU.

The kernels evaluate cos/sin of pos * f (f = theta^(-2i/D)) without FP64:
the host stores f * 2/pi as a 64-bit fixed-point fraction plus its integer
part mod 4 (from the exact product of f's significand with a 256-bit 2/pi),
and the device reduces pos * f modulo pi/2 with integer arithmetic, then
evaluates double-float Taylor series (csrc/rope_math.cuh, csrc/api.cu).

These tests check, on the CPU and without the library:
* the 256-bit constant in csrc/api.cu against 2/pi computed here from
  Machin's formula with Python integers;
* a model of the host table (the same bit extraction, on Python integers)
  against the exact rational product f * 2/pi;
* a model of the device arithmetic (integer steps exact, FP32 steps in numpy
  float32) against cos/sin of the exact angle evaluated to 60 digits: the
  absolute error stays below 1e-11 for positions up to 65536, far below a
  16-bit ulp of a rotated value.
The GPU tests check the kernels themselves (rotated K within one ulp of the
oracle at positions up to 65535).
"""
import os
import re
from fractions import Fraction

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "kv_cached_gqa_rope_gb300", "csrc")


def two_over_pi_bits(bits: int) -> int:
    """floor(2/pi * 2^bits) from Machin's formula pi/4 = 4 atan(1/5) - atan(1/239)."""
    guard = 64
    one = 1 << (bits + guard)

    def atan_inv(x):
        total = term = one // x
        n, sign = 1, -1
        while term:
            term //= x * x
            n += 2
            total += sign * (term // n)
            sign = -sign
        return total

    pi = 4 * (4 * atan_inv(5) - atan_inv(239))  # pi * 2^(bits + guard), to within a few units
    return ((2 << (2 * (bits + guard))) // pi) >> guard


def source_constant() -> int:
    text = open(os.path.join(CSRC, "api.cu")).read()
    body = re.search(r"kTwoOverPi256\[4\]\s*=\s*\{([^}]*)\}", text).group(1)
    words = [int(w.strip().rstrip("ull"), 16) for w in body.split(",")]
    return sum(w << (64 * i) for i, w in enumerate(words))


def test_two_over_pi_constant():
    assert source_constant() == two_over_pi_bits(256)


def quarter_turns(f: float, T: int):
    """Model of the host table: (fraction * 2^64, integer part mod 4) of f * 2/pi."""
    m, e = np.frexp(f)
    M = int(np.ldexp(m, 53))
    P = M * T  # f * 2/pi = P * 2^(e - 53 - 256)
    lo = 245 - int(e)
    full = P >> lo if lo >= 0 else P << -lo
    return full & ((1 << 64) - 1), (full >> 64) & 3


def frequencies():
    fs = []
    for theta, D in ((1e4, 64), (5e5, 128), (1e6, 128), (16.0, 8), (0.5, 128)):
        fs += [theta ** (-2.0 * i / D) for i in range(D // 2)]
    return fs


def test_host_table_is_the_exact_product():
    T = two_over_pi_bits(256)
    for f in frequencies() + [1.0, 0.0, 2.0 ** -30, 123.456]:
        frac, quad = quarter_turns(f, T)
        exact = Fraction(f) * Fraction(T, 1 << 256) * (1 << 64)  # f * 2/pi * 2^64 (2/pi to 2^-256)
        whole = exact.numerator // exact.denominator
        assert frac == whole % (1 << 64) and quad == (whole >> 64) & 3, f


# ---- the device arithmetic (FP32 steps as numpy float32; an FMA's product of
# two floats is exact in a double, so one double rounding models it)
f32 = np.float32


def _fma(a, b, c):
    return f32(float(a) * float(b) + float(c))


def _two_sum(a, b):
    s = f32(a + b)
    bb = f32(s - a)
    return s, f32(f32(a - f32(s - bb)) + f32(b - bb))


def _fast_two_sum(a, b):
    s = f32(a + b)
    return s, f32(b - f32(s - a))


def _add(a, b):
    s = _two_sum(a[0], b[0])
    return _fast_two_sum(s[0], f32(s[1] + f32(a[1] + b[1])))


def _add_f(a, b):
    s = _two_sum(a[0], b)
    return _fast_two_sum(s[0], f32(s[1] + a[1]))


def _mul(a, b):
    p = f32(a[0] * b[0])
    e = _fma(a[0], b[0], -p)
    e = _fma(a[0], b[1], e)
    e = _fma(a[1], b[0], e)
    return _fast_two_sum(p, e)


def _const(v):
    h = f32(v)
    return h, f32(v - float(h))


def cos_sin_model(pos: int, frac: int, quad: int):
    mask = (1 << 64) - 1
    lo = pos * (frac & 0xFFFFFFFF)
    hi = pos * (frac >> 32)
    f64 = (lo + (hi << 32)) & mask
    whole = ((hi >> 32) + (1 if f64 < lo else 0) + pos * quad) & 0xFFFFFFFF
    q = (whole + (f64 >> 63)) & 3
    r = ((f64 - (1 << 64)) if f64 >> 63 else f64) >> 16
    rd = _two_sum(f32(f32(r >> 24) * f32(16777216.0)), f32(r & 0xFFFFFF))
    x = _mul(rd, _const(1.5707963267948966 / 281474976710656.0))
    y = _mul(x, x)
    yh = y[0]
    ts = _fma(_fma(_fma(yh, f32(1 / 6227020800), f32(-1 / 39916800)), yh, f32(1 / 362880)), yh, f32(-1 / 5040))
    s3 = _add_f(_const(1 / 120), f32(yh * ts))
    s2 = _add(_const(-1 / 6), _mul(y, s3))
    s1 = _add(_const(1.0), _mul(y, s2))
    sx = _mul(x, s1)
    tc = _fma(_fma(yh, f32(1 / 479001600), f32(-1 / 3628800)), yh, f32(1 / 40320))
    c4 = _add_f(_const(-1 / 720), f32(yh * tc))
    c3 = _add(_const(1 / 24), _mul(y, c4))
    c2 = _add(_const(-0.5), _mul(y, c3))
    cx = _add(_const(1.0), _mul(y, c2))
    neg = lambda d: (-d[0], -d[1])  # noqa: E731
    c, s = {0: (cx, sx), 1: (neg(sx), cx), 2: (neg(cx), neg(sx)), 3: (sx, neg(cx))}[q]
    return float(c[0]) + float(c[1]), float(s[0]) + float(s[1])


def test_device_reduction_error_bound():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 60
    T = two_over_pi_bits(256)
    rng = np.random.default_rng(7)
    worst = 0.0
    for theta, D in ((1e4, 64), (5e5, 128), (1e6, 128)):
        freqs = [theta ** (-2.0 * i / D) for i in range(D // 2)]
        for pos in [0, 1, 2, 4095, 32768, 65535, 65536] + [int(v) for v in rng.integers(0, 65536, 12)]:
            for f in freqs[::3] + [freqs[-1]]:
                c, s = cos_sin_model(pos, *quarter_turns(f, T))
                ang = mpmath.mpf(pos) * mpmath.mpf(f)  # the exact angle
                worst = max(worst, abs(c - float(mpmath.cos(ang))), abs(s - float(mpmath.sin(ang))))
    assert worst < 1e-11, worst
