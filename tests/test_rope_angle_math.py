"""CPU check of the angle arithmetic the CUDA kernels use for RoPE (rope.cuh), emulated step by step
in numpy: the 64-bit fixed-point frequency F_k = round(theta_k / 2pi * 2^64), the 32-bit turn
fraction bits[32,64)(p * F_k) taken with one high multiply and one low multiply, the exact integer
reduction to the nearest quarter turn and the fitted sin/cos polynomials (fp32, fused multiply-add
emulated through float64).  The result must match cos/sin(p * theta_k) evaluated in float64 with
exact argument reduction to within 2.5e-7 for every pair k and positions up to 2^24 - 1."""
import math

import numpy as np
import pytest

S = [1.5707963705062866, -0.6459640860557556, 0.07968810945749283, -0.004624062217772007]
C = [1.0, -1.2337005138397217, 0.2536693811416626, -0.020861255005002022, 0.0009058757568709552]


def f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def fma32(a, b, c):
    return f32(a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64))


def sincos_turns(t):
    t = t.astype(np.uint64)
    q = ((t + 0x20000000) & 0xFFFFFFFF) >> 30
    rem = ((t - (q << 30)) & 0xFFFFFFFF).astype(np.int64)
    rem = np.where(rem >= 1 << 31, rem - (1 << 32), rem)
    r = f32(f32(rem) * np.float32(9.313225746154785e-10))
    z = f32(r * r)
    sp = fma32(fma32(fma32(f32(np.full_like(z, S[3])), z, f32(S[2])), z, f32(S[1])), z, f32(S[0]))
    sp = f32(sp * r)
    cp = fma32(fma32(fma32(fma32(f32(np.full_like(z, C[4])), z, f32(C[3])), z, f32(C[2])), z, f32(C[1])), z, f32(C[0]))
    c0 = np.where(q & 1, -sp, cp)
    s0 = np.where(q & 1, cp, sp)
    return np.where(q & 2, -c0, c0), np.where(q & 2, -s0, s0)


def turn_fraction(pos, theta):
    F = int(round(math.ldexp(theta / (2 * math.pi), 64)))
    lo, hi = F & 0xFFFFFFFF, F >> 32
    pos = pos.astype(np.uint64)
    return (((pos * np.uint64(lo)) >> np.uint64(32)) + pos * np.uint64(hi)) & np.uint64(0xFFFFFFFF), F


@pytest.mark.parametrize("d,base", [(64, 1e4), (128, 5e5), (128, 1e4)])
def test_cos_sin_of_positions(d, base):
    rng = np.random.default_rng(d)
    pos = np.concatenate([np.arange(0, 4096), rng.integers(0, 1 << 24, 20000), [1 << 15, 32767, (1 << 24) - 1]])
    worst = 0.0
    for k in range(d // 2):
        theta = base ** (-2.0 * k / d)
        t, F = turn_fraction(pos, theta)
        c, s = sincos_turns(t)
        # exact reference: the angle modulo one turn from the same rational frequency F / 2^64
        frac = np.array([(int(p) * F % (1 << 64)) / 2.0 ** 64 for p in pos])
        ang = 2 * np.pi * frac
        worst = max(worst, np.abs(c - np.cos(ang)).max(), np.abs(s - np.sin(ang)).max())
        # and F / 2^64 is theta / 2pi to double precision: angle error below 1e-10 rad at 2^24
        assert abs(F / 2.0 ** 64 - theta / (2 * math.pi)) * (1 << 24) * 2 * math.pi < 1e-8
    assert worst < 2.5e-7, worst


def test_quadrants_and_turn_wraparound():
    t = np.array([0, 1 << 30, 1 << 31, 3 << 30, (1 << 32) - 1, 0x20000000, 0x1FFFFFFF, 0xE0000000], dtype=np.uint64)
    c, s = sincos_turns(t)
    ang = 2 * np.pi * t.astype(np.float64) / 2.0 ** 32
    assert np.abs(c - np.cos(ang)).max() < 2.5e-7 and np.abs(s - np.sin(ang)).max() < 2.5e-7
