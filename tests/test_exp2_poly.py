"""The FMA-pipe exp2 used for part of the softmax exponentials.

Pinned on the CPU by re-running its exact float32 steps (round-to-nearest
range reduction with 1.5*2^23, degree-3 polynomial for 2^f on [-1/2, 1/2],
exponent add) in numpy and comparing with the exactly rounded 2^x: the
relative error must stay far below the bf16 rounding (2^-9) that P gets
next.  The coefficients are read from the CUDA header so the test checks
what the kernels compile.
"""
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bwd_jagged_flashattention_gb300",
                   "csrc", "ptx.cuh")


def _coeffs():
    text = open(HDR).read()
    m = re.search(r"constexpr float kExp2C0 = ([0-9.e+-]+)f, kExp2C1 = ([0-9.e+-]+)f, kExp2C2 = ([0-9.e+-]+)f, "
                  r"kExp2C3 = ([0-9.e+-]+)f;", text)
    assert m, "coefficients not found"
    return [np.float32(float(g)) for g in m.groups()]


def exp2_fma(x):
    """Bit-faithful float32 emulation of exp2_fma2 (one lane)."""
    c0, c1, c2, c3 = _coeffs()
    x = np.maximum(x.astype(np.float32), np.float32(-125.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    n = (t - magic).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = np.float32(np.float64(c3) * f + np.float64(c2))
    p = np.float32(np.float64(p) * f + np.float64(c1))
    p = np.float32(np.float64(p) * f + np.float64(c0))
    bits = (p.view(np.int32) + (t.view(np.int32) << 23)).astype(np.int32)
    return bits.view(np.float32)


def test_relative_error_over_softmax_range():
    x = np.linspace(-120.0, 8.0, 2_000_003, dtype=np.float32)
    y = exp2_fma(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y / ref - 1.0)
    assert rel.max() < 1e-4, rel.max()          # bf16 half-ulp is 2^-9 ~ 2e-3


def test_integer_and_half_points():
    x = np.array([-100, -10, -3, -1, 0, 1, 2, 7, -0.5, 0.5, -2.5, 3.5], dtype=np.float32)
    rel = np.abs(exp2_fma(x).astype(np.float64) / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() < 1e-4


def test_clamp_keeps_results_normal_and_tiny():
    y = exp2_fma(np.array([-125.0, -200.0, -1e30], dtype=np.float32))
    assert np.all(y > np.finfo(np.float32).tiny) and np.all(y < 1e-37)
