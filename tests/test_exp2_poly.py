"""The FMA-pipe exp2 kept in csrc/ptx.cuh (exp2_poly2), emulated in fp32 on the CPU.

No kernel calls it today: handing part of the exponentials to the FMA pipe
measured slower than the special-function unit alone on this GPU.  It
computes 2^x as 2^round(x) * p(x - round(x)) with the minimax
polynomial of csrc/exp2_poly.h (written by csrc/gen_exp2_poly.py from the
Remez exchange algorithm).  This test re-evaluates that sequence in float32
(products and sums rounded to float32 as the fused multiply-adds would be,
up to double rounding) over the range the kernel feeds it, and checks the
relative error against numpy's float64 exp2.
"""
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "causal_head_attention_mha_gb300", "csrc", "exp2_poly.h")


def coeffs():
    text = open(HDR).read()
    deg = int(re.search(r"MHA_EXP2_POLY_DEGREE (\d+)", text).group(1))
    return [np.float32(float(re.search(rf"MHA_EXP2_POLY_C{i} ([-0-9.e]+)f", text).group(1)))
            for i in range(deg + 1)]


def f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def fma32(a, b, c):
    return f32(a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64))


def exp2_poly(x):
    c = coeffs()
    shift = np.float32(12582912.0)
    x = np.minimum(np.maximum(f32(x), np.float32(-126.0)), np.float32(127.0))
    t = f32(x.astype(np.float64) + shift)
    n = f32(t.astype(np.float64) - shift)
    f = fma32(n, np.full_like(n, -1.0), x)
    p = np.full_like(f, c[-1])
    for ci in reversed(c[:-1]):
        p = fma32(p, f, np.full_like(f, ci))
    bits = (p.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))).astype(np.uint32)
    return bits.view(np.float32)


def test_relative_error_over_kernel_range():
    # the kernel's exponent arguments lie in [-inf, 64] on its fast path; below
    # -126 it clamps, and within one unit of the clamp the result reaches the
    # denormal boundary (~1e-38)
    x = np.concatenate([np.linspace(-125.0, 126.0, 2_000_001, dtype=np.float64),
                        np.arange(-125, 127, dtype=np.float64),
                        np.arange(-125, 126, dtype=np.float64) + 0.5]).astype(np.float32)
    y = exp2_poly(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y / ref - 1.0)
    assert np.all(np.isfinite(y)) and np.all(y > 0)
    assert rel.max() <= 1.0e-4, rel.max()


def test_clamped_inputs_stay_tiny_and_positive():
    y = exp2_poly(np.array([-np.inf, -1e30, -500.0, -127.0, -126.5, -125.5], np.float32))
    assert np.all(y > 0) and np.all(y < 2.0 ** -124)


def test_large_inputs_stay_huge_and_finite():
    # above 127 the input is clamped: the result stays >= 2^127, so a weight
    # past the kernel's 2^64 bound is still seen as one (never wraps to small)
    y = exp2_poly(np.array([127.0, 128.0, 200.0, 1e30, np.inf], np.float32))
    assert np.all(np.isfinite(y)) and np.all(y >= 2.0 ** 126)


def test_generator_reproduces_header():
    import subprocess
    import sys
    import tempfile
    src = os.path.join(os.path.dirname(HDR), "gen_exp2_poly.py")
    with tempfile.TemporaryDirectory() as d:
        import shutil
        shutil.copy(src, d)
        subprocess.run([sys.executable, os.path.join(d, "gen_exp2_poly.py"), "3"], check=True,
                       capture_output=True)
        assert open(os.path.join(d, "exp2_poly.h")).read() == open(HDR).read()
