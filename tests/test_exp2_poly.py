"""The prefill softmax computes some of its 2^x on the FMA pipe: range
reduction x = n + f (n = round(x), f in [-0.5, 0.5]), a degree-3 polynomial
for 2^f, and n added into the exponent field (sm100_ptx.cuh, exp2_poly2).
P is rounded to bf16 (relative step 2^-8), so a relative error well under
1e-4 is invisible in the output.

CPU: the same float32 steps in numpy, with the coefficients read from the
header, against 2^x in float64.  GPU: the device function against CUDA's
exp2f on the same arguments.
"""

from __future__ import annotations

import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from ragged_paged_attention_rpa_gb300 import build

HEADER = os.path.join(build.CSRC, "sm100_ptx.cuh")
BOUND = 1e-4


def coefficients():
    text = open(HEADER).read()
    body = text[text.index("exp2_poly2"):]
    vals = re.findall(r"f2_pack\((-?[0-9.]+(?:e-?[0-9]+)?)f, \1f\)", body)
    nums = [float(v) for v in vals]
    # shifter, -shifter, -1, then c3, c2, c1, c0 in Horner order
    assert nums[:3] == [12582912.0, -12582912.0, -1.0], nums[:3]
    c3, c2, c1, c0 = nums[3:7]
    return c0, c1, c2, c3


def emulate(x):
    f32 = np.float32
    c0, c1, c2, c3 = (f32(v) for v in coefficients())
    x0 = x.astype(f32)
    x = np.maximum(x0, f32(-125.0))
    t = (x + f32(12582912.0)).astype(f32)
    n = (t - f32(12582912.0)).astype(f32)
    fr = (x - n).astype(f32)
    p = (c3 * fr + c2).astype(f32)
    p = (p * fr + c1).astype(f32)
    p = (p * fr + c0).astype(f32)
    bits = p.view(np.int32) + (t.view(np.int32) << 23)
    return np.where(x0 < f32(-125.0), f32(0.0), bits.astype(np.int32).view(np.float32))


def test_masked_scores_give_exact_zero():
    x = np.array([-np.inf, -1e30, -200.0, -125.5], dtype=np.float32)
    assert (emulate(x) == 0.0).all()
    assert emulate(np.array([-125.0], dtype=np.float32))[0] > 0.0


def test_poly_exp2_matches_float64_on_the_softmax_range():
    x = np.concatenate([np.linspace(-125.0, 8.0, 400001, dtype=np.float64),
                        np.arange(-125, 9, dtype=np.float64)]).astype(np.float32)
    got = emulate(x).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(got - want) / want
    assert rel.max() < BOUND, rel.max()


def test_range_reduction_is_exact_at_integers():
    x = np.arange(-120, 9, dtype=np.float32)
    got = emulate(x).astype(np.float64)
    rel = np.abs(got / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() < BOUND


@pytest.mark.gpu
def test_poly_exp2_on_gpu_matches_exp2f(tmp_path):
    lib = str(tmp_path / "libexp2check.so")
    src = os.path.join(os.path.dirname(__file__), "csrc", "exp2_poly_check.cu")
    subprocess.run([build.nvcc()] + build.ARCH + ["-O3", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-I" + build.CSRC, "-o", lib, src], check=True)
    L = ctypes.CDLL(lib)
    x = np.concatenate([np.linspace(-125.0, 8.0, 200000), np.arange(-125, 9)]).astype(np.float32)
    if x.size % 2:
        x = x[:-1]
    poly = np.empty_like(x)
    ref = np.empty_like(x)
    vp = ctypes.c_void_p
    rc = L.exp2_poly_check(x.ctypes.data_as(vp), poly.ctypes.data_as(vp),
                           ref.ctypes.data_as(vp), ctypes.c_int(x.size))
    assert rc == 0
    rel = np.abs(poly.astype(np.float64) - ref) / ref
    assert rel.max() < BOUND, rel.max()
    # Masked scores (-inf) and arguments below the clamp give exactly 0.
    x = np.array([-np.inf, -1e30, -200.0, -125.5], dtype=np.float32)
    poly = np.empty_like(x)
    ref = np.empty_like(x)
    rc = L.exp2_poly_check(x.ctypes.data_as(vp), poly.ctypes.data_as(vp),
                           ref.ctypes.data_as(vp), ctypes.c_int(x.size))
    assert rc == 0 and (poly == 0.0).all(), poly
