"""The FMA-pipe exponential used by the kernels (exp2_fma in csrc/common.cuh):
its coefficients come from fit_exp2_poly.py and, with the kernel's range
reduction emulated in float32, it stays within 1e-4 relative error of 2^x on
the range the softmax uses (x <= 8 after the lazy-rescale threshold)."""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "sink_aware_masked_gb300", "csrc", "common.cuh")


def kernel_coefficients():
    with open(HDR) as f:
        src = f.read()
    body = src[src.index("SA_DEV float exp2_fma"):]
    body = body[:body.index("}")]
    nums = [float(x) for x in re.findall(r"(\d+\.\d+)f", body)]
    # fmaf(fmaf(fmaf(c3, f, c2), f, c1), f, c0) appear in the order c3, c2, c1, c0
    consts = [x for x in nums if x < 2.0][-4:]
    return consts[3], consts[2], consts[1], consts[0]


def emulate(x, c):
    x = np.maximum(x.astype(np.float32), np.float32(-125.0))
    t = (x + np.float32(12582912.0)).astype(np.float32)
    j = (t - np.float32(12582912.0)).astype(np.float32)
    f = (x - j).astype(np.float32)
    c0, c1, c2, c3 = (np.float32(v) for v in c)
    p = ((c3 * f + c2) * f + c1) * f + c0
    bits = p.view(np.int32) + (t.view(np.int32) << np.int32(23))
    return bits.view(np.float32)


def test_coefficients_match_fit():
    import importlib.util

    spec = importlib.util.spec_from_file_location("fitp", os.path.join(ROOT, "sink_aware_masked_gb300",
                                                                      "fit_exp2_poly.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    fitted = [float(v) for v in mod.fit()]
    assert np.allclose(kernel_coefficients(), fitted, rtol=1e-6, atol=1e-8)


def test_relative_error_bound():
    c = kernel_coefficients()
    x = np.concatenate([np.linspace(-120.0, 8.0, 400001), -np.linspace(0, 1, 10001)]).astype(np.float32)
    got = emulate(x, c).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(got / want - 1.0)) < 1e-4


def test_masked_scores_vanish():
    c = kernel_coefficients()
    got = emulate(np.array([-np.inf, -1e30, -200.0], dtype=np.float32), c)
    assert np.all(got > 0) and np.all(got < 3e-38)


def test_packed_variant_uses_same_polynomial():
    """exp2_fma2 (the f32x2 form) must carry exactly the scalar coefficients."""
    with open(HDR) as f:
        src = f.read()
    body = src[src.index("SA_DEV float2 exp2_fma2"):]
    body = body[:body.index("\n}")]
    nums = {float(x) for x in re.findall(r"(\d+\.\d+)f", body) if float(x) < 2.0}
    assert nums == set(kernel_coefficients())
