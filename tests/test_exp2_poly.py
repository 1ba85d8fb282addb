"""The FMA-pipe exp2 of the diagonal scan (`exp2_fma2` in csrc/diag_scan.cu, selected by
SSM_TUNE_DIAG_EXP_POLY): its coefficients are the ones csrc/fit_exp2.py fits, and its
range-reduced evaluation, emulated here in fp32 step by step, stays within 3e-7 of 2^x
(fp64) over the whole range the decays take, x in [-126, 0]."""
import importlib.util
import os
import re

import numpy as np

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "selective_state_space_143_b300", "csrc")


def _fit_module():
    spec = importlib.util.spec_from_file_location("fit_exp2", os.path.join(CSRC, "fit_exp2.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def kernel_coefficients() -> np.ndarray:
    src = open(os.path.join(CSRC, "diag_scan.cu")).read()
    found = dict(re.findall(r"kC(\d) = ([0-9.eE+-]+)f", src))
    assert sorted(found) == [str(i) for i in range(6)], found
    return np.array([float(found[str(i)]) for i in range(6)], dtype=np.float32)


def exp2_fma_emulated(x: np.ndarray, c: np.ndarray) -> np.ndarray:
    """exp2_fma2's steps in fp32 (each fused multiply-add rounded once, via fp64)."""
    f32 = np.float32
    x = np.maximum(x.astype(f32), f32(-126.0))
    t = (x + f32(12582912.0)).astype(f32)
    r = (t - f32(12582912.0)).astype(f32)
    f = (x - r).astype(f32)  # exact: rint(x) is within 1/2 of x
    p = np.full_like(f, c[5])
    for ci in c[4::-1]:
        p = (p.astype(np.float64) * f + np.float64(ci)).astype(f32)
    n = r.astype(np.int32)
    s = np.ldexp(np.ones_like(f), n).astype(f32)
    return (p * s).astype(f32)


def test_kernel_coefficients_are_the_fit():
    c = _fit_module().fit().astype(np.float32)
    np.testing.assert_array_equal(kernel_coefficients(), c)


def test_fit_is_close_to_the_minimax_bound():
    # a degree-5 fit of 2^f on [-1/2, 1/2]: the Taylor remainder is ~2.4e-6, the minimax
    # polynomial ~40x smaller; the fit must reach below one fp32 ulp
    c = _fit_module().fit()
    f = np.linspace(-0.5, 0.5, 200_001)
    err = np.max(np.abs(np.polyval(c[::-1], f) / np.exp2(f) - 1.0))
    assert err < 1.0e-7, err


def test_range_reduced_exp2_within_bound():
    c = kernel_coefficients()
    rng = np.random.default_rng(0)
    x = np.concatenate([np.linspace(-126.0, 0.0, 1_000_001), -rng.exponential(2.0, 200_000),
                        -rng.uniform(0.0, 1e-3, 10_000), [0.0, -0.5, -1.5, -125.5, -126.0]]).astype(np.float32)
    y = exp2_fma_emulated(x, c).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y / ref - 1.0)
    assert np.max(rel) <= 3e-7, (np.max(rel), x[np.argmax(rel)])


def test_below_range_clamps_to_smallest_normal():
    c = kernel_coefficients()
    y = exp2_fma_emulated(np.array([-127.0, -200.0, -1e30], dtype=np.float32), c)
    assert np.all(y > 0) and np.all(y <= np.float32(2.0 ** -126) * 1.000001)
