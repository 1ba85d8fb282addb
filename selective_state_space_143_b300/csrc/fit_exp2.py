"""Fit the polynomial p(f) ~ 2^f on [-1/2, 1/2] used by the FMA-pipe exp2 of the
diagonal scan (exp2_fma2 in diag_scan.cu): 2^x = 2^n * 2^f with n = rint(x).

Method: a weighted least-squares fit on Chebyshev nodes minimising the relative error
|p(f) / 2^f - 1|, then Lawson's iteratively reweighted least squares, which converges to
the minimax (equi-oscillating) relative-error polynomial of the given degree.
Coefficients are rounded to fp32 and the fp32 Horner evaluation is checked on a dense grid.

    python fit_exp2.py        # prints the coefficients c0..c5 and the error bounds
"""
import numpy as np

DEG = 5


def fit(deg: int = DEG, n: int = 4000, iters: int = 200) -> np.ndarray:
    k = np.arange(n)
    f = 0.5 * np.cos(np.pi * (k + 0.5) / n)
    y = np.exp2(f)
    V = np.vander(f, deg + 1, increasing=True) / y[:, None]  # relative error rows
    w = np.full(n, 1.0 / n)
    c = None
    for _ in range(iters):  # Lawson: reweight by the error, towards the minimax fit
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(V * sw[:, None], sw, rcond=None)
        e = np.abs(V @ c - 1.0)
        w = w * e
        w /= w.sum()
    return c


def horner_f32(c32: np.ndarray, f: np.ndarray) -> np.ndarray:
    p = np.full_like(f, c32[-1])
    for ci in c32[-2::-1]:
        p = (p * f + ci).astype(np.float32)
    return p


if __name__ == "__main__":
    c = fit()
    c32 = c.astype(np.float32)
    f = np.linspace(-0.5, 0.5, 2_000_001)
    rel64 = np.max(np.abs(np.polyval(c[::-1], f) / np.exp2(f) - 1.0))
    rel32 = np.max(np.abs(horner_f32(c32, f.astype(np.float32)).astype(np.float64) / np.exp2(f) - 1.0))
    for i, ci in enumerate(c32):
        print(f"c{i} = {float(ci):.9e}f  ({float(ci).hex()})")
    print(f"max relative error: fit {rel64:.3e}, fp32 Horner {rel32:.3e} (fp32 eps {np.finfo(np.float32).eps:.3e})")
