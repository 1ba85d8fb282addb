"""Pins for the oracle's backward pass: every gradient against central finite
differences of the forward oracle (itself pinned in test_oracle_pins.py), on tiny
problems in both modes, with and without the optional inputs.

The loss is L = sum(dout * out) + sum(dfinal * final_state) for fixed random dout and
dfinal, so dL/d(input) is exactly what the backward pass returns.  Central differences
with step 1e-6 in fp64 are accurate to about 1e-9 here, far below any plausible
mistake in the derivation (a dropped decay, a wrong sign, h_t for h_{t-1}, a missing
sigmoid or SiLU derivative).
"""
import numpy as np
import pytest

import oracle

INPUTS = ("x", "dt", "A", "B", "C", "D", "z", "dt_bias", "initial_state")
GRAD = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "z": "dz",
        "dt_bias": "ddt_bias", "initial_state": "dinit"}


def problem(rng, mode, b, T, H, P, N, G, gate=True, bias=True, skip=True, init=True):
    diag = mode == "diag"
    xs = (b, T, H) if diag else (b, T, H, P)
    st = (b, H, N) if diag else (b, H, P, N)
    arr = dict(
        x=rng.standard_normal(xs), dt=0.5 * rng.standard_normal((b, T, H)) - 0.5,
        A=(-rng.uniform(0.2, 1.5, (H, N)) if diag else -rng.uniform(0.2, 1.5, (H,))),
        B=rng.standard_normal((b, T, G, N)), C=rng.standard_normal((b, T, G, N)),
        D=rng.normal(1.0, 0.3, (H,)) if skip else None,
        z=rng.standard_normal(xs) if gate else None,
        dt_bias=rng.uniform(-0.5, 0.5, (H,)) if bias else None,
        initial_state=rng.standard_normal(st) if init else None,
    )
    dout = rng.standard_normal(xs)
    dfinal = rng.standard_normal(st)
    return arr, dout, dfinal


def loss(scan, arr, dout, dfinal):
    out, fs = scan(**arr)
    return float(np.sum(dout * out) + np.sum(dfinal * fs))


def finite_differences(scan, arr, dout, dfinal, eps=1e-6):
    grads = {}
    for name in INPUTS:
        v = arr[name]
        if v is None:
            continue
        g = np.zeros_like(v)
        flat = v.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + eps
            lp = loss(scan, arr, dout, dfinal)
            flat[i] = old - eps
            lm = loss(scan, arr, dout, dfinal)
            flat[i] = old
            g.reshape(-1)[i] = (lp - lm) / (2 * eps)
        grads[name] = g
    return grads


def mismatches(scan, scan_bwd, arr, dout, dfinal):
    """Names of the gradients where the backward pass and the differences disagree."""
    fd = finite_differences(scan, arr, dout, dfinal)
    bw = scan_bwd(**arr, dout=dout, dfinal=dfinal)
    bad = []
    for name, g in fd.items():
        got = bw[GRAD[name]]
        if got is None or not np.allclose(got, g, rtol=1e-6, atol=1e-8):
            bad.append(name)
    return bad


CASES = [
    ("diag", (1, 5, 2, 1, 3, 1), {}),
    ("diag", (2, 4, 4, 1, 2, 2), {}),
    ("diag", (1, 6, 2, 1, 3, 1), dict(gate=False, bias=False, skip=False, init=False)),
    ("ssd", (1, 5, 2, 2, 2, 1), {}),
    ("ssd", (1, 4, 4, 2, 3, 2), dict(gate=False, init=False)),
]


@pytest.mark.parametrize("mode,dims,opts", CASES, ids=[f"{c[0]}-{c[1]}-{len(c[2])}" for c in CASES])
def test_backward_matches_finite_differences(mode, dims, opts):
    rng = np.random.default_rng([len(mode), *dims, len(opts)])
    arr, dout, dfinal = problem(rng, mode, *dims, **opts)
    assert mismatches(oracle.scan, oracle.scan_bwd, arr, dout, dfinal) == []


def test_backward_without_final_state_gradient():
    rng = np.random.default_rng(4)
    arr, dout, _ = problem(rng, "diag", 1, 5, 2, 1, 3, 1)
    zero = np.zeros((1, 2, 3))
    a = oracle.scan_bwd(**arr, dout=dout, dfinal=None)
    b = oracle.scan_bwd(**arr, dout=dout, dfinal=zero)
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD", "dz", "ddt_bias", "dinit"):
        assert np.array_equal(a[k], b[k]), k


def test_backward_of_empty_sequence():
    """T = 0: the only path is initial_state -> final_state, so dinit = dfinal."""
    rng = np.random.default_rng(5)
    arr, dout, dfinal = problem(rng, "diag", 2, 0, 2, 1, 3, 1)
    g = oracle.scan_bwd(**arr, dout=dout, dfinal=dfinal)
    assert np.array_equal(g["dinit"], dfinal)
    assert np.all(g["dA"] == 0.0) and np.all(g["dD"] == 0.0)
