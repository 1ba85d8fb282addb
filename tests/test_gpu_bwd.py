"""GPU parity of the backward pass (ssm_scan_bwd, diagonal and SSD mode) against the fp64
oracle's backward, which is pinned by finite differences: every gradient, element by
element.

Tolerances: max relative error (floor 1e-2 of the largest reference value) 1e-4 for fp32
inputs, 2e-2 for bf16 inputs; all gradients are fp32.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_143_b300 as ssm
from selective_state_space_143_b300 import _lib
from selective_state_space_143_b300.inputs import WORKLOADS, make_inputs, random_inputs

from conftest import record_errors

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
DEV = "cuda:0"
NAMES = {"dx": "dx", "ddt": "ddt", "dA": "dA", "dB": "dB", "dC": "dC", "dD": "dD", "dz": "dz",
         "ddt_bias": "ddt_bias", "dinitial_state": "dinit"}


def grads_gpu(inp, dout, dfinal, init):
    d = {k: (None if v is None else v.to(DEV)) for k, v in inp.items()}
    g = ssm.scan_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                     dout=dout.to(DEV), dfinal_state=None if dfinal is None else dfinal.to(DEV),
                     initial_state=None if init is None else init.to(DEV))
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in g.items()}


def compare(w, inp, dout, dfinal, init):
    got = grads_gpu(inp, dout, dfinal, init)
    ref = oracle.scan_bwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                          inp["dt_bias"], None if init is None else init.numpy(),
                          dout=dout, dfinal=None if dfinal is None else dfinal.numpy())
    tol = TOL[w.dtype]
    errs = {}
    for k, rk in NAMES.items():
        if ref[rk] is None or got[k] is None:
            assert (ref[rk] is None) == (got[k] is None) or k == "dinitial_state", k
            continue
        if ref[rk].size == 0:
            continue
        assert np.all(np.isfinite(got[k])), f"{k}: non-finite"
        errs[k] = oracle.max_rel_error(got[k], ref[rk])
        assert errs[k] <= tol, f"{k}: max rel err {errs[k]:.3e} > {tol}"
    return errs


def extras(w, seed, with_init=True, with_dfinal=True):
    gen = torch.Generator().manual_seed(seed)
    ssd = w.mode == "ssd"
    xs = (w.batch, w.seqlen, w.nheads) + ((w.headdim,) if ssd else ())
    dout = torch.randn(xs, generator=gen)
    dout = dout.to(torch.bfloat16) if w.dtype == "bf16" else dout
    st = (w.batch, w.nheads) + ((w.headdim,) if ssd else ()) + (w.dstate,)
    dfinal = torch.randn(st, generator=gen) if with_dfinal else None
    init = torch.randn(st, generator=gen) if with_init else None
    return dout, dfinal, init


# (dtype, batch, T, D, N, G, gate, bias, skip, init, dfinal)
CASES = [
    ("f32", 1, 37, 16, 4, 1, True, True, True, True, True),
    ("f32", 2, 100, 32, 16, 2, True, True, True, False, True),
    ("f32", 1, 64, 24, 8, 1, False, False, False, True, False),
    ("bf16", 2, 257, 64, 16, 1, True, True, True, True, True),
    ("bf16", 1, 200, 32, 64, 1, True, True, True, True, True),    # two entries per lane
    ("bf16", 2, 129, 48, 24, 3, True, False, True, False, True),  # width 24, padded lanes
    ("bf16", 3, 1, 64, 16, 1, True, True, True, True, True),      # one step
    ("bf16", 2, 33, 40, 32, 1, False, True, False, True, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_backward_shapes(case):
    dtype, b, T, D, N, G, gate, bias, skip, init, dfin = case
    w, inp = random_inputs("diag", dtype, b, T, D, 1, N, ngroups=G, gate=gate, dt_bias=bias,
                           d_skip="normal" if skip else "none", seed=T + D + N)
    dout, dfinal, h0 = extras(w, seed=T, with_init=init, with_dfinal=dfin)
    compare(w, inp, dout, dfinal, h0)


@pytest.mark.parametrize("name", ["c0", "c1"])
def test_backward_workloads(name):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    dout, dfinal, _ = extras(w, seed=7, with_init=False)
    errs = compare(w, inp, dout, dfinal, None)
    print(name, {k: f"{v:.2e}" for k, v in errs.items()})


def test_backward_empty_sequence():
    w, inp = random_inputs("diag", "bf16", 2, 0, 64, 1, 16, seed=1)
    dout, dfinal, init = extras(w, seed=2)
    got = grads_gpu(inp, dout, dfinal, init)
    assert np.array_equal(got["dinitial_state"], dfinal.numpy())
    assert np.all(got["dA"] == 0) and np.all(got["dD"] == 0)


def test_backward_is_repeatable_where_no_atomics():
    """dx, ddt, dz and dinitial_state are written by one thread each: identical runs."""
    w, inp = random_inputs("diag", "bf16", 2, 300, 64, 1, 16, seed=4)
    dout, dfinal, init = extras(w, seed=5)
    a = grads_gpu(inp, dout, dfinal, init)
    b = grads_gpu(inp, dout, dfinal, init)
    for k in ("dx", "ddt", "dz", "dinitial_state"):
        assert np.array_equal(a[k], b[k]), k


# shapes whose channels alone fill the GPU (many thread blocks per group, full grids)
WIDE = [
    # (dtype, batch, T, D, N)
    ("bf16", 4, 40, 5120, 16),
    ("f32", 2, 24, 10240, 8),
    ("bf16", 2, 20, 1280, 64),
    ("f32", 4, 17, 9600, 4),        # bf16 rows of 4 entries are not 16-byte multiples
]


@pytest.mark.parametrize("case", WIDE, ids=lambda c: "-".join(map(str, c)))
def test_backward_many_channels(case):
    dtype, b, T, D, N = case
    w, inp = random_inputs("diag", dtype, b, T, D, 1, N, seed=T + N)
    dout, dfinal, h0 = extras(w, seed=T + 1)
    compare(w, inp, dout, dfinal, h0)


# SSD mode: A, Delta, D and dt_bias per head; dstate up to 256 (4 and 8 entries per lane,
# 8- and 4-step checkpoint segments)
# (dtype, batch, T, H, P, N, G, gate, bias, skip, init, dfinal)
SSD_CASES = [
    ("f32", 1, 37, 2, 8, 16, 1, True, True, True, True, True),
    ("f32", 2, 50, 4, 4, 64, 2, True, True, True, False, True),
    ("f32", 1, 30, 2, 4, 256, 1, False, True, False, True, True),
    ("bf16", 1, 100, 2, 64, 128, 1, True, True, True, True, True),
    ("bf16", 1, 45, 2, 16, 256, 1, True, False, True, True, True),
    ("bf16", 2, 64, 4, 32, 32, 2, False, True, False, False, True),
    ("bf16", 2, 1, 2, 8, 64, 1, True, True, True, True, True),     # one step
]


@pytest.mark.parametrize("case", SSD_CASES, ids=lambda c: "-".join(map(str, c)))
def test_backward_ssd_shapes(case):
    dtype, b, T, H, P, N, G, gate, bias, skip, init, dfin = case
    w, inp = random_inputs("ssd", dtype, b, T, H, P, N, ngroups=G, gate=gate, dt_bias=bias,
                           d_skip="normal" if skip else "none", seed=T + H + P + N)
    dout, dfinal, h0 = extras(w, seed=T + 3, with_init=init, with_dfinal=dfin)
    compare(w, inp, dout, dfinal, h0)


def test_backward_ssd_many_channels():
    """SSD with the channels of many thread blocks per group and head."""
    w, inp = random_inputs("ssd", "bf16", 2, 24, 16, 64, 128, ngroups=2, seed=11)
    dout, dfinal, h0 = extras(w, seed=12)
    compare(w, inp, dout, dfinal, h0)


# The chunked tensor-core backward (bf16, headdim 64, dstate 64 or 128, an even number of
# heads per group): chunks of 128 steps, ragged last chunks, groups, every optional input
# present or absent.  (dtype, batch, T, H, P, N, G, gate, bias, skip, init, dfinal)
TC_CASES = [
    ("bf16", 2, 300, 4, 64, 64, 1, True, True, True, True, True),
    ("bf16", 1, 128, 2, 64, 128, 1, False, False, False, False, False),
    ("bf16", 2, 257, 6, 64, 128, 3, True, True, True, False, True),
    ("bf16", 1, 1, 2, 64, 64, 1, True, True, True, True, True),
    ("bf16", 3, 129, 8, 64, 64, 2, True, False, True, True, False),
    ("bf16", 1, 1000, 2, 64, 128, 1, True, True, True, True, True),
]


@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: "-".join(map(str, c)))
def test_backward_ssd_tensor_core(case):
    dtype, b, T, H, P, N, G, gate, bias, skip, init, dfin = case
    w, inp = random_inputs("ssd", dtype, b, T, H, P, N, ngroups=G, gate=gate, dt_bias=bias,
                           d_skip="normal" if skip else "none", seed=T + H + N + 7)
    dout, dfinal, h0 = extras(w, seed=T + 5, with_init=init, with_dfinal=dfin)
    errs = compare(w, inp, dout, dfinal, h0)
    record_errors(f"ssd backward tc {case}", {k: {"gated": v} for k, v in errs.items()})


def test_backward_ssd_tensor_core_matches_recurrence_kernel():
    """The chunked tensor-core backward and the recurrence kernel (SSM_TUNE_SSD_CUDA_CORES)
    agree on the same inputs within the bf16 bound."""
    w, inp = random_inputs("ssd", "bf16", 2, 400, 4, 64, 128, gate=True, dt_bias=True, seed=41)
    dout, dfinal, h0 = extras(w, seed=42)
    tc = grads_gpu(inp, dout, dfinal, h0)
    with _lib.tuned(_lib.SSM_TUNE_SSD_CUDA_CORES, 1):
        rec = grads_gpu(inp, dout, dfinal, h0)
    for k in tc:
        if tc[k] is None:
            continue
        assert oracle.max_rel_error(tc[k], rec[k]) <= 2e-2, k
