"""GPU parity of the complex diagonal scan (SSM_MODE_CDIAG, the rotating state update
read for Mamba-3) against the fp64 oracle's complex scan, element by element.

Tolerances as for the real scans: max relative error (floor 1e-2 of the largest
reference value) 1e-4 for fp32 inputs, 2e-2 for bf16 inputs with fp32 state.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_143_b300 as ssm
from selective_state_space_143_b300.inputs import WORKLOADS, make_inputs, random_inputs

from conftest import record_errors

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
DEV = "cuda:0"


def run_gpu(inp, chunk=0, initial_state=None):
    d = {k: (None if v is None else v.to(DEV)) for k, v in inp.items()}
    out, fs = ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                           return_final_state=True, chunk=chunk,
                           initial_state=None if initial_state is None else initial_state.to(DEV))
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), fs.cpu().numpy()


def ref(inp, **kw):
    return oracle.scan_complex(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                               inp["z"], inp["dt_bias"], **kw)


def check(name, dtype, pairs):
    reports = {k: oracle.error_report(g, r) for k, (g, r) in pairs.items()}
    record_errors(name, reports)
    for k, (g, _) in pairs.items():
        assert np.all(np.isfinite(g)), f"{name}/{k}: non-finite"
        assert reports[k]["gated"] <= TOL[dtype], f"{name}/{k}: {reports[k]['gated']:.3e}"


CASES = [
    # (dtype, batch, T, D, N, G, chunk)
    ("f32", 1, 1, 8, 4, 1, 0),
    ("f32", 2, 37, 24, 8, 1, 0),
    ("f32", 1, 300, 16, 16, 2, 0),
    ("f32", 1, 200, 8, 32, 1, 48),      # largest state, forced time segments
    ("bf16", 2, 257, 64, 16, 1, 0),
    ("bf16", 1, 1000, 48, 8, 2, 0),     # few channels: time segments
    ("bf16", 3, 129, 40, 4, 1, 0),
    ("bf16", 2, 700, 64, 32, 1, 64),
    ("bf16", 1, 0, 16, 8, 1, 0),        # empty sequence: final state zero
]


@pytest.mark.parametrize("case", CASES, ids=str)
def test_complex_shapes(case):
    dtype, b, T, D, N, G, chunk = case
    _, inp = random_inputs("cdiag", dtype, b, T, D, 1, N, ngroups=G, seed=T + D + N)
    y, fs = run_gpu(inp, chunk=chunk)
    r, rfs = ref(inp)
    if T == 0:
        assert np.all(fs == 0.0)
        return
    check(f"complex {case}", dtype, {"out": (y, r), "final_state": (fs, rfs)})


def test_complex_cx1_full():
    w = WORKLOADS["cx1"]
    inp = make_inputs(w)
    y, fs = run_gpu(inp)
    r, rfs = ref(inp)
    check("cx1 full", "bf16", {"out": (y, r), "final_state": (fs, rfs)})


def test_complex_cx2_sampled():
    w = WORKLOADS["cx2"]
    inp = make_inputs(w)
    y, fs = run_gpu(inp)
    nch = w.batch * w.nheads
    sel = np.unique(np.concatenate([[0, nch - 1], np.random.default_rng(5).choice(nch, 62, replace=False)]))
    r, rfs = ref(inp, select=sel)
    yv = y.transpose(0, 2, 1).reshape(nch, w.seqlen)[sel]
    rv = r.transpose(0, 2, 1).reshape(nch, w.seqlen)[sel]
    check("cx2 sampled", "bf16", {"out": (yv, rv),
                                  "final_state": (fs.reshape(nch, -1)[sel], rfs.reshape(nch, -1)[sel])})


def test_complex_resume_from_state():
    """Two calls, the second starting from the first's final state, equal one call."""
    _, inp = random_inputs("cdiag", "bf16", 2, 600, 64, 1, 16, seed=3)
    cut = 256
    first = {k: (v[:, :cut].contiguous() if k in ("x", "dt", "B", "C", "z") and v is not None else v)
             for k, v in inp.items()}
    rest = {k: (v[:, cut:].contiguous() if k in ("x", "dt", "B", "C", "z") and v is not None else v)
            for k, v in inp.items()}
    _, s1 = run_gpu(first)
    y2, fs2 = run_gpu(rest, initial_state=torch.from_numpy(s1))
    r, rfs = ref(inp)
    check("complex resume", "bf16", {"out": (y2, r[:, cut:]), "final_state": (fs2, rfs)})


def test_complex_without_imaginary_parts_matches_real_scan():
    """Zero imaginary parts: the complex kernels give the real diagonal scan's result."""
    _, inp = random_inputs("cdiag", "f32", 2, 200, 32, 1, 16, seed=9)
    for k in ("A", "B", "C"):
        inp[k][..., 1] = 0.0
    y, fs = run_gpu(inp)
    real = dict(inp, A=inp["A"][..., 0].contiguous(), B=inp["B"][..., 0].contiguous(),
                C=inp["C"][..., 0].contiguous())
    d = {k: (None if v is None else v.to(DEV)) for k, v in real.items()}
    yr, fsr = ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                           return_final_state=True)
    torch.cuda.synchronize()
    assert oracle.max_rel_error(y, yr.cpu().numpy()) <= 1e-4
    assert oracle.max_rel_error(fs[..., 0], fsr.cpu().numpy()) <= 1e-4
    assert np.all(fs[..., 1] == 0.0)


def test_complex_delta_zero_gives_skip_only():
    _, inp = random_inputs("cdiag", "bf16", 2, 100, 64, 1, 8, seed=4)
    inp["dt"] = torch.full_like(inp["dt"], -1e4)
    inp["dt_bias"] = None
    y, fs = run_gpu(inp)
    r, _ = ref(inp)
    assert np.all(fs == 0.0)
    assert oracle.max_rel_error(y, r) <= 2e-2
