"""GPU parity at the workloads' full lengths and widths, where the oracle can only be run
on part of the problem.

Channels never interact in the forward recurrence, and in the backward pass only the
gradients of the shared inputs (B and C, and the per-head sums in SSD mode) combine
channels.  So a full-size GPU run is compared with the oracle run on a sub-problem that
keeps the sampled channels (heads in SSD mode) with every batch entry and every time
step: every per-channel quantity, and every per-head sum over the kept heads, must match.
The gradients that sum over all channels (dB, dC) are compared on problems of the same
length with fewer channels, with the kernels' time partitioning forced to what the full
workload uses.

Every comparison records the gated error and the informational measures
(oracle.error_report) through conftest.record_errors.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_143_b300 as ssm
from selective_state_space_143_b300 import _lib
from selective_state_space_143_b300.inputs import WORKLOADS, make_inputs, random_inputs, shapes

from conftest import record_errors

pytestmark = pytest.mark.gpu

TOL = 2e-2  # bf16 inputs, fp32 state and accumulation
DEV = "cuda:0"


def to_dev(inp):
    return {k: (None if v is None else v.to(DEV)) for k, v in inp.items()}


def check(name, pairs):
    """pairs: {quantity: (gpu array, oracle array)}; asserts the gated bound on each."""
    reports = {}
    for k, (g, r) in pairs.items():
        assert np.all(np.isfinite(g)), f"{name}/{k}: non-finite"
        reports[k] = oracle.error_report(g, r)
    record_errors(name, reports)
    for k, rep in reports.items():
        assert rep["gated"] <= TOL, f"{name}/{k}: max rel err {rep['gated']:.3e} > {TOL}"


def test_c4_forward_every_head():
    """c4 (1 x 131072 tokens, 32 heads x 64, N 256): two channels of every head, and
    their final states."""
    w = WORKLOADS["c4"]
    inp = make_inputs(w)
    d = to_dev(inp)
    out, fs = ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                           return_final_state=True, chunk=w.chunk)
    torch.cuda.synchronize()
    rng = np.random.default_rng(44)
    H, P = w.nheads, w.headdim
    sel = np.sort(np.concatenate([h * P + rng.choice(P, 2, replace=False) for h in range(H)]))
    ref, ref_fs = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["z"], inp["dt_bias"], select=sel)
    y = out.float().cpu().numpy()[0].reshape(w.seqlen, H * P)[:, sel]
    r = ref[0].reshape(w.seqlen, H * P)[:, sel]
    f = fs.cpu().numpy().reshape(H * P, w.dstate)[sel]
    rf = ref_fs.reshape(H * P, w.dstate)[sel]
    check("c4 forward, 2 channels of each of 32 heads", {"out": (y, r), "final_state": (f, rf)})


def _dout(w, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(tuple(shapes(w)["x"]), generator=g).to(torch.bfloat16)


def _gpu_bwd(inp, dout):
    d = to_dev(inp)
    g = ssm.scan_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                     dout=dout.to(DEV))
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in g.items()}


def _oracle_bwd(inp, dout):
    return oracle.scan_bwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                           inp["dt_bias"], None, dout=dout)


GRADS = {"dx": "dx", "ddt": "ddt", "dA": "dA", "dB": "dB", "dC": "dC", "dD": "dD", "dz": "dz",
         "ddt_bias": "ddt_bias", "dinitial_state": "dinit"}


def test_ssd_backward_c3_sampled_heads():
    """The SSD-mode backward of c3 itself (4 x 8192 tokens, 64 heads x 64, N 128; one time
    part, 4-step checkpoint segments), compared on two heads with every batch entry."""
    w = WORKLOADS["c3"]
    inp = make_inputs(w)
    dout = _dout(w, seed=9)
    got = _gpu_bwd(inp, dout)
    heads = np.array([5, 58])
    ht = torch.as_tensor(heads)
    sub = dict(inp)
    sub["x"] = inp["x"][:, :, ht].contiguous()
    sub["dt"] = inp["dt"][:, :, ht].contiguous()
    sub["A"] = inp["A"][ht].contiguous()
    sub["D"] = None if inp["D"] is None else inp["D"][ht].contiguous()
    sub["dt_bias"] = None if inp["dt_bias"] is None else inp["dt_bias"][ht].contiguous()
    sub["z"] = None if inp["z"] is None else inp["z"][:, :, ht].contiguous()
    ref = _oracle_bwd(sub, dout[:, :, ht].contiguous())
    pairs = {"dx": (got["dx"][:, :, heads], ref["dx"]), "ddt": (got["ddt"][:, :, heads], ref["ddt"]),
             "dA": (got["dA"][heads], ref["dA"]),
             "dinitial_state": (got["dinitial_state"][:, heads], ref["dinit"])}
    if ref["dD"] is not None:
        pairs["dD"] = (got["dD"][heads], ref["dD"])
    check("c3 SSD backward, heads 5 and 58 of 64", pairs)


@pytest.mark.parametrize("parts", [1, 0])
def test_ssd_backward_c3_length_all_gradients(parts):
    """Every gradient (dB and dC included) at c3's length and state width: 8192 tokens,
    N 128, two heads of 64.  parts=1 is c3's own plan (the channels fill the GPU, one
    time part); parts=0 lets the planner cut this few-channel shape into time parts."""
    w, inp = random_inputs("ssd", "bf16", 1, 8192, 2, 64, 128, seed=17)
    dout = _dout(w, seed=18)
    with _lib.tuned(_lib.SSM_TUNE_BWD_PARTS, parts):
        got = _gpu_bwd(inp, dout)
    ref = _oracle_bwd(inp, dout)
    pairs = {k: (got[k], ref[rk]) for k, rk in GRADS.items() if ref[rk] is not None and got[k] is not None}
    check(f"SSD backward 1x8192, 2 heads x 64, N 128, parts {parts or 'auto'}", pairs)


def test_ssd_backward_long_wide_state():
    """Every gradient at N 256 over 4096 tokens (32 lanes x 8 entries per channel)."""
    w, inp = random_inputs("ssd", "bf16", 1, 4096, 1, 64, 256, seed=19)
    dout = _dout(w, seed=20)
    got = _gpu_bwd(inp, dout)
    ref = _oracle_bwd(inp, dout)
    pairs = {k: (got[k], ref[rk]) for k, rk in GRADS.items() if ref[rk] is not None and got[k] is not None}
    check("SSD backward 1x4096, 1 head x 64, N 256", pairs)


def test_diag_backward_c2_sampled_channels():
    """The diagonal backward of c2 itself (4 x 8192 tokens, 5120 channels, N 16; 8 time
    parts), compared on 64 channels with every batch entry: every per-channel gradient."""
    w = WORKLOADS["c2"]
    inp = make_inputs(w)
    dout = _dout(w, seed=21)
    got = _gpu_bwd(inp, dout)
    rng = np.random.default_rng(22)
    ch = np.sort(np.concatenate([[0, w.nheads - 1], rng.choice(np.arange(1, w.nheads - 1), 62, replace=False)]))
    ct = torch.as_tensor(ch)
    sub = dict(inp)
    for k in ("x", "dt", "z"):
        sub[k] = None if inp[k] is None else inp[k][:, :, ct].contiguous()
    for k in ("A", "D", "dt_bias"):
        sub[k] = None if inp[k] is None else inp[k][ct].contiguous()
    ref = _oracle_bwd(sub, dout[:, :, ct].contiguous())
    pairs = {"dx": (got["dx"][:, :, ch], ref["dx"]), "ddt": (got["ddt"][:, :, ch], ref["ddt"]),
             "dA": (got["dA"][ch], ref["dA"]), "dinitial_state": (got["dinitial_state"][:, ch], ref["dinit"])}
    for k, rk in (("dz", "dz"), ("dD", "dD"), ("ddt_bias", "ddt_bias")):
        if ref[rk] is not None:
            idx = (slice(None), slice(None), ch) if k == "dz" else ch
            pairs[k] = (got[k][idx], ref[rk])
    check("c2 diagonal backward, 64 of 5120 channels", pairs)


def test_diag_backward_c2_length_all_gradients():
    """Every gradient (dB and dC included) at c2's length with c2's 8 time parts: 8192
    tokens, 512 channels, N 16."""
    w, inp = random_inputs("diag", "bf16", 1, 8192, 512, 1, 16, seed=23)
    dout = _dout(w, seed=24)
    with _lib.tuned(_lib.SSM_TUNE_BWD_PARTS, 8):
        got = _gpu_bwd(inp, dout)
    ref = _oracle_bwd(inp, dout)
    pairs = {k: (got[k], ref[rk]) for k, rk in GRADS.items() if ref[rk] is not None and got[k] is not None}
    check("diagonal backward 1x8192, 512 channels, N 16, 8 time parts", pairs)
