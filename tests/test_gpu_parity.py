"""GPU parity: the CUDA scan (through the C ABI) against the fp64 oracle on the same
seeded inputs, element by element.

Tolerances (max relative error with a floor at 1e-2 of the largest reference value):
1e-4 for fp32 inputs, 2e-2 for bf16 inputs (fp32 state and accumulation).  Full-size
workloads are compared on a sample of channels that the oracle evaluates one by one.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_143_b300 as ssm
from selective_state_space_143_b300 import _lib
from selective_state_space_143_b300.inputs import WORKLOADS, make_inputs, random_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
DEV = "cuda:0"


def to_dev(inp):
    return {k: (None if v is None else v.to(DEV)) for k, v in inp.items()}


def run_gpu(inp, w, chunk=None, final_state=True, initial_state=None):
    d = to_dev(inp)
    out, fs = ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                           return_final_state=True, chunk=w.chunk if chunk is None else chunk)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), fs.cpu().numpy()


def channel_view(a, w):
    """(b, T, H[, P]) -> (b*H*P, T) with the oracle's flat channel order."""
    if w.mode == "diag":
        return a.transpose(0, 2, 1).reshape(-1, a.shape[1])
    return a.transpose(0, 2, 3, 1).reshape(-1, a.shape[1])


def compare(w, inp, y, fs, select=None, chunk=None):
    ref, ref_fs = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["z"], inp["dt_bias"], select=select)
    if select is not None:
        yv, rv = channel_view(y, w)[select], channel_view(ref, w)[select]
        fv = fs.reshape(-1, w.dstate)[select]
        rfv = ref_fs.reshape(-1, w.dstate)[select]
    else:
        yv, rv, fv, rfv = y, ref, fs, ref_fs
    err = oracle.max_rel_error(yv, rv)
    err_fs = oracle.max_rel_error(fv, rfv)
    tol = TOL[w.dtype]
    assert np.all(np.isfinite(yv)), "non-finite output"
    assert err <= tol, f"out max rel err {err:.3e} > {tol}"
    assert err_fs <= tol, f"final_state max rel err {err_fs:.3e} > {tol}"
    return err, err_fs


@pytest.mark.parametrize("name", ["c0", "c1"])
def test_workload_full(name):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    y, fs = run_gpu(inp, w)
    err, err_fs = compare(w, inp, y, fs)
    print(f"{name}: out {err:.3e} final_state {err_fs:.3e}")


@pytest.mark.parametrize("px", [1, 2])
@pytest.mark.parametrize("shape", [dict(batch=8, seqlen=1024, nheads=512), dict(batch=4, seqlen=512, nheads=5120)],
                         ids=["c1-shape", "c2-widths"])
def test_diag_fma_pipe_exp2(px, shape):
    """SSM_TUNE_DIAG_EXP_POLY: 1 or 2 of every 2 decay pairs from the FMA-pipe polynomial
    exp2 (both lane layouts: 4 entries per lane with time segments, and 8 per lane)."""
    w, inp = random_inputs("diag", "bf16", headdim=1, dstate=16, seed=17, **shape)
    with _lib.tuned(_lib.SSM_TUNE_DIAG_EXP_POLY, px):
        y, fs = run_gpu(inp, w, chunk=0)
    err, err_fs = compare(w, inp, y, fs)
    print(f"px {px}: out {err:.3e} final_state {err_fs:.3e}")


@pytest.mark.parametrize("name", ["c2", "c3", "c4"])
def test_workload_full_size_sampled(name):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    y, fs = run_gpu(inp, w)
    nch = w.batch * w.d_inner
    rng = np.random.default_rng(123)
    k = 24 if name == "c4" else 96
    sel = np.unique(np.concatenate([[0, nch - 1], rng.choice(nch, k, replace=False)]))
    err, err_fs = compare(w, inp, y, fs, select=sel)
    print(f"{name}: out {err:.3e} final_state {err_fs:.3e} on {sel.size} channels")


DIAG_CASES = [
    # (dtype, batch, T, D, N, G, chunk)
    ("f32", 1, 1, 8, 4, 1, 0),
    ("f32", 2, 31, 24, 12, 1, 0),
    ("f32", 1, 33, 40, 16, 2, 0),
    ("bf16", 3, 257, 72, 16, 1, 0),
    ("bf16", 2, 1000, 48, 8, 2, 0),
    ("bf16", 1, 300, 96, 24, 3, 0),
    ("bf16", 2, 513, 64, 32, 1, 0),
    ("bf16", 1, 129, 40, 64, 1, 0),
    ("bf16", 2, 700, 64, 16, 1, 64),   # forced time segments
    ("bf16", 1, 1024, 32, 16, 1, 96),
    ("f32", 1, 450, 16, 8, 1, 32),
    ("f32", 2, 77, 8, 64, 1, 0),       # largest state (N = 64), fp32
    ("bf16", 4, 1, 16, 16, 2, 0),      # one token per sequence
]


@pytest.mark.parametrize("case", DIAG_CASES, ids=str)
def test_diag_shapes(case):
    dtype, b, T, D, N, G, chunk = case
    w, inp = random_inputs("diag", dtype, b, T, D, 1, N, ngroups=G, seed=T + D + N)
    y, fs = run_gpu(inp, w, chunk=chunk)
    compare(w, inp, y, fs)


SSD_CASES = [
    # (dtype, batch, T, H, P, N, G, chunk)
    ("f32", 1, 1, 2, 16, 16, 1, 0),
    ("bf16", 2, 200, 4, 64, 64, 1, 64),
    ("bf16", 1, 300, 4, 64, 128, 2, 128),
    ("bf16", 1, 513, 2, 64, 256, 1, 256),
    ("bf16", 2, 97, 3, 80, 32, 1, 32),
    ("f32", 1, 260, 2, 32, 16, 2, 0),
    ("bf16", 1, 150, 1, 256, 16, 1, 64),   # largest head dimension (P = 256)
    ("f32", 1, 70, 2, 16, 256, 1, 32),     # largest state (N = 256), fp32
    ("bf16", 1, 300, 4, 64, 128, 4, 256),  # one group per head
    ("bf16", 2, 777, 8, 64, 256, 1, 128),  # dstate 256 at chunk 128: every CTA a first half, ragged end
    ("bf16", 1, 1000, 16, 64, 256, 2, 256),  # dstate 256, two groups of 8 heads, ragged end
]


@pytest.mark.parametrize("case", SSD_CASES, ids=str)
def test_ssd_shapes(case):
    dtype, b, T, H, P, N, G, chunk = case
    w, inp = random_inputs("ssd", dtype, b, T, H, P, N, ngroups=G, seed=T + H + P + N)
    w = w.replace(chunk=chunk)
    y, fs = run_gpu(inp, w)
    compare(w, inp, y, fs)


@pytest.mark.parametrize("N,chunk", [(128, 256), (256, 256), (256, 128)])
def test_ssd_strong_and_weak_decay_heads(N, chunk):
    """Heads that barely decay within a chunk beside heads whose cumulative sums fall to
    the hundreds within a chunk (exp(cum_t - cum_s) spanning the whole fp32 range), in
    one launch: M' must stay exact where the decay underflows, with no overflow where it
    does not."""
    w, inp = random_inputs("ssd", "bf16", 1, 700, 8, 64, N, seed=N + chunk)
    w = w.replace(chunk=chunk)
    bias = inp["dt_bias"].clone()
    bias[::2] = 1.0  # Delta ~ 1.3-2.4: cumulative sums of -100s within a chunk
    inp["dt_bias"] = bias
    y, fs = run_gpu(inp, w)
    compare(w, inp, y, fs)


@pytest.mark.parametrize("mode", ["diag", "ssd"])
def test_delta_zero_gives_skip_only(mode):
    if mode == "diag":
        w, inp = random_inputs("diag", "bf16", 2, 100, 64, 1, 16, seed=3)
    else:
        w, inp = random_inputs("ssd", "bf16", 2, 100, 4, 64, 64, seed=3)
        w = w.replace(chunk=64)
    inp["dt"] = torch.full_like(inp["dt"], -1e4)
    inp["dt_bias"] = None
    y, fs = run_gpu(inp, w)
    D = inp["D"].numpy().astype(np.float64)
    x = inp["x"].float().numpy().astype(np.float64)
    z = inp["z"].float().numpy().astype(np.float64)
    Dv = D.reshape((1, 1, -1) if mode == "diag" else (1, 1, -1, 1))
    ref = Dv * x * z / (1 + np.exp(-z))
    assert oracle.max_rel_error(y, ref) < 1e-2
    assert np.all(fs == 0.0)


@pytest.mark.parametrize("mode", ["diag", "ssd"])
def test_causality_bit_exact(mode):
    if mode == "diag":
        w, inp = random_inputs("diag", "bf16", 1, 700, 64, 1, 16, seed=5)
    else:
        w, inp = random_inputs("ssd", "bf16", 1, 700, 2, 64, 64, seed=5)
        w = w.replace(chunk=128)
    y0, _ = run_gpu(inp, w)
    for t0 in (0, 300, 511, 699):
        pert = dict(inp)
        pert["x"] = inp["x"].clone()
        pert["x"][:, t0] += 2.0
        y1, _ = run_gpu(pert, w)
        assert np.array_equal(y0[:, :t0], y1[:, :t0])
        assert not np.array_equal(y0[:, t0:], y1[:, t0:])


@pytest.mark.parametrize("mode", ["diag", "ssd"])
def test_repeat_runs_bit_identical(mode):
    if mode == "diag":
        w, inp = random_inputs("diag", "bf16", 2, 600, 128, 1, 16, seed=8)
    else:
        w, inp = random_inputs("ssd", "bf16", 2, 600, 4, 64, 128, seed=8)
        w = w.replace(chunk=256)
    first = run_gpu(inp, w)
    for _ in range(3):
        again = run_gpu(inp, w)
        assert np.array_equal(first[0], again[0]) and np.array_equal(first[1], again[1])


def test_diag_segment_length_invariance():
    w, inp = random_inputs("diag", "bf16", 1, 2048, 64, 1, 16, seed=9)
    outs = [run_gpu(inp, w, chunk=c)[0] for c in (0, 64, 256, 2048)]
    for o in outs[1:]:
        assert oracle.max_rel_error(o, outs[0]) < 2e-2


def test_ssd_chunk_invariance():
    w, inp = random_inputs("ssd", "bf16", 1, 1024, 4, 64, 128, seed=10)
    outs = [run_gpu(inp, w, chunk=c)[0] for c in (64, 128, 256)]
    for o in outs[1:]:
        assert oracle.max_rel_error(o, outs[0]) < 2e-2


@pytest.mark.parametrize("mode", ["diag", "ssd"])
def test_empty_inputs(mode):
    if mode == "diag":
        w, inp = random_inputs("diag", "bf16", 2, 0, 64, 1, 16, seed=1)
    else:
        w, inp = random_inputs("ssd", "bf16", 2, 0, 4, 64, 64, seed=1)
    y, fs = run_gpu(inp, w)
    assert y.shape[1] == 0 and np.all(fs == 0.0)
    w0, inp0 = random_inputs("diag", "bf16", 0, 16, 64, 1, 16, seed=1)
    y0, fs0 = run_gpu(inp0, w0)
    assert y0.shape[0] == 0 and fs0.shape[0] == 0


def test_workspace_entry_matches_allocating_entry():
    w, inp = random_inputs("ssd", "bf16", 1, 512, 4, 64, 128, seed=12)
    w = w.replace(chunk=128)
    d = to_dev(inp)
    ref = ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                       chunk=128)
    n = ssm.workspace_size(d["x"], d["A"], d["B"], chunk=128)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    got = ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                       chunk=128, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(ref, got)


def test_launch_timing_records_every_kernel():
    """ssm_timing_enable / ssm_timing_collect: one record per launch, named per kernel,
    the same count as the launch counter, and the results unchanged."""
    w = WORKLOADS["c1"]
    inp = make_inputs(w)
    d = {k: (None if v is None else v.to(DEV)) for k, v in inp.items()}
    ref = ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"])
    from selective_state_space_143_b300 import _lib
    _lib.timing_collect()
    _lib.timing_enable(True)
    n0 = ssm.launch_count()
    for _ in range(3):
        out = ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"])
    torch.cuda.synchronize()
    _lib.timing_enable(False)
    kt = _lib.timing_collect()
    assert sum(v[0] for v in kt.values()) == ssm.launch_count() - n0
    assert "diag_scan_kernel (output pass)" in kt and kt["diag_scan_kernel (output pass)"][0] == 3
    assert all(v[1] > 0 for v in kt.values())
    assert torch.equal(out, ref)
