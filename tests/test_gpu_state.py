"""GPU parity of the carried state: a scan that starts from a given state, a long
sequence scanned in pieces that resume from each other's final state, and token-by-token
decoding with the state updated in place -- each against one fp64 oracle scan of the
whole sequence from the same initial state.

Initial states are the oracle's final state over an independent seeded prefix, so they
have the magnitudes a real resumed scan sees.  Tolerances as in the other parity tests:
max relative error (floor 1e-2 of the largest reference value) 1e-4 for fp32 inputs,
2e-2 for bf16 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_143_b300 as ssm
from selective_state_space_143_b300.inputs import random_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
DEV = "cuda:0"

# (mode, dtype, batch, T, H, P, N, G, chunk)
CASES = [
    ("diag", "f32", 2, 200, 32, 1, 16, 1, 0),
    ("diag", "bf16", 2, 700, 64, 1, 16, 1, 64),     # forced time segments
    ("diag", "bf16", 1, 300, 96, 1, 24, 3, 0),
    ("diag", "bf16", 2, 1024, 512, 1, 16, 1, 0),    # split across blocks by the default plan
    ("ssd", "f32", 1, 260, 2, 32, 16, 2, 0),         # CUDA-core SSD kernels
    ("ssd", "bf16", 2, 300, 4, 64, 128, 2, 128),     # tensor-core SSD kernels
    ("ssd", "bf16", 1, 513, 2, 64, 256, 1, 256),
]


def case_id(c):
    return "-".join(str(v) for v in c)


def inputs(case, seed_shift=0):
    mode, dtype, b, T, H, P, N, G, chunk = case
    w, inp = random_inputs(mode, dtype, b, T, H, P, N, ngroups=G, seed=T + H + N + seed_shift)
    return w.replace(chunk=chunk), inp


def prefix_state(case):
    """Oracle final state over an independent seeded prefix of 64 tokens."""
    mode, dtype, b, T, H, P, N, G, chunk = case
    _, pre = random_inputs(mode, dtype, b, 64, H, P, N, ngroups=G, seed=7 + H + N)
    _, fs = oracle.scan(pre["x"], pre["dt"], pre["A"], pre["B"], pre["C"], pre["D"], pre["z"],
                        pre["dt_bias"])
    return fs.astype(np.float32)


def dev(t):
    return None if t is None else t.to(DEV)


def piece(inp, s, e):
    """Tokens [s, e) of every per-token input (A, D and dt_bias are shared)."""
    out = {}
    for k, v in inp.items():
        if v is not None and k in ("x", "dt", "B", "C", "z"):
            out[k] = v[:, s:e].contiguous()
        else:
            out[k] = v
    return out


def check(w, y, fs, ref, ref_fs, what=""):
    tol = TOL[w.dtype]
    assert np.all(np.isfinite(y)), "non-finite output"
    err = oracle.max_rel_error(y, ref)
    err_fs = oracle.max_rel_error(fs, ref_fs)
    assert err <= tol, f"{what} out max rel err {err:.3e} > {tol}"
    assert err_fs <= tol, f"{what} final_state max rel err {err_fs:.3e} > {tol}"
    return err, err_fs


def scan_gpu(inp, w, init):
    d = {k: dev(v) for k, v in inp.items()}
    out, fs = ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                           return_final_state=True, chunk=w.chunk,
                           initial_state=None if init is None else dev(init))
    return out, fs


@pytest.mark.parametrize("case", CASES, ids=case_id)
def test_scan_from_initial_state(case):
    w, inp = inputs(case)
    h0 = prefix_state(case)
    ref, ref_fs = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["z"], inp["dt_bias"], initial_state=h0)
    out, fs = scan_gpu(inp, w, torch.from_numpy(h0))
    torch.cuda.synchronize()
    check(w, out.float().cpu().numpy(), fs.cpu().numpy(), ref, ref_fs)


@pytest.mark.parametrize("case", CASES, ids=case_id)
def test_split_sequence_resumes(case):
    """Three pieces of uneven length, each starting from the previous final state."""
    w, inp = inputs(case)
    T = w.seqlen
    h0 = prefix_state(case)
    ref, ref_fs = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["z"], inp["dt_bias"], initial_state=h0)
    cuts = [0, T // 3 + 5, (2 * T) // 3 - 1, T]
    state = torch.from_numpy(h0)
    ys = []
    for s, e in zip(cuts[:-1], cuts[1:]):
        out, state = scan_gpu(piece(inp, s, e), w, state)
        ys.append(out)
    torch.cuda.synchronize()
    y = torch.cat(ys, dim=1).float().cpu().numpy()
    check(w, y, state.cpu().numpy(), ref, ref_fs, "split")


def step_tensors(inp, t):
    """Token t of every per-token input, on the device, in ssm.step's layout."""
    d = {}
    for k in ("x", "dt", "z"):
        d[k] = None if inp[k] is None else dev(inp[k][:, t].contiguous())
    for k in ("B", "C"):
        d[k] = dev(inp[k][:, t].contiguous())  # (b, G, N)
    for k in ("A", "D", "dt_bias"):
        d[k] = dev(inp[k])
    return d


@pytest.mark.parametrize("case", CASES, ids=case_id)
def test_prefill_then_decode(case):
    """Scan a prefix, then decode the remaining tokens one ssm_step call at a time with
    the state updated in place; outputs and the final state match one oracle scan."""
    w, inp = inputs(case)
    T = w.seqlen
    n_dec = min(40, T // 2)
    h0 = prefix_state(case)
    ref, ref_fs = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["z"], inp["dt_bias"], initial_state=h0)
    out_pre, state = scan_gpu(piece(inp, 0, T - n_dec), w, torch.from_numpy(h0))
    ys = [out_pre.float()]
    for t in range(T - n_dec, T):
        d = step_tensors(inp, t)
        y = ssm.step(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                     state=state)
        ys.append(y.float().unsqueeze(1))
    torch.cuda.synchronize()
    y = torch.cat(ys, dim=1).cpu().numpy()
    check(w, y, state.cpu().numpy(), ref, ref_fs, "decode")
    # the decoded tokens alone, so a fault there is not hidden by the long prefix
    tol = TOL[w.dtype]
    err = oracle.max_rel_error(y[:, T - n_dec:], ref[:, T - n_dec:])
    assert err <= tol, f"decoded tokens max rel err {err:.3e}"


@pytest.mark.parametrize("mode,dtype,N", [("diag", "f32", 4), ("diag", "bf16", 64),
                                          ("ssd", "f32", 12), ("ssd", "bf16", 256)])
def test_step_ragged_state_widths(mode, dtype, N):
    """State rows that are not a multiple of the lanes a channel gets (N/4 not a power of
    two, or a full warp with several pieces each)."""
    H, P = (48, 1) if mode == "diag" else (6, 16)
    w, inp = random_inputs(mode, dtype, 3, 6, H, P, N, seed=N + H)
    h0 = np.random.default_rng(5).standard_normal((3, H, N) if mode == "diag" else (3, H, P, N))
    h0 = h0.astype(np.float32)
    ref, ref_fs = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["z"], inp["dt_bias"], initial_state=h0)
    state = torch.from_numpy(h0).to(DEV)
    ys = []
    for t in range(6):
        d = step_tensors(inp, t)
        ys.append(ssm.step(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"],
                           d["dt_bias"], state=state).float().unsqueeze(1))
    torch.cuda.synchronize()
    check(w, torch.cat(ys, 1).cpu().numpy(), state.cpu().numpy(), ref, ref_fs, "ragged step")


@pytest.mark.parametrize("mode", ["diag", "ssd"])
def test_empty_sequence_passes_state_through(mode):
    """seqlen 0: the final state is the initial state, bit for bit."""
    H, P, N = (64, 1, 16) if mode == "diag" else (4, 64, 64)
    w, inp = random_inputs(mode, "bf16", 2, 0, H, P, N, seed=1)
    h0 = torch.randn((2, H, N) if mode == "diag" else (2, H, P, N),
                     generator=torch.Generator().manual_seed(3))
    out, fs = scan_gpu(inp, w, h0)
    torch.cuda.synchronize()
    assert out.numel() == 0
    assert torch.equal(fs.cpu(), h0)


def test_step_matches_one_token_scan_bitwise_state_path():
    """ssm_step and a one-token scan from the same state agree (both within rounding of
    the oracle; the step kernel's output must not depend on the batch position)."""
    w, inp = random_inputs("ssd", "bf16", 4, 1, 8, 64, 128, seed=9)
    h0 = torch.from_numpy(np.random.default_rng(2).standard_normal((4, 8, 64, 128))
                          .astype(np.float32))
    ref, ref_fs = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["z"], inp["dt_bias"], initial_state=h0.numpy())
    state = h0.to(DEV)
    d = step_tensors(inp, 0)
    y = ssm.step(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                 state=state)
    torch.cuda.synchronize()
    check(w, y.float().unsqueeze(1).cpu().numpy(), state.cpu().numpy(), ref, ref_fs)
    # same inputs replicated across the batch give identical rows
    rep = {k: (None if v is None else v[:1].expand(4, *v.shape[1:]).contiguous())
           for k, v in d.items() if k not in ("A", "D", "dt_bias")}
    st2 = h0[:1].expand(4, *h0.shape[1:]).contiguous().to(DEV)
    y2 = ssm.step(rep["x"], rep["dt"], d["A"], rep["B"], rep["C"], d["D"], rep["z"], d["dt_bias"],
                  state=st2)
    torch.cuda.synchronize()
    for i in range(1, 4):
        assert torch.equal(y2[i], y2[0])
        assert torch.equal(st2[i], st2[0])


@pytest.mark.parametrize("mode,dtype,b,H,P,N", [
    ("diag", "bf16", 2048, 512, 1, 16),   # 64 MB carried state
    ("diag", "f32", 1400, 512, 1, 24),    # rows of 6 pieces on 4 lanes
    ("ssd", "bf16", 32, 64, 64, 128),
])
def test_step_large_batch(mode, dtype, b, H, P, N):
    """Decode steps over a carried state of 64 MB or more (serving-size batches), sampled
    channels against the oracle."""
    T = 3
    w, inp = random_inputs(mode, dtype, b, T, H, P, N, seed=N + b)
    rng = np.random.default_rng(4)
    shape = (b, H, N) if mode == "diag" else (b, H, P, N)
    h0 = rng.standard_normal(shape).astype(np.float32)
    state = torch.from_numpy(h0).to(DEV)
    ys = []
    for t in range(T):
        d = step_tensors(inp, t)
        ys.append(ssm.step(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                           state=state).float().unsqueeze(1))
    torch.cuda.synchronize()
    y = torch.cat(ys, 1).cpu().numpy()
    nch = b * H * P
    sel = np.unique(np.concatenate([[0, nch - 1], rng.choice(nch, 200, replace=False)]))
    ref, ref_fs = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["z"], inp["dt_bias"], initial_state=h0, select=sel)
    yv = (y.transpose(0, 2, 1) if mode == "diag" else y.transpose(0, 2, 3, 1)).reshape(nch, T)[sel]
    rv = (ref.transpose(0, 2, 1) if mode == "diag" else ref.transpose(0, 2, 3, 1)).reshape(nch, T)[sel]
    tol = TOL[dtype]
    assert oracle.max_rel_error(yv, rv) <= tol
    assert oracle.max_rel_error(state.cpu().numpy().reshape(nch, N)[sel], ref_fs.reshape(nch, N)[sel]) <= tol
