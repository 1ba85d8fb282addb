"""GPU parity of the causal depthwise convolution + SiLU ahead of the scan: the fused
diagonal-mode kernels and the SSD path (a convolution pass, then the SSD kernels: the
tensor-core ones on the split bf16 hi/lo convolved input where the shape allows) against
the fp64 oracle (convolution, then the sequential scan), the carried last inputs bit for
bit, and resume / token-by-token decoding with the convolution state carried.

Tolerances: max relative error (floor 1e-2 of the largest reference value) 1e-4 for fp32
inputs, 2e-2 for bf16 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_143_b300 as ssm
from selective_state_space_143_b300.inputs import WORKLOADS, conv_params, make_inputs, random_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
DEV = "cuda:0"

# (mode, dtype, batch, T, H, P, N, G, chunk, width, bias, x_prev)
CASES = [
    ("diag", "f32", 1, 100, 32, 1, 16, 1, 0, 4, True, False),
    ("diag", "f32", 2, 450, 16, 1, 8, 1, 32, 4, True, True),     # forced time segments
    ("diag", "bf16", 2, 700, 64, 1, 16, 1, 64, 4, True, True),
    ("diag", "bf16", 2, 1024, 512, 1, 16, 1, 0, 4, True, False),  # default plan splits time
    ("diag", "bf16", 1, 300, 96, 1, 24, 3, 0, 3, False, True),
    ("diag", "bf16", 3, 257, 72, 1, 16, 1, 0, 2, True, True),
    ("diag", "bf16", 2, 129, 64, 1, 32, 1, 0, 1, True, False),
    ("diag", "bf16", 2, 2, 64, 1, 16, 1, 0, 4, True, True),       # shorter than the kernel
    ("ssd", "f32", 1, 260, 2, 32, 16, 2, 0, 4, True, True),
    ("ssd", "bf16", 2, 300, 4, 64, 128, 2, 128, 4, True, True),
    ("ssd", "bf16", 1, 513, 2, 64, 256, 1, 256, 3, False, False),
    # tensor-core kernels on the split convolved input, 8 heads per CTA (x planes reloaded
    # for every head), both 128-row halves, ragged last chunk
    ("ssd", "bf16", 1, 600, 16, 64, 128, 1, 256, 4, True, True),
    ("ssd", "bf16", 2, 333, 8, 64, 64, 2, 128, 4, True, False),
    ("ssd", "bf16", 1, 270, 8, 64, 32, 1, 256, 2, False, True),
]


def cid(c):
    return "-".join(str(v) for v in c)


def setup(case):
    mode, dtype, b, T, H, P, N, G, chunk, K, bias, prev = case
    w, inp = random_inputs(mode, dtype, b, T, H, P, N, ngroups=G, seed=T + H + N + K)
    cp = conv_params(H * P, K, seed=T + K, bias=bias, batch=b if prev else 0, dtype=dtype)
    return w.replace(chunk=chunk), inp, cp


def dev(t):
    return None if t is None else t.to(DEV)


def gpu_scan(w, inp, cp, x_prev=None, initial_state=None, with_last=True):
    d = {k: dev(v) for k, v in inp.items()}
    K = cp["weight"].shape[1]
    ch = cp["weight"].shape[0]
    last = torch.empty((w.batch, K - 1, ch), dtype=d["x"].dtype, device=DEV) if with_last else None
    out, fs = ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                           return_final_state=True, chunk=w.chunk,
                           initial_state=dev(initial_state),
                           conv_weight=dev(cp["weight"]), conv_bias=dev(cp["bias"]),
                           conv_x_prev=dev(x_prev), conv_x_last=last)
    return out, fs, last


def ref_scan(inp, cp, x_prev=None, initial_state=None):
    return oracle.scan_conv(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                            inp["dt_bias"], conv_w=cp["weight"], conv_b=cp["bias"],
                            x_prev=x_prev, initial_state=initial_state)


def check(w, y, fs, ref, ref_fs, what=""):
    tol = TOL[w.dtype]
    assert np.all(np.isfinite(y)), "non-finite output"
    err = oracle.max_rel_error(y, ref)
    err_fs = oracle.max_rel_error(fs, ref_fs)
    assert err <= tol, f"{what} out max rel err {err:.3e} > {tol}"
    assert err_fs <= tol, f"{what} final_state max rel err {err_fs:.3e} > {tol}"


@pytest.mark.parametrize("case", CASES, ids=cid)
def test_scan_with_conv(case):
    w, inp, cp = setup(case)
    out, fs, last = gpu_scan(w, inp, cp, x_prev=cp["x_prev"])
    torch.cuda.synchronize()
    ref, ref_fs, ref_last = ref_scan(inp, cp, x_prev=cp["x_prev"])
    check(w, out.float().cpu().numpy(), fs.cpu().numpy(), ref, ref_fs)
    # the carried inputs are copies of x (or x_prev) values: exact
    assert np.array_equal(last.float().cpu().numpy().astype(np.float64), ref_last)


@pytest.mark.parametrize("case", [c for c in CASES if c[3] >= 100], ids=cid)
def test_conv_split_resumes(case):
    """Pieces that resume from the previous piece's final state and last inputs equal one
    oracle run over the whole sequence."""
    w, inp, cp = setup(case)
    T = w.seqlen
    ref, ref_fs, ref_last = ref_scan(inp, cp, x_prev=cp["x_prev"])
    cuts = [0, 1, T // 3 + 2, T]   # a one-token piece, shorter than the kernel
    state, prev, ys = None, cp["x_prev"], []
    for s0, e0 in zip(cuts[:-1], cuts[1:]):
        piece = {k: (v[:, s0:e0].contiguous() if v is not None and k in ("x", "dt", "B", "C", "z")
                     else v) for k, v in inp.items()}
        out, state, prev = gpu_scan(w.replace(seqlen=e0 - s0), piece, cp, x_prev=prev,
                                    initial_state=state)
        ys.append(out)
    torch.cuda.synchronize()
    y = torch.cat(ys, 1).float().cpu().numpy()
    check(w, y, state.cpu().numpy(), ref, ref_fs, "split")
    assert np.array_equal(prev.float().cpu().numpy().astype(np.float64), ref_last)


@pytest.mark.parametrize("case", [c for c in CASES if c[3] >= 100], ids=cid)
def test_conv_prefill_then_decode(case):
    """Prefill with the convolution, then decode with ssm_step_conv, the convolution state
    shifted in place; every output matches one oracle run."""
    w, inp, cp = setup(case)
    T = w.seqlen
    n_dec = 24
    ref, ref_fs, ref_last = ref_scan(inp, cp, x_prev=cp["x_prev"])
    pre = {k: (v[:, :T - n_dec].contiguous() if v is not None and k in ("x", "dt", "B", "C", "z")
               else v) for k, v in inp.items()}
    out, state, conv_state = gpu_scan(w.replace(seqlen=T - n_dec), pre, cp, x_prev=cp["x_prev"])
    ys = [out.float()]
    for t in range(T - n_dec, T):
        d = {k: dev(inp[k][:, t].contiguous()) if inp[k] is not None else None
             for k in ("x", "dt", "B", "C", "z")}
        y = ssm.step(d["x"], d["dt"], dev(inp["A"]), d["B"], d["C"], dev(inp["D"]), d["z"],
                     dev(inp["dt_bias"]), state=state, conv_weight=dev(cp["weight"]),
                     conv_bias=dev(cp["bias"]), conv_state=conv_state)
        ys.append(y.float().unsqueeze(1))
    torch.cuda.synchronize()
    y = torch.cat(ys, 1).cpu().numpy()
    check(w, y, state.cpu().numpy(), ref, ref_fs, "decode")
    err = oracle.max_rel_error(y[:, T - n_dec:], ref[:, T - n_dec:])
    assert err <= TOL[w.dtype], f"decoded tokens max rel err {err:.3e}"
    assert np.array_equal(conv_state.float().cpu().numpy().astype(np.float64), ref_last)


def test_c1_block_with_conv():
    """The Mamba-1 block workload (batch 8 x L 1024 x d_inner 512, N 16) with the width-4
    convolution ahead of the scan, all channels."""
    w = WORKLOADS["c1"]
    inp = make_inputs(w)
    cp = conv_params(w.d_inner, 4, seed=1)
    out, fs, last = gpu_scan(w.replace(final_state=True), inp, cp)
    torch.cuda.synchronize()
    ref, ref_fs, ref_last = ref_scan(inp, cp)
    check(w, out.float().cpu().numpy(), fs.cpu().numpy(), ref, ref_fs)
    assert np.array_equal(last.float().cpu().numpy().astype(np.float64), ref_last)
