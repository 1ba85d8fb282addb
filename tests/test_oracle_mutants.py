"""Plant mistakes in a copy of the oracle (on the CPU) and check the pins catch each.

Every mutant below is a plausible slip in writing the recurrence: a dropped term,
a flipped sign, the output read before the state update, B and C swapped, the
zero-order-hold input term instead of Delta*B, the bias or the gate misplaced,
the wrong group index, a wrong softplus or SiLU, an ignored initial state.  Each
one must make at least one pin fail; the unmodified copy must pass them all.
"""
import math
import os
import subprocess

import numpy as np
import pytest

import oracle
from test_oracle_pins import _bruteforce, _golden_arrays, _rand_problem, load_golden

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")

MUTANTS = {
    "drop_D": ("if (p->D) y += p->D[h] * xv;", ""),
    "flip_A_sign": ("exp(delta * oracle_acoef(p, h, n))", "exp(-delta * oracle_acoef(p, h, n))"),
    "read_before_update": (
        "state[n] = abar * state[n] + delta * Bt[n] * xv;\n            y += Ct[n] * state[n];",
        "y += Ct[n] * state[n];\n            state[n] = abar * state[n] + delta * Bt[n] * xv;"),
    "swap_B_C": (
        "state[n] = abar * state[n] + delta * Bt[n] * xv;\n            y += Ct[n] * state[n];",
        "state[n] = abar * state[n] + delta * Ct[n] * xv;\n            y += Bt[n] * state[n];"),
    "zoh_input": ("state[n] = abar * state[n] + delta * Bt[n] * xv;",
                  "state[n] = abar * state[n] + (abar - 1.0) / oracle_acoef(p, h, n) * Bt[n] * xv;"),
    "drop_dt_bias": ("const double v = p->dt[bt * H + h] + (p->dt_bias ? p->dt_bias[h] : 0.0);",
                     "const double v = p->dt[bt * H + h];"),
    "gate_before_D": ("if (p->D) y += p->D[h] * xv;\n        if (p->z) y *= oracle_silu(p->z[xi]);",
                      "if (p->z) y *= oracle_silu(p->z[xi]);\n        if (p->D) y += p->D[h] * xv;"),
    "group_index": ("const int64_t g = h / (H / G);\n    const int64_t sidx = ((b * H + h) * P + q) * N;\n    for (int64_t n = 0; n < N; ++n) state[n] = p->initial_state ? p->initial_state[sidx + n] : 0.0;\n    for (int64_t t = 0; t < T; ++t) {",
                    "const int64_t g = h % G;\n    const int64_t sidx = ((b * H + h) * P + q) * N;\n    for (int64_t n = 0; n < N; ++n) state[n] = p->initial_state ? p->initial_state[sidx + n] : 0.0;\n    for (int64_t t = 0; t < T; ++t) {"),
    "softplus_as_exp": ("return fmax(v, 0.0) + log1p(exp(-fabs(v)));", "return exp(v);"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "ignore_initial_state": (
        "for (int64_t n = 0; n < N; ++n) state[n] = p->initial_state ? p->initial_state[sidx + n] : 0.0;\n    for (int64_t t = 0; t < T; ++t) {",
        "for (int64_t n = 0; n < N; ++n) state[n] = 0.0;\n    for (int64_t t = 0; t < T; ++t) {"),
}


CONV_MUTANTS = {
    "conv_flipped": ("acc += w[c * K + k] * v;", "acc += w[c * K + (K - 1 - k)] * v;"),
    "conv_drop_bias": ("double acc = bias ? bias[c] : 0.0;", "double acc = 0.0;"),
    "conv_prev_offset": ("v = x_prev[(b * (K - 1) + (K - 1 + s)) * channels + c];\n"
                         "                    acc += w[c * K + k] * v;",
                         "v = x_prev[(b * (K - 1) + (K - 2 + s)) * channels + c];\n"
                         "                    acc += w[c * K + k] * v;"),
    "conv_no_silu": ("xc[(b * seqlen + t) * channels + c] = oracle_silu(acc);",
                     "xc[(b * seqlen + t) * channels + c] = acc;"),
    "conv_last_off_by_one": ("const int64_t s = seqlen - K + 1 + j;", "const int64_t s = seqlen - K + j;"),
}


BWD_MUTANTS = {
    "bwd_no_decay_carry": ("g[n] *= abar; /* now dL/dh_{t-1} */", "/* carry dropped */"),
    "bwd_dA_uses_h_t": ("const double da = g[n] * abar * delta * hprev[n];",
                        "const double da = g[n] * abar * delta * hcur[n];"),
    "bwd_no_softplus_derivative": ("ddt[bt * H + h] += ddelta * sig_v;", "ddt[bt * H + h] += ddelta;"),
    "bwd_silu_derivative": ("dz[xi] = dout[xi] * y * sz * (1.0 + zv * (1.0 - sz));",
                            "dz[xi] = dout[xi] * y * sz;"),
    "bwd_dC_uses_h_prev": ("dC[(bt * G + grp) * N + n] += dy * hcur[n];",
                           "dC[(bt * G + grp) * N + n] += dy * hprev[n];"),
    "bwd_dx_no_skip": ("double dxv = D ? dy * D[h] : 0.0;", "double dxv = 0.0;"),
    "bwd_ddelta_no_decay_term": ("ddelta += g[n] * (Bt[n] * xv + abar * an * hprev[n]);",
                                 "ddelta += g[n] * (Bt[n] * xv);"),
    "bwd_gate_ignored": ("const double dy = dout[xi] * gate;", "const double dy = dout[xi];"),
}


def _bwd_pins(lib):
    """The backward pins (finite differences of this copy's own forward) on two cases."""
    from test_oracle_bwd_pins import mismatches, problem
    bad = []
    for mode, dims in (("diag", (1, 5, 2, 1, 3, 1)), ("ssd", (1, 4, 2, 2, 2, 1))):
        arr, dout, dfinal = problem(np.random.default_rng(9), mode, *dims)
        bad += [f"{mode}:{n}" for n in mismatches(oracle.scan, lib.scan_bwd, arr, dout, dfinal)]
    return bad


def _conv_pins(conv):
    """The convolution pins against ``conv`` (numpy.convolve per channel, resume)."""
    failed = []
    rng = np.random.default_rng(77)
    x = rng.standard_normal((2, 9, 3))
    w = rng.standard_normal((3, 4))
    bias = rng.standard_normal(3)
    prev = rng.standard_normal((2, 3, 3))
    xc, last = conv(x, w, bias, prev)
    for b in range(2):
        for c in range(3):
            seq = np.concatenate([prev[b, :, c], x[b, :, c]])
            pre = np.convolve(seq, w[c, ::-1])[3:12] + bias[c]
            if not np.allclose(xc[b, :, c], pre / (1 + np.exp(-pre)), rtol=1e-12, atol=1e-14):
                failed.append("numpy_convolve")
            if not np.array_equal(last[b, :, c], seq[-3:]):
                failed.append("last_inputs")
    return failed


def _pins(scan):
    """Run the pins against ``scan``; return the names of those that fail."""
    failed = []
    for case in load_golden():
        out, fs = scan(**_golden_arrays(case))
        if not (np.allclose(out.ravel(), case["out"], rtol=1e-12, atol=1e-14)
                and np.allclose(fs.ravel(), case["final_state"], rtol=1e-12, atol=1e-14)):
            failed.append("golden:" + case["name"])
    rng = np.random.default_rng(21)
    for mode, dims in (("diag", (1, 9, 2, 1, 3, 1)), ("ssd", (1, 8, 4, 2, 2, 2))):
        arr = _rand_problem(rng, mode, *dims)
        out, _ = scan(**arr)
        if not np.allclose(out, _bruteforce(arr, mode), rtol=1e-10, atol=1e-12):
            failed.append("bruteforce:" + mode)
    # closed-form impulse response of the time-invariant case
    T = 10
    delta = math.log1p(math.exp(0.3))
    x = np.zeros((1, T, 1))
    x[0, 0, 0] = 1.0
    out, _ = scan(x=x, dt=np.full((1, T, 1), 0.3), A=np.array([[-0.5]]),
                  B=np.full((1, T, 1, 1), 0.9), C=np.full((1, T, 1, 1), 1.2), D=np.array([0.4]))
    ref = 1.2 * delta * 0.9 * np.exp(-0.5 * delta) ** np.arange(T)
    ref[0] += 0.4
    if not np.allclose(out[0, :, 0], ref, rtol=1e-12, atol=1e-14):
        failed.append("closed_form")
    # split / resume through the initial state
    arr = _rand_problem(rng, "diag", 1, 12, 2, 1, 3, 1)
    y, _ = scan(**arr)
    cut = {k: (v[:, :5] if k in ("x", "dt", "B", "C", "z") and v is not None else v)
           for k, v in arr.items()}
    rest = {k: (v[:, 5:] if k in ("x", "dt", "B", "C", "z") and v is not None else v)
            for k, v in arr.items()}
    _, s1 = scan(**cut)
    y2, _ = scan(**rest, initial_state=s1)
    if not np.allclose(y2, y[:, 5:], rtol=1e-12, atol=1e-13):
        failed.append("split_resume")
    return failed


def _build_variant(tmp_path, name, old, new):
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    path_c = tmp_path / f"{name}.c"
    path_c.write_text(mutated, encoding="utf-8")
    path_so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(path_so), str(path_c), "-lm"], check=True)
    return oracle.OracleLib(str(path_so))


def test_unmutated_copy_passes(tmp_path):
    lib = _build_variant(tmp_path, "identity", "oracle_softplus", "oracle_softplus")
    assert _pins(lib.scan) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _build_variant(tmp_path, name, old, new)
    assert _pins(lib.scan), f"mutant {name} passed every pin"


def test_unmutated_conv_passes(tmp_path):
    lib = _build_variant(tmp_path, "identity_conv", "oracle_silu", "oracle_silu")
    assert _conv_pins(lib.conv_silu) == []


@pytest.mark.parametrize("name", sorted(CONV_MUTANTS))
def test_conv_mutant_is_caught(tmp_path, name):
    old, new = CONV_MUTANTS[name]
    lib = _build_variant(tmp_path, name, old, new)
    assert _conv_pins(lib.conv_silu), f"mutant {name} passed every pin"


def test_unmutated_backward_passes(tmp_path):
    lib = _build_variant(tmp_path, "identity_bwd", "oracle_silu", "oracle_silu")
    assert _bwd_pins(lib) == []


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_backward_mutant_is_caught(tmp_path, name):
    old, new = BWD_MUTANTS[name]
    lib = _build_variant(tmp_path, name, old, new)
    assert _bwd_pins(lib), f"mutant {name} passed every pin"
