"""Pins of the oracle's complex diagonal scan (the rotating state update read for Mamba-3),
each independent of the oracle's own code, and planted mistakes that the pins must catch.

The pages describe Mamba-3's state update only in words: an input-dependent rotation,
read as underdamped oscillation ("状态空间模型与 Mamba：不用注意力读取长序列的方法", the
Mamba-3 paragraph) and a complex-valued state update ("基础知识：Mamba 与混合 SSM 架构",
section 6).  What pins the reading:
  * with every imaginary part zero it is exactly the real diagonal scan (the oracle's
    pinned real recurrence, a separate code path);
  * the materialised semiseparable matrix, built here from explicit products of the
    per-step complex decays;
  * the closed-form impulse and step responses of a damped oscillator (constant Delta,
    A = -alpha + i omega, B = C = 1): y_t = Delta e^{-alpha Delta t} cos(omega Delta t);
  * pure rotation (Re A = 0) conserves the state's magnitude and is periodic when
    omega Delta = 2 pi / k;
  * Delta = 0 leaves only the skip term; causality; split / resume through the state.
"""
import math
import os
import subprocess

import numpy as np
import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")


def softplus(v):
    return max(v, 0.0) + math.log1p(math.exp(-abs(v)))


def rand_problem(rng, b, T, D, N, G=1, gate=True, skip=True, bias=True):
    A = np.stack([-rng.uniform(0.1, 1.5, (D, N)), rng.uniform(-3.0, 3.0, (D, N))], axis=-1)
    bshape = (b, T, N, 2) if G == 1 else (b, T, G, N, 2)
    return dict(
        x=rng.standard_normal((b, T, D)), dt=rng.standard_normal((b, T, D)) * 0.5 - 1.0, A=A,
        B=rng.standard_normal(bshape), C=rng.standard_normal(bshape),
        D=rng.standard_normal(D) if skip else None,
        z=rng.standard_normal((b, T, D)) if gate else None,
        dt_bias=rng.uniform(-1.0, 0.5, D) if bias else None)


def bruteforce(p):
    """y = (M x + D x) SiLU(z) with M[j, i] = Re sum_n C_j[n] (prod_{k=i+1..j} e^{Delta_k A_n})
    Delta_i B_i[n], the products written out term by term."""
    x, dt, A = p["x"], p["dt"], p["A"]
    b, T, D = x.shape
    N = A.shape[1]
    G = 1 if p["B"].ndim == 4 else p["B"].shape[2]
    Bc = (p["B"][..., 0] + 1j * p["B"][..., 1]).reshape(b, T, G, N)
    Cc = (p["C"][..., 0] + 1j * p["C"][..., 1]).reshape(b, T, G, N)
    Ac = A[..., 0] + 1j * A[..., 1]
    y = np.zeros((b, T, D))
    for bb in range(b):
        for c in range(D):
            g = c // (D // G)
            bias = p["dt_bias"][c] if p["dt_bias"] is not None else 0.0
            delta = [softplus(dt[bb, t, c] + bias) for t in range(T)]
            for j in range(T):
                acc = 0.0
                for i in range(j + 1):
                    m = 0.0 + 0.0j
                    for n in range(N):
                        prod = 1.0 + 0.0j
                        for k in range(i + 1, j + 1):
                            prod *= np.exp(delta[k] * Ac[c, n])
                        m += Cc[bb, j, g, n] * prod * delta[i] * Bc[bb, i, g, n]
                    acc += m.real * x[bb, i, c]
                if p["D"] is not None:
                    acc += p["D"][c] * x[bb, j, c]
                if p["z"] is not None:
                    zz = p["z"][bb, j, c]
                    acc *= zz / (1.0 + math.exp(-zz))
                y[bb, j, c] = acc
    return y


def _cut(p, a, b_):
    return {k: (v[:, a:b_] if k in ("x", "dt", "B", "C", "z") and v is not None else v)
            for k, v in p.items()}


def complex_pins(scan_complex):
    """Run every pin against ``scan_complex``; return the names of those that fail."""
    failed = []
    rng = np.random.default_rng(5)

    # 1. no imaginary parts: the real diagonal scan
    p = rand_problem(rng, 2, 12, 3, 4, G=1)
    for k in ("A", "B", "C"):
        p[k][..., 1] = 0.0
    out, fs = scan_complex(**p)
    ref, ref_fs = oracle.scan(p["x"], p["dt"], p["A"][..., 0], p["B"][..., 0], p["C"][..., 0],
                              p["D"], p["z"], p["dt_bias"])
    if not (np.allclose(out, ref, rtol=1e-12, atol=1e-13)
            and np.allclose(fs[..., 0], ref_fs, rtol=1e-12, atol=1e-13)
            and np.all(fs[..., 1] == 0.0)):
        failed.append("real_reduction")

    # 2. materialised semiseparable matrix, with groups
    for G in (1, 2):
        p = rand_problem(rng, 1, 7, 2, 3, G=G)
        out, _ = scan_complex(**p)
        if not np.allclose(out, bruteforce(p), rtol=1e-10, atol=1e-12):
            failed.append(f"bruteforce_G{G}")

    # 3. damped oscillator: impulse and step responses in closed form
    T, alpha, omega, dtv, Dv = 24, 0.3, 1.7, 0.2, 0.25
    delta = softplus(dtv)
    base = dict(dt=np.full((1, T, 1), dtv), A=np.array([[[-alpha, omega]]]),
                B=np.tile(np.array([1.0, 0.0]), (1, T, 1, 1)),
                C=np.tile(np.array([1.0, 0.0]), (1, T, 1, 1)), D=np.array([Dv]))
    t = np.arange(T)
    x = np.zeros((1, T, 1))
    x[0, 0, 0] = 1.0
    out, fs = scan_complex(x=x, **base)
    ref = delta * np.exp(-alpha * delta * t) * np.cos(omega * delta * t)
    ref[0] += Dv
    h_last = delta * np.exp((-alpha + 1j * omega) * delta * (T - 1))
    if not (np.allclose(out[0, :, 0], ref, rtol=1e-12, atol=1e-14)
            and np.allclose(fs[0, 0, 0], [h_last.real, h_last.imag], rtol=1e-12, atol=1e-14)):
        failed.append("impulse_oscillation")
    q = np.exp((-alpha + 1j * omega) * delta)
    out, _ = scan_complex(x=np.ones((1, T, 1)), **base)
    ref = (delta * (1 - q ** (t + 1)) / (1 - q)).real + Dv
    if not np.allclose(out[0, :, 0], ref, rtol=1e-12, atol=1e-13):
        failed.append("step_oscillation")

    # 4. pure rotation: |h| conserved after an impulse; period k when omega Delta = 2 pi / k
    k = 7
    rot = dict(base, A=np.array([[[0.0, 2 * math.pi / (k * delta)]]]), D=None)
    out, fs = scan_complex(x=x, **rot)
    if not (abs(np.hypot(*fs[0, 0, 0]) - delta) < 1e-12
            and np.allclose(out[0, k:2 * k, 0], out[0, :k, 0], rtol=1e-10, atol=1e-12)):
        failed.append("pure_rotation")

    # 5. Delta = 0: only the gated skip term, state zero
    p = rand_problem(rng, 1, 6, 2, 3)
    p["dt"] = np.full_like(p["dt"], -1e4)
    p["dt_bias"] = None
    out, fs = scan_complex(**p)
    zz = p["z"]
    if not (np.allclose(out, p["D"] * p["x"] * zz / (1 + np.exp(-zz)), rtol=1e-14, atol=0)
            and np.all(fs == 0.0)):
        failed.append("delta_zero")

    # 6. causality and split / resume through the state
    p = rand_problem(rng, 1, 10, 2, 3)
    y, _ = scan_complex(**p)
    p2 = {kk: (v.copy() if v is not None else None) for kk, v in p.items()}
    p2["x"][:, 6] += 1.0
    y2, _ = scan_complex(**p2)
    if not (np.array_equal(y[:, :6], y2[:, :6]) and not np.allclose(y[:, 6], y2[:, 6])):
        failed.append("causality")
    _, s1 = scan_complex(**_cut(p, 0, 4))
    y3, _ = scan_complex(**_cut(p, 4, 10), initial_state=s1)
    if not np.allclose(y3, y[:, 4:], rtol=1e-12, atol=1e-13):
        failed.append("split_resume")
    return failed


def test_complex_oracle_passes_its_pins():
    assert complex_pins(oracle.scan_complex) == []


def test_complex_selection_matches_full_run():
    rng = np.random.default_rng(8)
    p = rand_problem(rng, 2, 9, 5, 3)
    y, fs = oracle.scan_complex(**p)
    sel = np.array([1, 7, 9])
    ys, fss = oracle.scan_complex(**p, select=sel)
    yv = y.transpose(0, 2, 1).reshape(10, 9)
    ysv = ys.transpose(0, 2, 1).reshape(10, 9)
    assert np.array_equal(ysv[sel], yv[sel])
    assert np.array_equal(fss.reshape(10, 3, 2)[sel], fs.reshape(10, 3, 2)[sel])
    assert np.all(np.isnan(np.delete(ysv, sel, axis=0)))


# Planted mistakes in copies of the complex oracle; each must fail a pin.
MUTANTS = {
    "conjugate_C": ("acc += cn * state[n];", "acc += conj(cn) * state[n];"),
    "rotation_sign": ("state[n] = cexp(delta * an) * state[n] + delta * bn * xv;",
                      "state[n] = cexp(delta * conj(an)) * state[n] + delta * bn * xv;"),
    "drop_imag_B": ("const double complex bn = Bt[2 * n] + I * Bt[2 * n + 1];",
                    "const double complex bn = Bt[2 * n];"),
    "read_imag_part": ("double y = creal(acc);", "double y = cimag(acc);"),
    "decay_without_rotation": ("state[n] = cexp(delta * an) * state[n] + delta * bn * xv;",
                               "state[n] = exp(delta * creal(an)) * state[n] + delta * bn * xv;"),
    "im_re_swapped_A": ("const double complex an = A[2 * (c * N + n)] + I * A[2 * (c * N + n) + 1];",
                        "const double complex an = A[2 * (c * N + n) + 1] + I * A[2 * (c * N + n)];"),
    "output_before_update": (
        "state[n] = cexp(delta * an) * state[n] + delta * bn * xv;\n            acc += cn * state[n];",
        "acc += cn * state[n];\n            state[n] = cexp(delta * an) * state[n] + delta * bn * xv;"),
}


def _variant(tmp_path, name, old, new):
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation site for {name} not found"
    path_c = tmp_path / f"{name}.c"
    path_c.write_text(src.replace(old, new), encoding="utf-8")
    path_so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(path_so), str(path_c), "-lm"], check=True)
    return oracle.OracleLib(str(path_so))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_complex_mutant_is_caught(tmp_path, name):
    lib = _variant(tmp_path, name, *MUTANTS[name])
    assert complex_pins(lib.scan_complex), f"mutant {name} passed every pin"
