"""Pins for the fp64 oracle against facts fixed outside the oracle itself.

Each check is chosen so that a plausible mistake in the oracle (a dropped term,
a wrong sign or index, a transposed operand, output read before the update,
the wrong discretisation) fails at least one of them:

* hand-worked golden values (tests/golden/hand_worked.txt)
* the materialised lower-triangular semiseparable matrix, y = (L o M) x
  ("Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里", section 第二步),
  built from explicit products of per-step decays on tiny inputs
* closed-form impulse and step responses of the time-invariant special case
  ("状态空间模型与 Mamba：不用注意力读取长序列的方法", section 工作原理: with fixed
  parameters the recurrence is a convolution)
* A = 0 reduces to causally masked linear attention tril(C B^T) (Delta x)
  ("引言：Attention的天花板" article, section Mamba2的改进: SSM as a special
  linear attention)
* invariants: Delta = 0, causality, linearity, split/resume, chunk-size
  invariance, SSD == diagonal mode with tied A, and the direction of the
  Delta effect ("Mamba-2 ..." explainer, section 第一步: large Delta updates
  the state quickly, small Delta keeps it).
* the causal depthwise convolution + SiLU ahead of the scan ("论文解读：Mamba —
  线性时间的序列建模革命", section 五 Mamba块架构): numpy's own convolution routine
  on every channel, the identity and pure-delay kernels, and resuming from the
  previous call's last inputs.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.txt")


def _softplus_ref(v):
    # ln(1 + e^v) through numpy's log-add-exp routine: ln(e^0 + e^v).
    return np.logaddexp(0.0, v)


def _silu_ref(z):
    return z * (0.5 * (1.0 + np.tanh(0.5 * z)))  # sigmoid via tanh identity


def load_golden():
    cases = []
    env = {"ln2": math.log(2.0), "ln3": math.log(3.0), "__builtins__": {}}
    cur = None
    with open(GOLDEN, encoding="utf-8") as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case "):
                _, name, mode, b, T, H, P, N, G = line.split()
                cur = dict(name=name, mode=mode, dims=tuple(int(v) for v in (b, T, H, P, N, G)))
                cases.append(cur)
                continue
            key, vals = line.split(":", 1)
            cur[key.strip()] = np.array([eval(tok, env) for tok in vals.split()], dtype=np.float64)
    return cases


def _golden_arrays(case):
    b, T, H, P, N, G = case["dims"]
    diag = case["mode"] == "diag"
    xs = (b, T, H) if diag else (b, T, H, P)
    arr = dict(
        x=case["x"].reshape(xs), dt=case["dt"].reshape(b, T, H),
        A=case["A"].reshape((H, N) if diag else (H,)),
        B=case["B"].reshape(b, T, G, N), C=case["C"].reshape(b, T, G, N),
        D=case.get("D"), z=None if "z" not in case else case["z"].reshape(xs),
        dt_bias=case.get("dt_bias"),
    )
    return arr


@pytest.mark.parametrize("case", load_golden(), ids=lambda c: c["name"])
def test_golden_hand_worked(case):
    arr = _golden_arrays(case)
    out, fs = oracle.scan(**arr)
    np.testing.assert_allclose(out.ravel(), case["out"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(fs.ravel(), case["final_state"], rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------------------
# tiny random problems


def _rand_problem(rng, mode, b, T, H, P, N, G, gate=True, bias=True, skip=True):
    diag = mode == "diag"
    xs = (b, T, H) if diag else (b, T, H, P)
    return dict(
        x=rng.standard_normal(xs), dt=0.5 * rng.standard_normal((b, T, H)) - 1.0,
        A=(-rng.uniform(0.2, 2.0, (H, N)) if diag else -rng.uniform(0.2, 2.0, (H,))),
        B=rng.standard_normal((b, T, G, N)), C=rng.standard_normal((b, T, G, N)),
        D=rng.normal(1.0, 0.3, (H,)) if skip else None,
        z=rng.standard_normal(xs) if gate else None,
        dt_bias=rng.uniform(-1.0, 0.5, (H,)) if bias else None,
    )


def _bruteforce(arr, mode):
    """Materialise M per channel from explicit decay products; y = M x + D x, gated."""
    x, dt, A, B, C = arr["x"], arr["dt"], arr["A"], arr["B"], arr["C"]
    diag = mode == "diag"
    if diag:
        b, T, H = x.shape
        P = 1
        x4 = x[..., None]
    else:
        b, T, H, P = x.shape
        x4 = x
    G, N = B.shape[2], B.shape[3]
    out = np.zeros_like(x4)
    for bi in range(b):
        for h in range(H):
            g = h // (H // G)
            v = dt[bi, :, h] + (arr["dt_bias"][h] if arr["dt_bias"] is not None else 0.0)
            delta = _softplus_ref(v)
            an = A[h] if diag else np.full(N, A[h])
            M = np.zeros((T, T))
            for j in range(T):
                for i in range(j + 1):
                    prod = np.ones(N)
                    for k in range(i + 1, j + 1):
                        prod = prod * np.exp(delta[k] * an)
                    M[j, i] = np.sum(C[bi, j, g] * prod * delta[i] * B[bi, i, g])
            for p in range(P):
                y = M @ x4[bi, :, h, p]
                if arr["D"] is not None:
                    y = y + arr["D"][h] * x4[bi, :, h, p]
                if arr["z"] is not None:
                    zz = arr["z"][bi, :, h] if diag else arr["z"][bi, :, h, p]
                    y = y * _silu_ref(zz)
                out[bi, :, h, p] = y
    return out[..., 0] if diag else out


@pytest.mark.parametrize("mode,dims", [
    ("diag", (2, 13, 3, 1, 4, 1)),
    ("diag", (1, 24, 4, 1, 3, 2)),
    ("ssd", (2, 11, 4, 3, 2, 2)),
    ("ssd", (1, 20, 2, 2, 4, 1)),
])
def test_bruteforce_semiseparable(mode, dims):
    rng = np.random.default_rng(11)
    arr = _rand_problem(rng, mode, *dims)
    out, _ = oracle.scan(**arr)
    ref = _bruteforce(arr, mode)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("mode", ["diag", "ssd"])
def test_closed_form_lti(mode):
    """Constant Delta, A, B, C: impulse and step responses in closed form."""
    T, N = 40, 3
    H, P = (1, 1) if mode == "diag" else (1, 2)
    A_n = np.array([-0.3, -1.1, -2.5]) if mode == "diag" else np.full(N, -0.7)
    Bv = np.array([0.8, -1.3, 0.4])
    Cv = np.array([1.5, 0.6, -0.9])
    dtv, Dv = 0.25, 0.7
    delta = math.log1p(math.exp(dtv))
    a = np.exp(delta * A_n)
    t = np.arange(T)
    for kind in ("impulse", "step"):
        xs = (1, T, H) if mode == "diag" else (1, T, H, P)
        x = np.zeros(xs)
        if kind == "impulse":
            x[0, 0] = 1.0
        else:
            x[:] = 1.0
        arr = dict(x=x, dt=np.full((1, T, H), dtv),
                   A=A_n.reshape(1, N) if mode == "diag" else np.array([A_n[0]]),
                   B=np.broadcast_to(Bv, (1, T, 1, N)).copy(),
                   C=np.broadcast_to(Cv, (1, T, 1, N)).copy(), D=np.array([Dv]))
        out, fs = oracle.scan(**arr)
        w = Cv * delta * Bv
        if kind == "impulse":
            ref = (w[None, :] * a[None, :] ** t[:, None]).sum(1) + Dv * (t == 0)
            ref_fs = delta * Bv * a ** (T - 1)
        else:
            ref = (w[None, :] * (1 - a[None, :] ** (t[:, None] + 1)) / (1 - a[None, :])).sum(1) + Dv
            ref_fs = delta * Bv * (1 - a ** T) / (1 - a)
        y = out.reshape(T, -1)
        for p in range(y.shape[1]):
            np.testing.assert_allclose(y[:, p], ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(fs.reshape(-1, N), np.broadcast_to(ref_fs, (fs.size // N, N)),
                                   rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("mode", ["diag", "ssd"])
def test_A_zero_is_masked_linear_attention(mode):
    rng = np.random.default_rng(5)
    b, T, H, P, N, G = (2, 17, 3, 1, 4, 1) if mode == "diag" else (2, 17, 2, 3, 4, 1)
    arr = _rand_problem(rng, mode, b, T, H, P, N, G, gate=False, skip=False)
    arr["A"] = np.zeros_like(arr["A"])
    out, _ = oracle.scan(**arr)
    for bi in range(b):
        for h in range(H):
            delta = _softplus_ref(arr["dt"][bi, :, h] + arr["dt_bias"][h])
            S = np.tril(arr["C"][bi, :, 0] @ arr["B"][bi, :, 0].T)  # (T, T)
            xh = arr["x"][bi, :, h][:, None] if mode == "diag" else arr["x"][bi, :, h]
            ref = S @ (delta[:, None] * xh)
            got = out[bi, :, h][:, None] if mode == "diag" else out[bi, :, h]
            np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode", ["diag", "ssd"])
def test_delta_zero(mode):
    rng = np.random.default_rng(6)
    dims = (2, 19, 3, 1, 4, 1) if mode == "diag" else (1, 19, 2, 3, 4, 1)
    arr = _rand_problem(rng, mode, *dims, bias=False)
    arr["dt"][:] = -1e4  # softplus underflows to exactly zero
    out, fs = oracle.scan(**arr)
    H = dims[2]
    Dh = arr["D"].reshape((1, 1, H) if mode == "diag" else (1, 1, H, 1))
    ref = Dh * arr["x"] * _silu_ref(arr["z"])
    np.testing.assert_allclose(out, ref, rtol=1e-14, atol=0)
    assert np.all(fs == 0.0)


@pytest.mark.parametrize("mode", ["diag", "ssd"])
def test_causality(mode):
    rng = np.random.default_rng(7)
    dims = (1, 30, 3, 1, 4, 1) if mode == "diag" else (1, 30, 2, 2, 4, 1)
    arr = _rand_problem(rng, mode, *dims)
    out0, _ = oracle.scan(**arr)
    for t0 in (0, 11, 29):
        pert = {k: (None if v is None else np.array(v, copy=True)) for k, v in arr.items()}
        pert["x"][:, t0] += 3.0
        pert["B"][:, t0] -= 1.0
        pert["dt"][:, t0] += 0.5
        out1, _ = oracle.scan(**pert)
        assert np.array_equal(out0[:, :t0], out1[:, :t0])
        assert not np.allclose(out0[:, t0:], out1[:, t0:])


@pytest.mark.parametrize("mode", ["diag", "ssd"])
def test_linearity_in_x(mode):
    rng = np.random.default_rng(8)
    dims = (2, 25, 3, 1, 4, 1) if mode == "diag" else (1, 25, 2, 3, 4, 1)
    arr = _rand_problem(rng, mode, *dims, gate=False)
    x2 = rng.standard_normal(arr["x"].shape)
    y1, s1 = oracle.scan(**arr)
    y2, s2 = oracle.scan(**{**arr, "x": x2})
    y3, s3 = oracle.scan(**{**arr, "x": 2.5 * arr["x"] - 0.75 * x2})
    np.testing.assert_allclose(y3, 2.5 * y1 - 0.75 * y2, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(s3, 2.5 * s1 - 0.75 * s2, rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("mode", ["diag", "ssd"])
def test_split_resume(mode):
    rng = np.random.default_rng(9)
    dims = (2, 40, 3, 1, 5, 1) if mode == "diag" else (1, 40, 2, 3, 5, 1)
    arr = _rand_problem(rng, mode, *dims)
    y, fs = oracle.scan(**arr)
    T1 = 17
    head = {k: (v[:, :T1] if k in ("x", "dt", "B", "C", "z") and v is not None else v)
            for k, v in arr.items()}
    tail = {k: (v[:, T1:] if k in ("x", "dt", "B", "C", "z") and v is not None else v)
            for k, v in arr.items()}
    y1, fs1 = oracle.scan(**head)
    y2, fs2 = oracle.scan(**tail, initial_state=fs1)
    np.testing.assert_allclose(np.concatenate([y1, y2], axis=1), y, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(fs2, fs, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("mode", ["diag", "ssd"])
@pytest.mark.parametrize("Q", [1, 7, 64, 256])
def test_chunked_equals_sequential(mode, Q):
    rng = np.random.default_rng(10)
    dims = (2, 300, 3, 1, 4, 1) if mode == "diag" else (1, 300, 2, 2, 3, 1)
    arr = _rand_problem(rng, mode, *dims)
    y, fs = oracle.scan(**arr)
    yc, fsc = oracle.scan(**arr, chunk=Q)
    assert oracle.max_rel_error(yc, y) < 1e-10
    assert oracle.max_rel_error(fsc, fs) < 1e-10


def test_ssd_equals_diag_with_tied_A():
    rng = np.random.default_rng(12)
    b, T, H, P, N = 2, 33, 3, 4, 5
    arr = _rand_problem(rng, "ssd", b, T, H, P, N, 1)
    y, fs = oracle.scan(**arr)
    Dc = H * P
    diag = dict(
        x=arr["x"].reshape(b, T, Dc), dt=np.repeat(arr["dt"], P, axis=2),
        A=np.repeat(arr["A"], P)[:, None] * np.ones((1, N)),
        B=arr["B"], C=arr["C"], D=np.repeat(arr["D"], P), z=arr["z"].reshape(b, T, Dc),
        dt_bias=np.repeat(arr["dt_bias"], P),
    )
    yd, fsd = oracle.scan(**diag)
    np.testing.assert_allclose(yd.reshape(y.shape), y, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(fsd.reshape(fs.shape), fs, rtol=1e-13, atol=1e-14)


def test_larger_delta_updates_state_faster():
    """Constant input x = 1, B = C = 1, A = -1: the state's progress toward its
    steady value after t steps is 1 - exp(-Delta (t + 1)), which grows with Delta;
    an impulse decays as exp(-Delta t), faster for larger Delta."""
    T = 12
    prog, decay = [], []
    for dtv in (-3.0, -1.0, 0.0, 1.5):
        delta = _softplus_ref(dtv)
        base = dict(dt=np.full((1, T, 1), dtv), A=np.array([[-1.0]]),
                    B=np.ones((1, T, 1, 1)), C=np.ones((1, T, 1, 1)))
        y, _ = oracle.scan(x=np.ones((1, T, 1)), **base)
        steady = delta / (1.0 - math.exp(-delta))
        prog.append(y[0, 5, 0] / steady)
        imp = np.zeros((1, T, 1))
        imp[0, 0, 0] = 1.0
        yi, _ = oracle.scan(x=imp, **base)
        decay.append(yi[0, 6, 0] / yi[0, 0, 0])
        np.testing.assert_allclose(prog[-1], 1.0 - math.exp(-6 * delta), rtol=1e-12)
    assert all(p1 < p2 for p1, p2 in zip(prog, prog[1:]))
    assert all(d1 > d2 for d1, d2 in zip(decay, decay[1:]))


@pytest.mark.parametrize("v", [-60.0, -20.0, -2.0, 0.0, 3.0, 40.0])
def test_softplus_has_no_cutoff(v):
    """With A = 0, B = C = x = 1 and one step, y equals Delta = ln(1 + e^v) exactly
    across the whole range (no threshold where softplus is replaced by v or 0)."""
    arr = dict(x=np.ones((1, 1, 1)), dt=np.full((1, 1, 1), v), A=np.zeros((1, 1)),
               B=np.ones((1, 1, 1, 1)), C=np.ones((1, 1, 1, 1)))
    y, _ = oracle.scan(**arr)
    np.testing.assert_allclose(y[0, 0, 0], _softplus_ref(v), rtol=1e-15, atol=0)


def test_select_matches_full():
    rng = np.random.default_rng(13)
    arr = _rand_problem(rng, "ssd", 2, 21, 3, 4, 3, 1)
    y, fs = oracle.scan(**arr)
    sel = [0, 5, 13, 23]
    ys, fss = oracle.scan(**arr, select=sel)
    flat_y = y.transpose(0, 2, 3, 1).reshape(-1, 21)
    flat_ys = ys.transpose(0, 2, 3, 1).reshape(-1, 21)
    assert np.array_equal(flat_y[sel], flat_ys[sel])
    assert np.array_equal(fs.reshape(-1, 3)[sel], fss.reshape(-1, 3)[sel])
    others = np.setdiff1d(np.arange(flat_y.shape[0]), sel)
    assert np.all(np.isnan(flat_ys[others]))


def test_empty_sequence():
    arr = dict(x=np.zeros((2, 0, 3)), dt=np.zeros((2, 0, 3)), A=-np.ones((3, 4)),
               B=np.zeros((2, 0, 1, 4)), C=np.zeros((2, 0, 1, 4)))
    y, fs = oracle.scan(**arr)
    assert y.shape == (2, 0, 3)
    assert np.all(fs == 0.0)


def test_max_rel_error_definition():
    ref = np.array([1.0, -2.0, 1e-9, 0.0])
    y = ref + np.array([1e-3, 0.0, 2e-6, 0.0])
    # floor = 1e-2 * 2 = 2e-2 for the tiny entries
    assert abs(oracle.max_rel_error(y, ref) - 1e-3) < 1e-15
    y2 = ref + np.array([0.0, 0.0, 2e-2, 0.0])
    assert abs(oracle.max_rel_error(y2, ref) - 1.0) < 1e-12


def _fp32_recurrence(arr, diag):
    """The recurrence evaluated step by step in float32 with numpy's exp/log1p."""
    f = np.float32
    x = arr["x"].astype(f)
    x = x[..., None] if diag else x
    b, T, H, P = x.shape
    B, C = arr["B"].astype(f), arr["C"].astype(f)
    G, N = B.shape[2], B.shape[3]
    g = np.arange(H) // (H // G)
    A = arr["A"].astype(f)
    h = np.zeros((b, H, P, N), f)
    y = np.zeros((b, T, H, P), f)
    for t in range(T):
        v = arr["dt"][:, t].astype(f) + (arr["dt_bias"].astype(f) if arr["dt_bias"] is not None else f(0))
        de = (np.maximum(v, 0) + np.log1p(np.exp(-np.abs(v)))).astype(f)
        a = np.exp(de[:, :, None, None] * (A[None, :, None, :] if diag else A[None, :, None, None])).astype(f)
        h = (a * h + (de[:, :, None] * x[:, t])[..., None] * B[:, t][:, g][:, :, None, :]).astype(f)
        y[:, t] = np.einsum("bhpn,bhn->bhp", h, C[:, t][:, g]).astype(f)
    return (y[..., 0] if diag else y), h.reshape((b, H, N) if diag else (b, H, P, N))


def test_error_report_definitions():
    """The informational measures, on values worked by hand."""
    ref = np.array([10.0, -0.5, 0.0, 0.02])
    y = np.array([10.01, -0.5, 0.001, 0.021])
    r = oracle.error_report(y, ref)
    # gated: floors at 0.1 (1% of 10): errors 0.01/10, 0, 0.001/0.1, 0.001/0.1
    assert abs(r["gated"] - 0.01) < 1e-12
    # floor 1e-3 of 10 = 0.01: 0.001/0.01 (the zero), 0.001/0.02
    assert abs(r["floor_1e-3"] - 0.1) < 1e-12
    # unfloored over nonzero references: 0.001/0.02 = 0.05 (the zero is left out)
    assert abs(r["unfloored"] - 0.05) < 1e-12
    # normwise: max error 0.01 over max |ref| 10
    assert abs(r["normwise"] - 0.001) < 1e-12


@pytest.mark.parametrize("mode", ["diag", "ssd"])
def test_error_measure_leaves_margin_for_exact_fp32(mode):
    """The fp32 bound (1e-4) must be met with margin by an exactly rounded fp32
    evaluation; the floor of the error measure is chosen so that it is (scores
    about 1e-5), while a floor of 1e-3 puts exact fp32 at the bound itself."""
    rng = np.random.default_rng(14)
    dims = (2, 200, 8, 1, 16, 1) if mode == "diag" else (1, 260, 2, 32, 16, 2)
    arr = _rand_problem(rng, mode, *dims, gate=False, skip=False)
    y32, h32 = _fp32_recurrence(arr, mode == "diag")
    y, h = oracle.scan(**arr)
    assert oracle.max_rel_error(y32, y) < 2e-5
    assert oracle.max_rel_error(h32, h) < 2e-5


# ---------------------------------------------------------------- convolution ahead of the scan

def _conv_problem(rng, b, T, ch, K):
    return (rng.standard_normal((b, T, ch)), rng.standard_normal((ch, K)),
            rng.standard_normal(ch), rng.standard_normal((b, K - 1, ch)))


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_conv_matches_numpy_convolution(K):
    """Every channel against numpy.convolve: the causal correlation
    sum_k w[k] x[t-K+1+k] is the full convolution with the reversed kernel, cut to
    the first T outputs; the previous call's inputs are prepended."""
    rng = np.random.default_rng(40 + K)
    x, w, bias, x_prev = _conv_problem(rng, 2, 17, 5, K)
    for prev in (None, x_prev):
        xc, x_last = oracle.conv_silu(x, w, bias, prev)
        for b in range(2):
            for c in range(5):
                head = np.zeros(K - 1) if prev is None else prev[b, :, c]
                seq = np.concatenate([head, x[b, :, c]])
                pre = np.convolve(seq, w[c, ::-1])[K - 1:K - 1 + 17] + bias[c]
                assert np.allclose(xc[b, :, c], _silu_ref(pre), rtol=1e-13, atol=1e-14)
                assert np.array_equal(x_last[b, :, c], seq[len(seq) - (K - 1):] if K > 1
                                      else np.zeros(0))


def test_conv_identity_and_delay_kernels():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((1, 9, 4))
    ident = np.zeros((4, 4))
    ident[:, 3] = 1.0
    xc, _ = oracle.conv_silu(x, ident)
    assert np.allclose(xc, _silu_ref(x), rtol=1e-14, atol=0)
    delay = np.zeros((4, 4))
    delay[:, 0] = 1.0
    xc, _ = oracle.conv_silu(x, delay)
    assert np.all(xc[:, :3] == 0.0)
    assert np.allclose(xc[:, 3:], _silu_ref(x[:, :-3]), rtol=1e-14, atol=0)


def test_conv_resume_from_last_inputs():
    """Two calls, the second fed the first one's last inputs, equal one call -- also
    when the first piece is shorter than the kernel."""
    rng = np.random.default_rng(8)
    x, w, bias, x_prev = _conv_problem(rng, 2, 12, 3, 4)
    whole, last = oracle.conv_silu(x, w, bias, x_prev)
    for cut in (1, 2, 7):
        a, la = oracle.conv_silu(x[:, :cut], w, bias, x_prev)
        bb, lb = oracle.conv_silu(x[:, cut:], w, bias, la)
        assert np.array_equal(np.concatenate([a, bb], axis=1), whole)
        assert np.array_equal(lb, last)


def test_scan_conv_equals_scan_of_convolved_input():
    """The skip term reads the convolved input too: with Delta = 0 the output is
    D * x' * SiLU(z)."""
    rng = np.random.default_rng(12)
    arr = _rand_problem(rng, "diag", 1, 10, 3, 1, 2, 1)
    w = rng.standard_normal((3, 4))
    cb = rng.standard_normal(3)
    arr["dt"] = np.full_like(arr["dt"], -1e4)
    arr["dt_bias"] = None
    out, fs, _ = oracle.scan_conv(**arr, conv_w=w, conv_b=cb)
    xc, _ = oracle.conv_silu(arr["x"], w, cb)
    assert np.allclose(out, arr["D"] * xc * _silu_ref(arr["z"]), rtol=1e-14, atol=1e-15)
    assert np.all(fs == 0.0)
