"""fp64 CPU oracle for the selective state-space scan (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python
binding) never does, and this package never imports the product path: the two
meet only at the seeded input generator, which holds none of the method's
arithmetic.

The arithmetic lives in ``ssm_oracle.c`` (plain C, fp64, OpenMP over independent
channels).  This module compiles it on first use and marshals numpy arrays.

What it computes (cited by page title and section):
  * "Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里", 背景问题 and
    第一步: h_t = Abar_t h_{t-1} + Bbar_t x_t, y_t = C_t h_t, Delta_t = softplus(.)
  * "引言：Attention的天花板" article, 基本原理: the D x_t skip term
  * "论文解读：Mamba — 线性时间的序列建模革命", 五 Mamba块架构: the SiLU(z) gate
with Abar = exp(Delta A), Bbar = Delta B.  ``scan(..., chunk=Q)`` evaluates the
same operator through its semiseparable block form (Mamba-2 explainer, 第二步 and
关键技术点 1) and serves to pin chunk-size invariance.  ``scan_complex`` is the
complex-valued, rotating state update read for Mamba-3 ("状态空间模型与 Mamba：不用注意力
读取长序列的方法", the Mamba-3 paragraph; "基础知识：Mamba 与混合 SSM 架构", section 6).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None

MODE_DIAG = 0
MODE_SSD = 1


def build(force: bool = False, src: str = _SRC, lib: str = _LIB) -> str:
    """Compile the oracle with gcc (fp64, no fast-math, no FMA contraction, OpenMP)."""
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src):
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-Wall", "-o", lib + ".tmp", src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(lib + ".tmp", lib)
    return lib


class OracleLib:
    """ctypes view of one compiled copy of ``ssm_oracle.c``."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        lib.oracle_scan.argtypes = [ctypes.c_int] + [i64] * 6 + [dp] * 9 + [dp, dp, ip, i64,
                                                                          ctypes.c_int]
        lib.oracle_scan.restype = ctypes.c_int
        lib.oracle_scan_chunked.argtypes = [ctypes.c_int] + [i64] * 7 + [dp] * 9 + [
            dp, dp, ip, i64, ctypes.c_int]
        lib.oracle_scan_chunked.restype = ctypes.c_int
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_scan_bwd.argtypes = [ctypes.c_int] + [i64] * 6 + [dp] * 20
        lib.oracle_scan_bwd.restype = ctypes.c_int
        lib.oracle_conv_silu.argtypes = [i64] * 4 + [dp] * 6
        lib.oracle_conv_silu.restype = ctypes.c_int
        lib.oracle_scan_complex.argtypes = [i64] * 5 + [dp] * 11 + [ip, i64, ctypes.c_int]
        lib.oracle_scan_complex.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def scan(self, *args, **kw):
        return _scan(self.lib, *args, **kw)

    def conv_silu(self, *args, **kw):
        return _conv_silu(self.lib, *args, **kw)

    def scan_bwd(self, *args, **kw):
        return _scan_bwd(self.lib, *args, **kw)

    def scan_complex(self, *args, **kw):
        return _scan_complex(self.lib, *args, **kw)


def _load():
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
    return _default.lib


def conv_silu(*args, **kw):
    """Run the oracle's convolution + SiLU; see ``_conv_silu``."""
    return _conv_silu(_load(), *args, **kw)


def _conv_silu(lib, x, w, bias=None, x_prev=None):
    """Causal depthwise convolution + SiLU ahead of the scan (fp64).

    x: (b, T, H) or (b, T, H, P); w: (channels, K) with channels = H*P; bias: (channels,);
    x_prev: (b, K-1, channels) inputs before t = 0 (None: zeros).
    Returns ``(x_conv, x_last)``: x_conv shaped like x, x_last (b, K-1, channels) the
    K-1 inputs that precede the end of the sequence.
    """
    x, w, bias, x_prev = (_f64(v) for v in (x, w, bias, x_prev))
    b, T = x.shape[0], x.shape[1]
    ch = int(np.prod(x.shape[2:]))
    if w.ndim != 2 or w.shape[0] != ch:
        raise ValueError("conv weight must be (channels, width)")
    K = w.shape[1]
    if bias is not None and bias.shape != (ch,):
        raise ValueError("conv bias must be (channels,)")
    if x_prev is not None and x_prev.size != b * (K - 1) * ch:
        raise ValueError("x_prev must be (batch, width-1, channels)")
    xc = np.empty(x.shape, dtype=np.float64)
    x_last = np.empty((b, K - 1, ch), dtype=np.float64)
    rc = lib.oracle_conv_silu(b, T, ch, K, _ptr(x), _ptr(w), _ptr(bias), _ptr(x_prev),
                                  _ptr(xc), _ptr(x_last))
    if rc != 0:
        raise RuntimeError(f"oracle returned status {rc}")
    return xc, x_last


def scan_conv(x, dt, A, B, C, D=None, z=None, dt_bias=None, *, conv_w, conv_b=None,
              x_prev=None, **kw):
    """The scan with the convolution + SiLU ahead of it: ``conv_silu`` then ``scan`` on
    the convolved input.  Returns ``(out, final_state, x_last)``."""
    xc, x_last = conv_silu(x, conv_w, conv_b, x_prev)
    out, fs = scan(xc, dt, A, B, C, D, z, dt_bias, **kw)
    return out, fs, x_last


def scan_bwd(*args, **kw):
    """Run the oracle's backward pass; see ``_scan_bwd``."""
    return _scan_bwd(_load(), *args, **kw)


def _scan_bwd(lib, x, dt, A, B, C, D=None, z=None, dt_bias=None, initial_state=None, *, dout,
              dfinal=None):
    """Gradients of the scan (fp64, serial over channels).

    Arguments as ``scan``; ``dout`` has x's shape, ``dfinal`` the final state's.
    Returns a dict with dx, ddt, dA, dB, dC (always) and dD, dz, ddt_bias, dinit (None
    where the matching input is None).
    """
    x, dt, A, B, C = (_f64(v) for v in (x, dt, A, B, C))
    D, z, dt_bias, initial_state, dout, dfinal = (
        _f64(v) for v in (D, z, dt_bias, initial_state, dout, dfinal))
    mode, b, T, H, P, N, G = _shape(x, dt, A, B)
    Bs = B.reshape(b, T, G, N)
    out = {
        "dx": np.empty(x.shape), "ddt": np.empty(dt.shape), "dA": np.empty(A.shape),
        "dB": np.empty(Bs.shape), "dC": np.empty(Bs.shape),
        "dD": None if D is None else np.empty(D.shape),
        "dz": None if z is None else np.empty(z.shape),
        "ddt_bias": None if dt_bias is None else np.empty(dt_bias.shape),
        "dinit": np.empty((b, H, N) if mode == MODE_DIAG else (b, H, P, N)),
    }
    if dout.shape != x.shape:
        raise ValueError("dout must have x's shape")
    rc = lib.oracle_scan_bwd(mode, b, T, H, P, N, G,
                             *(_ptr(v) for v in (x, dt, A, Bs, C.reshape(Bs.shape), D, z, dt_bias,
                                                 initial_state, dout, dfinal)),
                             *(_ptr(out[k]) for k in ("dx", "ddt", "dA", "dB", "dC", "dD", "dz",
                                                      "ddt_bias", "dinit")))
    if rc != 0:
        raise RuntimeError(f"oracle returned status {rc}")
    out["dB"] = out["dB"].reshape(B.shape)
    out["dC"] = out["dC"].reshape(B.shape)
    return out


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # a torch tensor: read exactly the values it holds
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shape(x, dt, A, B):
    """Infer (mode, batch, seqlen, nheads, headdim, dstate, ngroups)."""
    if A.ndim == 2:  # DIAG: x (b, T, D), A (D, N)
        if x.ndim != 3:
            raise ValueError("diagonal mode expects x of shape (batch, seqlen, d_inner)")
        b, T, H = x.shape
        P = 1
        mode = MODE_DIAG
        if A.shape[0] != H:
            raise ValueError("A must be (d_inner, dstate)")
    elif A.ndim == 1:  # SSD: x (b, T, H, P), A (H,)
        if x.ndim != 4:
            raise ValueError("SSD mode expects x of shape (batch, seqlen, nheads, headdim)")
        b, T, H, P = x.shape
        mode = MODE_SSD
        if A.shape[0] != H:
            raise ValueError("A must be (nheads,)")
    else:
        raise ValueError("A must be 1-D (SSD) or 2-D (diagonal)")
    if B.ndim == 3:
        G, N = 1, B.shape[2]
    else:
        G, N = B.shape[2], B.shape[3]
    if mode == MODE_DIAG and A.shape[1] != N:
        raise ValueError("A's second dimension must equal dstate")
    if dt.shape[:2] != (b, T) or dt.size != b * T * H:
        raise ValueError("dt must be (batch, seqlen, nheads)")
    return mode, b, T, H, P, N, G


def scan(*args, **kw):
    """Run the oracle; see ``_scan`` for arguments.  Returns ``(out, final_state)``."""
    return _scan(_load(), *args, **kw)


def _scan(lib, x, dt, A, B, C, D=None, z=None, dt_bias=None, initial_state=None, select=None,
          chunk: int = 0, nthreads: int = 0, out=None):
    """Run the oracle; returns ``(out, final_state)`` as float64 arrays.

    Shapes: DIAG x/z (b, T, D), dt (b, T, D), A (D, N), B/C (b, T, N) or (b, T, G, N),
    D/dt_bias (D,), states (b, D, N).  SSD x/z (b, T, H, P), dt (b, T, H), A (H,),
    B/C (b, T, G, N), D/dt_bias (H,), states (b, H, P, N).

    ``select``: optional flat channel indices b*H*P + h*P + p; only those channels
    are evaluated (the others stay NaN).  ``chunk`` > 0 selects the chunked
    (semiseparable block) evaluation with that chunk length.
    """
    x, dt, A, B, C = (_f64(v) for v in (x, dt, A, B, C))
    D, z, dt_bias, initial_state = (_f64(v) for v in (D, z, dt_bias, initial_state))
    mode, b, T, H, P, N, G = _shape(x, dt, A, B)
    if C.shape != B.shape:
        raise ValueError("B and C must have the same shape")
    if z is not None and z.shape != x.shape:
        raise ValueError("z must have x's shape")
    for name, v in (("D", D), ("dt_bias", dt_bias)):
        if v is not None and v.shape != (H,):
            raise ValueError(f"{name} must have shape ({H},)")
    st_shape = (b, H, N) if mode == MODE_DIAG else (b, H, P, N)
    if initial_state is not None and initial_state.size != b * H * P * N:
        raise ValueError("initial_state has the wrong size")
    if out is None:
        out = np.full(x.shape, np.nan, dtype=np.float64)
    fs = np.full(st_shape, np.nan, dtype=np.float64)
    sel = None
    nsel = 0
    if select is not None:
        sel = np.ascontiguousarray(np.asarray(select, dtype=np.int64))
        nsel = sel.size
    selp = sel.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if sel is not None else \
        ctypes.POINTER(ctypes.c_int64)()
    common = (x, dt, A, B, C, D, z, dt_bias, initial_state)
    if chunk and chunk > 0:
        rc = lib.oracle_scan_chunked(mode, b, T, H, P, N, G, int(chunk), *(_ptr(v) for v in common),
                                     _ptr(out), _ptr(fs), selp, nsel, int(nthreads))
    else:
        rc = lib.oracle_scan(mode, b, T, H, P, N, G, *(_ptr(v) for v in common), _ptr(out),
                             _ptr(fs), selp, nsel, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle returned status {rc}")
    return out, fs


def max_rel_error(y, ref, floor_frac: float = 1e-2) -> float:
    """max_i |y_i - r_i| / max(|r_i|, floor_frac * max_j |r_j|)  (0 for empty input).

    The error measure used against the stated tolerances: elementwise relative error
    with a floor at 1% of the largest reference magnitude, so that values near zero
    (cancellation in C.h or in a state entry) do not turn the conditioning of the
    sum into the score.  With this floor an exactly rounded fp32 evaluation of the
    recurrence scores about 1e-5, ten times inside the fp32 bound of 1e-4.
    """
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    scale = np.max(np.abs(ref))
    denom = np.maximum(np.abs(ref), floor_frac * scale)
    denom = np.where(denom == 0, 1.0, denom)
    return float(np.max(np.abs(y - ref) / denom))


def error_report(y, ref) -> dict:
    """Every error measure recorded next to the gated one, for information:
    ``gated`` (the measure the tolerances apply to, floor 1e-2), ``floor_1e-3`` (the same
    with a floor of 1e-3 of the largest reference magnitude), ``unfloored``
    (max_i |y_i - r_i| / |r_i| over the nonzero r_i) and ``normwise``
    (max_i |y_i - r_i| / max_i |r_i|)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return {"gated": 0.0, "floor_1e-3": 0.0, "unfloored": 0.0, "normwise": 0.0}
    diff = np.abs(y - ref)
    nz = ref != 0
    scale = float(np.max(np.abs(ref)))
    return {"gated": max_rel_error(y, ref), "floor_1e-3": max_rel_error(y, ref, 1e-3),
            "unfloored": float(np.max(diff[nz] / np.abs(ref[nz]))) if nz.any() else 0.0,
            "normwise": float(np.max(diff) / scale) if scale > 0 else float(np.max(diff))}


def scan_complex(*args, **kw):
    """Run the oracle's complex diagonal scan; see ``_scan_complex``."""
    return _scan_complex(_load(), *args, **kw)


def _scan_complex(lib, x, dt, A, B, C, D=None, z=None, dt_bias=None, initial_state=None,
                  select=None, nthreads: int = 0):
    """Complex diagonal scan (the rotating state update read for Mamba-3), fp64.

    x, z, dt (b, T, D); A (D, N, 2); B, C (b, T, N, 2) or (b, T, G, N, 2), each complex
    number an (re, im) pair; D, dt_bias (D,); initial_state (b, D, N, 2).  Returns
    ``(out (b, T, D), final_state (b, D, N, 2))``; ``select`` as for ``scan`` with flat
    channels b*D + c (unselected channels stay NaN).
    """
    x, dt, A, B, C = (_f64(v) for v in (x, dt, A, B, C))
    D, z, dt_bias, initial_state = (_f64(v) for v in (D, z, dt_bias, initial_state))
    if x.ndim != 3 or A.ndim != 3 or A.shape[2] != 2:
        raise ValueError("complex scan expects x (b, T, D) and A (D, N, 2)")
    b, T, H = x.shape
    N = A.shape[1]
    if A.shape[0] != H:
        raise ValueError("A must be (d_inner, dstate, 2)")
    if B.ndim == 4:
        G = 1
    elif B.ndim == 5:
        G = B.shape[2]
    else:
        raise ValueError("B must be (b, T, N, 2) or (b, T, G, N, 2)")
    if B.shape[-2:] != (N, 2) or C.shape != B.shape or B.shape[:2] != (b, T):
        raise ValueError("B and C must be (b, T[, G], N, 2)")
    if dt.shape != x.shape or (z is not None and z.shape != x.shape):
        raise ValueError("dt and z must have x's shape")
    if initial_state is not None and initial_state.size != b * H * N * 2:
        raise ValueError("initial_state must be (b, D, N, 2)")
    out = np.full(x.shape, np.nan)
    fs = np.full((b, H, N, 2), np.nan)
    sel = None if select is None else np.ascontiguousarray(np.asarray(select, dtype=np.int64))
    selp = sel.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if sel is not None else \
        ctypes.POINTER(ctypes.c_int64)()
    rc = lib.oracle_scan_complex(b, T, H, N, G, *(_ptr(v) for v in (x, dt, A, B, C, D, z, dt_bias,
                                                                     initial_state, out, fs)),
                                 selp, 0 if sel is None else sel.size, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle returned status {rc}")
    return out, fs
