"""Seeded synthetic inputs for the selective-scan workloads.

This module is shared by the tests, the benchmark and the CPU oracle's callers.
It only draws random numbers and rounds them to the storage dtype; it holds none
of the scan's arithmetic (no softplus, exponentials or recurrences).

Workloads (shapes follow the Mamba block used on the pages: a ``Mamba(d_model=256,
d_state=16, d_conv=4, expand=2)`` layer on a (8, 1024, 256) input gives d_inner 512;
the larger ones are a 3B-width Mamba-1 layer and two Mamba-2/SSD layers):

  c0  diagonal A, fp32:  batch 1,  L 256,    d_inner 64,    N 16, no gate, D = 1
  c1  diagonal A, bf16:  batch 8,  L 1024,   d_inner 512,   N 16, gate, dt_bias, D
  c2  diagonal A, bf16:  batch 4,  L 8192,   d_inner 5120,  N 16, gate, dt_bias, D, final state
  c3  SSD, bf16:         batch 4,  L 8192,   64 heads x 64, N 128, chunk 256, D
  c4  SSD, bf16:         batch 1,  L 131072, 32 heads x 64, N 256, chunk 256, D, final state
  cx1 complex diagonal A (the rotating state update read for Mamba-3) at c1's shape
  cx2 complex diagonal A at c2's shape, final state

Distributions: x, z, B, C ~ N(0, 1); dt = 0.5 N(0, 1) - 2 (the kernel applies
softplus(dt + dt_bias)); dt_bias ~ U(-4, -2) per channel; D ~ N(1, 0.1) (c0: D = 1);
diagonal A[c, n] = -(n + 1); SSD A_h = -U(1, 16); complex diagonal A[c, n] =
-(n + 1) + i U(-pi, pi) (the real part as the diagonal workloads, an angular frequency
per entry), B and C with N(0, 1) real and imaginary parts.  Values are drawn in float32
from numpy's PCG64 stream in the fixed order x, dt, B, C, z, D, dt_bias, A and then
rounded (round-to-nearest-even) to the workload's dtype; both the CUDA path and
the oracle read the rounded values.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    mode: str            # "diag" (Mamba-1), "ssd" (Mamba-2) or "cdiag" (complex diagonal A)
    dtype: str           # "f32" or "bf16": storage type of x, dt, B, C, z and out
    batch: int
    seqlen: int
    nheads: int          # diag: d_inner; ssd: number of heads
    headdim: int         # diag: 1
    dstate: int
    ngroups: int = 1
    chunk: int = 0       # 0: implementation default
    gate: bool = False
    dt_bias: bool = False
    d_skip: str = "normal"   # "ones", "normal" (N(1, 0.1)) or "none"
    final_state: bool = False
    seed: int = 0

    @property
    def d_inner(self) -> int:
        return self.nheads * self.headdim

    @property
    def token_channels(self) -> int:
        return self.batch * self.seqlen * self.d_inner

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "c0": Workload("c0", "diag", "f32", 1, 256, 64, 1, 16, gate=False, dt_bias=False,
                   d_skip="ones", seed=0),
    "c1": Workload("c1", "diag", "bf16", 8, 1024, 512, 1, 16, gate=True, dt_bias=True,
                   seed=1),
    "c2": Workload("c2", "diag", "bf16", 4, 8192, 5120, 1, 16, gate=True, dt_bias=True,
                   final_state=True, seed=2),
    "c3": Workload("c3", "ssd", "bf16", 4, 8192, 64, 64, 128, chunk=256, seed=3),
    "c4": Workload("c4", "ssd", "bf16", 1, 131072, 32, 64, 256, chunk=256,
                   final_state=True, seed=4),
    "cx1": Workload("cx1", "cdiag", "bf16", 8, 1024, 512, 1, 16, gate=True, dt_bias=True,
                    seed=11),
    "cx2": Workload("cx2", "cdiag", "bf16", 4, 8192, 5120, 1, 16, gate=True, dt_bias=True,
                    final_state=True, seed=12),
}

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(w: Workload):
    return _TORCH_DTYPE[w.dtype]


def shapes(w: Workload) -> dict:
    b, T, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    if w.mode == "diag":
        s = dict(x=(b, T, H), dt=(b, T, H), A=(H, N), B=(b, T, G, N), C=(b, T, G, N),
                 state=(b, H, N))
    elif w.mode == "cdiag":
        s = dict(x=(b, T, H), dt=(b, T, H), A=(H, N, 2), B=(b, T, G, N, 2), C=(b, T, G, N, 2),
                 state=(b, H, N, 2))
    else:
        s = dict(x=(b, T, H, P), dt=(b, T, H), A=(H,), B=(b, T, G, N), C=(b, T, G, N),
                 state=(b, H, P, N))
    s.update(z=s["x"], out=s["x"], D=(H,), dt_bias=(H,))
    return s


def _store(a: np.ndarray, dtype) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t if dtype == torch.float32 else t.to(dtype)


def make_inputs(w: Workload, seed: int | None = None) -> dict:
    """Draw one input set for workload ``w`` as CPU torch tensors.

    x, dt, B, C, z carry the workload dtype; A, D and dt_bias are float32.
    Absent optional inputs map to None.  B and C are (b, T, G, N).
    """
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    s = shapes(w)
    dt_ = torch_dtype(w)
    f32 = np.float32
    x = rng.standard_normal(s["x"], dtype=f32)
    dt = rng.standard_normal(s["dt"], dtype=f32)
    dt *= f32(0.5)
    dt -= f32(2.0)
    B = rng.standard_normal(s["B"], dtype=f32)
    C = rng.standard_normal(s["C"], dtype=f32)
    z = rng.standard_normal(s["z"], dtype=f32) if w.gate else None
    if w.d_skip == "ones":
        D = np.ones(s["D"], dtype=f32)
    elif w.d_skip == "normal":
        D = (1.0 + 0.1 * rng.standard_normal(s["D"])).astype(f32)
    else:
        D = None
    dt_bias = rng.uniform(-4.0, -2.0, s["dt_bias"]).astype(f32) if w.dt_bias else None
    if w.mode == "diag":
        A = -np.broadcast_to(np.arange(1, w.dstate + 1, dtype=f32), s["A"]).copy()
    elif w.mode == "cdiag":
        A = np.empty(s["A"], dtype=f32)
        A[..., 0] = -np.arange(1, w.dstate + 1, dtype=f32)
        A[..., 1] = rng.uniform(-np.pi, np.pi, s["A"][:2]).astype(f32)
    else:
        A = (-rng.uniform(1.0, 16.0, s["A"])).astype(f32)
    return dict(
        x=_store(x, dt_), dt=_store(dt, dt_), B=_store(B, dt_), C=_store(C, dt_),
        z=None if z is None else _store(z, dt_),
        A=torch.from_numpy(A), D=None if D is None else torch.from_numpy(D),
        dt_bias=None if dt_bias is None else torch.from_numpy(dt_bias),
    )


def random_inputs(mode: str, dtype: str, batch: int, seqlen: int, nheads: int, headdim: int,
                  dstate: int, ngroups: int = 1, gate: bool = True, dt_bias: bool = True,
                  d_skip: str = "normal", seed: int = 0) -> tuple[Workload, dict]:
    """Inputs for an arbitrary shape with the same distributions as the workloads."""
    w = Workload("custom", mode, dtype, batch, seqlen, nheads, headdim if mode == "ssd" else 1,
                 dstate, ngroups=ngroups, gate=gate, dt_bias=dt_bias, d_skip=d_skip, seed=seed)
    return w, make_inputs(w)


def conv_params(channels: int, width: int = 4, seed: int = 0, bias: bool = True,
                batch: int = 0, dtype: str = "bf16") -> dict:
    """Seeded parameters of the depthwise convolution ahead of the scan.

    weight (channels, width) and bias (channels,) ~ U(-1/sqrt(width), 1/sqrt(width)),
    PyTorch's default Conv1d initialisation for one input channel per group; with
    ``batch`` > 0 also ``x_prev`` (batch, width-1, channels) ~ N(0, 1) in ``dtype``, the
    inputs of an earlier call.  float32 CPU tensors except x_prev.
    """
    rng = np.random.Generator(np.random.PCG64(1000 + seed))
    bound = 1.0 / np.sqrt(width)
    w = rng.uniform(-bound, bound, (channels, width)).astype(np.float32)
    b = rng.uniform(-bound, bound, channels).astype(np.float32) if bias else None
    out = dict(weight=torch.from_numpy(w), bias=None if b is None else torch.from_numpy(b),
               x_prev=None)
    if batch > 0:
        xp = rng.standard_normal((batch, width - 1, channels), dtype=np.float32)
        out["x_prev"] = _store(xp, torch.bfloat16 if dtype == "bf16" else torch.float32)
    return out
