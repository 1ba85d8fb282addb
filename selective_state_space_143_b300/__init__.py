"""B300-native selective state-space scan (Mamba-1 diagonal form and Mamba-2 SSD form).

Python binding of libssmscan.so.  Every step of the scan runs in the library's CUDA
kernels; this module only checks tensor metadata and passes device pointers and the
current CUDA stream through the C ABI (include/ssm_scan.h).  PyTorch provides device
memory and streams.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import SsmError, ssm_conv, ssm_shape

__all__ = ["scan_fwd", "scan_bwd", "step", "workspace_size", "make_shape", "launch_count", "SsmError",
           "ssm_shape"]

_DTYPES = {torch.float32: _lib.SSM_F32, torch.bfloat16: _lib.SSM_BF16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def make_shape(x: torch.Tensor, A: torch.Tensor, B: torch.Tensor, chunk: int = 0) -> ssm_shape:
    """Build the ``ssm_shape`` descriptor from tensor shapes.

    DIAG (Mamba-1): x (b, T, D), A (D, N).  SSD (Mamba-2): x (b, T, H, P), A (H,).
    B: (b, T, N) or (b, T, G, N).  CDIAG (complex A, the rotating state update read for
    Mamba-3): x (b, T, D), A (D, N, 2), B (b, T, N, 2) or (b, T, G, N, 2), every complex
    number an (re, im) pair.
    """
    if x.dtype not in _DTYPES:
        raise TypeError(f"x must be float32 or bfloat16, got {x.dtype}")
    s = ssm_shape()
    s.dtype = _DTYPES[x.dtype]
    if A.dim() == 3:
        if x.dim() != 3 or A.shape[2] != 2:
            raise ValueError("complex mode: x must be (batch, seqlen, d_inner), A (d_inner, dstate, 2)")
        s.mode = _lib.SSM_MODE_CDIAG
        s.batch, s.seqlen, s.nheads = x.shape
        s.headdim = 1
        if B.dim() == 4:
            s.ngroups, s.dstate = 1, B.shape[2]
        elif B.dim() == 5:
            s.ngroups, s.dstate = B.shape[2], B.shape[3]
        else:
            raise ValueError("complex mode: B must be (batch, seqlen, dstate, 2) or "
                             "(batch, seqlen, ngroups, dstate, 2)")
        s.chunk = int(chunk)
        s.flags = 0
        return s
    if A.dim() == 2:
        if x.dim() != 3:
            raise ValueError("diagonal mode: x must be (batch, seqlen, d_inner)")
        s.mode = _lib.SSM_MODE_DIAG
        s.batch, s.seqlen, s.nheads = x.shape
        s.headdim = 1
    elif A.dim() == 1:
        if x.dim() != 4:
            raise ValueError("SSD mode: x must be (batch, seqlen, nheads, headdim)")
        s.mode = _lib.SSM_MODE_SSD
        s.batch, s.seqlen, s.nheads, s.headdim = x.shape
    else:
        raise ValueError("A must be 2-D (d_inner, dstate) or 1-D (nheads,)")
    if B.dim() == 3:
        s.ngroups, s.dstate = 1, B.shape[2]
    elif B.dim() == 4:
        s.ngroups, s.dstate = B.shape[2], B.shape[3]
    else:
        raise ValueError("B must be (batch, seqlen, dstate) or (batch, seqlen, ngroups, dstate)")
    s.chunk = int(chunk)
    s.flags = 0
    return s


def _check(name, t, shape, dtype, device):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def workspace_size(x, A, B, chunk: int = 0) -> int:
    """Device scratch bytes ``scan_fwd`` needs for these shapes (0 when none)."""
    s = make_shape(x, A, B, chunk)
    n = _lib.load().ssm_scan_workspace_size(ctypes.byref(s))
    if n == ctypes.c_size_t(-1).value:
        raise SsmError(_lib.SSM_ERR_SHAPE, "ssm_scan_workspace_size")
    return int(n)


def _conv_struct(name, weight, bias, x_prev, x_last, x, b, ch, dev):
    """Check the convolution tensors and build the ``ssm_conv`` descriptor."""
    if weight.dim() != 2 or weight.shape[0] != ch:
        raise ValueError(f"{name}: conv_weight must be ({ch}, width)")
    K = int(weight.shape[1])
    _check("conv_weight", weight, (ch, K), torch.float32, dev)
    _check("conv_bias", bias, (ch,), torch.float32, dev)
    _check("conv_x_prev", x_prev, (b, K - 1, ch), x.dtype, dev)
    _check("conv_x_last", x_last, (b, K - 1, ch), x.dtype, dev)
    c = ssm_conv()
    c.weight, c.bias = weight.data_ptr(), None if bias is None else bias.data_ptr()
    c.x_prev = None if x_prev is None else x_prev.data_ptr()
    c.x_last = None if x_last is None else x_last.data_ptr()
    c.width = K
    return c


def scan_fwd(x, dt, A, B, C, D=None, z=None, dt_bias=None, *, out=None, final_state=None,
             return_final_state: bool = False, chunk: int = 0, workspace=None, stream=None,
             initial_state=None, conv_weight=None, conv_bias=None, conv_x_prev=None,
             conv_x_last=None):
    """Selective scan forward on the GPU.

    out_t = (C_t . h_t + D x_t) * SiLU(z_t),  h_t = exp(Delta_t A) h_{t-1} + Delta_t B_t x_t,
    Delta_t = softplus(dt_t + dt_bias).  Shapes as in ``make_shape``; dt is (b, T, D) for
    the diagonal mode and (b, T, H) for SSD; D and dt_bias are (D,) / (H,) float32.

    Returns ``out``, or ``(out, final_state)`` when ``return_final_state`` is set or a
    ``final_state`` tensor is passed.  Runs asynchronously on ``stream`` (default: the
    current torch stream).  ``workspace``: optional uint8 CUDA tensor of at least
    ``workspace_size`` bytes; otherwise the library draws scratch from the stream-ordered
    allocator.  ``initial_state``: optional float32 state entering t = 0 (the layout of
    ``final_state``; must not share memory with it), for resuming a split sequence.

    ``conv_weight`` (channels, width) float32 puts the causal depthwise convolution + SiLU
    ahead of the scan (channels = d_inner, or nheads*headdim); ``conv_bias`` (channels,),
    ``conv_x_prev`` (b, width-1, channels) the inputs before t = 0, and ``conv_x_last``
    a tensor of that shape to receive this call's last inputs.
    """
    s = make_shape(x, A, B, chunk)
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("scan_fwd runs on CUDA tensors only")
    b, T, H, P, N, G = s.batch, s.seqlen, s.nheads, s.headdim, s.dstate, s.ngroups
    diag = s.mode == _lib.SSM_MODE_DIAG
    cplx = s.mode == _lib.SSM_MODE_CDIAG
    _check("x", x, x.shape, x.dtype, dev)
    _check("dt", dt, (b, T, H), x.dtype, dev)
    _check("A", A, (H, N, 2) if cplx else (H, N) if diag else (H,), torch.float32, dev)
    _check("B", B, B.shape, x.dtype, dev)
    _check("C", C, B.shape, x.dtype, dev)
    _check("D", D, (H,), torch.float32, dev)
    _check("z", z, x.shape, x.dtype, dev)
    _check("dt_bias", dt_bias, (H,), torch.float32, dev)
    if out is None:
        out = torch.empty_like(x)
    _check("out", out, x.shape, x.dtype, dev)
    want_state = return_final_state or final_state is not None
    st_shape = (b, H, N, 2) if cplx else (b, H, N) if diag else (b, H, P, N)
    if want_state and final_state is None:
        final_state = torch.empty(st_shape, device=dev, dtype=torch.float32)
    _check("final_state", final_state, st_shape, torch.float32, dev)
    _check("initial_state", initial_state, st_shape, torch.float32, dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = ctypes.c_void_p(stream.cuda_stream)
    lib = _lib.load()
    with torch.cuda.device(dev):
        if workspace is not None and workspace.device != dev:
            raise ValueError("workspace must be on x's device")
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        if conv_weight is not None:
            cv = _conv_struct("scan_fwd", conv_weight, conv_bias, conv_x_prev, conv_x_last, x,
                              b, H * P, dev)
            rc = lib.ssm_scan_fwd_conv(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                       _ptr(z), _ptr(dt_bias), ctypes.byref(cv),
                                       _ptr(initial_state), _ptr(out), _ptr(final_state),
                                       ctypes.byref(s), _ptr(workspace), ws_bytes, handle)
        elif initial_state is not None:
            rc = lib.ssm_scan_fwd_state(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                        _ptr(z), _ptr(dt_bias), _ptr(initial_state), _ptr(out),
                                        _ptr(final_state), ctypes.byref(s), _ptr(workspace),
                                        ws_bytes, handle)
        elif workspace is None:
            rc = lib.ssm_scan_fwd(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                  _ptr(dt_bias), _ptr(out), _ptr(final_state), ctypes.byref(s),
                                  handle)
        else:
            rc = lib.ssm_scan_fwd_ws(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                     _ptr(z), _ptr(dt_bias), _ptr(out), _ptr(final_state),
                                     ctypes.byref(s), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), handle)
    if rc != _lib.SSM_OK:
        raise SsmError(rc, "ssm_scan_fwd")
    return (out, final_state) if want_state else out


def scan_bwd(x, dt, A, B, C, D=None, z=None, dt_bias=None, *, dout, dfinal_state=None,
             initial_state=None, workspace=None, stream=None, grads=None):
    """Gradients of the scan, diagonal mode (2-D A) or SSD mode (1-D A per head).

    ``dout`` is the gradient of the output (x's shape and dtype), ``dfinal_state`` that of
    the final state (float32, optional).  Returns a dict of float32 tensors: dx, ddt, dA,
    dB, dC (B's shape), and dD, dz, ddt_bias, dinitial_state where the matching input was
    given (dinitial_state always); each has its input's shape (SSD: ddt (b, T, H), dA
    (H,), dinitial_state (b, H, P, N)).  ``grads``: optional dict of preallocated float32
    tensors with those names and shapes, written in place instead of new ones.
    """
    s = make_shape(x, A, B, 0)
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("scan_bwd runs on CUDA tensors only")
    ssd = s.mode == _lib.SSM_MODE_SSD
    b, T, H, P, N = s.batch, s.seqlen, s.nheads, s.headdim, s.dstate
    st = (b, H, P, N) if ssd else (b, H, N)
    a_shape = (H,) if ssd else (H, N)
    for name, t, shp, dt_ in (("x", x, x.shape, x.dtype), ("dt", dt, (b, T, H), x.dtype),
                              ("A", A, a_shape, torch.float32), ("B", B, B.shape, x.dtype),
                              ("C", C, B.shape, x.dtype), ("D", D, (H,), torch.float32),
                              ("z", z, x.shape, x.dtype), ("dt_bias", dt_bias, (H,), torch.float32),
                              ("dout", dout, x.shape, x.dtype),
                              ("dfinal_state", dfinal_state, st, torch.float32),
                              ("initial_state", initial_state, st, torch.float32)):
        _check(name, t, shp, dt_, dev)
    f32 = dict(device=dev, dtype=torch.float32)
    g = {"dx": torch.empty(x.shape, **f32), "ddt": torch.empty((b, T, H), **f32),
         "dA": torch.empty(a_shape, **f32), "dB": torch.empty(B.shape, **f32),
         "dC": torch.empty(B.shape, **f32),
         "dD": None if D is None else torch.empty((H,), **f32),
         "dz": None if z is None else torch.empty(x.shape, **f32),
         "ddt_bias": None if dt_bias is None else torch.empty((H,), **f32),
         "dinitial_state": torch.empty(st, **f32)}
    if grads is not None:
        for k, v in grads.items():
            if k not in g or g[k] is None:
                raise ValueError(f"grads: unexpected {k}")
            _check(k, v, g[k].shape, torch.float32, dev)
            g[k] = v
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        rc = _lib.load().ssm_scan_bwd(
            *(_ptr(t) for t in (x, dt, A, B, C, D, z, dt_bias, initial_state, dout, dfinal_state,
                                g["dx"], g["ddt"], g["dA"], g["dB"], g["dC"], g["dD"], g["dz"],
                                g["ddt_bias"], g["dinitial_state"])),
            ctypes.byref(s), _ptr(workspace), ws_bytes, ctypes.c_void_p(stream.cuda_stream))
    if rc != _lib.SSM_OK:
        raise SsmError(rc, "ssm_scan_bwd")
    return g


def step(x, dt, A, B, C, D=None, z=None, dt_bias=None, *, state, out=None, stream=None,
         conv_weight=None, conv_bias=None, conv_state=None):
    """One token of recurrent decoding; ``state`` (float32) is updated in place.

    With ``conv_weight`` (channels, width) the convolution + SiLU runs ahead of the scan;
    ``conv_state`` (b, width-1, channels) in x's dtype holds the previous inputs and is
    shifted in place (None: zeros, nothing kept).

    DIAG: x, z (b, D), dt (b, D), A (D, N), B, C (b, N) or (b, G, N), state (b, D, N).
    SSD: x, z (b, H, P), dt (b, H), A (H,), B, C (b, N) or (b, G, N), state (b, H, P, N).
    Returns ``out`` (shaped like x).  Equivalent to ``scan_fwd`` over one token with
    ``initial_state=state`` and the final state written back to ``state``.
    """
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("step runs on CUDA tensors only")
    if x.dtype not in _DTYPES:
        raise TypeError(f"x must be float32 or bfloat16, got {x.dtype}")
    s = ssm_shape()
    s.dtype = _DTYPES[x.dtype]
    s.seqlen = 1
    if A.dim() == 2:
        if x.dim() != 2:
            raise ValueError("diagonal mode: x must be (batch, d_inner)")
        s.mode = _lib.SSM_MODE_DIAG
        (s.batch, s.nheads), s.headdim = x.shape, 1
    elif A.dim() == 1:
        if x.dim() != 3:
            raise ValueError("SSD mode: x must be (batch, nheads, headdim)")
        s.mode = _lib.SSM_MODE_SSD
        s.batch, s.nheads, s.headdim = x.shape
    else:
        raise ValueError("A must be 2-D (d_inner, dstate) or 1-D (nheads,)")
    if B.dim() == 2:
        s.ngroups, s.dstate = 1, B.shape[1]
    elif B.dim() == 3:
        s.ngroups, s.dstate = B.shape[1], B.shape[2]
    else:
        raise ValueError("B must be (batch, dstate) or (batch, ngroups, dstate)")
    s.chunk, s.flags = 0, 0
    b, H, P, N = s.batch, s.nheads, s.headdim, s.dstate
    diag = s.mode == _lib.SSM_MODE_DIAG
    _check("x", x, x.shape, x.dtype, dev)
    _check("dt", dt, (b, H), x.dtype, dev)
    _check("A", A, (H, N) if diag else (H,), torch.float32, dev)
    _check("B", B, B.shape, x.dtype, dev)
    _check("C", C, B.shape, x.dtype, dev)
    _check("D", D, (H,), torch.float32, dev)
    _check("z", z, x.shape, x.dtype, dev)
    _check("dt_bias", dt_bias, (H,), torch.float32, dev)
    _check("state", state, (b, H, N) if diag else (b, H, P, N), torch.float32, dev)
    if out is None:
        out = torch.empty_like(x)
    _check("out", out, x.shape, x.dtype, dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        if conv_weight is not None:
            cv = _conv_struct("step", conv_weight, conv_bias, conv_state, conv_state, x, b, H * P,
                              dev)
            rc = _lib.load().ssm_step_conv(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                           _ptr(z), _ptr(dt_bias), ctypes.byref(cv), _ptr(state),
                                           _ptr(out), ctypes.byref(s),
                                           ctypes.c_void_p(stream.cuda_stream))
        else:
            rc = _lib.load().ssm_step(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                      _ptr(z), _ptr(dt_bias), _ptr(state), _ptr(out),
                                      ctypes.byref(s), ctypes.c_void_p(stream.cuda_stream))
    if rc != _lib.SSM_OK:
        raise SsmError(rc, "ssm_step")
    return out


def device_status(clear: bool = True, stream=None) -> int:
    """Status of the library's bounded device-side waits (and, in a bounds-checked build,
    its store bounds checks) on the current device, after the work queued on ``stream``
    (default: the current torch stream): ``_lib.SSM_OK``, ``_lib.SSM_ERR_TIMEOUT`` (a
    kernel gave up a wait; its outputs are not valid) or ``_lib.SSM_ERR_BOUNDS`` (a store
    fell outside its buffer and was skipped).  ``clear`` resets the status word."""
    if stream is None:
        stream = torch.cuda.current_stream()
    rc = _lib.load().ssm_device_status(1 if clear else 0, ctypes.c_void_p(stream.cuda_stream))
    if rc not in (_lib.SSM_OK, _lib.SSM_ERR_TIMEOUT, _lib.SSM_ERR_BOUNDS):
        raise SsmError(rc, "ssm_device_status")
    return rc


def bounds_check_enabled() -> bool:
    """True when the loaded library was built with SSM_BOUNDS_CHECK."""
    return bool(_lib.load().ssm_bounds_check_enabled())


def selftest_bounds(buf: torch.Tensor, nbytes: int, index: int, stream=None) -> None:
    """Store to ``buf[index]`` through the bounds check against the first ``nbytes`` of the
    fp32 device tensor ``buf`` (see ``ssm_selftest_bounds``; ``buf`` must hold ``index``).
    Bounds-checked builds only; read the outcome with ``device_status``."""
    if buf.dtype != torch.float32 or not buf.is_cuda or index >= buf.numel():
        raise ValueError("buf must be a CUDA fp32 tensor that holds element `index`")
    if stream is None:
        stream = torch.cuda.current_stream()
    rc = _lib.load().ssm_selftest_bounds(ctypes.c_void_p(buf.data_ptr()), int(nbytes), int(index),
                                         ctypes.c_void_p(stream.cuda_stream))
    if rc != _lib.SSM_OK:
        raise SsmError(rc, "ssm_selftest_bounds")


def selftest_bounded_wait(max_checks: int = 1000, stream=None) -> None:
    """Launch the bounded-wait self-test (a wait nothing completes; see
    ``ssm_selftest_bounded_wait``); read the outcome with ``device_status``."""
    if stream is None:
        stream = torch.cuda.current_stream()
    rc = _lib.load().ssm_selftest_bounded_wait(int(max_checks), ctypes.c_void_p(stream.cuda_stream))
    if rc != _lib.SSM_OK:
        raise SsmError(rc, "ssm_selftest_bounded_wait")


def launch_count() -> int:
    """Kernels launched by libssmscan.so in this process so far."""
    return _lib.launch_count()
