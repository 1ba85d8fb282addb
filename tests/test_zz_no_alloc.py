"""The no-allocation entry point, ssm_scan_fwd_noalloc, against ssm_scan_fwd.

ssm_scan_fwd_noalloc serves callers that must not allocate device memory during a
scan (an application that owns all device memory through its own allocator, or a
latency-critical loop where an allocation could stall or fail): it takes its scratch
from a fixed 64 MiB array inside the library instead.  This file is named so that
pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_143_b300 as ssm
from selective_state_space_143_b300 import _lib
from selective_state_space_143_b300.inputs import random_inputs

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(None if t is None else t.data_ptr())


def _noalloc(d, out, fs, shape, stream):
    return _lib.load().ssm_scan_fwd_noalloc(
        _ptr(d["x"]), _ptr(d["dt"]), _ptr(d["A"]), _ptr(d["B"]), _ptr(d["C"]), _ptr(d["D"]),
        _ptr(d["z"]), _ptr(d["dt_bias"]), _ptr(out), _ptr(fs), ctypes.byref(shape),
        ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("mode", ["ssd", "diag"])
def test_noalloc_matches_allocating_entry_twice(mode):
    if mode == "ssd":
        w, inp = random_inputs("ssd", "bf16", 2, 700, 4, 64, 128, seed=31)
        chunk = 256
    else:
        w, inp = random_inputs("diag", "bf16", 1, 900, 64, 1, 16, seed=32)
        chunk = 128  # several time segments, so the scan uses scratch
    d = {k: (None if v is None else v.to("cuda:0")) for k, v in inp.items()}
    shape = ssm.make_shape(d["x"], d["A"], d["B"], chunk=chunk)
    assert ssm.workspace_size(d["x"], d["A"], d["B"], chunk=chunk) > 0
    ref, ref_fs = ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"],
                               d["dt_bias"], return_final_state=True, chunk=chunk)
    stream = torch.cuda.current_stream()
    for _ in range(2):  # the second call runs on scratch left over from the first
        out = torch.full_like(d["x"], float("nan"))
        fs = torch.full_like(ref_fs, float("nan"))
        rc = _noalloc(d, out, fs, shape, stream)
        assert rc == _lib.SSM_OK, _lib.strerror(rc)
        torch.cuda.synchronize()
        assert oracle.max_rel_error(out.float().cpu().numpy(), ref.float().cpu().numpy()) <= 2e-2
        assert oracle.max_rel_error(fs.cpu().numpy(), ref_fs.cpu().numpy()) <= 2e-2
        assert torch.isfinite(out.float()).all()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # an SSD shape whose chunk states need far more than 64 MiB of scratch
    shape = _lib.ssm_shape()
    shape.mode, shape.dtype = _lib.SSM_MODE_SSD, _lib.SSM_BF16
    shape.batch, shape.seqlen, shape.nheads, shape.headdim = 1, 131072, 32, 64
    shape.dstate, shape.ngroups, shape.chunk, shape.flags = 256, 1, 256, 0
    assert _lib.load().ssm_scan_workspace_size(ctypes.byref(shape)) > (64 << 20)
    vp = ctypes.c_void_p
    rc = _lib.load().ssm_scan_fwd_noalloc(vp(1 << 12), vp(2 << 12), vp(3 << 12), vp(4 << 12),
                                          vp(5 << 12), None, None, None, vp(6 << 12), None,
                                          ctypes.byref(shape), None)
    assert rc == _lib.SSM_ERR_ALLOC
