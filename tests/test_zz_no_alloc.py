"""The no-allocation entry point, ssm_scan_fwd_noalloc, against ssm_scan_fwd.

ssm_scan_fwd_noalloc serves callers that must not allocate device memory during a
scan (an application that owns all device memory through its own allocator, or a
latency-critical loop where an allocation could stall or fail): it takes its scratch
from a fixed 64 MiB array inside the library instead.  The array keeps whatever the
previous call left, so each test first runs the entry point on other inputs (another
seed, more time segments or chunks) and only then on the checked inputs.  The
no-allocation call runs the same kernels with the same scratch layout as the
allocating one, so their results must be bit-identical; the oracle bound is checked
as well.  This file is named so that pytest collects it last; the test that the entry
point rejects shapes beyond its scratch is a host check in tests/test_abi_host.py.
"""
import ctypes

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


def _case(mode, seed, seqlen):
    if mode == "ssd":
        w, inp = random_inputs("ssd", "bf16", 2, seqlen, 4, 64, 128, seed=seed)
        chunk = 256
    else:
        w, inp = random_inputs("diag", "bf16", 1, seqlen, 64, 1, 16, seed=seed)
        chunk = 128  # several time segments, so the scan uses scratch
    d = {k: (None if v is None else v.to("cuda:0")) for k, v in inp.items()}
    return inp, d, chunk


@pytest.mark.parametrize("mode", ["ssd", "diag"])
def test_noalloc_matches_allocating_entry_twice(mode):
    stream = torch.cuda.current_stream()
    # other inputs first, with more scratch in use than the checked call needs, so that
    # the checked call starts on stale scratch contents
    _, d0, chunk = _case(mode, seed=131, seqlen=1500)
    shape0 = ssm.make_shape(d0["x"], d0["A"], d0["B"], chunk=chunk)
    out0 = torch.empty_like(d0["x"])
    fs0 = torch.empty((d0["x"].shape[0],) + tuple(d0["A"].shape[:1]) +
                      ((d0["x"].shape[3],) if mode == "ssd" else ()) + (d0["B"].shape[-1],),
                      device="cuda:0", dtype=torch.float32)
    assert _noalloc(d0, out0, fs0, shape0, stream) == _lib.SSM_OK
    torch.cuda.synchronize()

    inp, d, chunk = _case(mode, seed=31 if mode == "ssd" else 32, seqlen=700 if mode == "ssd" else 900)
    shape = ssm.make_shape(d["x"], d["A"], d["B"], chunk=chunk)
    assert ssm.workspace_size(d["x"], d["A"], d["B"], chunk=chunk) > 0
    ref, ref_fs = ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"],
                               d["dt_bias"], return_final_state=True, chunk=chunk)
    torch.cuda.synchronize()
    orc, orc_fs = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["z"], inp["dt_bias"])
    for _ in range(2):  # the second call runs on the scratch the first one left
        out = torch.full_like(d["x"], float("nan"))
        fs = torch.full_like(ref_fs, float("nan"))
        rc = _noalloc(d, out, fs, shape, stream)
        assert rc == _lib.SSM_OK, _lib.strerror(rc)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), "no-allocation result differs from ssm_scan_fwd"
        assert torch.equal(fs, ref_fs), "no-allocation final state differs from ssm_scan_fwd"
        assert oracle.max_rel_error(out.float().cpu().numpy(), orc) <= 2e-2
        assert oracle.max_rel_error(fs.cpu().numpy(), orc_fs) <= 2e-2
