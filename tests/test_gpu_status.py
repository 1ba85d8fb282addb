"""Bounded device-side waits report SSM_ERR_TIMEOUT through the status word instead of
hanging: a self-test kernel waits on an mbarrier that nothing completes (a bound of a
few hundred polls), the host reads the timeout with ssm_device_status, clears it, and the
same context then runs a tensor-core SSD scan that matches the oracle with a clean status.
"""
import pytest
import torch

import oracle
import selective_state_space_143_b300 as ssm
from selective_state_space_143_b300 import _lib
from selective_state_space_143_b300.inputs import random_inputs

pytestmark = pytest.mark.gpu


def test_wait_that_never_ends_reports_timeout_and_context_survives():
    torch.cuda.init()
    assert ssm.device_status(clear=True) == _lib.SSM_OK
    ssm.selftest_bounded_wait(max_checks=300)
    assert ssm.device_status(clear=False) == _lib.SSM_ERR_TIMEOUT
    assert ssm.device_status(clear=True) == _lib.SSM_ERR_TIMEOUT   # read, then cleared
    assert ssm.device_status(clear=True) == _lib.SSM_OK
    # the context is usable: a tensor-core SSD scan (mbarrier waits that do complete)
    w, inp = random_inputs("ssd", "bf16", 1, 300, 2, 64, 64, seed=21)
    d = {k: (None if v is None else v.to("cuda:0")) for k, v in inp.items()}
    out, fs = ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                           return_final_state=True, chunk=128)
    torch.cuda.synchronize()
    assert ssm.device_status(clear=True) == _lib.SSM_OK
    ref, _ = oracle.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                         inp["dt_bias"])
    assert oracle.max_rel_error(out.float().cpu().numpy(), ref) <= 2e-2
