"""The bounds-checked build (-DSSM_BOUNDS_CHECK, libssmscan_bc.so): the debugging
stand-in for a memory checker.  Every kernel checks each global store against the byte
range of the buffer it writes and, outside it, skips the store and records
SSM_ERR_BOUNDS in the device status word, without trapping.

1. The check's path on demand: a self-test stores through the check to an index past
   the range it is given, inside a buffer that really holds that index (the address is
   valid whatever the check does): the store is skipped and SSM_ERR_BOUNDS read back.
2. No false alarms, and the checks change no result: the GPU parity tests of the forward
   scans, the state/decode paths, the convolution, the complex scan and the backward run
   in a child process on the bounds-checked library, each followed by a clean status.
"""
import os
import subprocess
import sys

import pytest
import torch

from selective_state_space_143_b300 import build as _build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bc_lib():
    return _build.build_bounds_checked()


def _child(bc_lib, args, timeout):
    env = dict(os.environ, SSM_LIB_PATH=bc_lib, SSM_EXPECT_BOUNDS_CHECK="1")
    return subprocess.run([sys.executable, *args], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=timeout)


SELFTEST = r"""
import torch
import selective_state_space_143_b300 as ssm
from selective_state_space_143_b300 import _lib
assert ssm.bounds_check_enabled()
assert ssm.device_status(clear=True) == _lib.SSM_OK
buf = torch.zeros(64, dtype=torch.float32, device="cuda:0")
ssm.selftest_bounds(buf, 32 * 4, 40)          # past the given range, inside buf
assert ssm.device_status(clear=False) == _lib.SSM_ERR_BOUNDS
assert ssm.device_status(clear=True) == _lib.SSM_ERR_BOUNDS
assert ssm.device_status(clear=True) == _lib.SSM_OK
assert float(buf[40]) == 0.0, "the out-of-range store was not skipped"
ssm.selftest_bounds(buf, 32 * 4, 10)          # in range: stored, no status
assert ssm.device_status(clear=True) == _lib.SSM_OK
assert float(buf[10]) == 1.0
print("selftest ok")
"""


def test_bounds_check_records_and_skips(bc_lib):
    r = _child(bc_lib, ["-c", SELFTEST], 300)
    assert r.returncode == 0 and "selftest ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]


def test_parity_suite_on_bounds_checked_library(bc_lib):
    files = ["tests/test_gpu_parity.py", "tests/test_gpu_state.py", "tests/test_gpu_conv.py",
             "tests/test_gpu_complex.py", "tests/test_gpu_bwd.py"]
    r = _child(bc_lib, ["-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *files], 1200)
    tail = r.stdout[-3000:] + r.stderr[-2000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout, tail


def test_normal_build_has_no_checks():
    import selective_state_space_143_b300 as ssm
    from selective_state_space_143_b300 import _lib
    if os.environ.get("SSM_LIB_PATH"):
        pytest.skip("another library is loaded")
    assert not ssm.bounds_check_enabled()
    buf = torch.zeros(4, dtype=torch.float32, device="cuda:0")
    with pytest.raises(ssm.SsmError) as e:
        ssm.selftest_bounds(buf, 16, 1)
    assert e.value.status == _lib.SSM_ERR_UNSUPPORTED
