"""Runs tests/test_abi_host.py in a child process that sees no GPU.

Those tests pass made-up device addresses that the library's host checks must reject
before any launch.  In a process with a visible GPU a regression in one of those checks
could launch a kernel on invalid addresses, so on a GPU machine the module skips itself
and this test runs it with CUDA_VISIBLE_DEVICES empty: a broken check then fails with
SSM_ERR_CUDA (no device) instead of touching the GPU.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_host_checks_run_in_a_process_without_a_gpu():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_abi_host.py")],
                       env=env, cwd=os.path.dirname(HERE), capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "skipped" not in r.stdout.splitlines()[-1], r.stdout[-2000:]
