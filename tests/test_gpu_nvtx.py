"""NVTX ranges around every kernel launch.

A child process loads tests/nvtx_record.c (built here with gcc) as its NVTX injection
library and runs a diagonal scan and a tensor-core SSD scan; the recorded ranges must
name each launched kernel and close every range they open.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))

CHILD = textwrap.dedent("""
    import torch
    import selective_state_space_143_b300 as ssm
    from selective_state_space_143_b300.inputs import random_inputs
    for mode, kw in (("diag", dict(headdim=1, dstate=16, nheads=256)),
                     ("ssd", dict(headdim=64, dstate=128, nheads=8))):
        w, inp = random_inputs(mode, "bf16", batch=1, seqlen=512, **kw)
        d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
        ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                     chunk=256 if mode == "ssd" else 0)
    torch.cuda.synchronize()
""")


def test_every_launch_is_an_nvtx_range(tmp_path):
    lib = tmp_path / "nvtx_record.so"
    subprocess.run(["gcc", "-shared", "-fPIC", "-O2", "-I", "/usr/local/cuda/include", "-o", str(lib),
                    os.path.join(HERE, "nvtx_record.c")], check=True)
    log = tmp_path / "ranges.txt"
    env = dict(os.environ, NVTX_INJECTION64_PATH=str(lib), SSM_NVTX_LOG=str(log))
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=os.path.dirname(HERE),
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    lines = log.read_text().splitlines()
    depth, names = 0, []
    for ln in lines:
        if ln.startswith("push "):
            depth += 1
            names.append(ln[5:])
        else:
            assert ln == "pop", ln
            depth -= 1
        assert 0 <= depth <= 1, "launch ranges nest or pop unopened"
    assert depth == 0
    assert "diag_scan_kernel (output pass)" in names
    assert {"ssd_state_tc", "ssd_state_pass_split", "ssd_scan_tc"} <= set(names), names
