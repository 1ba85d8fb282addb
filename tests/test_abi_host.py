"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function include/ssm_scan.h declares, and rejects bad arguments with the documented
status before touching the device.

Many of these tests pass made-up device addresses that the host checks must reject
before anything is launched.  They never run in a process that sees a GPU: where one
is visible, this module is skipped and tests/test_host_checks_child.py runs it in a
child process with CUDA_VISIBLE_DEVICES empty, so that a regression in a host check
fails a test (SSM_ERR_CUDA instead of the expected status) rather than launching a
kernel on invalid addresses."""
import ctypes
import os
import re

import pytest
import torch

pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="made-up device addresses: run without a visible GPU "
                                       "(tests/test_host_checks_child.py)")

import selective_state_space_143_b300 as ssm
from selective_state_space_143_b300 import _lib
from selective_state_space_143_b300.inputs import WORKLOADS

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "ssm_scan.h")


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(ssm_[a-z_0-9]+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_expected_functions():
    assert declared_functions() == sorted(_lib.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = _lib.load()
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_strerror_and_version():
    for st in range(0, 9):
        assert _lib.strerror(st)
    assert "unknown" in _lib.strerror(99)
    assert _lib.load().ssm_abi_version() >> 16 == 1


def _shape(**kw):
    s = _lib.ssm_shape()
    base = dict(mode=0, dtype=1, batch=2, seqlen=64, nheads=64, headdim=1, dstate=16, ngroups=1,
                chunk=0, flags=0)
    base.update(kw)
    for k, v in base.items():
        setattr(s, k, v)
    return s


def _ws(s):
    return _lib.load().ssm_scan_workspace_size(ctypes.byref(s))


BAD = ctypes.c_size_t(-1).value


@pytest.mark.parametrize("kw,valid", [
    (dict(), True),
    (dict(mode=7), False), (dict(dtype=5), False), (dict(flags=1), False),
    (dict(batch=-1), False), (dict(nheads=0), False), (dict(ngroups=3), False),
    (dict(headdim=2), False),                   # diagonal mode needs headdim 1
    (dict(dstate=72), False),                   # diagonal N limit 64
    (dict(dstate=12), False),                   # bf16 B/C rows must be 16-byte multiples
    (dict(nheads=60), False),                   # bf16 channel rows must be 16-byte multiples
    (dict(chunk=48), False),                    # diagonal segment length multiple of 32
    (dict(mode=1, headdim=64, nheads=8, dstate=128, chunk=256), True),
    (dict(mode=1, headdim=64, nheads=8, dstate=300), False),
    (dict(mode=1, headdim=64, nheads=8, dstate=128, chunk=100), False),
    (dict(mode=1, headdim=64, nheads=8, dstate=128, chunk=512), False),
    (dict(mode=1, dtype=0, headdim=3, nheads=4, dstate=1, ngroups=4), False),  # P*N % 4
    (dict(mode=1, dtype=0, headdim=4, nheads=4, dstate=1, ngroups=4), True),
])
def test_workspace_query_validates_shape(kw, valid):
    n = _ws(_shape(**kw))
    assert (n != BAD) == valid


def test_workspace_sizes_of_workloads():
    for name, w in WORKLOADS.items():
        s = _shape(mode=0 if w.mode == "diag" else 1, dtype=1 if w.dtype == "bf16" else 0,
                   batch=w.batch, seqlen=w.seqlen, nheads=w.nheads, headdim=w.headdim,
                   dstate=w.dstate, ngroups=w.ngroups, chunk=w.chunk)
        n = _ws(s)
        assert n != BAD, name
        if w.mode == "ssd":
            assert n > 0


def _call(s, x=1 << 12, dt=2 << 12, A=3 << 12, B=4 << 12, C=5 << 12, out=6 << 12, **opt):
    lib = _lib.load()
    vp = ctypes.c_void_p
    return lib.ssm_scan_fwd(vp(x), vp(dt), vp(A), vp(B), vp(C), vp(opt.get("D")), vp(opt.get("z")),
                            vp(opt.get("dt_bias")), vp(out), vp(opt.get("fs")),
                            ctypes.byref(s) if s is not None else None, None)


def test_argument_errors_are_reported_before_any_launch():
    s = _shape()
    assert _call(None) == _lib.SSM_ERR_NULL
    assert _call(s, x=0) == _lib.SSM_ERR_NULL
    assert _call(s, out=0) == _lib.SSM_ERR_NULL
    assert _call(s, dt=(2 << 12) + 8) == _lib.SSM_ERR_ALIGN
    assert _call(s, z=(7 << 12) + 2) == _lib.SSM_ERR_ALIGN
    assert _call(_shape(dtype=9)) == _lib.SSM_ERR_DTYPE
    assert _call(_shape(flags=2)) == _lib.SSM_ERR_UNSUPPORTED
    assert _call(_shape(nheads=12, ngroups=5)) == _lib.SSM_ERR_SHAPE
    assert _call(_shape(mode=1, nheads=8, headdim=64, dstate=512)) == _lib.SSM_ERR_UNSUPPORTED


def test_workspace_entry_rejects_small_or_misaligned_workspace():
    lib = _lib.load()
    s = _shape(mode=1, nheads=8, headdim=64, dstate=128, chunk=64, seqlen=256)
    need = _ws(s)
    assert need > 0
    vp = ctypes.c_void_p
    args = [vp(1 << 12), vp(2 << 12), vp(3 << 12), vp(4 << 12), vp(5 << 12), None, None, None,
            vp(6 << 12), None, ctypes.byref(s)]
    assert lib.ssm_scan_fwd_ws(*args, None, 0, None) == _lib.SSM_ERR_ALLOC
    assert lib.ssm_scan_fwd_ws(*args, vp(1 << 20), need - 1, None) == _lib.SSM_ERR_ALLOC
    assert lib.ssm_scan_fwd_ws(*args, vp((1 << 20) + 16), need, None) == _lib.SSM_ERR_ALIGN


def test_binding_shape_descriptor():
    x = torch.zeros(2, 10, 4, 8, dtype=torch.bfloat16)
    A = torch.zeros(4)
    B = torch.zeros(2, 10, 2, 16, dtype=torch.bfloat16)
    s = ssm.make_shape(x, A, B, chunk=64)
    assert (s.mode, s.dtype, s.batch, s.seqlen, s.nheads, s.headdim, s.dstate, s.ngroups,
            s.chunk) == (1, 1, 2, 10, 4, 8, 16, 2, 64)
    x3 = torch.zeros(1, 5, 32)
    s3 = ssm.make_shape(x3, torch.zeros(32, 8), torch.zeros(1, 5, 8))
    assert (s3.mode, s3.dtype, s3.nheads, s3.headdim, s3.dstate, s3.ngroups) == (0, 0, 32, 1, 8, 1)


def test_binding_refuses_cpu_tensors():
    x = torch.zeros(1, 4, 8)
    with pytest.raises(ValueError):
        ssm.scan_fwd(x, x, torch.zeros(8, 4), torch.zeros(1, 4, 4), torch.zeros(1, 4, 4))


def _step(s, x=1 << 12, dt=2 << 12, A=3 << 12, B=4 << 12, C=5 << 12, state=6 << 12,
          out=7 << 12, **opt):
    lib = _lib.load()
    vp = ctypes.c_void_p
    return lib.ssm_step(vp(x), vp(dt), vp(A), vp(B), vp(C), vp(opt.get("D")), vp(opt.get("z")),
                        vp(opt.get("dt_bias")), vp(state), vp(out),
                        ctypes.byref(s) if s is not None else None, None)


def test_step_argument_errors():
    one = dict(seqlen=1)
    assert _step(None) == _lib.SSM_ERR_NULL
    assert _step(_shape(seqlen=2)) == _lib.SSM_ERR_SHAPE            # one token per call
    assert _step(_shape(**one), state=0) == _lib.SSM_ERR_NULL
    assert _step(_shape(**one), x=0) == _lib.SSM_ERR_NULL
    assert _step(_shape(**one), state=(6 << 12) + 4) == _lib.SSM_ERR_ALIGN
    assert _step(_shape(mode=1, nheads=8, headdim=8, dstate=2, ngroups=8, dtype=1, seqlen=1)) \
        == _lib.SSM_ERR_ALIGN                                      # dstate % 4
    # out inside the state: the in-place update would overwrite it
    assert _step(_shape(**one), out=(6 << 12) + 256) == _lib.SSM_ERR_SHAPE
    # nothing to do
    assert _step(_shape(batch=0, seqlen=1), x=0, dt=0, B=0, C=0, state=0, out=0) == _lib.SSM_OK


def test_scan_with_initial_state_argument_errors():
    lib = _lib.load()
    vp = ctypes.c_void_p
    s = _shape()

    def call(init, fs, ws=None, nbytes=0):
        return lib.ssm_scan_fwd_state(vp(1 << 12), vp(2 << 12), vp(3 << 12), vp(4 << 12),
                                      vp(5 << 12), None, None, None, vp(init), vp(6 << 12),
                                      vp(fs), ctypes.byref(s), vp(ws), nbytes, None)

    assert call((8 << 12) + 4, None) == _lib.SSM_ERR_ALIGN
    st_bytes = 2 * 64 * 16 * 4
    assert call(8 << 20, (8 << 20) + st_bytes - 16) == _lib.SSM_ERR_SHAPE  # overlap
    s2 = _shape(mode=1, nheads=8, headdim=64, dstate=128, chunk=64, seqlen=256)
    need = _ws(s2)
    assert lib.ssm_scan_fwd_state(vp(1 << 12), vp(2 << 12), vp(3 << 12), vp(4 << 12),
                                  vp(5 << 12), None, None, None, vp(8 << 20), vp(6 << 12), None,
                                  ctypes.byref(s2), vp(1 << 20), need - 1, None) \
        == _lib.SSM_ERR_ALLOC


def test_step_binding_refuses_cpu_tensors():
    x = torch.zeros(1, 8)
    with pytest.raises(ValueError):
        ssm.step(x, x, torch.zeros(8, 4), torch.zeros(1, 4), torch.zeros(1, 4),
                 state=torch.zeros(1, 8, 4))


def test_conv_argument_errors():
    lib = _lib.load()
    vp = ctypes.c_void_p
    s = _shape()  # DIAG bf16, batch 2, seqlen 64, 64 channels

    def conv(weight=9 << 20, bias=None, x_prev=None, x_last=None, width=4):
        c = _lib.ssm_conv()
        c.weight, c.bias, c.x_prev, c.x_last, c.width = weight, bias, x_prev, x_last, width
        return c

    def call(c):
        return lib.ssm_scan_fwd_conv(vp(1 << 12), vp(2 << 12), vp(3 << 12), vp(4 << 12),
                                     vp(5 << 12), None, None, None,
                                     None if c is None else ctypes.byref(c), None,
                                     vp(6 << 20), None, ctypes.byref(s), None, 0, None)

    assert call(None) == _lib.SSM_ERR_NULL
    assert call(conv(weight=None)) == _lib.SSM_ERR_NULL
    assert call(conv(width=5)) == _lib.SSM_ERR_UNSUPPORTED
    assert call(conv(width=0)) == _lib.SSM_ERR_UNSUPPORTED
    assert call(conv(x_prev=(10 << 20) + 4)) == _lib.SSM_ERR_ALIGN
    # x_last inside x (x is 2*64*64 bf16 = 16 KB at 4 KB): written while x is read
    assert call(conv(x_last=(1 << 12) + 256)) == _lib.SSM_ERR_SHAPE
    # x_last overlapping x_prev
    assert call(conv(x_prev=10 << 20, x_last=(10 << 20) + 16)) == _lib.SSM_ERR_SHAPE
    # the SSD path keeps the convolved input in scratch
    s2 = _shape(mode=1, nheads=8, headdim=64, dstate=128, chunk=64, seqlen=256)
    plain = _ws(s2)
    with_conv = lib.ssm_scan_conv_workspace_size(ctypes.byref(s2))
    assert with_conv >= plain + 2 * 256 * 8 * 64 * 4
    # the diagonal path fuses it and needs no extra scratch
    assert lib.ssm_scan_conv_workspace_size(ctypes.byref(s)) == _ws(s)


def test_step_conv_state_may_be_updated_in_place():
    lib = _lib.load()
    vp = ctypes.c_void_p
    c = _lib.ssm_conv()
    c.weight, c.bias, c.width = 9 << 20, None, 4
    c.x_prev = c.x_last = 10 << 20
    s = _shape(batch=0, seqlen=1)
    # nothing to compute, so only the argument checks run
    assert lib.ssm_step_conv(None, None, vp(3 << 12), None, None, None, None, None,
                             ctypes.byref(c), None, None, ctypes.byref(s), None) == _lib.SSM_OK
    c.x_last = (10 << 20) + 16  # partial overlap is refused
    s = _shape(batch=2, seqlen=1)
    assert lib.ssm_step_conv(vp(1 << 12), vp(2 << 12), vp(3 << 12), vp(4 << 12), vp(5 << 12),
                             None, None, None, ctypes.byref(c), vp(6 << 20), vp(7 << 20),
                             ctypes.byref(s), None) == _lib.SSM_ERR_SHAPE


def test_backward_argument_errors():
    lib = _lib.load()
    vp = ctypes.c_void_p
    s = _shape()
    ptrs = [vp((i + 1) << 12) for i in range(20)]

    def call(shape, **over):
        args = list(ptrs)
        names = ["x", "dt", "A", "B", "C", "D", "z", "dt_bias", "init", "dout", "dfinal", "dx",
                 "ddt", "dA", "dB", "dC", "dD", "dz", "ddt_bias", "dinit"]
        for k, v in over.items():
            args[names.index(k)] = None if v is None else vp(v)
        return lib.ssm_scan_bwd(*args, ctypes.byref(shape), None, 0, None)

    def parts_extra(n, ch, N):
        """The scratch beyond the checkpoints: per time part a local end state, a local
        adjoint (ch x N fp32 each) and a Delta sum per channel (256-byte aligned)."""
        for p in range(1, 17):
            hq = 0 if p == 1 else -(-(ch * p * N * 4) // 256) * 256
            d = 0 if p == 1 else -(-(ch * p * 4) // 256) * 256
            if n == 2 * hq + d:
                return p
        return None

    # SSD mode on the recurrence kernel (fp32, or dstate 256): the state of every (head, p)
    # channel every 4 steps at dstate 128 and 256; with this many channels the sequence is
    # not split into time parts
    ssd = _shape(mode=1, dtype=0, batch=16, nheads=64, headdim=64, dstate=128, chunk=64)
    assert lib.ssm_scan_bwd_workspace_size(ctypes.byref(ssd)) == 16 * (64 // 4) * 64 * 64 * 128 * 4
    ssd256 = _shape(mode=1, batch=16, nheads=64, headdim=64, dstate=256)
    assert lib.ssm_scan_bwd_workspace_size(ctypes.byref(ssd256)) == 16 * (64 // 4) * 64 * 64 * 256 * 4
    # SSD mode on the chunked tensor-core backward (bf16, headdim 64, dstate 64 or 128):
    # chunks of 128 steps; Delta and the cumulative sums, the forward and the adjoint chunk
    # states, y before the gate and the two dy planes
    a256 = lambda n: -(-n // 256) * 256
    for b_, T_, H_, N_ in ((16, 64, 64, 128), (3, 300, 4, 64)):
        tcs = _shape(mode=1, batch=b_, seqlen=T_, nheads=H_, headdim=64, dstate=N_)
        nc = -(-T_ // 128)
        want = (2 * a256(b_ * H_ * nc * 128 * 4) + 2 * a256(b_ * nc * H_ * 64 * N_ * 4)
                + 3 * a256(b_ * T_ * H_ * 64 * 2))
        assert lib.ssm_scan_bwd_workspace_size(ctypes.byref(tcs)) == want
    # few channels: the checkpoints plus the summaries of several time parts
    small = _shape(mode=1, dtype=0, nheads=8, headdim=64, dstate=128, chunk=64)
    ckpt = 2 * (64 // 4) * 8 * 64 * 128 * 4
    n = lib.ssm_scan_bwd_workspace_size(ctypes.byref(small))
    assert n > ckpt and (parts_extra(n - ckpt, 2 * 8 * 64, 128) or 0) > 1
    assert call(small, dB=(15 << 12) + 8) == _lib.SSM_ERR_ALIGN
    assert lib.ssm_scan_bwd_workspace_size(ctypes.byref(_shape(mode=1, dstate=300))) == BAD
    assert call(s, dx=None) == _lib.SSM_ERR_NULL
    assert call(s, dout=None) == _lib.SSM_ERR_NULL
    assert call(s, dA=None) == _lib.SSM_ERR_NULL
    assert call(s, dB=(15 << 12) + 8) == _lib.SSM_ERR_ALIGN
    n = lib.ssm_scan_bwd_workspace_size(ctypes.byref(s))
    ckpt = 2 * (64 // 8) * 64 * 16 * 4   # the state every 8 steps (4 entries per lane)
    assert n >= ckpt and parts_extra(n - ckpt, 2 * 64, 16) is not None


def test_timing_collect_without_launches():
    lib = _lib.load()
    lib.ssm_timing_enable(1)
    assert lib.ssm_timing_collect(None, 0) == 0   # nothing launched, nothing recorded
    lib.ssm_timing_enable(0)
    assert _lib.timing_collect() == {}


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # an SSD shape whose chunk states need far more than the 64 MiB fixed scratch
    shape = _shape(mode=1, batch=1, seqlen=131072, nheads=32, headdim=64, dstate=256, chunk=256)
    assert _ws(shape) > (64 << 20)
    vp = ctypes.c_void_p
    rc = _lib.load().ssm_scan_fwd_noalloc(vp(1 << 12), vp(2 << 12), vp(3 << 12), vp(4 << 12),
                                          vp(5 << 12), None, None, None, vp(6 << 12), None,
                                          ctypes.byref(shape), None)
    assert rc == _lib.SSM_ERR_ALLOC


def test_injected_allocation_failure_is_reported():
    """A failing stream-ordered allocation (injected on the host) surfaces as
    SSM_ERR_ALLOC with nothing queued, for the forward and the backward entry points."""
    lib = _lib.load()
    vp = ctypes.c_void_p
    s = _shape(mode=1, nheads=8, headdim=64, dstate=128, chunk=64, seqlen=256)
    assert _ws(s) > 0
    lib.ssm_inject_alloc_failures(1)
    try:
        assert _call(s) == _lib.SSM_ERR_ALLOC
    finally:
        lib.ssm_inject_alloc_failures(0)
    assert lib.ssm_scan_bwd_workspace_size(ctypes.byref(s)) > 0
    ptrs = [vp((i + 1) << 12) for i in range(20)]
    lib.ssm_inject_alloc_failures(1)
    try:
        assert lib.ssm_scan_bwd(*ptrs, ctypes.byref(s), None, 0, None) == _lib.SSM_ERR_ALLOC
    finally:
        lib.ssm_inject_alloc_failures(0)


def test_tuning_knobs():
    lib = _lib.load()
    assert lib.ssm_tuning_set(99, 1) == _lib.SSM_ERR_UNSUPPORTED
    assert lib.ssm_tuning_set(_lib.SSM_TUNE_BWD_PARTS, -1) == _lib.SSM_ERR_SHAPE
    assert lib.ssm_tuning_get(99) == 0
    s = _shape(mode=1, dtype=0, nheads=8, headdim=64, dstate=128, chunk=64)  # recurrence kernel
    default = lib.ssm_scan_bwd_workspace_size(ctypes.byref(s))
    with _lib.tuned(_lib.SSM_TUNE_BWD_PARTS, 1):
        assert _lib.tuning_get(_lib.SSM_TUNE_BWD_PARTS) == 1
        one_part = lib.ssm_scan_bwd_workspace_size(ctypes.byref(s))
    assert _lib.tuning_get(_lib.SSM_TUNE_BWD_PARTS) == 0
    # one time part needs only the checkpoints; the default plan splits this few-channel
    # shape into several parts, each with its own summaries
    assert one_part < default
    assert lib.ssm_scan_bwd_workspace_size(ctypes.byref(s)) == default
    # the CUDA-core knob moves a bf16 SSD backward from the chunked tensor-core path (its
    # own scratch) to the recurrence kernel
    t = _shape(mode=1, nheads=8, headdim=64, dstate=128)
    tc_ws = lib.ssm_scan_bwd_workspace_size(ctypes.byref(t))
    with _lib.tuned(_lib.SSM_TUNE_SSD_CUDA_CORES, 1):
        rec_ws = lib.ssm_scan_bwd_workspace_size(ctypes.byref(t))
    assert tc_ws != rec_ws and lib.ssm_scan_bwd_workspace_size(ctypes.byref(t)) == tc_ws
    # the FMA-pipe exponential knob exists, round-trips, and leaves the scratch size alone
    d = _shape(mode=0, dtype=1, nheads=512, headdim=1, dstate=16, batch=8, seqlen=1024)
    diag_ws = _ws(d)
    for px in (1, 2):
        with _lib.tuned(_lib.SSM_TUNE_DIAG_EXP_POLY, px):
            assert _lib.tuning_get(_lib.SSM_TUNE_DIAG_EXP_POLY) == px
            assert _ws(d) == diag_ws
    assert _lib.tuning_get(_lib.SSM_TUNE_DIAG_EXP_POLY) == 0


def test_complex_mode_shapes_and_unsupported_entry_points():
    lib = _lib.load()
    vp = ctypes.c_void_p
    cd = dict(mode=2, nheads=64, dstate=16)
    assert _ws(_shape(**cd)) != BAD
    assert _ws(_shape(mode=2, nheads=64, dstate=33)) == BAD          # at most 32 complex entries
    assert _ws(_shape(mode=2, nheads=64, dstate=2)) == BAD           # bf16 rows: 16-byte multiples
    assert _ws(_shape(mode=2, dtype=0, nheads=64, dstate=2)) != BAD  # fp32: 2 x 2 x 4 bytes
    assert _ws(_shape(mode=2, nheads=64, dstate=16, headdim=2)) == BAD
    assert _call(_shape(mode=2, nheads=64, dstate=40)) == _lib.SSM_ERR_UNSUPPORTED
    # few channels: the sequence is split into segments, with their summaries as scratch
    assert _ws(_shape(mode=2, nheads=64, dstate=16, seqlen=4096)) > 0
    s = _shape(**cd)
    assert lib.ssm_scan_conv_workspace_size(ctypes.byref(s)) == BAD
    assert lib.ssm_scan_bwd_workspace_size(ctypes.byref(s)) == BAD
    assert _step(_shape(seqlen=1, **cd)) == _lib.SSM_ERR_UNSUPPORTED
    ptrs = [vp((i + 1) << 12) for i in range(20)]
    assert lib.ssm_scan_bwd(*ptrs, ctypes.byref(s), None, 0, None) == _lib.SSM_ERR_UNSUPPORTED
    c = _lib.ssm_conv()
    c.weight, c.bias, c.x_prev, c.x_last, c.width = 9 << 20, None, None, None, 4
    assert lib.ssm_scan_fwd_conv(vp(1 << 12), vp(2 << 12), vp(3 << 12), vp(4 << 12), vp(5 << 12),
                                 None, None, None, ctypes.byref(c), None, vp(6 << 20), None,
                                 ctypes.byref(s), None, 0, None) == _lib.SSM_ERR_UNSUPPORTED


def test_bounds_check_entry_points_without_checks():
    """The normal build has no store checks: it says so, and the bounds self-test is
    refused before any launch."""
    lib = _lib.load()
    if os.environ.get("SSM_LIB_PATH"):
        pytest.skip("another library is loaded")
    assert lib.ssm_bounds_check_enabled() == 0
    assert lib.ssm_selftest_bounds(None, 16, 1, None) == _lib.SSM_ERR_UNSUPPORTED
    assert lib.ssm_strerror(_lib.SSM_ERR_BOUNDS).decode().startswith("a store address")


def test_bounds_checked_library_exports_and_host_checks():
    """libssmscan_bc.so (built with -DSSM_BOUNDS_CHECK) exports the same symbols, reports
    its checks, and rejects a NULL or malformed self-test before any launch."""
    from selective_state_space_143_b300 import build as _build
    path = _build.OUT_BC
    if not os.path.exists(path):
        pytest.skip("bounds-checked library not built (build.py --bounds-check)")
    bc = ctypes.CDLL(path)
    for name in _lib.EXPORTED:
        assert hasattr(bc, name), name
    bc.ssm_bounds_check_enabled.restype = ctypes.c_int
    bc.ssm_selftest_bounds.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64, ctypes.c_void_p]
    bc.ssm_selftest_bounds.restype = ctypes.c_int
    assert bc.ssm_bounds_check_enabled() == 1
    assert bc.ssm_selftest_bounds(None, 16, 1, None) == _lib.SSM_ERR_NULL
    assert bc.ssm_selftest_bounds(ctypes.c_void_p(0x1000), 16, -1, None) == _lib.SSM_ERR_SHAPE
    assert bc.ssm_selftest_bounds(ctypes.c_void_p(0x1000), 15, 1, None) == _lib.SSM_ERR_SHAPE
