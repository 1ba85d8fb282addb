"""ctypes view of libssmscan.so (the C ABI declared in include/ssm_scan.h).

Argument marshalling only: no arithmetic of the scan happens in Python.  The
library must be present (or buildable with nvcc); there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

SSM_OK = 0
SSM_ERR_NULL = 1
SSM_ERR_SHAPE = 2
SSM_ERR_DTYPE = 3
SSM_ERR_ALIGN = 4
SSM_ERR_UNSUPPORTED = 5
SSM_ERR_ALLOC = 6
SSM_ERR_CUDA = 7
SSM_ERR_TIMEOUT = 8
SSM_ERR_BOUNDS = 9

SSM_MODE_DIAG = 0
SSM_MODE_SSD = 1
SSM_MODE_CDIAG = 2
SSM_F32 = 0
SSM_BF16 = 1

# Every function declared in include/ssm_scan.h.
EXPORTED = ("ssm_scan_fwd", "ssm_scan_fwd_ws", "ssm_scan_workspace_size", "ssm_scan_fwd_noalloc",
            "ssm_scan_fwd_state", "ssm_step", "ssm_scan_fwd_conv", "ssm_scan_conv_workspace_size",
            "ssm_step_conv", "ssm_scan_bwd", "ssm_scan_bwd_workspace_size", "ssm_timing_enable",
            "ssm_timing_collect", "ssm_device_status", "ssm_selftest_bounded_wait", "ssm_strerror",
            "ssm_kernel_launch_count", "ssm_abi_version", "ssm_tuning_set", "ssm_tuning_get",
            "ssm_inject_alloc_failures", "ssm_bounds_check_enabled", "ssm_selftest_bounds")

SSM_TUNE_DIAG_NPT = 0
SSM_TUNE_SSD_CUDA_CORES = 1
SSM_TUNE_BWD_PARTS = 2
SSM_TUNE_BWD_LPC = 3
SSM_TUNE_DIAG_EXP_POLY = 4


class ssm_shape(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("dtype", ctypes.c_int32), ("batch", ctypes.c_int64),
                ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64), ("headdim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64), ("chunk", ctypes.c_int64),
                ("flags", ctypes.c_uint32)]


class ssm_conv(ctypes.Structure):
    _fields_ = [("weight", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("x_prev", ctypes.c_void_p), ("x_last", ctypes.c_void_p),
                ("width", ctypes.c_int32)]


class ssm_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 64), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


class SsmError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {strerror(status)} (status {status})")
        self.status = status


_lock = threading.Lock()
_lib = None


def path() -> str:
    """The library this process loads: SSM_LIB_PATH if set (another build of the same
    sources, e.g. with different compile-time options), else the in-tree build."""
    return os.environ.get("SSM_LIB_PATH") or _build.OUT


def load() -> ctypes.CDLL:
    """Load (building first if the sources are newer) and declare the C ABI."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if path() == _build.OUT and not _build.up_to_date():
            try:
                _build.build()
            except Exception as exc:  # no nvcc or a compile error: fail loudly
                if not os.path.exists(_build.OUT):
                    raise RuntimeError(
                        "libssmscan.so is missing and could not be built "
                        f"({exc}); run `python -m selective_state_space_143_b300.build`") from exc
        lib = ctypes.CDLL(path())
        vp = ctypes.c_void_p
        fp = ctypes.POINTER(ctypes.c_float)
        sp = ctypes.POINTER(ssm_shape)
        lib.ssm_scan_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sp, vp]
        lib.ssm_scan_fwd.restype = ctypes.c_int
        lib.ssm_scan_fwd_ws.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sp, vp,
                                        ctypes.c_size_t, vp]
        lib.ssm_scan_fwd_ws.restype = ctypes.c_int
        lib.ssm_scan_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sp, vp]
        lib.ssm_scan_fwd_noalloc.restype = ctypes.c_int
        lib.ssm_scan_fwd_state.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sp, vp,
                                           ctypes.c_size_t, vp]
        lib.ssm_scan_fwd_state.restype = ctypes.c_int
        lib.ssm_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sp, vp]
        lib.ssm_step.restype = ctypes.c_int
        cp = ctypes.POINTER(ssm_conv)
        lib.ssm_scan_fwd_conv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, cp, vp, vp, vp, sp, vp,
                                          ctypes.c_size_t, vp]
        lib.ssm_scan_fwd_conv.restype = ctypes.c_int
        lib.ssm_scan_conv_workspace_size.argtypes = [sp]
        lib.ssm_scan_conv_workspace_size.restype = ctypes.c_size_t
        lib.ssm_step_conv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, cp, vp, vp, sp, vp]
        lib.ssm_step_conv.restype = ctypes.c_int
        lib.ssm_scan_bwd.argtypes = [vp] * 20 + [sp, vp, ctypes.c_size_t, vp]
        lib.ssm_scan_bwd.restype = ctypes.c_int
        lib.ssm_scan_bwd_workspace_size.argtypes = [sp]
        lib.ssm_scan_bwd_workspace_size.restype = ctypes.c_size_t
        lib.ssm_timing_enable.argtypes = [ctypes.c_int]
        lib.ssm_timing_enable.restype = None
        lib.ssm_timing_collect.argtypes = [ctypes.POINTER(ssm_kernel_time), ctypes.c_int]
        lib.ssm_timing_collect.restype = ctypes.c_int
        lib.ssm_scan_workspace_size.argtypes = [sp]
        lib.ssm_scan_workspace_size.restype = ctypes.c_size_t
        lib.ssm_strerror.argtypes = [ctypes.c_int]
        lib.ssm_strerror.restype = ctypes.c_char_p
        lib.ssm_kernel_launch_count.argtypes = []
        lib.ssm_kernel_launch_count.restype = ctypes.c_uint64
        lib.ssm_abi_version.argtypes = []
        lib.ssm_abi_version.restype = ctypes.c_int
        lib.ssm_device_status.argtypes = [ctypes.c_int, ctypes.c_void_p]
        lib.ssm_device_status.restype = ctypes.c_int
        lib.ssm_selftest_bounded_wait.argtypes = [ctypes.c_uint32, ctypes.c_void_p]
        lib.ssm_selftest_bounded_wait.restype = ctypes.c_int
        lib.ssm_tuning_set.argtypes = [ctypes.c_int, ctypes.c_int64]
        lib.ssm_tuning_set.restype = ctypes.c_int
        lib.ssm_tuning_get.argtypes = [ctypes.c_int]
        lib.ssm_tuning_get.restype = ctypes.c_int64
        lib.ssm_inject_alloc_failures.argtypes = [ctypes.c_int]
        lib.ssm_inject_alloc_failures.restype = None
        lib.ssm_bounds_check_enabled.argtypes = []
        lib.ssm_bounds_check_enabled.restype = ctypes.c_int
        lib.ssm_selftest_bounds.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64, ctypes.c_void_p]
        lib.ssm_selftest_bounds.restype = ctypes.c_int
        del fp
        _lib = lib
        return lib


def tuning_set(knob: int, value: int) -> None:
    """Set a plan override (ssm_tuning_set); 0 restores the library's own choice."""
    rc = load().ssm_tuning_set(int(knob), int(value))
    if rc != SSM_OK:
        raise SsmError(rc, "ssm_tuning_set")


def tuning_get(knob: int) -> int:
    return int(load().ssm_tuning_get(int(knob)))


class tuned:
    """Context manager: ``with tuned(SSM_TUNE_BWD_PARTS, 8): ...`` sets a plan override
    for the block and restores the previous setting afterwards."""

    def __init__(self, knob: int, value: int):
        self.knob, self.value, self.prev = knob, value, 0

    def __enter__(self):
        self.prev = tuning_get(self.knob)
        tuning_set(self.knob, self.value)
        return self

    def __exit__(self, *exc):
        tuning_set(self.knob, self.prev)
        return False


def strerror(status: int) -> str:
    return load().ssm_strerror(int(status)).decode()


def launch_count() -> int:
    return int(load().ssm_kernel_launch_count())


def timing_enable(on: bool) -> None:
    """Bracket every library launch with CUDA events on its stream (see ssm_timing_enable)."""
    load().ssm_timing_enable(1 if on else 0)


def timing_collect() -> dict:
    """{kernel name: (launches, total ms)} since the last collect; clears the records."""
    buf = (ssm_kernel_time * 64)()  # the library has far fewer distinct kernels
    n = load().ssm_timing_collect(buf, 64)
    if n < 0:
        raise SsmError(-n, "ssm_timing_collect")
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms))
            for i in range(min(n, 64))}
