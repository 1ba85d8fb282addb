"""Build libssmscan.so in-tree with nvcc for sm_103a.

Usage: ``python -m selective_state_space_143_b300.build [--force] [-v] [--bounds-check]``.
Each .cu under csrc/ is compiled to an object, then linked into one shared library
with the CUDA runtime linked statically, so the library loads without a GPU.
``--bounds-check`` builds the same sources with -DSSM_BOUNDS_CHECK into
libssmscan_bc.so: every kernel store checks its address against its buffer and
records SSM_ERR_BOUNDS instead of writing outside it (load it through SSM_LIB_PATH).
"""
from __future__ import annotations

import argparse
import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT = os.path.join(HERE, "libssmscan.so")
BUILD_DIR = os.path.join(HERE, "_build")
OUT_BC = os.path.join(HERE, "libssmscan_bc.so")
BUILD_DIR_BC = os.path.join(HERE, "_build_bc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    out = sources()
    for d in (CSRC, INCLUDE):
        out += [os.path.join(d, f) for f in os.listdir(d) if f.endswith((".cuh", ".h"))]
    return out


def up_to_date(out: str = OUT) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          out: str = OUT, build_dir: str = BUILD_DIR) -> str:
    """Compile every .cu under csrc/ and link ``out``; ``extra`` adds nvcc flags."""
    if not force and up_to_date(out):
        return out
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    objs, cmds = [], []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *FLAGS, *(extra or []), "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
            print(" ".join(cmd), flush=True)
        cmds.append(cmd)
        objs.append(obj)
    # the translation units are independent: compile them concurrently
    workers = max(1, min(len(cmds), os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as pool:
        for f in [pool.submit(subprocess.run, c, check=True) for c in cmds]:
            f.result()
    tmp = out + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true", help="print ptxas register/smem usage")
    ap.add_argument("--bounds-check", action="store_true",
                    help="build libssmscan_bc.so with -DSSM_BOUNDS_CHECK")
    args = ap.parse_args(argv)
    if args.bounds_check:
        print(build_bounds_checked(force=args.force, verbose=args.verbose))
    else:
        print(build(force=args.force, verbose=args.verbose))
    return 0


def build_bounds_checked(force: bool = False, verbose: bool = False) -> str:
    """The bounds-checked library (stores checked against their buffers)."""
    return build(force=force, verbose=verbose, extra=["-DSSM_BOUNDS_CHECK"], out=OUT_BC,
                 build_dir=BUILD_DIR_BC)


if __name__ == "__main__":
    sys.exit(main())
