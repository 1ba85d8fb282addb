#!/usr/bin/env python3
"""Benchmark of the B300 selective-scan library.

One step = one ``ssm_scan_fwd`` call (the whole hot path: softplus discretisation,
decay and input terms, the scan, skip term, gate, store) over one batch of the
workload's synthetic inputs, which are resident in HBM before timing starts.  L2
is flushed (a 256 MB write) before every timed step; each step is bracketed by CUDA
events on the stream the library launches on.

Prints ONE JSON line (rank 0).  Under torchrun every rank runs the same workload
on its own GPU with no collective on the data path (weak scaling); ``value`` is the
total token-channels of all ranks divided by the slowest rank's time.

``--impl reference`` times the fp64 CPU oracle instead (host cores, rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SSM scan Gtoken·ch/s and % of HBM / tensor roofline, 1 B300, vs CPU oracle"
UNIT = "Gtoken·ch/s"
L2_FLUSH_BYTES = 256 << 20

DESCRIPTIONS = {
    "c0": "Mamba-1 selective scan (diagonal A), fp32, batch 1 x L 256 x d_inner 64, N 16, D=1",
    "c1": "Mamba-1 block scan (diagonal A), bf16 in / fp32 state, batch 8 x L 1024 x d_inner 512, "
          "N 16, dt_bias, D, SiLU(z) gate",
    "c2": "Mamba-1 scan at 3B-layer width, bf16 in / fp32 state, batch 4 x L 8192 x d_inner 5120, "
          "N 16, dt_bias, D, SiLU(z) gate, final_state",
    "c3": "Mamba-2 SSD scan (scalar A per head), bf16, batch 4 x L 8192, 64 heads x 64, N 128, "
          "1 group, chunk 256, D",
    "c4": "Mamba-2 SSD long sequence, bf16, batch 1 x L 131072, 32 heads x 64, N 256, 1 group, "
          "chunk 256, D, final_state",
    "cx1": "complex diagonal A (the rotating state update read for Mamba-3) at c1's shape, bf16, "
           "batch 8 x L 1024 x d_inner 512, N 16 complex, dt_bias, D, SiLU(z) gate",
    "cx2": "complex diagonal A at c2's shape, bf16, batch 4 x L 8192 x d_inner 5120, N 16 complex, "
           "dt_bias, D, SiLU(z) gate, final_state",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c4", choices=sorted(DESCRIPTIONS),
                    help="the timed workload (default c4, the largest by token-channels)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload block (c0..c4) of the forward scan line")
    ap.add_argument("--chunk", type=int, default=None, help="override the workload's chunk")
    ap.add_argument("--seqlen", type=int, default=None,
                    help="override the workload's sequence length (reduced cases for profiling; "
                         "not a bench line of the named workload)")
    ap.add_argument("--quick", action="store_true",
                    help="skip the clock soak, CPU baseline and end-to-end legs (profiling runs)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--conv", action="store_true",
                    help="put the width-4 causal depthwise convolution + SiLU ahead of the scan")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (ssm_scan_bwd, diagonal mode) of the workload")
    ap.add_argument("--decode", action="store_true",
                    help="time single-token recurrent steps (ssm_step) at the workload's widths")
    ap.add_argument("--decode-batch", type=int, default=0,
                    help="sequences decoded per step (0: enough for a 256 MB carried state)")
    ap.add_argument("--tune", action="append", default=[], metavar="KNOB=VALUE",
                    help="plan override through ssm_tuning_set, e.g. DIAG_EXP_POLY=1 "
                         "(SSM_TUNE_<KNOB>; recorded in the line's config)")
    return ap.parse_args()


TUNING: dict = {}


def emit(line: dict) -> None:
    """Print one JSON result line; plan overrides in force go into its config."""
    if TUNING and isinstance(line.get("config"), dict):
        line["config"]["tuning"] = dict(TUNING)
    print(json.dumps(line), flush=True)


def apply_tuning(specs) -> None:
    from selective_state_space_143_b300 import _lib
    for spec in specs:
        name, _, value = spec.partition("=")
        knob = getattr(_lib, "SSM_TUNE_" + name.strip().upper(), None)
        if knob is None or not value.strip().lstrip("-").isdigit():
            raise SystemExit(f"--tune {spec}: expected KNOB=VALUE with KNOB one of the SSM_TUNE_* names")
        _lib.tuning_set(knob, int(value))
        TUNING["SSM_TUNE_" + name.strip().upper()] = int(value)


# ---------------------------------------------------------------------------- helpers

def algorithmic_bytes(w) -> int:
    """Bytes the method must move: inputs, outputs, parameters, final state."""
    E = 2 if w.dtype == "bf16" else 4
    b, T, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    per_tok_ch = (2 + (1 if w.gate else 0)) * E  # x, out, z (dt below)
    nbytes = b * T * H * P * per_tok_ch
    nbytes += b * T * H * E                      # dt: per channel (diag) or per head (ssd)
    cpl = 2 if w.mode == "cdiag" else 1           # complex: (re, im) pairs
    nbytes += 2 * b * T * G * N * E * cpl        # B, C
    nbytes += (H * N * cpl if w.mode != "ssd" else H) * 4   # A
    nbytes += H * 4 * ((1 if w.d_skip != "none" else 0) + (1 if w.dt_bias else 0))
    if w.final_state:
        nbytes += b * H * P * N * 4 * cpl
    return int(nbytes)


def algorithmic_flops(w) -> float:
    """Tensor-core FLOPs of the SSD chunk form (dense tiles, causal half of Q x Q terms)."""
    if w.mode != "ssd":
        return 0.0
    Q = w.chunk or 256
    nchunks = math.ceil(w.seqlen / Q)
    per_chunk_group = Q * Q * w.dstate               # causal half of 2 Q^2 N (C B^T)
    per_chunk_head = Q * Q * w.headdim + 2 * Q * w.headdim * w.dstate * 2
    return float(w.batch * nchunks * (w.ngroups * per_chunk_group + w.nheads * per_chunk_head))


def backward_flops(w) -> float:
    """Tensor-core FLOPs of the chunked SSD backward (chunk 128): per chunk and head the
    causal halves of M^T dY (Q^2 P), dY X^T (Q^2 P), Z B and Z^T C (Q^2 N each), the
    inter-chunk products B R^T, dY h_in, X R and the adjoint chunk state (4 Q P N), the
    recomputed forward chunk state (Q P N); per chunk and group the causal half of C B^T."""
    if w.mode != "ssd":
        return 0.0
    Q, P, N = 128, w.headdim, w.dstate
    nchunks = math.ceil(w.seqlen / Q)
    mac_head = Q * Q * P / 2 * 2 + Q * Q * N / 2 * 2 + 5 * Q * P * N
    mac_group = Q * Q * N / 2
    return 2.0 * w.batch * nchunks * (w.nheads * mac_head + w.ngroups * mac_group)


def _packed(specs, pinned, dev=None):
    """One contiguous buffer holding tensors of the given {name: (shape, dtype)} at
    256-byte aligned offsets; returns (buffer, {name: view})."""
    offs, total = {}, 0
    for k, (shape, dtype) in specs.items():
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        offs[k] = (total, n)
        total += (n + 255) // 256 * 256
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device=dev)
    if pinned:
        buf = buf.pin_memory()
    views = {k: buf[o:o + n].view(specs[k][1]).view(specs[k][0]) for k, (o, n) in offs.items()}
    return buf, views


def pipelined_e2e(dev, host, run, out_specs, K, dist):
    """End-to-end steps through the public API: each step copies its inputs from pinned
    host memory, runs the library call, and copies its outputs back to pinned host memory.
    The inputs of a step travel as one packed buffer and so do its outputs (one copy each
    way per step); copy-in, compute and copy-out run on three streams with two buffer
    sets, so that one step's copies overlap its neighbours' compute (the way a caller
    streaming batches would drive the library).

    host: {name: CPU tensor or None}; out_specs: {name: (shape, dtype)};
    run(device_inputs, device_outputs) writes the outputs.  Returns (ms per step, max over
    ranks; bytes copied in; bytes copied out)."""
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_specs = {k: (tuple(v.shape), v.dtype) for k, v in host.items() if v is not None}
    hbuf, hviews = _packed(in_specs, pinned=True)
    for k, v in hviews.items():
        v.copy_(host[k])
    dins = [_packed(in_specs, pinned=False, dev=dev) for _ in range(2)]
    douts = [_packed(out_specs, pinned=False, dev=dev) for _ in range(2)]
    houts = [_packed(out_specs, pinned=True) for _ in range(2)]
    h_done = [torch.cuda.Event() for _ in range(2)]
    c_done = [torch.cuda.Event() for _ in range(2)]
    o_done = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        sl = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(c_done[sl])  # step i-2's compute has read this input set
            dins[sl][0].copy_(hbuf, non_blocking=True)
            h_done[sl].record(s_in)
        comp.wait_event(h_done[sl])
        if i >= 2:
            comp.wait_event(o_done[sl])  # step i-2's copy-out has read this output set
        run({k: dins[sl][1].get(k) for k in host}, douts[sl][1])
        c_done[sl].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(c_done[sl])
            houts[sl][0].copy_(douts[sl][0], non_blocking=True)
            o_done[sl].record(s_out)

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    e0.record(s_in)
    for i in range(K):
        step(i)
    s_out.wait_stream(comp)
    e1.record(s_out)
    torch.cuda.synchronize()
    return (max_over_ranks(dist, e0.elapsed_time(e1) / K), hbuf.numel(), houts[0][0].numel())


E2E_NOTE = ("inputs copied from pinned host memory and outputs read back every step, one "
            "packed copy each way; copy-in, compute and copy-out on three streams with two "
            "buffer sets")


def kernel_times(ssm, K, step, flush=None):
    """Per-kernel device times from a second pass of K steps with the library's launch
    events on (kept out of the headline pass: the events add a gap between kernels)."""
    ssm._lib.timing_collect()
    ssm._lib.timing_enable(True)
    for i in range(K):
        if flush is not None:
            flush.zero_()
        step(i)
    torch.cuda.synchronize()
    ssm._lib.timing_enable(False)
    return ssm._lib.timing_collect()


def kernel_roofline(kt, nbytes, calls, peak_gbs, peak_kind, whole):
    """Roofline of the dominant kernel from the library's launch timing ``kt``
    ({name: (launches, total ms)} over K steps of the same workload): the call's
    algorithmic bytes, all of which that kernel reads or writes, over its average
    event-timed duration."""
    if not kt:
        return whole
    name, (n, ms) = max(kt.items(), key=lambda kv: kv[1][1])
    avg_ms = ms / max(n, 1)
    per_call = n / max(calls, 1)  # launches of that kernel per call
    achieved = nbytes / per_call / (avg_ms * 1e-3) / 1e9
    total = sum(v[1] for v in kt.values())
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak_gbs, "unit": "GB/s",
            "frac": achieved / peak_gbs, "traffic": None, "kernel": name,
            "kernel_avg_us": avg_ms * 1e3, "algorithmic_bytes_per_launch": int(nbytes / per_call),
            "peak_source": peak_kind,
            "kernels": {k: {"launches": v[0], "avg_us": 1e3 * v[1] / max(v[0], 1),
                            "share": v[1] / total} for k, v in kt.items()},
            "call": whole}
    return roof


# DRAM traffic per launch of a kernel (dram__bytes_read.sum + dram__bytes_write.sum) comes
# from profiles/dram_traffic.json: one entry per (bench mode, workload, kernel) with the
# ncu command it was read from and a digest of the library sources at capture time.  An
# entry counts only while the sources are unchanged; otherwise the traffic is null.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
CSRC = os.path.join(ROOT, "selective_state_space_143_b300", "csrc")


def sources_digest() -> str:
    """sha256 over the library's kernel sources (every file under csrc/, sorted)."""
    import hashlib
    h = hashlib.sha256()
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(f.encode())
            with open(os.path.join(CSRC, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()


def traffic_entry(key):
    try:
        with open(TRAFFIC_FILE) as f:
            entries = json.load(f)
    except (OSError, ValueError):
        return None, "no capture file"
    digest = sources_digest()
    for e in entries:
        if (e.get("mode"), e.get("workload"), e.get("kernel")) == key:
            if e.get("sources_sha256") != digest:
                return None, "the kernel sources changed since the capture"
            return int(e["bytes_per_launch"]), e.get("command", "")
    return None, "no capture of this kernel and workload"


def with_traffic(roof, key):
    t, how = traffic_entry(key + (roof.get("kernel"),))
    roof["traffic"] = t
    roof["traffic_source"] = (f"ncu capture (bytes per launch): {how}" if t is not None else how)
    return roof


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock and throttle-reason sampling in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.strip().split(",") for r in self.file.read().splitlines() if r.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return dist, world, rank, local
    return None, 1, 0, local


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------- CPU oracle

def oracle_sample(w, inp, seconds: float, max_reps: int = 1000, conv=None):
    """Time the oracle on whole channels of the workload until ``seconds`` pass.
    Returns (token-channels processed, elapsed seconds, threads, description, last) with
    ``last`` = (selected flat channels, oracle out of the last call) for a parity check.
    With ``conv`` (weight, bias) each call also runs the oracle's convolution over the
    input."""
    import oracle
    nch = w.batch * w.d_inner
    per_channel = w.seqlen

    def run(sel):
        x = inp["x"]
        if conv is not None:
            x, _ = oracle.conv_silu(x, conv["weight"], conv["bias"])
        fn = oracle.scan_complex if w.mode == "cdiag" else oracle.scan
        out, _ = fn(x, inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                    inp["dt_bias"], select=sel)
        return out

    # pick a channel block sized to ~1 s per call (at most the time budget)
    t0 = time.perf_counter()
    probe = np.arange(min(nch, 16))
    run(probe)
    dt_probe = max(time.perf_counter() - t0, 1e-4)
    per_call = int(min(nch, max(16, probe.size * min(1.0, seconds) / dt_probe)))
    done, elapsed, reps = 0, 0.0, 0
    rng = np.random.default_rng(0)
    last = None
    while (elapsed < seconds and reps < max_reps) or reps == 0:
        sel = np.sort(rng.choice(nch, per_call, replace=False)) if per_call < nch else np.arange(nch)
        t0 = time.perf_counter()
        out = run(sel)
        elapsed += time.perf_counter() - t0
        done += sel.size * per_channel
        reps += 1
        last = (sel, out)
    desc = (f"{reps} oracle calls of {per_call} whole channels (of {nch}) x L {w.seqlen}, "
            f"fp64, OpenMP over channels")
    return done, elapsed, oracle.max_threads(), desc, last


def channel_view(a, mode):
    """(b, T, H[, P]) -> (b*H*P, T), the oracle's flat channel order."""
    if mode != "ssd":
        return a.transpose(0, 2, 1).reshape(-1, a.shape[1])
    return a.transpose(0, 2, 3, 1).reshape(-1, a.shape[1])


def parity_of(w, gpu_out, last):
    """Error measures of the GPU output against the oracle on the sampled channels."""
    import oracle
    sel, ref = last
    y = channel_view(gpu_out, w.mode)[sel]
    r = channel_view(ref, w.mode)[sel]
    rep = oracle.error_report(y, r)
    tol = 1e-4 if w.dtype == "f32" else 2e-2
    return {**{k: float(f"{v:.4g}") for k, v in rep.items()}, "tolerance": tol,
            "pass": bool(rep["gated"] <= tol), "channels": int(len(sel)),
            "what": "out on the oracle sample's channels, whole sequences"}


# ---------------------------------------------------------------------------- arms

def host_inputs(w):
    from selective_state_space_143_b300.inputs import make_inputs
    return make_inputs(w)


def run_reference(args, w):
    dist, world, rank, _ = dist_setup()
    if rank != 0:
        barrier(dist)
        return 0
    inp = host_inputs(w)
    import oracle
    nch = w.batch * w.d_inner
    # per step: a bounded sample of whole channels (about 1 s of CPU work)
    done_probe, el_probe, threads, _, _ = oracle_sample(w, inp, seconds=0.5, max_reps=1)
    per_sec = done_probe / el_probe / w.seqlen  # channels per second
    per_step = int(max(1, min(nch, per_sec * 1.0)))
    rng = np.random.default_rng(1)
    times, units = [], 0
    for i in range(args.warmup + args.steps):
        sel = np.sort(rng.choice(nch, per_step, replace=False))
        t0 = time.perf_counter()
        fn = oracle.scan_complex if w.mode == "cdiag" else oracle.scan
        fn(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["dt_bias"],
           select=sel)
        el = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(el)
            units += per_step * w.seqlen
    total = sum(times)
    value = units / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: {DESCRIPTIONS[w.name]}",
                   "sample_per_step": f"{per_step} of {nch} whole channels"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{per_step} whole channels x L {w.seqlen} per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    emit(line)
    barrier(dist)
    return 0


def measure_forward(args, w, dev, dist, rank, world, K, warmup, headline, cpu_seconds):
    """Time ssm_scan_fwd on workload ``w``: K steps after ``warmup``, L2 flushed before
    each; the library's per-kernel event times from a second pass; roofline of the
    dominant kernel and of the whole call.  With ``headline`` also the clock record
    during a load soak and the end-to-end leg.  On rank 0 the oracle baseline on a
    bounded sample, and the parity of the GPU output on that sample."""
    import selective_state_space_143_b300 as ssm
    chunk = w.chunk if args.chunk is None or not headline else args.chunk
    inp = host_inputs(w)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    out = torch.empty_like(d["x"])
    st_shape = {"diag": (w.batch, w.nheads, w.dstate), "cdiag": (w.batch, w.nheads, w.dstate, 2)}.get(
        w.mode, (w.batch, w.nheads, w.headdim, w.dstate))
    fs = torch.empty(st_shape, device=dev, dtype=torch.float32) if w.final_state else None
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    conv, cp = {}, None
    if args.conv:
        from selective_state_space_143_b300.inputs import conv_params
        cp = conv_params(w.d_inner, 4, seed=w.seed)
        conv = dict(conv_weight=cp["weight"].to(dev), conv_bias=cp["bias"].to(dev))

    def step():
        ssm.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                     out=out, final_state=fs, chunk=chunk, stream=stream, **conv)

    for _ in range(max(warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device())
    soak = headline and not args.quick
    if soak:
        clocks.start()
        # keep the GPU busy for about a second so that the clock samples see load
        t_end = time.perf_counter() + 1.0
        while time.perf_counter() < t_end:
            for _ in range(20):
                step()
            torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier(dist)
    torch.cuda.synchronize()
    n0 = ssm.launch_count()
    # Hold the GPU in a spin kernel while the K steps are queued, so that the event
    # pairs time device execution only, not the host's launch rate.
    torch.cuda._sleep(int(min(2e9, 2e6 + K * 4e5)))
    for i in range(K):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    launches = ssm.launch_count() - n0
    kt = kernel_times(ssm, K, lambda i: step(), flush)
    barrier(dist)
    ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms_step = max_over_ranks(dist, sum(ms) / K)
    clk = clocks.stop() if soak else {"sm_mhz": None, "sm_max_mhz": None,
                                     "reasons": ["not sampled (--quick)"]}
    units = w.token_channels * world
    value = units / (ms_step * 1e-3) / 1e9

    # ---- roofline of the call (all its kernels) against the measured peaks
    peaks, peak_kind = measured_peaks()
    nbytes = algorithmic_bytes(w) + (w.d_inner * 5 * 4 if args.conv else 0)
    hbm_gbs = nbytes / (ms_step * 1e-3) / 1e9
    whole = {"achieved": hbm_gbs, "frac": hbm_gbs / peaks["hbm_gbs"], "unit": "GB/s",
             "ms": ms_step, "algorithmic_bytes": nbytes,
             "what": "all kernels of one ssm_scan_fwd call"}
    roof = kernel_roofline(kt, nbytes, K, peaks["hbm_gbs"], peak_kind, whole)
    roof = with_traffic(roof, ("conv" if args.conv else "scan",
                               w.name if args.seqlen is None else f"{w.name}@L{w.seqlen}"))
    sm_mhz = float(peaks.get("sm_max_mhz", 2032.0))
    if w.mode == "ssd":
        fl = algorithmic_flops(w)
        roof["tensor_tflops"] = fl / (ms_step * 1e-3) / 1e12
        roof["tensor_frac"] = roof["tensor_tflops"] / peaks["bf16_tflops"]
        roof["tensor_note"] = ("algorithmic FLOPs of the chunk form over the whole call's time, "
                               "against the measured bf16 dense peak")
    elif w.mode == "diag":
        # The diagonal scan needs one exponential per state entry and step; B300's SFU
        # retires 32 ex2 per clock per SM (measured), so its ceiling is
        # SMs x 32 x SM clock.
        nsm = torch.cuda.get_device_properties(dev).multi_processor_count
        sfu_peak = nsm * 32 * sm_mhz * 1e6
        exps = float(w.token_channels * w.dstate)
        t_sfu = roof.get("kernel_avg_us", ms_step * 1e3) * 1e-6
        roof["sfu"] = {"achieved": exps / t_sfu, "peak": sfu_peak, "unit": "exp/s",
                       "frac": exps / t_sfu / sfu_peak,
                       "note": f"one ex2 per state entry and step in the output pass; peak = "
                               f"{nsm} SMs x 32/clk x max SM clock"}

    # ---- end to end through the public API from pinned host buffers
    e2e = None
    if headline and not args.quick:
        specs = {"out": (tuple(out.shape), out.dtype)}
        if fs is not None:
            specs["final_state"] = (tuple(fs.shape), torch.float32)

        def run(dd, oo):
            ssm.scan_fwd(dd["x"], dd["dt"], dd["A"], dd["B"], dd["C"], dd["D"], dd["z"],
                         dd["dt_bias"], out=oo["out"], final_state=oo.get("final_state"),
                         chunk=chunk, stream=torch.cuda.current_stream(dev), **conv)

        e2e_ms, h2d, d2h = pipelined_e2e(dev, inp, run, specs, K, dist)
        e2e = {"value": units / (e2e_ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "how": E2E_NOTE}

    cpu = parity = None
    if rank == 0 and not args.quick:
        done, el, threads, desc, last = oracle_sample(w, inp, cpu_seconds,
                                                      conv=cp if args.conv else None)
        cpu = {"value": done / el / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": desc, "seconds": el}
        step()
        torch.cuda.synchronize()
        parity = parity_of(w, out.float().cpu().numpy(), last)
    res = {"value": value, "ms_per_step": ms_step, "launches": int(launches), "roofline": roof,
           "cpu_baseline": cpu, "parity": parity, "e2e": e2e, "clocks": clk, "chunk": chunk}
    del d, out, fs, flush
    torch.cuda.empty_cache()
    return res


def config_summary(w, r):
    roof = r["roofline"]
    item = {"workload": f"{w.name}: {DESCRIPTIONS[w.name]}", "value": r["value"], "unit": UNIT,
            "ms_per_step": r["ms_per_step"],
            "kernel": roof.get("kernel"), "kernel_avg_us": roof.get("kernel_avg_us"),
            "frac": roof.get("frac"), "achieved_gbs": roof.get("achieved"),
            "traffic": roof.get("traffic"), "call_frac": roof.get("call", {}).get("frac"),
            "cpu_baseline": r["cpu_baseline"], "parity": r["parity"],
            "gpu_launches": r["launches"]}
    if "tensor_frac" in roof:
        item["tensor_frac"] = roof["tensor_frac"]
    if "sfu" in roof:
        item["sfu_frac"] = roof["sfu"]["frac"]
    return item


def run_ours(args, w):
    from selective_state_space_143_b300.inputs import WORKLOADS
    dist, world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    head = measure_forward(args, w, dev, dist, rank, world, args.steps, args.warmup, True,
                           args.cpu_seconds)
    configs = None
    if not args.no_configs and not args.quick and not args.conv and args.seqlen is None:
        configs = {}
        for name in sorted(WORKLOADS):
            if name == w.name:
                configs[name] = config_summary(w, head)
                continue
            wn = WORKLOADS[name]
            r = measure_forward(args, wn, dev, dist, rank, world, 10, 3, False, 3.0)
            configs[name] = config_summary(wn, r)
    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic",
            "config": {"workload": f"{w.name}: {DESCRIPTIONS[w.name]}" +
                                   (", width-4 causal conv1d + SiLU ahead of the scan" if args.conv else "") +
                                   (f", sequence length reduced to {w.seqlen} (profiling case)"
                                    if args.seqlen is not None else ""),
                       "l2": "flushed before every timed step (256 MB write)",
                       "chunk": head["chunk"], "parallelism": f"replicas x{world} (independent batches)"},
            "roofline": head["roofline"], "cpu_baseline": head["cpu_baseline"],
            "parity": head["parity"], "e2e": head["e2e"], "clocks": head["clocks"],
            "gpu_launches": head["launches"],
        }
        if configs is not None:
            line["configs"] = configs
        emit(line)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def decode_workload(args, w):
    """The workload's widths with a serving batch: one token per sequence per step."""
    per_seq = w.nheads * w.headdim * w.dstate * 4
    batch = args.decode_batch or max(1, math.ceil((256 << 20) / per_seq))
    return w.replace(name=w.name, batch=batch, seqlen=1, final_state=False, chunk=0), batch


def decode_bytes(w) -> int:
    """Bytes one decode step must move: the state read and written, the token's inputs
    and output, the parameters."""
    E = 2 if w.dtype == "bf16" else 4
    b, H, P, N, G = w.batch, w.nheads, w.headdim, w.dstate, w.ngroups
    nbytes = 2 * b * H * P * N * 4
    nbytes += b * H * P * (2 + (1 if w.gate else 0)) * E + b * H * E + 2 * b * G * N * E
    nbytes += (H * N if w.mode == "diag" else H) * 4
    nbytes += H * 4 * ((1 if w.d_skip != "none" else 0) + (1 if w.dt_bias else 0))
    return int(nbytes)


def run_decode(args, w0):
    """ssm_step over a batch of carried states; each step depends on the previous one."""
    import selective_state_space_143_b300 as ssm
    from selective_state_space_143_b300.inputs import make_inputs
    dist, world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w, batch = decode_workload(args, w0)
    ntok = 4  # distinct token inputs, used in turn
    wt = w.replace(seqlen=ntok)
    inp = make_inputs(wt)
    diag = w.mode == "diag"

    def token(t, src):
        out = {}
        for k in ("x", "dt", "z"):
            v = src[k]
            out[k] = None if v is None else v[:, t].contiguous()
        for k in ("B", "C"):
            out[k] = src[k][:, t].contiguous()
        for k in ("A", "D", "dt_bias"):
            out[k] = src[k]
        return out

    toks = [{k: (None if v is None else v.to(dev)) for k, v in token(t, inp).items()}
            for t in range(ntok)]
    st_shape = (batch, w.nheads, w.dstate) if diag else (batch, w.nheads, w.headdim, w.dstate)
    gen = torch.Generator().manual_seed(11)
    state0 = torch.randn(st_shape, generator=gen)
    state = state0.to(dev)
    outs = [torch.empty_like(toks[0]["x"]) for _ in range(ntok)]
    stream = torch.cuda.current_stream(dev)

    def step(i):
        d = toks[i % ntok]
        ssm.step(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                 state=state, out=outs[i % ntok], stream=stream)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    if not args.quick:
        clocks.start()
        t_end = time.perf_counter() + 1.0
        while time.perf_counter() < t_end:
            for i in range(50):
                step(i)
            torch.cuda.synchronize()
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier(dist)
    torch.cuda.synchronize()
    n0 = ssm.launch_count()
    torch.cuda._sleep(int(min(2e9, 2e6 + K * 4e5)))
    for i in range(K):
        starts[i].record(stream)
        step(i)
        ends[i].record(stream)
    torch.cuda.synchronize()
    launches = ssm.launch_count() - n0
    kt = kernel_times(ssm, K, step)
    barrier(dist)
    ms_step = max_over_ranks(dist, sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / K)
    clk = clocks.stop() if not args.quick else {"sm_mhz": None, "sm_max_mhz": None,
                                               "reasons": ["not sampled (--quick)"]}
    units = batch * w.nheads * w.headdim * world
    value = units / (ms_step * 1e-3) / 1e9
    peaks, peak_kind = measured_peaks()
    nbytes = decode_bytes(w)
    gbs = nbytes / (ms_step * 1e-3) / 1e9
    whole = {"achieved": gbs, "frac": gbs / peaks["hbm_gbs"], "unit": "GB/s", "ms": ms_step,
             "algorithmic_bytes": nbytes, "what": "one ssm_step call"}
    roof = kernel_roofline(kt, nbytes, K, peaks["hbm_gbs"], peak_kind, whole)
    roof = with_traffic(roof, ("decode", f"{w0.name}/{batch}"))

    cpu = e2e = None
    if not args.quick:
        # end to end: the token's inputs copied in and its output copied out every step
        host = {k: v for k, v in token(0, inp).items() if k not in ("A", "D", "dt_bias")}
        specs = {"out": (tuple(outs[0].shape), outs[0].dtype)}

        def run(dd, oo):
            ssm.step(dd["x"], dd["dt"], toks[0]["A"], dd["B"], dd["C"], toks[0]["D"], dd["z"],
                     toks[0]["dt_bias"], state=state, out=oo["out"],
                     stream=torch.cuda.current_stream(dev))

        e2e_ms, h2d, d2h = pipelined_e2e(dev, host, run, specs, K, dist)
        e2e = {"value": units / (e2e_ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "how": E2E_NOTE}
        if rank == 0:
            import oracle
            # one-token scans from the carried state over whole sequences until the
            # sample time is used up
            t_used, done, reps = 0.0, 0, 0
            seqs = min(batch, 64)
            h0 = state0[:seqs].numpy()
            sub = {k: (None if v is None or k in ("A", "D", "dt_bias") else v[:seqs, :1])
                   for k, v in inp.items()}
            while t_used < args.cpu_seconds and reps < 10000:
                t0 = time.perf_counter()
                oracle.scan(sub["x"], sub["dt"], inp["A"], sub["B"], sub["C"], inp["D"],
                            sub["z"], inp["dt_bias"], initial_state=h0)
                t_used += time.perf_counter() - t0
                done += seqs * w.nheads * w.headdim
                reps += 1
            cpu = {"value": done / t_used / 1e9, "unit": UNIT, "cores": oracle.max_threads(),
                   "kind": "oracle", "seconds": t_used,
                   "sample": f"{reps} one-token oracle scans of {seqs} sequences from a carried state"}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": f"{w0.name}-decode: one token per step for {batch} sequences "
                                   f"at the widths of {w0.name} ({DESCRIPTIONS[w0.name]})",
                       "l2": f"carried state {batch * w.nheads * w.headdim * w.dstate * 4 >> 20} MB "
                             "(larger than L2), not flushed",
                       "parallelism": f"replicas x{world} (independent batches)"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": int(launches),
        }
        emit(line)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def backward_bytes(w) -> int:
    """Bytes the backward pass must move: the forward inputs and dout read, every
    gradient written (fp32)."""
    E = 2 if w.dtype == "bf16" else 4
    b, T, H, N, G = w.batch, w.seqlen, w.nheads, w.dstate, w.ngroups
    P = w.headdim if w.mode == "ssd" else 1                      # channels per head
    na = H if w.mode == "ssd" else H * N                         # entries of A
    nbytes = b * T * H * P * E * (2 + (1 if w.gate else 0))      # x, dout, z
    nbytes += b * T * H * (E + 4)                                # dt, ddt
    nbytes += 2 * b * T * G * N * E                              # B, C
    nbytes += b * T * H * P * 4 * (1 + (1 if w.gate else 0))     # dx, dz
    nbytes += 2 * b * T * G * N * 4                              # dB, dC
    nbytes += 2 * na * 4 + 4 * H * 4                             # A, dA, D, dD, dt_bias, ddt_bias
    nbytes += 2 * b * H * P * N * 4                              # dfinal, dinitial_state
    return int(nbytes)


def run_backward(args, w):
    """ssm_scan_bwd over the workload; one step = one backward call."""
    import selective_state_space_143_b300 as ssm
    dist, world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = host_inputs(w)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    gen = torch.Generator().manual_seed(w.seed + 100)
    dout_h = torch.randn(d["x"].shape, generator=gen).to(d["x"].dtype)
    st_shape = (w.batch, w.nheads) + ((w.headdim,) if w.mode == "ssd" else ()) + (w.dstate,)
    dfin_h = torch.randn(st_shape, generator=gen)
    dout, dfin = dout_h.to(dev), dfin_h.to(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    s = ssm.make_shape(d["x"], d["A"], d["B"])
    ws = torch.empty(max(1, int(ssm._lib.load().ssm_scan_bwd_workspace_size(ctypes_byref(s)))),
                     dtype=torch.uint8, device=dev)

    def step():
        return ssm.scan_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                            dout=dout, dfinal_state=dfin, workspace=ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    if not args.quick:
        clocks.start()
        t_end = time.perf_counter() + 1.0
        while time.perf_counter() < t_end:
            for _ in range(10):
                step()
            torch.cuda.synchronize()
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier(dist)
    torch.cuda.synchronize()
    n0 = ssm.launch_count()
    torch.cuda._sleep(int(min(2e9, 2e6 + K * 4e5)))
    for i in range(K):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    launches = ssm.launch_count() - n0
    kt = kernel_times(ssm, K, lambda i: step(), flush)
    barrier(dist)
    ms_step = max_over_ranks(dist, sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / K)
    clk = clocks.stop() if not args.quick else {"sm_mhz": None, "sm_max_mhz": None,
                                               "reasons": ["not sampled (--quick)"]}
    units = w.token_channels * world
    value = units / (ms_step * 1e-3) / 1e9
    peaks, peak_kind = measured_peaks()
    nbytes = backward_bytes(w)
    gbs = nbytes / (ms_step * 1e-3) / 1e9
    whole = {"achieved": gbs, "frac": gbs / peaks["hbm_gbs"], "unit": "GB/s", "ms": ms_step,
             "algorithmic_bytes": nbytes, "what": "one ssm_scan_bwd call (zeroing + kernel)"}
    roof = kernel_roofline(kt, nbytes, K, peaks["hbm_gbs"], peak_kind, whole)
    roof = with_traffic(roof, ("backward", w.name if args.seqlen is None else f"{w.name}@L{w.seqlen}"))
    sm_mhz = float(peaks.get("sm_max_mhz", 2032.0))
    if "ssd_bwd_chunk_tc" in kt:
        # the chunked tensor-core backward: algorithmic FLOPs of its products over the call
        fl = backward_flops(w)
        roof["tensor_tflops"] = fl / (ms_step * 1e-3) / 1e12
        roof["tensor_frac"] = roof["tensor_tflops"] / peaks["bf16_tflops"]
        roof["tensor_note"] = ("algorithmic FLOPs of the chunked backward's products (causal halves, "
                               "chunk 128) over the whole call's time, against the measured bf16 dense peak")
    else:
        nsm = torch.cuda.get_device_properties(0).multi_processor_count
        exps = 3.0 * w.token_channels * w.dstate  # the decay is formed in three sweeps
        roof["sfu"] = {"achieved": exps / (ms_step * 1e-3), "peak": nsm * 32 * sm_mhz * 1e6,
                       "unit": "exp/s", "frac": exps / (ms_step * 1e-3) / (nsm * 32 * sm_mhz * 1e6),
                       "note": "three exponentials per state entry and step (forward sweep, "
                               f"recompute, reverse); peak = {nsm} SMs x 32/clk x max SM clock"}
    cpu = e2e = None
    if not args.quick:
        host = dict(inp, dout=dout_h, dfinal=dfin_h)
        xs, f32 = tuple(inp["x"].shape), torch.float32
        H, N = w.nheads, w.dstate
        specs = {"dx": (xs, f32), "ddt": (tuple(inp["dt"].shape), f32),
                 "dA": (tuple(inp["A"].shape), f32),
                 "dB": (tuple(inp["B"].shape), f32), "dC": (tuple(inp["C"].shape), f32),
                 "dinitial_state": (st_shape, f32)}
        if inp["D"] is not None:
            specs["dD"] = ((H,), f32)
        if inp["z"] is not None:
            specs["dz"] = (xs, f32)
        if inp["dt_bias"] is not None:
            specs["ddt_bias"] = ((H,), f32)

        def run(dd, oo):
            ssm.scan_bwd(dd["x"], dd["dt"], dd["A"], dd["B"], dd["C"], dd["D"], dd["z"],
                         dd["dt_bias"], dout=dd["dout"], dfinal_state=dd["dfinal"],
                         workspace=ws, stream=torch.cuda.current_stream(dev), grads=oo)

        e2e_ms, h2d, d2h = pipelined_e2e(dev, host, run, specs, K, dist)
        e2e = {"value": units / (e2e_ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "how": E2E_NOTE}
        if rank == 0:
            import oracle
            # the oracle's backward over the first sequence and a block of channels (SSD: of
            # heads)
            nch = min(w.nheads, 64 if w.mode == "diag" else 2)
            sub = {k: (None if v is None else v) for k, v in inp.items()}
            cut = lambda t: t[:1, :, :nch].contiguous()
            sl = dict(x=cut(sub["x"]), dt=cut(sub["dt"]), A=sub["A"][:nch], B=sub["B"][:1],
                      C=sub["C"][:1], D=None if sub["D"] is None else sub["D"][:nch],
                      z=None if sub["z"] is None else cut(sub["z"]),
                      dt_bias=None if sub["dt_bias"] is None else sub["dt_bias"][:nch])
            t_used, reps = 0.0, 0
            while t_used < args.cpu_seconds and reps < 1000:
                t0 = time.perf_counter()
                oracle.scan_bwd(**sl, dout=dout_h[:1, :, :nch], dfinal=dfin_h[:1, :nch])
                t_used += time.perf_counter() - t0
                reps += 1
            per_head = w.headdim if w.mode == "ssd" else 1
            cpu = {"value": reps * w.seqlen * nch * per_head / t_used / 1e9, "unit": UNIT,
                   "cores": 1, "kind": "oracle", "seconds": t_used,
                   "sample": f"{reps} oracle backward passes over 1 sequence x {nch * per_head} "
                             f"channels x L {w.seqlen} (fp64, one thread)"}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": f"{w.name}-backward: gradients of every input of "
                                   f"{DESCRIPTIONS[w.name]}, from dout and dfinal_state",
                       "l2": "flushed before every timed step (256 MB write)",
                       "parallelism": f"replicas x{world} (independent batches)"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": int(launches),
        }
        emit(line)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def ctypes_byref(s):
    import ctypes
    return ctypes.byref(s)


def main():
    args = parse()
    from selective_state_space_143_b300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.seqlen is not None:
        w = w.replace(seqlen=args.seqlen)
    if args.impl == "reference":
        return run_reference(args, w)
    apply_tuning(args.tune)
    if args.decode:
        return run_decode(args, w)
    if args.backward:
        return run_backward(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
