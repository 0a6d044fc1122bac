"""Benchmark of the head-wise RNN recurrence (forward; forward+backward for the
training workload) on GB300.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole recurrence over one synthetic batch of the
workload (default: LSTM, 12 heads x 64, B=16, T=1024, bf16 inputs / fp32
state), inputs resident in HBM.  L2 is flushed (a write larger than L2)
before every timed step, outside the timed events.  ``value`` is recurrent
TFLOP/s = 2*B*NH*Dh*G*Dh*T / step time (backward counts twice that), summed
over ranks (weak scaling: every rank runs its own independent batch).
``e2e`` repeats the measurement through the same C ABI with pinned host
buffers: host->device transfer of the step's inputs and device->host transfer
of h_seq inside the timed region (forward workloads: rnn_fwd_host's automatic
mode -- staged copies pipelined over eight time chunks, or, for a Wx stream
under 64 GB/s, the kernel reading and writing the mapped host buffers; the
training workload: double-buffered copies).  ``--impl reference`` times the fp64 CPU
oracle (the reference arm) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import atexit
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import WORKLOADS, workload_inputs  # noqa: E402

DEFAULT_WORKLOAD = "lstm_bf16_12x64_b16_t1024"
METRIC = "fwd recurrent TFLOP/s & steps/s, LSTM 12x64 heads B=16 T=1024; % roofline"
GATES = {"lstm": 4, "gru": 3, "slstm": 4}


def flops_per_step(w):
    f = 2.0 * w["B"] * w["NH"] * w["Dh"] * GATES[w["cell"]] * w["Dh"] * w["T"]
    return f * (3.0 if w["backward"] else 1.0)  # bwd: dh_rec + dR contractions


def algorithmic_bytes_fwd(w):
    """Bytes the forward must move: Wx in, h_seq out, R, bias, final states."""
    e = 2 if w["dtype"] == "bf16" else 4
    G, T, B, NH, Dh = GATES[w["cell"]], w["T"], w["B"], w["NH"], w["Dh"]
    per_step = B * NH * G * Dh * e + B * NH * Dh * e
    once = NH * Dh * G * Dh * e + NH * G * Dh * 4 + 2 * B * NH * Dh * 4
    if w["backward"]:  # training stash written: gate activations + c_t, fp32
        per_step += B * NH * Dh * 5 * 4
    return per_step, per_step * T + once


def algorithmic_bytes_bwd(w):
    """Bytes the backward must move: dh_seq, the training stash and h_seq in,
    dWx out, R in, dR / db out (once)."""
    e = 2 if w["dtype"] == "bf16" else 4
    G, T, B, NH, Dh = GATES[w["cell"]], w["T"], w["B"], w["NH"], w["Dh"]
    nstash = 6 if w["cell"] == "slstm" else 5
    per_step = B * NH * Dh * e + B * NH * Dh * nstash * 4 + B * NH * Dh * e + B * NH * G * Dh * e
    once = NH * Dh * G * Dh * (e + 4) + NH * G * Dh * 4 + 3 * B * NH * Dh * 4
    return per_step * T + once


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples (every 50 ms) of the SM clock and throttle reasons of
    this process's GPU while the steps run.

    Every GPU is queried with its UUID and the lines of ours are kept (the UUID
    torch reports, matched without its "GPU-" prefix; with a single visible
    GPU its line is taken).  nvidia-smi needs a few hundred ms to start, so the
    sampler is started before the warm-up and ``wait_first`` holds the timing
    back until the first sample has arrived; samples cover the untimed
    clock soak and the timed region, both of which run the measured steps."""

    Q = ("uuid,clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = str(uuid).lower().removeprefix("gpu-")
        self.proc = None
        self.lines = []
        self.first = threading.Event()

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())
            self.first.set()

    def wait_first(self, timeout=5.0):
        if self.proc is not None:
            self.first.wait(timeout)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def _ours(self):
        rows = [[x.strip() for x in ln.split(",")] for ln in self.lines]
        rows = [r for r in rows if len(r) >= 8]
        uuids = {r[0].lower().removeprefix("gpu-") for r in rows}
        if self.uuid in uuids:
            return [r for r in rows if r[0].lower().removeprefix("gpu-") == self.uuid]
        return rows if len(uuids) == 1 else []

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for parts in self._ours():
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_rate(w, d, budget_s=10.0):
    """fp64 oracle forward (+backward) on the host cores: TFLOP/s over a bounded
    sample.  Also returns the threads it kept busy on average: process CPU time
    (all threads, numpy's BLAS included) over wall time."""
    from oracle import rnn_oracle as O
    f_full = flops_per_step(w)
    c0 = time.process_time()
    t0 = time.perf_counter()
    reps = 0
    while True:
        if w["backward"]:
            O.backward(w["cell"], d["Wx"], d["R"], d["b"], d["h0"], d["c0"], dh_seq=d["dh"])
        else:
            O.forward(w["cell"], d["Wx"], d["R"], d["b"], d["h0"], d["c0"], d["n0"], d["m0"])
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 1000:
            break
    busy = (time.process_time() - c0) / max(el, 1e-9)
    return f_full * reps / el / 1e12, reps, el, busy


SINGLE_THREAD_ENV = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS",
                     "BLIS_NUM_THREADS", "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS")


def oracle_rate_single_thread(workload, max_T, budget_s):
    """The oracle's rate on one host thread: a child process whose BLAS thread
    pools are limited to one before numpy loads (no GPU work in it)."""
    env = dict(os.environ)
    for k in SINGLE_THREAD_ENV:
        env[k] = "1"
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "from synth import workload_inputs; "
            "w = bench.sample_workload(dict(bench.WORKLOADS[%r]), %d); "
            "d = workload_inputs(%r, T=w['T']); "
            "r, reps, el, busy = bench.oracle_rate(w, d, budget_s=%r); "
            "print(json.dumps({'value': r, 'reps': reps, 'seconds': el, 'busy': busy}))"
            % (ROOT, workload, max_T, workload, budget_s))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    if r.returncode != 0:
        return None
    return json.loads(r.stdout.strip().splitlines()[-1])


def threads_used(busy):
    """Threads the oracle kept busy, rounded (at least 1), for ``cores``."""
    return max(1, int(round(busy)))


def sample_workload(w, max_T):
    """Same workload with the time axis cut to max_T steps (CPU sample)."""
    s = dict(w)
    s["T"] = min(w["T"], max_T)
    return s


def run_reference(args, w, rank):
    if rank != 0:
        return None
    # bounded sample: the full batch/head shape, time axis cut so a step is ~seconds
    sw = sample_workload(w, 256 if w["Dh"] <= 256 else 64)
    d = workload_inputs(args.workload, T=sw["T"])
    for _ in range(args.warmup):
        oracle_rate(sw, d, budget_s=0.0)
    times, busy = [], []
    for _ in range(args.steps):
        rate, reps, el, b = oracle_rate(sw, d, budget_s=0.0)
        times.append(el)
        busy.append(b)
    t = sum(times) / len(times)
    value = flops_per_step(sw) / t / 1e12
    cores = threads_used(statistics.mean(busy))
    sample = (f"{args.workload} with T cut to {sw['T']} steps, one oracle pass per step "
              f"(mean of {args.steps}); {statistics.mean(busy):.2f} threads busy on average "
              f"of {os.cpu_count()} host cores")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, **{k: w[k] for k in ("cell", "NH", "Dh", "B", "T")},
                       "sample_T": sw["T"]},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# host-only sources (argument checks, the launch plan, the multi-launch
# runtimes): no device code.  The plan's effect on a measured launch is its
# shape, which the committed traffic entries record and ncu_traffic compares.
HOST_ONLY_SOURCES = ("api.h", "capi.cu", "plan.cu", "runtime.cu")


def kernel_source_hash():
    """Hash of the sources that hold device code (every file under csrc but the
    host-only ones): ncu counters taken at another hash no longer describe the
    kernels that run."""
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "sequential_rnn_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f in HOST_ONLY_SOURCES:
            continue
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:12]


def tu_source_hash(tu):
    """Hash of one kernel translation unit under csrc and every local header it
    includes, recursively: ncu counters taken at another hash no longer
    describe the kernel that runs (changes elsewhere in csrc do not matter)."""
    import re
    csrc = os.path.join(ROOT, "sequential_rnn_gb300", "csrc")
    seen, todo = set(), [tu]
    while todo:
        f = todo.pop()
        if f in seen or not os.path.exists(os.path.join(csrc, f)):
            continue
        seen.add(f)
        with open(os.path.join(csrc, f)) as fh:
            todo += re.findall(r'^#include "([^"/]+)"', fh.read(), flags=re.M)
    h = hashlib.sha1()
    for f in sorted(seen):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:12]


def ncu_traffic(workload, launch=None):
    """DRAM bytes per launch from a committed ncu summary, if it matches the
    sources of the captured kernel (its translation unit and headers) and (when
    both are known) the forward's launch shape."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    e = j.get(workload)
    if not e:
        return None
    want = tu_source_hash(e["tu"]) if "tu" in e else kernel_source_hash()
    if e.get("source_hash") != want:
        return None
    shape = e.get("launch")
    if shape and launch and any(shape[k] != launch.get(k) for k in shape):
        return None
    return e.get("dram_bytes_per_launch")


def run_ours(args, w, rank, world, local_rank):
    import torch
    import sequential_rnn_gb300 as S
    from sequential_rnn_gb300 import build as B

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    d = workload_inputs(args.workload, seed=rank)
    cell = w["cell"]
    dt = torch.bfloat16 if w["dtype"] == "bf16" else torch.float32
    g = {k: torch.from_numpy(np.ascontiguousarray(d[k])).to(dev, dt) for k in ("Wx", "R")}
    for k in ("b", "h0", "c0", "n0", "m0"):
        g[k] = torch.from_numpy(np.ascontiguousarray(d[k])).to(dev, torch.float32)
    if w["backward"]:
        g["dh"] = torch.from_numpy(np.ascontiguousarray(d["dh"])).to(dev, dt)
    T, Bsz, NH, Dh = w["T"], w["B"], w["NH"], w["Dh"]
    G = GATES[cell]
    flags = S.RNN_FLAG_TRAIN if w["backward"] else 0
    desc = S.make_desc(cell, w["dtype"], T, Bsz, NH, Dh, flags, args.cluster)
    cfg = S.rnn_fwd_config(desc)
    f32 = dict(dtype=torch.float32, device=dev)
    h_seq = torch.empty((T, Bsz, NH, Dh), dtype=dt, device=dev)
    hT = torch.empty((Bsz, NH, Dh), **f32)
    cT = torch.empty((Bsz, NH, Dh), **f32) if cell != "gru" else None
    nT = torch.empty((Bsz, NH, Dh), **f32) if cell == "slstm" else None
    mT = torch.empty((Bsz, NH, Dh), **f32) if cell == "slstm" else None
    ws = torch.zeros(S.rnn_workspace_size(desc, 0), dtype=torch.uint8, device=dev)
    stash = torch.empty(max(S.rnn_stash_size(desc) // 4, 1), **f32) if w["backward"] else None
    if w["backward"]:
        gr = {"dWx": torch.empty_like(g["Wx"]), "dR": torch.empty((NH, Dh, G * Dh), **f32),
              "db": torch.empty((NH, G * Dh), **f32), "dh0": torch.empty((Bsz, NH, Dh), **f32),
              "dc0": torch.empty((Bsz, NH, Dh), **f32)}
        wsb = torch.zeros(S.rnn_workspace_size(desc, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    launches_per_step = 1

    def step(Wx=None, R=None, bev=None):
        st = S.rnn_fwd(desc, g["Wx"] if Wx is None else Wx, g["R"] if R is None else R, g["b"],
                       g["h0"], g["c0"], g["n0"] if cell == "slstm" else None,
                       g["m0"] if cell == "slstm" else None, h_seq, hT, cT, nT, mT, stash, ws,
                       stream)
        if st:
            raise S.RnnError(st, "rnn_fwd")
        if w["backward"]:
            if bev is not None:
                bev[0].record(stream)
            st = S.rnn_bwd(desc, g["R"] if R is None else R, g["h0"], g["c0"], None, h_seq, stash,
                           g["dh"], None, None, None, gr["dWx"], gr["dR"], gr["db"], gr["dh0"],
                           gr["dc0"], None, wsb, stream)
            if bev is not None:
                bev[1].record(stream)
            if st:
                raise S.RnnError(st, "rnn_bwd")

    if w["backward"]:
        launches_per_step = 5  # fwd, h0->bf16, bwd recurrence, dR GEMM, db reduce

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    clk = ClockSampler(torch.cuda.get_device_properties(dev).uuid).__enter__()
    atexit.register(clk.__exit__, None, None, None)  # no stray nvidia-smi on an error
    w0 = time.perf_counter()
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if S.rnn_read_status(ws):
        raise S.RnnError(S.rnn_read_status(ws), "warm-up (device)")
    t1 = (time.perf_counter() - w0) / max(args.warmup, 3)
    if args.steps is None:  # ~2 s of timed work
        args.steps = int(min(3000, max(20, 2.0 / max(t1, 1e-5))))
    # untimed clock soak: the same steps for ~1 s (and until nvidia-smi has
    # reported), so that the clock record covers the GPU under this load even
    # when the timed region itself is a few ms long
    clk.wait_first()
    soak0 = time.perf_counter()
    while time.perf_counter() - soak0 < 1.0:
        for _ in range(max(1, int(0.05 / max(t1, 1e-5)))):
            flush.fill_(0.0)
            step()
        torch.cuda.synchronize(dev)

    # ---- device-resident timing: events around each step, L2 flushed between
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    # training: the reverse pass (the dominant launch) is also timed on its own
    bev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)] if w["backward"] else None
    barrier()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        step(bev=bev[i] if bev else None)
        ev[i][1].record(stream)
    barrier()
    wall = time.perf_counter() - wall0
    clk.__exit__(None, None, None)
    per = [a.elapsed_time(b) for a, b in ev]  # ms
    t_step = sum(per) / len(per) / 1e3
    t_bwd = (sum(a.elapsed_time(b) for a, b in bev) / len(bev) / 1e3) if bev else None
    # the job takes as long as its slowest rank
    from sequential_rnn_gb300.dist import max_over_ranks
    t_step = max_over_ranks(t_step, device=dev)
    if S.rnn_read_status(ws):
        raise S.RnnError(S.rnn_read_status(ws), "timed region (device)")

    # ---- sync floor of the same launch shape, and of every other shape the
    #      library admits for this workload (CTAs per head 1..16): the smallest
    #      is the floor no launch choice can go below
    fl_ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    fe = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))

    def sync_floor(cluster):
        fdesc = S.make_desc(cell, w["dtype"], T, Bsz, NH, Dh, 0, cluster)
        for _ in range(3):
            S.rnn_sync_floor(fdesc, T, fl_ws, stream)
        fl = []
        for _ in range(10):
            fe[0].record(stream)
            st = S.rnn_sync_floor(fdesc, T, fl_ws, stream)
            fe[1].record(stream)
            torch.cuda.synchronize(dev)
            if st:
                raise S.RnnError(st, "rnn_sync_floor")
            fl.append(fe[0].elapsed_time(fe[1]) / 1e3)
        return statistics.median(fl) / T

    t_floor = sync_floor(args.cluster)
    floors = {}
    for cs in ((1,) if w["dtype"] == "f32" else (1, 2, 4, 8, 16)):
        try:
            S.rnn_fwd_config(S.make_desc(cell, w["dtype"], T, Bsz, NH, Dh, flags, cs))
        except S.RnnError:
            continue  # no variant for this split
        floors[cs] = sync_floor(cs)

    # ---- end to end through the C ABI with pinned host buffers: every step copies
    #      that step's Wx in from host memory and h_seq back out.  Forward: the
    #      host-memory entry point (rnn_fwd_host), which pipelines the copies with
    #      the recurrence over time chunks; training: Wx and R double-buffered on
    #      the device, step i+1's copied in on a copy stream while step i runs, and
    #      h_seq copied out after each step.
    hWx = g["Wx"].cpu().pin_memory()
    hh = torch.empty(h_seq.shape, dtype=dt).pin_memory()
    e2e_steps = max(3, min(args.steps, 50))
    ee = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    if not w["backward"]:
        hws = torch.empty(max(S.rnn_fwd_host_workspace_size(desc, 0), 256), dtype=torch.uint8,
                          device=dev)

        def e2e_step():
            st = S.rnn_fwd_host(desc, 0, hWx, g["R"], g["b"], g["h0"], g["c0"],
                                g["n0"] if cell == "slstm" else None,
                                g["m0"] if cell == "slstm" else None, hh, hT, cT, nT, mT, hws,
                                stream)
            if st:
                raise S.RnnError(st, "rnn_fwd_host")
        h2d = hWx.numel() * hWx.element_size()
    else:
        hR = g["R"].cpu().pin_memory()
        bufs = [(torch.empty_like(g["Wx"]), torch.empty_like(g["R"])) for _ in range(2)]
        cstream = torch.cuda.Stream(dev)
        ready = [torch.cuda.Event() for _ in range(2)]  # buffer b holds the next inputs
        done = [torch.cuda.Event() for _ in range(2)]   # the step reading buffer b ended
        nstep = [0]

        def upload(b):
            cstream.wait_event(done[b])
            with torch.cuda.stream(cstream):
                bufs[b][0].copy_(hWx, non_blocking=True)
                bufs[b][1].copy_(hR, non_blocking=True)
            ready[b].record(cstream)

        def e2e_step():
            b = nstep[0] & 1
            if nstep[0] == 0:
                upload(0)
            stream.wait_event(ready[b])
            upload(1 - b)  # the next step's inputs, while this one runs
            step(*bufs[b])
            done[b].record(stream)
            hh.copy_(h_seq, non_blocking=True)
            nstep[0] += 1
        h2d = hWx.numel() * hWx.element_size() + hR.numel() * hR.element_size()
    for _ in range(2):
        e2e_step()
    barrier()
    ee[0].record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    if w["backward"]:  # the last upload (inputs of the step after) is inside the region too
        stream.wait_event(ready[nstep[0] & 1])
    ee[1].record(stream)
    barrier()
    if not w["backward"] and S.rnn_read_status(hws):
        raise S.RnnError(S.rnn_read_status(hws), "end-to-end (device)")
    t_e2e = ee[0].elapsed_time(ee[1]) / 1e3 / e2e_steps
    d2h = hh.numel() * hh.element_size()

    fl_step = flops_per_step(w)
    hbm, tflops_peak, peak_kind = load_peaks()
    pipe = "bf16 tensor (measured cuBLAS)"
    if w["dtype"] == "f32":
        # the fp32 path runs on the FMA pipe (no tensor cores, no TF32): its peak
        # from unit counts and clock -- SMs x 128 fp32 FMA lanes x 2 FLOP x SM clock
        props = torch.cuda.get_device_properties(dev)
        mhz = float(clk.summary().get("sm_max_mhz") or 2070.0)
        tflops_peak = props.multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12
        pipe = f"fp32 FMA ({props.multi_processor_count} SMs x 128 lanes x 2 FLOP x {mhz:.0f} MHz)"
    per_step_bytes, total_bytes = algorithmic_bytes_fwd(w)
    # per-step roofline: slower of bytes at HBM and flops at the tensor pipe, plus the floor
    t_bytes = per_step_bytes / (hbm * 1e9)
    t_flop = 2.0 * Bsz * NH * Dh * G * Dh / (tflops_peak * 1e12)
    t_roof = max(t_bytes, t_flop) + t_floor
    t_meas_step = t_step / T
    t_floor_min = min(floors.values()) if floors else t_floor
    if w["backward"]:
        # dominant launch of the training step: the reverse recurrence (rnn_bwd)
        roof_bytes = algorithmic_bytes_bwd(w)
        achieved_gbs = roof_bytes / t_bwd / 1e9
        roof_note = (f"rnn_bwd (reverse recurrence + dR GEMM + db): algorithmic bytes {roof_bytes} "
                     f"per launch / its event time {t_bwd * 1e3:.3f} ms; peak {peak_kind} HBM copy bandwidth")
    else:
        achieved_gbs = total_bytes / t_step / 1e9
        roof_note = (f"algorithmic bytes {total_bytes} per launch / event time; "
                     f"peak {peak_kind} HBM copy bandwidth")
    res = {
        "metric": METRIC, "value": world * fl_step / t_step / 1e12, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic",
        "config": {"workload": args.workload, "cell": cell, "NH": NH, "Dh": Dh, "B": Bsz, "T": T,
                   "l2": "flushed before every timed step (2x L2 write, outside the events)",
                   "launch": cfg, "parallelism": f"weak x{world}: one independent batch per GPU"},
        "steps_per_s": world * T / t_step,
        "per_step_ns": t_meas_step * 1e9,
        "per_step_roofline": {
            "bytes_ns": t_bytes * 1e9, "flops_ns": t_flop * 1e9, "sync_floor_ns": t_floor * 1e9,
            "roofline_ns": t_roof * 1e9, "frac": t_roof / t_meas_step,
            "floors_ns_by_ctas_per_head": {str(k): v * 1e9 for k, v in floors.items()},
            "frac_min_floor": (max(t_bytes, t_flop) + t_floor_min) / t_meas_step,
            "note": ("frac: the floor of the launch shape that ran; frac_min_floor: the "
                     "smallest floor among the shapes the library admits for this workload"),
            "peaks": f"HBM {peak_kind} {hbm} GB/s; pipe {pipe} {tflops_peak:.1f} TFLOP/s"},
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": achieved_gbs / hbm, "traffic": ncu_traffic(args.workload, cfg),
                     "note": roof_note},
        "e2e": {"value": world * fl_step / t_e2e / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": {**clk.summary(),
                   "window": "nvidia-smi every 50 ms over a 1 s untimed soak of the same steps "
                             "and the timed region"},
        "wall_timed_s": wall,
    }
    return res


def free_port() -> int:
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as so:
        so.bind(("127.0.0.1", 0))
        return so.getsockname()[1]


def rank_launch_cmd(n: int, script: str, argv: list) -> list:
    """torch.distributed.run command that starts ``script`` as n ranks on this
    node (one per GPU), rendezvous on 127.0.0.1."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            f"--nproc-per-node={int(n)}", "--master-addr", "127.0.0.1",
            "--master-port", str(free_port()), script, *argv]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for ~2 s of timed work, 20..3000)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cluster", type=int, default=0, help="CTAs per head (0 = automatic)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()

    if args.gpus > 1 and "WORLD_SIZE" not in os.environ and args.impl == "ours":
        # no launcher around us: start one rank per GPU ourselves
        cmd = rank_launch_cmd(args.gpus, os.path.abspath(__file__), sys.argv[1:])
        sys.exit(subprocess.call(cmd))

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = dict(WORKLOADS[args.workload])

    if args.impl == "reference":
        if args.steps is None:
            args.steps = 3
        res = run_reference(args, w, rank)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return

    # CPU baseline first (before any GPU work): the oracle on the host cores
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        sw = sample_workload(w, 256 if w["Dh"] <= 256 else 64)
        d = workload_inputs(args.workload, T=sw["T"])
        rate, reps, el, busy = oracle_rate(sw, d, budget_s=10.0)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": threads_used(busy), "kind": "oracle",
               "sample": (f"{args.workload} with T cut to {sw['T']}, {reps} oracle passes in "
                          f"{el:.1f} s; {busy:.2f} threads busy on average of {os.cpu_count()} "
                          "host cores")}
        one = oracle_rate_single_thread(args.workload, sw["T"], 5.0)
        if one is not None:
            cpu["single_thread"] = {
                "value": one["value"], "unit": "TFLOP/s", "cores": 1,
                "sample": (f"same sample, BLAS thread pools limited to one: {one['reps']} passes "
                           f"in {one['seconds']:.1f} s ({one['busy']:.2f} threads busy)")}

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
        world = dist.get_world_size()  # n_gpus: the ranks that joined
    res = run_ours(args, w, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        res["cpu_baseline"] = cpu
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
