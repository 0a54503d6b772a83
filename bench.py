#!/usr/bin/env python3
"""Benchmark of the decomposed collective matmul on one GB300.

One step = the whole hot path over one batch: the fc1 AllGather->GEMM
(cm_ag_gemm) and the fc2 GEMM->ReduceScatter (cm_gemm_rs) of a Megatron-SP
MLP with h=8192, ffn=28672, s=8192, N=8 logical ranks on the GPU, one chunk
per shard, unidirectional ring (synthetic bf16 data, inputs resident in HBM).

Prints one JSON line (rank 0).  Metric: TFLOP/s (sum over ranks of 2*M*K*n
per op), with the roofline of the persistent kernel against the measured
dense bf16 peak, the same metric end to end through the C ABI with host
buffers, the oracle timed on the host cores, and SM clocks sampled during the
timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--sweep]   # the N x chunks x ring sweep, one JSON line per point
                  [--configs] # every configuration's ops with roofline fractions

For --gpus N > 1 (launched by torch.distributed.run), every rank runs an
independent replica of the step on its own GPU (the path does not shard
across GPUs); value = all ranks' FLOPs / max-over-ranks time.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "AG-GEMM / GEMM-RS bf16 TFLOP/s and % of dense tensor peak on 1 GB300"
UNIT = "TFLOP/s"
WORKLOAD = "mlp_h8192_ffn28672_s8192"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}  # of fallback
# every source that decides what the kernels do (tile order, task table, launch shape)
KERNEL_SOURCES = ["cm_kernel.cu", "cm_kernel_pair.cu", "cm_device.cuh", "cm_kernel.cuh", "cm_kernel_common.cuh",
                  "cm_api.cu", "cm_plan.cpp", "cm_internal.h"]


# ---- distributed host logic (also exercised by the gloo tests on CPU) ---------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def dist_barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def dist_max(value: float, device=None) -> float:
    """Max of a float over ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(flops_per_step_per_rank: float, steps: int, world: int, seconds_max: float) -> float:
    """Whole-job TFLOP/s: every rank's work over the slowest rank's time."""
    return flops_per_step_per_rank * steps * world / seconds_max / 1e12


# ---- helpers ------------------------------------------------------------------------

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def code_of(text: str) -> str:
    """C/C++/CUDA source without its comments and blank lines: what the
    compiler sees, so that a comment edit does not retire a measurement."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "collective_matmul_decomposition_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(code_of(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, if it matches this kernel."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_hash") != kernel_hash():
        return None
    return d


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.gpu_id is not None:
            cmd += ["-i", str(self.gpu_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        # samples under load: power well above idle
        load = [s for s, p in zip(sm, pw) if p is not None and pw and p > 0.5 * max(pw)] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


def physical_gpu_id(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return local_rank


# ---- the workload ---------------------------------------------------------------------

def make_step_inputs(N: int, device):
    """fc1 AG-GEMM and fc2 GEMM-RS operands (CPU copies kept for the oracle)."""
    from collective_matmul_decomposition_gb300 import inputs as gen
    s = gen.mlp_shapes(N)
    a, r = s["ag"], s["rs"]
    wl = gen.WORKLOADS[WORKLOAD]
    x1, w1 = gen.ag_inputs(N, a["m"], a["K"], a["n"], wl["ag"]["x"], wl["ag"]["w"], wl["ag"]["seed"], "nk")
    x2, w2 = gen.rs_inputs(N, r["M"], r["k"], r["n"], wl["rs"]["x"], wl["rs"]["w"], wl["rs"]["seed"], "nk")
    return dict(shapes=s, cpu=(x1, w1, x2, w2))


def flops(s, N):
    a, r = s["ag"], s["rs"]
    ag = 2.0 * N * (N * a["m"]) * a["K"] * a["n"]        # sum over ranks of 2*M*K*n
    rs = 2.0 * r["M"] * r["k"] * r["n"] * N
    return ag, rs


class Step:
    """Device buffers and plans of one step; run() enqueues both ops."""

    def __init__(self, N, chunks, direction, data, device, y_dtype=None):
        import torch
        from collective_matmul_decomposition_gb300 import cm
        self.cm = cm
        self.N = N
        s = data["shapes"]
        a, r = s["ag"], s["rs"]
        x1, w1, x2, w2 = data["cpu"]
        yd = y_dtype or torch.bfloat16
        self.x1, self.w1 = x1.to(device), w1.to(device)
        self.x2, self.w2 = x2.to(device), w2.to(device)
        self.y1 = torch.empty(N, N * a["m"], a["n"], dtype=yd, device=device)
        self.y2 = torch.empty(N, r["M"] // N, r["n"], dtype=yd, device=device)
        self.plan = cm.Plan(N, chunks, direction)
        self.ws1 = torch.empty(self.plan.ag_workspace_size(a["m"], a["K"]), dtype=torch.uint8, device=device)
        self.ws2 = torch.empty(self.plan.rs_workspace_size(r["M"], r["n"]), dtype=torch.uint8, device=device)

    def set_rs_in_place(self, v):
        """CM_OPT_RS_IN_PLACE for this step's plan (the RS workspace is resized)."""
        import torch
        self.plan.set_option(self.cm.CM_OPT_RS_IN_PLACE, int(v))
        M, n = self.x2.shape[1], self.y2.shape[2]
        self.ws2 = torch.empty(self.plan.rs_workspace_size(M, n), dtype=torch.uint8, device=self.x2.device)
        return self

    def ag(self):
        self.cm.cm_ag_gemm(self.plan, self.x1, self.w1, self.y1, self.ws1, "nk")

    def rs(self):
        self.cm.cm_gemm_rs(self.plan, self.x2, self.w2, self.y2, self.ws2, "nk")

    def rs_pipe(self):
        """The pipelined GEMM->ReduceScatter on the same inputs (own workspace)."""
        if not hasattr(self, "ws3"):
            import torch
            r = self.x2.shape
            n = self.y2.shape[2]
            self.ws3 = torch.empty(self.plan.rs_pipelined_workspace_size(r[1], n), dtype=torch.uint8,
                                   device=self.x2.device)
        self.cm.cm_gemm_rs_pipelined(self.plan, self.x2, self.w2, self.y2, self.ws3, "nk")

    def check(self, ops=("ag", "rs")):
        """Device status of the last call of each op in `ops` (only ops that ran)."""
        for op in ops:
            ws = {"ag": self.ws1, "rs": self.ws2, "rs_pipe": getattr(self, "ws3", None)}[op]
            st, info = self.cm.cm_check_status(ws)
            if st != 0:
                raise RuntimeError(f"{op}: device status {st} {info}")


class EndToEnd:
    """One step through the C ABI starting from pinned host buffers.

    Serial: H2D of the four inputs, both calls, D2H of both outputs, then the
    host reads the result. Pipelined: the same per-step work, but the H2D of
    step i+1 (into the other device buffer set) and the D2H of step i-1 run on
    their own streams while step i computes; the host reads step i-1's result
    once its copy has landed. Every step still moves all of its inputs and
    outputs across the host link."""

    def __init__(self, st, data, torch):
        self.torch = torch
        self.st = st
        self.host_in = [t.pin_memory() for t in data["cpu"]]
        self.host_out = [[torch.empty(st.y1.shape, dtype=st.y1.dtype).pin_memory(),
                          torch.empty(st.y2.shape, dtype=st.y2.dtype).pin_memory()] for _ in range(2)]
        self.dev_in = [[st.x1, st.w1, st.x2, st.w2], [torch.empty_like(t) for t in (st.x1, st.w1, st.x2, st.w2)]]
        self.dev_out = [[st.y1, st.y2], [torch.empty_like(st.y1), torch.empty_like(st.y2)]]
        self.h2d = sum(t.numel() * t.element_size() for t in self.host_in)
        self.d2h = sum(t.numel() * t.element_size() for t in self.host_out[0])
        self.s_in = torch.cuda.Stream()
        self.s_out = torch.cuda.Stream()

    def compute(self, b):
        cm, st = self.st.cm, self.st
        x1, w1, x2, w2 = self.dev_in[b]
        y1, y2 = self.dev_out[b]
        cm.cm_ag_gemm(st.plan, x1, w1, y1, st.ws1, "nk")
        cm.cm_gemm_rs(st.plan, x2, w2, y2, st.ws2, "nk")

    def run_serial(self, n):
        torch = self.torch
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            for d, h in zip(self.dev_in[0], self.host_in):
                d.copy_(h, non_blocking=True)
            self.compute(0)
            for h, d in zip(self.host_out[0], self.dev_out[0]):
                h.copy_(d, non_blocking=True)
            torch.cuda.synchronize()
            float(self.host_out[0][1][0, 0, 0])
        return time.perf_counter() - t0

    def run_pipelined(self, n):
        torch = self.torch
        main = torch.cuda.current_stream()
        ev = lambda: torch.cuda.Event()
        in_ready, comp_done, out_done = [ev() for _ in range(n)], [ev() for _ in range(n)], [ev() for _ in range(n)]
        torch.cuda.synchronize()
        t0 = time.perf_counter()

        def load(i):
            b = i % 2
            with torch.cuda.stream(self.s_in):
                if i >= 2:
                    self.s_in.wait_event(comp_done[i - 2])      # step i-2 has read this buffer set
                for d, h in zip(self.dev_in[b], self.host_in):
                    d.copy_(h, non_blocking=True)
                in_ready[i].record(self.s_in)

        load(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                load(i + 1)
            main.wait_event(in_ready[i])
            if i >= 2:
                main.wait_event(out_done[i - 2])               # step i-2's outputs have left
            self.compute(b)
            comp_done[i].record(main)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(comp_done[i])
                for h, d in zip(self.host_out[b], self.dev_out[b]):
                    h.copy_(d, non_blocking=True)
                out_done[i].record(self.s_out)
            if i >= 1:
                out_done[i - 1].synchronize()
                float(self.host_out[(i - 1) % 2][1][0, 0, 0])
        out_done[n - 1].synchronize()
        float(self.host_out[(n - 1) % 2][1][0, 0, 0])
        dt = time.perf_counter() - t0
        torch.cuda.synchronize()
        return dt


def time_loop(fn, iters, torch, warmup=3):
    """Mean ms per call of fn() over iters calls after `warmup` untimed calls
    (CUDA events, synchronised)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def time_interleaved(fns, iters, torch, warmup=3):
    """Median ms per call of each fn in the dict `fns`, calling them in turn
    (one of each per round, `iters` rounds) so that all see the same clocks
    and power state. CUDA events around every call, synchronised once."""
    for _ in range(warmup):
        for fn in fns.values():
            fn()
    torch.cuda.synchronize()
    ev = {k: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(iters)] for k in fns}
    for i in range(iters):
        for k, fn in fns.items():
            ev[k][i][0].record()
            fn()
            ev[k][i][1].record()
    torch.cuda.synchronize()
    return {k: statistics.median(a.elapsed_time(b) for a, b in ev[k]) for k in fns}


def concat_operands(st, shapes, N):
    """The undecomposed operands of one step for torch.matmul: fc1 X [N*m, K] and
    W [N*n, K]; fc2 X [M, N*k] and W [n, N*k] (contiguous copies)."""
    a, r = shapes["ag"], shapes["rs"]
    X1 = st.x1.reshape(N * a["m"], a["K"])
    W1 = st.w1.reshape(N * a["n"], a["K"])
    X2 = st.x2.permute(1, 0, 2).reshape(r["M"], N * r["k"]).contiguous()
    W2 = st.w2.permute(1, 0, 2).reshape(r["n"], N * r["k"]).contiguous()
    return X1, W1, X2, W2


def oracle_sample(cpu, shapes, N, seconds: float, seed=0):
    """Time the fp64 oracle on sampled output rows for about `seconds`.
    Returns (flops done, seconds taken, threads, description)."""
    import numpy as np
    import oracle
    from collective_matmul_decomposition_gb300 import inputs as gen
    x1, w1, x2, w2 = cpu
    xb1, wb1, xb2, wb2 = (gen.bf16_bits(t) for t in cpu)
    a, r = shapes["ag"], shapes["rs"]
    rng = np.random.default_rng(seed)
    f_ag_row = 2.0 * a["K"] * a["n"]
    f_rs_row = 2.0 * r["k"] * r["n"] * N

    def run(n_ag, n_rs):
        ranks = rng.integers(0, N, n_ag)
        rows = rng.integers(0, N * a["m"], n_ag)
        owners = rng.integers(0, N, n_rs)
        rrows = rng.integers(0, r["M"] // N, n_rs)
        t0 = time.perf_counter()
        oracle.ag_gemm_rows(xb1, wb1, ranks, rows, "nk")
        oracle.gemm_rs_rows(xb2, wb2, owners, rrows, "nk")
        return time.perf_counter() - t0, n_ag * f_ag_row + n_rs * f_rs_row

    nthr = oracle.threads()
    dt, fl = run(nthr, max(1, nthr // 4))               # calibration
    rate = fl / max(dt, 1e-6)
    target = max(seconds * rate, fl)
    # same mix as the step: equal flops for the two ops
    n_ag = max(1, int(target / 2 / f_ag_row))
    n_rs = max(1, int(target / 2 / f_rs_row))
    dt, fl = run(n_ag, n_rs)
    desc = (f"{n_ag} AG-GEMM output rows + {n_rs} GEMM-RS output rows of the {WORKLOAD} step at "
            f"N={N} (fp64 oracle, OpenMP {nthr} threads)")
    return fl, dt, nthr, desc


# ---- arms -----------------------------------------------------------------------------

def run_reference(args):
    """The oracle, as it stands, timed on the host cores over bounded samples."""
    rank, world, _ = dist_env()
    if world > 1:
        dist_init("gloo")
        if rank != 0:
            return 0
    import oracle
    oracle.build()
    N = 8
    data = make_step_inputs(N, "cpu")
    shapes = data["shapes"]
    budget = args.ref_seconds  # seconds of oracle work for the whole run
    per_step = budget / max(1, args.steps + args.warmup)
    for _ in range(args.warmup):
        oracle_sample(data["cpu"], shapes, N, per_step)
    tot_f, tot_t, thr, desc = 0.0, 0.0, 1, ""
    for i in range(args.steps):
        f, t, thr, desc = oracle_sample(data["cpu"], shapes, N, per_step, seed=i + 1)
        tot_f += f
        tot_t += t
    value = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": step_config(N, 1, "uni", shapes),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle",
                             "sample": "each step: " + desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def choose_peak(peaks, timed_s, clocks):
    """The measured dense bf16 peak that matches the clocks the kernel ran at.
    The burst figure (a GEMM timed alone, at full clocks) when the median SM
    clock sampled under load during the timed region stayed at its maximum;
    the sustained figure (seconds of back-to-back GEMMs under the power cap,
    whose clocks came down the same way) when it did not.  Without clock
    samples, the length of the timed region decides (under 1 s: burst)."""
    burst, sust = float(peaks["bf16_tflops"]), float(peaks["bf16_tflops_sustained"])
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if sm is not None and mx:
        if sm >= 0.97 * mx:
            return burst, "burst", f"median SM clock {sm:.0f} MHz, at its maximum {mx:.0f}"
        return sust, "sustained", (f"median SM clock {sm:.0f} MHz under load, below its maximum {mx:.0f} "
                                   f"(reasons {','.join(clocks.get('reasons') or []) or 'none'})")
    if timed_s < 1.0:
        return burst, "burst", f"no clock samples; timed region {timed_s:.3f} s < 1 s"
    return sust, "sustained", f"no clock samples; timed region {timed_s:.2f} s"


def step_config(N, chunks, direction, shapes):
    a, r = shapes["ag"], shapes["rs"]
    return {"workload": WORKLOAD, "logical_ranks": N, "chunks": chunks, "ring": direction,
            "ops": ["fc1 AG-GEMM", "fc2 GEMM-RS"],
            "ag": {"x": [N, a["m"], a["K"]], "w": [N, a["n"], a["K"]], "y": [N, N * a["m"], a["n"]]},
            "rs": {"x": [N, r["M"], r["k"]], "w": [N, r["n"], r["k"]], "y": [N, r["M"] // N, r["n"]]},
            "w_layout": "nk", "accumulate": "fp32", "out": "bf16",
            "l2": "inputs larger than L2 (fc1 598 MB, fc2 940 MB of operands per op), no flush",
            "parallelism": "logical ranks on one GPU; replicas across GPUs"}


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist_init("nccl")
    device = torch.device("cuda", torch.cuda.current_device())
    import __graft_entry__
    __graft_entry__.build()
    N, chunks, direction = 8, 1, "uni"
    data = make_step_inputs(N, device)
    shapes = data["shapes"]
    f_ag, f_rs = flops(shapes, N)
    st = Step(N, chunks, direction, data, device)

    def step():
        st.ag()
        st.rs()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st.check()

    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_barrier()
    torch.cuda.synchronize()
    with ClockSampler(physical_gpu_id(local)) as clk:
        t_start.record()
        for i in range(K):
            evs[i][0].record()
            st.ag()
            evs[i][1].record()
            st.rs()
            evs[i][2].record()
        t_end.record()
        torch.cuda.synchronize()
    dist_barrier()
    st.check()
    elapsed = t_start.elapsed_time(t_end) / 1e3
    elapsed_max = dist_max(elapsed, device)
    ag_ms = [e[0].elapsed_time(e[1]) for e in evs]
    rs_ms = [e[1].elapsed_time(e[2]) for e in evs]
    value = aggregate(f_ag + f_rs, K, world, elapsed_max)
    clocks = clk.summary()

    peaks, peak_kind = load_peaks()
    peak, peak_which, peak_why = choose_peak(peaks, elapsed_max, clocks)
    peak_burst = float(peaks["bf16_tflops"])
    peak_sust = float(peaks["bf16_tflops_sustained"])
    launch_ms = statistics.mean(ag_ms + rs_ms)
    achieved = (f_ag + f_rs) / 2 / (launch_ms / 1e3) / 1e12
    ach_ag = f_ag / (statistics.mean(ag_ms) / 1e3) / 1e12
    ach_rs = f_rs / (statistics.mean(rs_ms) / 1e3) / 1e12
    traffic = ncu_traffic()

    # comparators on the same data -- the undecomposed op in this kernel and
    # cuBLAS (torch.matmul on the concatenated operands) -- timed interleaved
    # with the decomposed calls so that all see the same clocks
    detail = {}
    if rank == 0:
        iters = max(5, min(20, K))
        mono = Step(N, 1, "none", {"shapes": shapes, "cpu": data["cpu"]}, device)
        X1, W1, X2, W2 = concat_operands(st, shapes, N)
        variants = {"ag": st.ag, "none_ag": mono.ag, "torch_ag": lambda: torch.matmul(X1, W1.t()),
                    "rs": st.rs, "none_rs": mono.rs, "torch_rs": lambda: torch.matmul(X2, W2.t())}
        ms = time_interleaved(variants, iters, torch)
        st.check()
        mono.check()
        for k in variants:
            detail[f"{k}_ms_interleaved"] = ms[k]
        detail["ag_ms"] = statistics.mean(ag_ms)
        detail["rs_ms"] = statistics.mean(rs_ms)
        detail["ag_tflops"] = f_ag / (detail["ag_ms"] / 1e3) / 1e12
        detail["rs_tflops"] = f_rs / (detail["rs_ms"] / 1e3) / 1e12
        for op in ("ag", "rs"):
            mine = detail[f"{op}_ms_interleaved"]
            detail[f"{op}_vs_torch_time"] = mine / detail[f"torch_{op}_ms_interleaved"]
            detail[f"{op}_vs_none_time"] = mine / detail[f"none_{op}_ms_interleaved"]
        detail["comparators"] = ("each op, its undecomposed form in this kernel and torch.matmul on the "
                                 f"concatenated operands, interleaved {iters} times after the timed region (median)")
        del X2, W2, mono, variants

    # end to end through the C ABI with host buffers: every step copies all four
    # inputs from pinned host memory, runs both calls and copies both outputs
    # back, and the host reads each step's result
    e2e = None
    if rank == 0 or world > 1:
        n_e2e = max(3, min(10, K))
        runner = EndToEnd(st, data, torch)
        runner.run_serial(1)
        runner.run_pipelined(2)
        dist_barrier()
        dt_serial = runner.run_serial(n_e2e)
        # five rounds of n_e2e pipelined steps; the median round is reported
        # (host-link throughput varies from round to round), every round listed
        rounds = []
        for _ in range(5):
            dist_barrier()
            rounds.append(dist_max(runner.run_pipelined(n_e2e), device))
        dt_max = statistics.median(rounds)
        e2e = {"value": aggregate(f_ag + f_rs, n_e2e, world, dt_max), "unit": UNIT,
               "h2d_bytes_per_step": runner.h2d, "d2h_bytes_per_step": runner.d2h,
               "ms_per_step": dt_max / n_e2e * 1e3, "steps": n_e2e,
               "how": ("copies of step i+1's inputs and of step i-1's outputs overlap step i's calls "
                       "(two device buffer sets, one copy stream each way); median of 5 rounds"),
               "round_ms_per_step": [r / n_e2e * 1e3 for r in rounds],
               "serial_ms_per_step": dt_serial / n_e2e * 1e3,
               "serial_value": (f_ag + f_rs) * world / (dt_serial / n_e2e) / 1e12}
        st.check()
        del runner

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, t, thr, desc = oracle_sample(data["cpu"], shapes, N, args.cpu_seconds)
        cpu_baseline = {"value": f / t / 1e12, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": desc,
                        "seconds": t}

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": elapsed_max / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights)",
        "config": step_config(N, chunks, direction, shapes),
        "pct_of_peak": value / peak,
        "pct_of_burst_peak": value / peak_burst,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "frac_ag": ach_ag / peak, "frac_rs": ach_rs / peak,
                     "achieved_ag": ach_ag, "achieved_rs": ach_rs,
                     "frac_of_burst": achieved / peak_burst, "frac_of_sustained": achieved / peak_sust,
                     "traffic": traffic["bytes_per_launch"] if traffic else None,
                     "kernel": "cm_pair_kernel (one launch per op; AG and RS averaged)",
                     "peak_source": f"{peak_which} dense bf16 of {peak_kind} ({peak_why})"},
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": 2 * K,
        "gpu_launch_note": "one persistent kernel per op per step (plus one flag memset each)",
        "cpu_baseline": cpu_baseline,
        "detail": detail,
    }
    print(json.dumps(line), flush=True)
    return 0


def sweep_best(points):
    """The fastest point of each op among sweep lines (dicts with op, N,
    chunks, ring, ms, frac_of_peak): one summary dict per op, in first-seen
    op order."""
    best = {}
    for p in points:
        b = best.get(p["op"])
        if b is None or p["ms"] < b["ms"]:
            best[p["op"]] = p
    return [{"sweep_best": p["op"], "N": p["N"], "chunks": p["chunks"], "ring": p["ring"],
             "ms": p["ms"], "frac_of_peak": p["frac_of_peak"],
             "vs_undecomposed_time": p.get("vs_undecomposed_time"),
             "vs_torch_time": p.get("vs_torch_time")} for p in best.values()]


def run_sweep(args):
    """All points of the MLP sweep: N in {4,8,16} x chunks {1,2,4} x {uni,bidi} x {AG, RS},
    then the fastest point of each op (pipelined RS included)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    device = torch.device("cuda", 0)
    peaks, kind = load_peaks()
    peak = float(peaks["bf16_tflops"])
    points = []
    for N in (4, 8, 16):
        data = make_step_inputs(N, device)
        shapes = data["shapes"]
        f_ag, f_rs = flops(shapes, N)
        fl = {"ag": f_ag, "rs": f_rs}
        # every point runs interleaved with the undecomposed op in this kernel
        # and with torch.matmul on the concatenated operands, so that the
        # ratios compare calls made under the same clocks
        mono = Step(N, 1, "none", data, device)
        X1, W1, X2, W2 = concat_operands(mono, shapes, N)
        comp = {"ag": {"none": mono.ag, "torch": lambda: torch.matmul(X1, W1.t())},
                "rs": {"none": mono.rs, "torch": lambda: torch.matmul(X2, W2.t())}}

        def emit(op, chunks, ring, fn, check):
            t = time_interleaved({"dec": fn, **comp[op]}, max(20, args.steps), torch, warmup=args.warmup)
            check()
            tf = fl[op] / (t["dec"] / 1e3) / 1e12
            pt = {"sweep": WORKLOAD, "op": op, "N": N, "chunks": chunks, "ring": ring,
                  "ms": t["dec"], "tflops": tf, "frac_of_peak": tf / peak,
                  "vs_undecomposed_time": t["dec"] / t["none"],
                  "vs_torch_time": t["dec"] / t["torch"],
                  "ms_undecomposed": t["none"], "ms_torch": t["torch"],
                  "peak_source": kind}
            points.append(pt)
            print(json.dumps(pt), flush=True)

        for direction in ("uni", "bidi"):
            for chunks in (1, 2, 4):
                st = Step(N, chunks, direction, data, device)
                emit("ag", chunks, direction, st.ag, lambda: st.check(("ag",)))
                emit("rs", chunks, direction, st.rs, lambda: st.check(("rs",)))
                del st
        # pipeline-chunk ReduceScatter ([HTP] section 6) next to the moving bucket
        for chunks in (1, 2, 4):
            st = Step(N, chunks, "uni", data, device)
            emit("rs", chunks, "pipelined", st.rs_pipe, lambda: st.check(("rs_pipe",)))
            del st
        mono.check()
        del mono, X1, W1, X2, W2, comp
        del data
        torch.cuda.empty_cache()
    for line in sweep_best(points):
        print(json.dumps(line), flush=True)
    return 0


def named_workload_inputs(name):
    """(N, inputs) of a named workload other than the MLP sweep; an op the
    workload does not define gets a tiny stand-in so that Step can be built."""
    from collective_matmul_decomposition_gb300 import inputs as gen
    wl = gen.WORKLOADS[name]
    N = wl["N"]
    a = wl.get("ag") or {"m": 128, "K": 128, "n": 256, "x": gen.NORMAL1, "w": gen.NORMAL002, "seed": 1}
    r = wl.get("rs") or {"M": 128 * N, "k": 128, "n": 256, "x": gen.NORMAL1, "w": gen.NORMAL002, "seed": 2}
    x1, w1 = gen.ag_inputs(N, a["m"], a["K"], a["n"], a["x"], a["w"], a["seed"], "nk")
    x2, w2 = gen.rs_inputs(N, r["M"], r["k"], r["n"], r["x"], r["w"], r["seed"], "nk")
    return N, {"shapes": {"ag": dict(m=a["m"], K=a["K"], n=a["n"]), "rs": dict(M=r["M"], k=r["k"], n=r["n"])},
               "cpu": (x1, w1, x2, w2)}


def algorithmic_bytes(op, N, sh, out_bytes):
    """Bytes an op must move at least: the ring's traffic (AG: every shard
    written into N - 1 receive slots and read back; RS: every partial bucket
    of N - 1 hops written and read as fp32) plus reading the operands and
    writing the output once."""
    if op == "ag":
        m, K, n = sh["m"], sh["K"], sh["n"]
        ring = 2 * N * (N - 1) * m * K * 2
        return ring, ring + N * m * K * 2 + N * K * n * 2 + N * N * m * n * out_bytes
    M, k, n = sh["M"], sh["k"], sh["n"]
    ring = 2 * N * (N - 1) * (M // N) * n * 4
    return ring, ring + N * M * k * 2 + N * k * n * 2 + M * n * out_bytes


# The five workloads, each op with the ring the configuration names, plus the
# other ring for the GPT-3 layer (its configuration names the bidirectional one).
CONFIG_RUNS = [
    ("tiny_n2", "ag", "uni", 1), ("tiny_n2", "rs", "uni", 1),
    ("sp_mlp_fc1_ag_n8", "ag", "uni", 1), ("sp_mlp_fc2_rs_n8", "rs", "uni", 1),
    ("gpt3_h12288_s2048_n8", "ag", "bidi", 1), ("gpt3_h12288_s2048_n8", "rs", "bidi", 1),
    ("gpt3_h12288_s2048_n8", "ag", "uni", 1), ("gpt3_h12288_s2048_n8", "rs", "uni", 1),
    (WORKLOAD, "ag", "uni", 1), (WORKLOAD, "rs", "uni", 1),
]


def run_configs(args):
    """Every configuration's ops: ms per call (median of interleaved rounds
    with the undecomposed op in this kernel and torch.matmul on the
    concatenated operands), TFLOP/s, and the roofline fractions (tensor
    against the measured dense bf16 peak that matches the clocks sampled
    during the rounds, see choose_peak, and HBM against the measured copy
    bandwidth for the algorithmic bytes), one JSON line each."""
    import torch
    import __graft_entry__
    from collective_matmul_decomposition_gb300 import inputs as gen
    __graft_entry__.build()
    device = torch.device("cuda", 0)
    peaks, kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    cache = {}
    for name, op, ring, chunks in CONFIG_RUNS:
        if name not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            if name == WORKLOAD:
                N, data = 8, make_step_inputs(8, device)
            else:
                N, data = named_workload_inputs(name)
            yd = torch.float32 if gen.WORKLOADS[name]["y_dtype"] == "f32" else torch.bfloat16
            mono = Step(N, 1, "none", data, device, yd)
            X1, W1, X2, W2 = concat_operands(mono, data["shapes"], N)
            cache[name] = (N, data, yd, mono, X1, W1, X2, W2)
        N, data, yd, mono, X1, W1, X2, W2 = cache[name]
        st = Step(N, chunks, ring, data, device, yd)
        torch_fn = (lambda: torch.matmul(X1, W1.t())) if op == "ag" else (lambda: torch.matmul(X2, W2.t()))
        fns = {"dec": getattr(st, op), "none": getattr(mono, op), "torch": torch_fn}
        alt = None
        if op == "rs" and ring != "none":   # the same ring with one buffer per (rank, step)
            alt = Step(N, chunks, ring, data, device, yd).set_rs_in_place(0)
            fns["per_step"] = alt.rs
        with ClockSampler(physical_gpu_id(0)) as clk:
            t = time_interleaved(fns, max(20, args.steps), torch, warmup=args.warmup)
        st.check((op,))
        mono.check((op,))
        if alt is not None:
            alt.check(("rs",))
        clocks = clk.summary()
        timed_s = max(20, args.steps) * sum(t.values()) / 1e3
        peak, peak_which, peak_why = choose_peak(peaks, timed_s, clocks)
        # the decomposed output against torch.matmul of the same operands
        # (normwise max relative error; the parity tests hold the oracle's)
        with torch.no_grad():
            ref = torch_fn().float()
            if op == "ag":
                sh = data["shapes"]["ag"]
                ref = ref.reshape(N * sh["m"], N, sh["n"]).permute(1, 0, 2)
                got = st.y1.float()
            else:
                ref = ref.reshape(N, -1, ref.shape[-1])
                got = st.y2.float()
            err_vs_torch = float((got - ref).abs().max() / ref.abs().max())
        f_ag, f_rs = flops(data["shapes"], N)
        fl = f_ag if op == "ag" else f_rs
        tf = fl / (t["dec"] / 1e3) / 1e12
        ring_b, alg_b = algorithmic_bytes(op, N, data["shapes"][op], 4 if yd == torch.float32 else 2)
        gbs = alg_b / (t["dec"] / 1e3) / 1e9
        ai = fl / alg_b
        bound = "tensor" if ai >= peak * 1e12 / (hbm * 1e9) else "hbm"
        print(json.dumps({
            "config": name, "op": op, "N": N, "chunks": chunks, "ring": ring,
            "ms": t["dec"], "tflops": tf, "bound": bound,
            "frac_tensor": tf / peak, "algorithmic_bytes": alg_b, "ring_bytes": ring_b,
            "achieved_gbs": gbs, "frac_hbm": gbs / hbm, "flop_per_byte": ai,
            "frac": tf / peak if bound == "tensor" else gbs / hbm,
            "ms_undecomposed": t["none"], "ms_torch": t["torch"],
            "vs_undecomposed_time": t["dec"] / t["none"], "vs_torch_time": t["dec"] / t["torch"],
            "ms_rs_per_step_buffers": t.get("per_step"),
            "max_rel_err_vs_torch": err_vs_torch,
            "rounds": max(20, args.steps), "clocks": clocks,
            "peak_source": f"{peak_which} dense bf16 {peak} ({peak_why}) and hbm_gbs {hbm} of {kind}"}), flush=True)
        del st, alt
    return 0


# NVLink-class per-GPU rates for the gate's projection (one direction of one
# link to a ring neighbour, and the native collective's bandwidth through the
# same fabric); a stated assumption, not a measurement of this box.
NVLINK_GBS, NVLINK_HOP_US = 900.0, 2.0


def run_gate(args):
    """The cost model against measurement, with rates calibrated on this GPU.

    For each workload and op: the decomposed and the undecomposed op timed
    interleaved, and the model's prediction of both.  The model's one-GPU
    rates are measured separately from the decomposed op they predict:
    - compute: each rank's share of this GPU's rate on the undecomposed op of
      the same shape (so the undecomposed prediction equals its measurement
      by construction; the decomposed prediction is the test);
    - ring: GEMM->ReduceScatter, each rank's share of the ring's own
      throughput, from the same ring run with almost no compute (a
      contraction of 64): the bytes one hop carries, summed over ranks and
      steps, over that call's time; AllGather->GEMM, each rank's share of
      the HBM copy rate (the same kind of run, with 256 output columns, is
      latency-bound and is printed for reference);
    - the native collective moves nothing on one GPU (every partial already
      sits in one memory), a message costs one flag round trip (1 us), and
      the realigning addition runs at each rank's share of the HBM copy rate.
    Each line gives the predictions, the relative error of the decomposed
    one, the model's choice and whether measurement agrees (within 5 %), the
    choice under NVLink-class rates as a labelled projection, and the
    Einsum-level choice (which collective to decompose) for the same shapes
    under those rates."""
    import torch
    import __graft_entry__
    from collective_matmul_decomposition_gb300 import cm
    from collective_matmul_decomposition_gb300 import inputs as gen
    __graft_entry__.build()
    device = torch.device("cuda", 0)
    peaks, kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    cases = [("sp_mlp_fc1_ag_n8", ("ag",), None), ("sp_mlp_fc2_rs_n8", ("rs",), None),
             ("gpt3_h12288_s2048_n8", ("ag", "rs"), None), ("gpt3_h12288_s2048_n8", ("ag", "rs"), "uni")]
    cases += [(f"{WORKLOAD}:N={N}", ("ag", "rs"), None) for N in (4, 8, 16)]
    for name, ops, ring_override in cases:
        if name.startswith(WORKLOAD):
            N = int(name.split("=")[1])
            data, direction, chunks = make_step_inputs(N, device), "uni", 1
        else:
            N, data = named_workload_inputs(name)
            direction, chunks = gen.WORKLOADS[name]["direction"], gen.WORKLOADS[name]["chunks"]
        direction = ring_override or direction
        f_ag, f_rs = flops(data["shapes"], N)
        dec, mono = Step(N, chunks, direction, data, device), Step(N, 1, "none", data, device)
        for op in ops:
            fl = f_ag if op == "ag" else f_rs
            # interleaved, so that both forms run under the same clocks
            t = time_interleaved({"dec": getattr(dec, op), "none": getattr(mono, op)}, max(20, args.steps), torch,
                                 warmup=args.warmup)
            ms_dec, ms_none = t["dec"], t["none"]
            dec.check((op,))
            mono.check((op,))
            sh = data["shapes"][op]
            rows, K, n = (sh["m"], sh["K"], sh["n"]) if op == "ag" else (sh["M"], sh["k"], sh["n"])
            code = cm.CM_OP_AG_GEMM if op == "ag" else cm.CM_OP_GEMM_RS
            ring_bytes, ms_ring = ring_calibration(cm, torch, device, op, N, direction, chunks, rows, K, n)
            rate = fl / (ms_none / 1e3) / 1e12   # this GPU's rate on the undecomposed op
            ring_gbs = ring_bytes / (ms_ring / 1e3) / 1e9
            # AG: a forward reads and writes each byte once, so a rank's link is
            # its share of the HBM copy rate (the peak-rate reading); the
            # calibration run, with one column tile per row tile, forwards from
            # a few tiles at a time and measures their latency instead (kept in
            # the line for reference).  RS: the calibration runs the real bucket
            # epilogue on every tile, so its rate is the ring's.
            ring_model = hbm / 2 if op == "ag" else ring_gbs
            one_gpu = dict(gemm_tflops=rate / N, ring_gbs=ring_model / N, coll_gbs=1e12, hop_us=1.0,
                           mem_gbs=hbm / 2 / N)
            pred_dec = cm.cost_estimate(N, chunks, direction, code, rows, K, n, one_gpu) / 1e3
            pred_none = cm.cost_estimate(N, 1, "none", code, rows, K, n, one_gpu) / 1e3
            # the same rates for both ring directions: which one the model prefers
            pred_ring = {d: cm.cost_estimate(N, chunks, d, code, rows, K, n, one_gpu) / 1e3 for d in ("uni", "bidi")}
            pick = cm.plan_choose(N, code, rows, K, n, one_gpu)
            nvl = dict(gemm_tflops=rate, ring_gbs=NVLINK_GBS, coll_gbs=NVLINK_GBS, hop_us=NVLINK_HOP_US, mem_gbs=hbm)
            pick_nvl = cm.plan_choose(N, code, rows, K, n, nvl)
            m_e = rows if op == "ag" else rows // N
            k_e = K
            ein = cm.plan_choose_einsum(N, m_e, k_e, n, nvl)
            faster = "decomposed" if ms_dec < ms_none else "undecomposed"
            # within 5 % either way is a tie, and a tie agrees with either choice
            agrees = (ms_none <= ms_dec * 1.05) if pick[1] == "none" else (ms_dec <= ms_none * 1.05)
            print(json.dumps({"gate": name, "op": op, "N": N, "chunks": chunks, "ring": direction,
                              "measured_ms": {"decomposed": ms_dec, "undecomposed": ms_none, "faster": faster},
                              "calibration": {"ring_bytes": ring_bytes, "ring_ms": ms_ring, "ring_gbs": ring_gbs,
                                              "gemm_tflops": rate},
                              "one_gpu_model": {"rates": one_gpu, "decomposed_ms": pred_dec,
                                                "undecomposed_ms": pred_none,
                                                "decomposed_rel_err": (pred_dec - ms_dec) / ms_dec,
                                                "undecomposed_rel_err": (pred_none - ms_none) / ms_none,
                                                "choice": {"chunks": pick[0], "ring": pick[1]},
                                                "agrees_with_measurement": agrees,
                                                "decomposed_ms_by_ring": pred_ring},
                              "nvlink_projection": {"rates": nvl, "choice": {"chunks": pick_nvl[0], "ring": pick_nvl[1]},
                                                    "predicted_ms": pick_nvl[2] / 1e3,
                                                    "einsum_offering_both": {"decompose": ein[0], "chunks": ein[1],
                                                                             "ring": ein[2],
                                                                             "predicted_ms": ein[3] / 1e3,
                                                                             "m": m_e, "K": k_e, "n": n}},
                              "peak_source": kind}), flush=True)
        del dec, mono, data
        torch.cuda.empty_cache()
    return 0


def ring_calibration(cm, torch, device, op, N, direction, chunks, rows, K, n):
    """The ring's own throughput with almost no compute: (bytes one hop
    carries, summed over ranks and steps; median ms of one call).  AG: the
    same shards (m x K) rotated, 256 output columns; RS: the same buckets
    ((rows/N) x n fp32) circulated, a contraction of 64."""
    from collective_matmul_decomposition_gb300 import inputs as gen
    plan = cm.Plan(N, chunks, direction)
    hops = N - 1
    if op == "ag":
        n_cal = 256
        x, w = gen.ag_inputs(N, rows, K, n_cal, gen.NORMAL1, gen.NORMAL002, seed=77, w_layout="nk")
        x, w = x.to(device), w.to(device)
        y = torch.empty(N, N * rows, n_cal, dtype=torch.bfloat16, device=device)
        ws = torch.empty(plan.ag_workspace_size(rows, K), dtype=torch.uint8, device=device)
        fn = lambda: cm.cm_ag_gemm(plan, x, w, y, ws, "nk")
        ring_bytes = N * hops * rows * K * 2
    else:
        k_cal = 64
        x, w = gen.rs_inputs(N, rows, k_cal, n, gen.NORMAL1, gen.NORMAL002, seed=78, w_layout="nk")
        x, w = x.to(device), w.to(device)
        y = torch.empty(N, rows // N, n, dtype=torch.bfloat16, device=device)
        ws = torch.empty(plan.rs_workspace_size(rows, n), dtype=torch.uint8, device=device)
        fn = lambda: cm.cm_gemm_rs(plan, x, w, y, ws, "nk")
        ring_bytes = N * hops * (rows // N) * n * 4
    ms = time_interleaved({"ring": fn}, 20, torch, warmup=3)["ring"]
    st, info = cm.cm_check_status(ws)
    if st != 0:
        raise RuntimeError(f"ring calibration: device status {st} {info}")
    return ring_bytes, ms


def run_backward(args):
    """The backward pair of the MLP fc1 (column-parallel) layer at N ranks: data
    gradient (GEMM-RS of dY_r @ W_r) and weight gradient (dY_r^T @ gathered X),
    with the gather on a second stream under the GEMM-RS (bulk overlap) and
    without; the data gradient alone next to them."""
    import torch
    import __graft_entry__
    from collective_matmul_decomposition_gb300 import cm
    from collective_matmul_decomposition_gb300 import inputs as gen
    __graft_entry__.build()
    device = torch.device("cuda", 0)
    peaks, kind = load_peaks()
    for N in (4, 8, 16):
        sh = gen.mlp_shapes(N)["ag"]
        m, K, n = sh["m"], sh["K"], sh["n"]
        T = N * m
        x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=6000, w_layout="nk")
        dy, _ = gen.ag_inputs(N, T, n, 1, gen.NORMAL1, gen.NORMAL1, seed=6001)
        x, w, dy = x.to(device), w.to(device), dy.to(device)
        dx = torch.empty(N, m, K, dtype=torch.bfloat16, device=device)
        dw = torch.empty(N, n, K, dtype=torch.bfloat16, device=device)
        plan = cm.Plan(N, 1, "uni")
        ws = torch.empty(plan.backward_pair_workspace_size(m, K, n), dtype=torch.uint8, device=device)
        flops = 4.0 * N * T * n * K
        res = {}
        for overlap in (1, 0):
            plan.set_option(cm.CM_OPT_BULK_OVERLAP, overlap)
            ms = time_loop(lambda: cm.cm_backward_pair(plan, x, w, dy, dx, dw, ws), args.steps, torch,
                           warmup=args.warmup)
            st, info = cm.cm_check_status(ws)
            if st != 0:
                raise RuntimeError(f"backward pair: device status {st} {info}")
            res["overlap" if overlap else "serial"] = ms
        ms_dgrad = time_loop(lambda: cm.cm_gemm_rs(plan, dy, w, dx, ws, "kn"), args.steps, torch, warmup=args.warmup)
        print(json.dumps({"backward_pair": WORKLOAD, "N": N, "m": m, "K": K, "n": n,
                          "ms_bulk_overlap": res["overlap"], "ms_serial_gather": res["serial"],
                          "ms_dgrad_alone": ms_dgrad,
                          "tflops_bulk_overlap": flops / (res["overlap"] / 1e3) / 1e12,
                          "frac_of_peak": flops / (res["overlap"] / 1e3) / 1e12 / float(peaks["bf16_tflops"]),
                          "gather_bytes": N * N * m * K * 2, "peak_source": kind}), flush=True)
        del x, w, dy, dx, dw, ws
        torch.cuda.empty_cache()
    return 0


def run_cannon(args):
    """Cannon-style 2-D rotation on q x q logical ranks for C = A @ B with
    A, B, C of 8192 x 8192 (bf16 in, bf16 out), against the same GEMM as one
    launch of this kernel (N=1) and torch.matmul."""
    import torch
    import __graft_entry__
    from collective_matmul_decomposition_gb300 import cm
    from collective_matmul_decomposition_gb300 import inputs as gen
    __graft_entry__.build()
    device = torch.device("cuda", 0)
    peaks, kind = load_peaks()
    S = 8192
    for q in (2, 4):
        b_ = S // q
        a, _ = gen.ag_inputs(q * q, b_, b_, 1, gen.NORMAL1, gen.NORMAL002, seed=7000)
        b, _ = gen.ag_inputs(q * q, b_, b_, 1, gen.NORMAL1, gen.NORMAL002, seed=7001)   # blocks [bn][bk]
        a, b = a.to(device), b.to(device)
        c = torch.empty(q * q, b_, b_, dtype=torch.bfloat16, device=device)
        plan = cm.Plan(q * q, 1, "uni")
        ws = torch.empty(plan.cannon_workspace_size(b_, b_, b_), dtype=torch.uint8, device=device)
        ms = time_loop(lambda: cm.cm_cannon_gemm(plan, a, b, c, ws, "nk"), args.steps, torch, warmup=args.warmup)
        st, info = cm.cm_check_status(ws)
        if st != 0:
            raise RuntimeError(f"cannon: device status {st} {info}")
        A = a.reshape(q, q, b_, b_).permute(0, 2, 1, 3).reshape(S, S).contiguous()
        Bt = b.reshape(q, q, b_, b_).permute(1, 2, 0, 3).reshape(S, S).contiguous()   # [n][K]
        one = cm.Plan(1, 1, "uni")
        y1 = torch.empty(1, S, S, dtype=torch.bfloat16, device=device)
        ws1 = torch.empty(one.ag_workspace_size(S, S), dtype=torch.uint8, device=device)
        ms_mono = time_loop(lambda: cm.cm_ag_gemm(one, A[None], Bt[None], y1, ws1, "nk"), args.steps, torch,
                            warmup=args.warmup)
        ms_torch = time_loop(lambda: torch.matmul(A, Bt.t()), args.steps, torch, warmup=args.warmup)
        fl = 2.0 * S ** 3
        print(json.dumps({"cannon": f"{S}x{S}x{S}", "q": q, "ms": ms, "tflops": fl / (ms / 1e3) / 1e12,
                          "ms_monolithic_same_kernel": ms_mono, "ms_torch": ms_torch,
                          "rotation_bytes_per_step": 2 * q * q * b_ * b_ * 2, "peak_source": kind}), flush=True)
        del a, b, c, ws, A, Bt, y1, ws1
        torch.cuda.empty_cache()
    return 0


def run_profile_case(args):
    """A few calls of one op of one workload, nothing else: the command ncu captures."""
    import torch
    import __graft_entry__
    from collective_matmul_decomposition_gb300 import inputs as gen
    __graft_entry__.build()
    device = torch.device("cuda", 0)
    N = args.ranks
    if args.workload == WORKLOAD:
        data = make_step_inputs(N, device)
    else:
        N, data = named_workload_inputs(args.workload)
    st = Step(N, args.chunks, args.ring, data, device)
    st.plan.set_option(st.cm.CM_OPT_KERNEL, args.kernel)
    st.plan.set_option(st.cm.CM_OPT_STATIC_TILES, args.static_tiles)
    if args.tile_group:
        st.plan.set_option(st.cm.CM_OPT_TILE_GROUP, args.tile_group)
    if args.l2_hints >= 0:
        st.plan.set_option(st.cm.CM_OPT_L2_HINTS, args.l2_hints)
    if args.l2_promotion >= 0:
        st.plan.set_option(st.cm.CM_OPT_L2_PROMOTION, args.l2_promotion)
    if args.row_band >= 0:
        st.plan.set_option(st.cm.CM_OPT_ROW_BAND, args.row_band)
    if args.rs_preload >= 0:
        st.plan.set_option(st.cm.CM_OPT_RS_PRELOAD, args.rs_preload)
    if args.rs_in_place >= 0:
        st.set_rs_in_place(args.rs_in_place)
    if args.rs_epilogue >= 0:
        st.plan.set_option(st.cm.CM_OPT_RS_EPILOGUE, args.rs_epilogue)
    if args.task_order >= 0:
        st.plan.set_option(st.cm.CM_OPT_TASK_ORDER, args.task_order)
    if args.rs_col_slabs >= 0:
        st.plan.set_option(st.cm.CM_OPT_RS_COL_SLABS, args.rs_col_slabs)
    fn = {"ag": st.ag, "rs": st.rs, "rs_pipe": st.rs_pipe}[args.profile]
    f_ag, f_rs = flops(data["shapes"], N)
    ms = time_loop(fn, args.steps, torch, warmup=args.warmup)
    st.check((args.profile,))
    fl = f_ag if args.profile == "ag" else f_rs
    print(json.dumps({"profile_case": args.workload, "op": args.profile, "N": N, "chunks": args.chunks,
                      "ring": args.ring, "kernel": args.kernel, "static_tiles": args.static_tiles, "tile_group": args.tile_group, "l2_hints": args.l2_hints, "l2_promotion": args.l2_promotion, "row_band": args.row_band, "rs_preload": args.rs_preload, "rs_in_place": args.rs_in_place,
                      "rs_epilogue": args.rs_epilogue, "task_order": args.task_order,
                      "rs_col_slabs": args.rs_col_slabs,
                      "ms": ms, "tflops": fl / (ms / 1e3) / 1e12}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--gate", action="store_true", help="the cost model's choices against measurement")
    ap.add_argument("--backward", action="store_true", help="the backward pair of the MLP fc1 layer")
    ap.add_argument("--cannon", action="store_true", help="Cannon-style 2-D rotation, 8192^3")
    ap.add_argument("--configs", action="store_true",
                    help="every configuration's ops with roofline fractions, one JSON line each")
    ap.add_argument("--profile", choices=["ag", "rs", "rs_pipe"], default=None,
                    help="run only --steps calls of one op (for ncu captures)")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--ranks", type=int, default=8)
    ap.add_argument("--chunks", type=int, default=1)
    ap.add_argument("--ring", choices=["uni", "bidi", "none"], default="uni")
    ap.add_argument("--kernel", type=int, default=0, help="CM_OPT_KERNEL for --profile")
    ap.add_argument("--static-tiles", type=int, default=0, help="CM_OPT_STATIC_TILES for --profile")
    ap.add_argument("--tile-group", type=int, default=0, help="CM_OPT_TILE_GROUP for --profile (0 = default)")
    ap.add_argument("--l2-hints", type=int, default=-1, help="CM_OPT_L2_HINTS for --profile (-1 = default)")
    ap.add_argument("--l2-promotion", type=int, default=-1, help="CM_OPT_L2_PROMOTION for --profile (-1 = default)")
    ap.add_argument("--row-band", type=int, default=-1, help="CM_OPT_ROW_BAND for --profile (-1 = default)")
    ap.add_argument("--rs-preload", type=int, default=-1, help="CM_OPT_RS_PRELOAD for --profile (-1 = default)")
    ap.add_argument("--rs-in-place", type=int, default=-1, help="CM_OPT_RS_IN_PLACE for --profile (-1 = default)")
    ap.add_argument("--rs-epilogue", type=int, default=-1, help="CM_OPT_RS_EPILOGUE for --profile (-1 = default)")
    ap.add_argument("--task-order", type=int, default=-1, help="CM_OPT_TASK_ORDER for --profile (-1 = default)")
    ap.add_argument("--rs-col-slabs", type=int, default=-1, help="CM_OPT_RS_COL_SLABS for --profile (-1 = default)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="oracle seconds for the cpu_baseline of the default arm")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="oracle seconds for a whole --impl reference run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)        # at least 3 untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.gate:
        return run_gate(args)
    if args.backward:
        return run_backward(args)
    if args.cannon:
        return run_cannon(args)
    if args.configs:
        return run_configs(args)
    if args.profile:
        return run_profile_case(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
