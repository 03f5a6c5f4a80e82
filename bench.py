#!/usr/bin/env python3
"""Benchmark of the fused MoE expert forward on GB300.

One step = the whole hot path on one batch: top-k routing of the router
logits, then the fused expert forward (schedule tables + gather, L1 grouped
GEMM + SwiGLU/requant epilogue, L2 grouped GEMM, combine), all in this
repository's CUDA kernels through the C ABI.

The headline workload is the prefill shape (T=8192, H=7168, I=2048, E=256,
top-8), the largest configuration and the compute-bound one; the
decode shape (T=128, same model) is timed after it in the same run and
reported under "per_workload" (device-timed, with its own roofline).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line.  N > 1 runs under torchrun as independent replicas
(the path has no data exchange on one GPU), barrier + max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_expert_ffn_route_gb300 import synth  # noqa: E402

METRIC = "fused MoE fwd tokens/s & TFLOP/s, % of roofline (1×GB300)"
DEFAULT_WORKLOAD = "prefill"          # the largest single-GPU configuration (compute-bound)
ALSO_TIMED = ("decode",)              # timed after the headline in the same run (weight-streaming)
L2_BYTES = 129 * 1024 * 1024
KERNELS_PER_STEP = 5      # route, layout count, dispatch/gather, grouped GEMM (L1 + L2), combine


def peaks():
    """Measured HBM GB/s and FP8-rate (block-scaled mxf8f6f4) TFLOP/s."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        m = json.load(open(path))
        # the block-scaled FP8xFP4 MMA runs at the FP8 rate: 2x bf16 (nominal 4.5 / 2.25)
        return dict(hbm_gbs=m["hbm_gbs"], fp8_tflops=2.0 * m["bf16_tflops"],
                    fp8_tflops_sustained=2.0 * m["bf16_tflops_sustained"], source="measured")
    return dict(hbm_gbs=6800.0, fp8_tflops=3800.0, fp8_tflops_sustained=3400.0, source="fallback")


def algorithmic(wl, counts):
    """Useful FLOPs and algorithmic HBM bytes of one forward (and of the L1
    GEMM launch alone), counting only experts that receive rows."""
    N = wl.N
    H, I = wl.H, wl.I
    touched = int((counts > 0).sum())
    f_l1 = 2.0 * N * 2 * H * I
    f_l2 = 2.0 * N * H * I
    w1 = touched * 2 * I * H * (0.5 + 1 / 32)          # E2M1 + UE8M0
    w2 = touched * H * I * (0.5 + 1 / 32)
    act_x = N * H * (1 + 1 / 32)                        # gathered E4M3 rows + scales
    act_h = N * I * (1 + 1 / 32)
    y_pool = 2.0 * N * H
    b_l1 = w1 + act_x + act_h                           # reads W1 and X, writes H
    b_l2 = w2 + act_h + y_pool                          # reads W2 and H, writes Y rows
    total_b = w1 + w2 + act_x + 2 * act_h + y_pool      # the pages' byte model plus scales
    return dict(flops=f_l1 + f_l2, bytes=total_b, l1_flops=f_l1, l1_bytes=b_l1,
                l2_flops=f_l2, l2_bytes=b_l2, touched=touched)


class ClockSampler:
    """nvidia-smi samples every 20 ms (as fast as it answers) while running.
    Entering waits for the first sample, so the samples taken between enter
    and exit fall inside the caller's timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.lines = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.perf_counter()
            while not self.lines and time.perf_counter() - t0 < 5.0 and self.proc.poll() is None:
                time.sleep(0.005)
            self.lines = []
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi -lms 20"}


class NvmlSampler:
    """The same record read through NVML every 2 ms by a thread while running
    (nvidia-smi answers every ~20 ms, which leaves a timed region of a few ms
    without a sample).  Reads only; raises OSError where NVML or the device's
    handle is unavailable, and the caller falls back to ClockSampler."""

    REASONS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40), ("sw_thermal_slowdown", 0x20),
               ("sw_power_cap", 0x4))

    def __init__(self, dev):
        import ctypes
        import torch
        self.ct = ctypes
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError as e:
            raise OSError(f"no NVML: {e}")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(dev)
        bus = getattr(props, "pci_bus_id", None)
        if bus is not None:
            busid = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), bus, getattr(props, "pci_device_id", 0))
            rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(busid.encode(), ctypes.byref(self.h))
        else:
            n = ctypes.c_uint()
            if self.lib.nvmlDeviceGetCount_v2(ctypes.byref(n)) != 0 or n.value != torch.cuda.device_count():
                raise OSError("cannot match the CUDA device to an NVML device")
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(dev.index, ctypes.byref(self.h))
        if rc != 0:
            raise OSError(f"no NVML handle ({rc})")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        if self.reasons_fn is None:
            self.reasons_fn = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0 else None
        self.samples = []
        self.stop = threading.Event()
        if self._sample() is None:
            raise OSError("NVML clock query failed")

    def _sample(self):
        ct = self.ct
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk)) != 0:   # 1: NVML_CLOCK_SM
            return None
        if self.reasons_fn(self.h, ct.byref(rs)) != 0:
            return None
        return float(clk.value), int(rs.value)

    def _poll(self):
        while not self.stop.is_set():
            v = self._sample()
            if v is not None:
                self.samples.append(v)
            self.stop.wait(0.002)

    def __enter__(self):
        self.samples = []
        self.thread = threading.Thread(target=self._poll, daemon=True)
        self.thread.start()
        return self

    def __exit__(self, *exc):
        self.stop.set()
        self.thread.join(timeout=5)

    def summary(self):
        reasons = sorted({n for _, r in self.samples for n, bit in self.REASONS if r & bit})
        sm = [c for c, _ in self.samples]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(sm), "source": "nvml, every 2 ms"}


def clock_sampler(dev):
    """NVML sampler where the driver's library answers, else nvidia-smi."""
    try:
        return NvmlSampler(dev)
    except Exception:
        return ClockSampler(dev.index)


def traffic_from_profile(kernel_src_hash: str, workload: str, units_scale: float):
    """DRAM bytes per grouped-GEMM launch from the committed ncu summary, if it
    was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "grouped_gemm_traffic.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_hash = re.search(r"kernel source sha256:\s*([0-9a-f]{16,64})", text)
    m_val = re.search(rf"dram bytes per launch \({workload}\):\s*([0-9.eE+]+)", text)
    if not m_hash or not m_val or not kernel_src_hash.startswith(m_hash.group(1)):
        return None
    return float(m_val.group(1)) * units_scale


def kernel_hash() -> str:
    """sha256 of the GEMM kernel's source with `//` comments, trailing spaces
    and blank lines removed: a change of comments keeps a profile valid."""
    h = hashlib.sha256()
    for f in ("gemm_kernels.cu", "common.cuh"):
        text = open(os.path.join(ROOT, "moe_expert_ffn_route_gb300", "csrc", f)).read()
        for line in text.splitlines():
            code = re.sub(r"//.*$", "", line).rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()


def cpu_baseline(wl, inp, idx, w, budget_s: float = 10.0):
    """The oracle as it stands on this host's cores, on a bounded token sample."""
    import oracle
    rng = np.random.default_rng(0)
    n = min(8, wl.T)
    t0 = time.perf_counter()
    oracle.forward(inp, idx, w, tokens=rng.choice(wl.T, n, replace=False))
    dt = time.perf_counter() - t0
    n2 = int(min(wl.T, max(n, n * budget_s / max(dt, 1e-3))))
    toks = rng.choice(wl.T, n2, replace=False)
    t0 = time.perf_counter()
    oracle.forward(inp, idx, w, tokens=toks)
    dt = time.perf_counter() - t0
    return {"value": n2 / dt, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n2} of {wl.T} tokens of workload {wl.name}, all k slots, fp64 direct loop"}


def setup_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks of the process group (the value
    itself without one): the job is as slow as its slowest replica."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, max_ms: float) -> float:
    """Units per second of the whole job: every replica processes
    `units_per_rank` units; the job takes the slowest replica's time."""
    return units_per_rank * world / (max_ms / 1e3)


def run_reference(args, wl):
    """--impl reference: the oracle, timed on this host's cores (rank 0 only)."""
    world, rank, _ = setup_dist()
    if rank != 0:
        return
    import oracle
    inp = synth.make_inputs(wl)
    idx, w = oracle.route(inp["logits"], wl.k)
    rng = np.random.default_rng(1)
    n = min(wl.T, 8)
    t0 = time.perf_counter()
    oracle.forward(inp, idx, w, tokens=rng.choice(wl.T, n, replace=False))
    per_tok = (time.perf_counter() - t0) / n
    # each step: a token sample sized so that warmup + steps take about two minutes
    n_step = int(max(1, min(wl.T, 120.0 / max(args.steps + args.warmup, 1) / max(per_tok, 1e-6))))
    for _ in range(args.warmup):
        oracle.forward(inp, idx, w, tokens=rng.choice(wl.T, n_step, replace=False))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.forward(inp, idx, w, tokens=rng.choice(wl.T, n_step, replace=False))
    dt = time.perf_counter() - t0
    value = n_step * args.steps / dt
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy generator)",
            "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
                       "tokens_per_step": n_step},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{n_step} random tokens of {wl.T} per step, all k slots"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


class DeviceRun:
    """One workload resident on the device: inputs, prepared weights, workspace
    and output, plus the timed device steps."""

    def __init__(self, wl, dev, mb):
        import torch
        self.wl, self.dev, self.mb = wl, dev, mb
        self.inp = synth.make_inputs(wl)
        T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
        self.prob = mb.problem(T, H, I, E, k)
        # the same forward with the two layers as two launches (per-layer times)
        self.prob_split = mb.problem(T, H, I, E, k, debug_flags=mb.DEBUG_SPLIT_LAYERS)
        self.tile_n = mb.tile_n(self.prob)

        def up(a):
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint32:
                a = a.view(np.int32)
            return torch.from_numpy(a).to(dev)

        inp = self.inp
        self.prepared = mb.prepare_weights(self.prob, up(inp["w1"]), up(inp["w1_sf"]), up(inp["w2"]),
                                           up(inp["w2_sf"]))
        self.logits, self.x, self.x_sf = up(inp["logits"]), up(inp["x"]), up(inp["x_sf"])
        self.idx = torch.empty((T, k), dtype=torch.int64, device=dev)
        self.wts = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.ws = mb.empty_workspace(self.prob, dev)
        self.y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream()

    def step(self, events=None, logits=None, x=None, x_sf=None, y=None, split=False):
        """One pass of the whole hot path: routing, then the fused forward."""
        mb, k = self.mb, self.wl.k
        logits = self.logits if logits is None else logits
        x = self.x if x is None else x
        x_sf = self.x_sf if x_sf is None else x_sf
        y = self.y if y is None else y
        prob = self.prob_split if split else self.prob
        mb.route_topk(logits, k, self.idx, self.wts)
        if events is None:
            mb.forward(prob, x, x_sf, self.idx, self.wts, self.prepared, self.ws, y)
        else:
            mb.forward_profiled(prob, x, x_sf, self.idx, self.wts, self.prepared, self.ws, y, events)

    def warm(self, W):
        import torch
        for _ in range(W):
            self.step()
            self.flush.fill_(1)
        torch.cuda.synchronize()
        st, code, _ = self.mb.device_status(self.prob, self.ws)
        if st != self.mb.OK:
            raise SystemExit(f"device status {self.mb.STATUS[st]} ({code})")
        counts = self.mb.query(self.prob, self.ws, "counts").view(torch.int32)[: self.wl.E].cpu().numpy()
        self.alg = algorithmic(self.wl, counts)

    def timed(self, K, world):
        """K steps, each bracketed by CUDA events on the launching stream, the L2
        flushed between steps outside the timed intervals; then steps with
        events between the stages.  Returns (per-step ms, stage ms, clocks, wall s)."""
        import torch
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        with clock_sampler(self.dev) as clocks:
            wall0 = time.perf_counter()
            for i in range(K):
                starts[i].record(self.stream)
                self.step()
                ends[i].record(self.stream)
                self.flush.fill_(i & 0xFF)
            torch.cuda.synchronize()
            wall = time.perf_counter() - wall0
        step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        # per-stage times from separate steps with events between the stages (the
        # events keep one kernel from starting before the previous one ends, so
        # these steps are not the timed ones); then the same with the two layers
        # as two launches, for per-layer times
        KP = min(K, 20)
        stage_ms = []
        for split in (False, True):
            stages = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(KP)]
            for i in range(KP):
                self.step(stages[i], split=split)
                self.flush.fill_(i & 0xFF)
            torch.cuda.synchronize()
            stage_ms.append(np.array([[ev[j].elapsed_time(ev[j + 1]) for j in range(4)] for ev in stages]))
        return step_ms, stage_ms, clocks.summary(), wall


def gemm_roofline(alg, gemm_ms, pk):
    """The grouped-GEMM launch (L1 and L2 items) against the bound its
    arithmetic intensity sets.  A tensor-bound launch is timed inside steps
    that run back to back for the whole timed region (tens to hundreds of ms,
    under the board's power cap), so its peak is the sustained FP8-rate figure;
    the fraction of the burst figure is reported beside it."""
    flops = alg["l1_flops"] + alg["l2_flops"]
    nbytes = alg["l1_bytes"] + alg["l2_bytes"]
    compute_bound = flops / (pk["fp8_tflops"] * 1e12) >= nbytes / (pk["hbm_gbs"] * 1e9)
    if compute_bound:
        achieved = flops / (gemm_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["fp8_tflops_sustained"], "unit": "TFLOP/s"}
    else:
        achieved = nbytes / (gemm_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if compute_bound:
        roof["frac_of_burst_peak"] = achieved / pk["fp8_tflops"]
    roof["kernel"] = "grouped_gemm_kernel (L1 items with the SwiGLU/requant epilogue, then L2 items; one launch)"
    roof["peak_source"] = (f"{pk['source']}: MEASURED_PEAKS bf16 sustained x2 (FP8-rate block-scaled MMA, "
                           f"timed inside a long run of steps); of measured"
                           if compute_bound else f"{pk['source']}: MEASURED_PEAKS hbm_gbs; of measured")
    return roof


def step_roofline_time(alg, pk, sustained=False):
    """max(F / P_tc, B / BW): P_tc the burst FP8-rate figure (the stricter
    bound), or the sustained one."""
    p_tc = pk["fp8_tflops_sustained"] if sustained else pk["fp8_tflops"]
    return max(alg["flops"] / (p_tc * 1e12), alg["bytes"] / (pk["hbm_gbs"] * 1e9))


def stage_summary(stage_ms):
    """Stage means of the one-launch forward, and the layer times of the
    two-launch form of the same forward."""
    one, two = stage_ms
    return {"tables+gather": float(one[:, 0].mean()), "grouped_gemm": float(one[:, 1:3].sum(axis=1).mean()),
            "combine": float(one[:, 3].mean()),
            "two_launches": {"l1_gemm": float(two[:, 1].mean()), "l2_gemm": float(two[:, 2].mean())}}


def gemm_ms_of(stage_ms):
    return float(stage_ms[0][:, 1:3].sum(axis=1).mean())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--also", default=",".join(ALSO_TIMED),
                    help="comma-separated workloads timed after the headline (device-timed only); '' for none")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    wl = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
        return

    import torch
    from moe_expert_ffn_route_gb300 import binding as mb

    world, rank, local = setup_dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    R = DeviceRun(wl, dev, mb)
    T, H, k = wl.T, wl.H, wl.k
    R.warm(args.warmup)
    alg = R.alg
    K = args.steps
    step_ms, stage_ms, clock_summary, wall = R.timed(K, world)
    total_ms = max_over_ranks(float(sum(step_ms)), dev)
    if world > 1:
        torch.distributed.barrier()
    ms_per_step = total_ms / K
    value = whole_job_rate(T * K, world, total_ms)

    # e2e through host buffers: pinned inputs -> device, route + forward, y -> pinned host
    inp = R.inp
    h_logits = torch.from_numpy(inp["logits"]).pin_memory()
    h_x = torch.from_numpy(inp["x"]).pin_memory()
    h_xsf = torch.from_numpy(inp["x_sf"].view(np.int32)).pin_memory()
    h_y = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    h2d = h_logits.numel() * 4 + h_x.numel() + h_xsf.numel() * 4
    d2h = T * H * 2
    stream = R.stream
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = 0.0
    for i in range(K):
        e_s.record(stream)
        R.logits.copy_(h_logits, non_blocking=True)
        R.x.copy_(h_x, non_blocking=True)
        R.x_sf.copy_(h_xsf, non_blocking=True)
        R.step()
        h_y.copy_(R.y, non_blocking=True)
        e_e.record(stream)
        torch.cuda.synchronize()
        e2e_ms += e_s.elapsed_time(e_e)
    e2e_ms = max_over_ranks(e2e_ms, dev)

    # the same steps pipelined as a server would run them: two buffer sets, inputs
    # copied in on one stream and y copied out on another, so that the copies of
    # step i overlap the kernels of steps i - 1 and i + 1 (every step still moves
    # its own inputs in and its own y out inside the timed region)
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sets = [{"logits": torch.empty_like(R.logits), "x": torch.empty_like(R.x), "x_sf": torch.empty_like(R.x_sf),
             "y": torch.empty_like(R.y)} for _ in range(2)]
    h_ys = [h_y, torch.empty((T, H), dtype=torch.bfloat16).pin_memory()]
    ready, done, out_done = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    p_s, p_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    p_s.record(cin)
    for i in range(K):
        b = i & 1
        S = sets[b]
        if i >= 2:
            cin.wait_event(done[b])            # step i - 2 no longer reads this set's inputs
        with torch.cuda.stream(cin):
            S["logits"].copy_(h_logits, non_blocking=True)
            S["x"].copy_(h_x, non_blocking=True)
            S["x_sf"].copy_(h_xsf, non_blocking=True)
        ready[b].record(cin)
        stream.wait_event(ready[b])
        if i >= 2:
            stream.wait_event(out_done[b])     # step i - 2's y has left this set
        R.step(logits=S["logits"], x=S["x"], x_sf=S["x_sf"], y=S["y"])
        done[b].record(stream)
        cout.wait_event(done[b])
        with torch.cuda.stream(cout):
            h_ys[b].copy_(S["y"], non_blocking=True)
        out_done[b].record(cout)
    p_e.record(cout)
    torch.cuda.synchronize()
    e2e_pipe_ms = max_over_ranks(p_s.elapsed_time(p_e), dev)

    # further workloads, device-timed in the same process (the other configuration
    # the throughput target names: decode, weight-streaming)
    pk = peaks()
    also = {}
    for name in [a for a in args.also.split(",") if a and a != wl.name]:
        R2 = DeviceRun(synth.WORKLOADS[name], dev, mb)
        R2.warm(args.warmup)
        s2, st2, c2, _ = R2.timed(K, world)
        ms2 = max_over_ranks(float(sum(s2)), dev) / K
        w2 = R2.wl
        also[name] = {
            "config": {"workload": name, "T": w2.T, "H": w2.H, "I": w2.I, "E": w2.E, "k": w2.k,
                       "tile_n": R2.tile_n, "touched_experts": R2.alg["touched"]},
            "value": whole_job_rate(w2.T * K, world, ms2 * K), "unit": "tokens/s",
            "ms_per_step": ms2, "ms_per_step_median": float(np.median(s2)),
            "tflops": R2.alg["flops"] / (ms2 / 1e3) / 1e12 * world,
            "hbm_gbs": R2.alg["bytes"] / (ms2 / 1e3) / 1e9,
            "roofline_step_frac": step_roofline_time(R2.alg, pk) / (ms2 / 1e3),
            "roofline_step_frac_sustained": step_roofline_time(R2.alg, pk, True) / (ms2 / 1e3),
            "stage_ms": stage_summary(st2),
            "roofline": gemm_roofline(R2.alg, gemm_ms_of(st2), pk),
            "clocks": c2,
        }
        also[name]["roofline"]["traffic"] = traffic_from_profile(kernel_hash(), name, 1.0)
        del R2
        torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    roof = gemm_roofline(alg, gemm_ms_of(stage_ms), pk)
    roof["traffic"] = traffic_from_profile(kernel_hash(), wl.name, 1.0)
    t_roof = step_roofline_time(alg, pk)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step,
        "ms_per_step_median": float(np.median(step_ms)), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxf8f6f4 (e4m3 x e2m1, ue8m0/32, fp32 accum, bf16 out)",
        "data": "synthetic (seeded numpy generator; random-init expert weights)",
        "config": {"workload": wl.name, "T": T, "H": H, "I": wl.I, "E": wl.E, "k": k, "tile_n": R.tile_n,
                   "l2": "flushed between steps (256 MiB write outside the timed intervals)",
                   "touched_experts": alg["touched"]},
        "tflops": alg["flops"] / (ms_per_step / 1e3) / 1e12 * world,
        "hbm_gbs": alg["bytes"] / (ms_per_step / 1e3) / 1e9,
        "roofline_step_frac": t_roof / (ms_per_step / 1e3),
        "roofline_step_frac_sustained": step_roofline_time(alg, pk, True) / (ms_per_step / 1e3),
        "stage_ms": stage_summary(stage_ms),
        "roofline": roof,
        "e2e": {"value": whole_job_rate(T * K, world, e2e_pipe_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "mode": "pipelined: inputs in and y out on two copy streams, two buffer sets"},
        "e2e_serial": {"value": whole_job_rate(T * K, world, e2e_ms), "unit": "tokens/s",
                       "mode": "copy in, route + forward, copy out, synchronise; per step"},
        "gpu_launches": KERNELS_PER_STEP * K,
        "wall_s": wall,
    }
    line["clocks"] = clock_summary
    if also:
        line["per_workload"] = also
    if not args.no_cpu_baseline and world == 1:
        import oracle
        ridx, rw = oracle.route(inp["logits"], k)
        line["cpu_baseline"] = cpu_baseline(wl, inp, ridx, rw)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
