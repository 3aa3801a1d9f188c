#!/usr/bin/env python3
"""Throughput of the Mamba-1 selective scan forward + backward on GB300.

One step = ssm_scan_fwd + ssm_scan_bwd (through the C ABI) over one batch of
the Mamba-1.4B-like layer workload: batch 8, seqlen 2048, dinner 4096,
dstate 16, bf16 activations (u, delta_raw, z, B, C, dout), fp32 A_log / D,
fp32 state and accumulation, Euler B.  Inputs are seeded synthetic data with
the distributions of the workload; they are resident in HBM and larger than
L2 (805 MB of activations per step), so no flush is needed between steps.

Prints one JSON line (rank 0).  `value` is whole-job tokens/s in Mtokens/s:
batch*seqlen tokens per step per rank.  Several GPUs run independent
replicas (weak scaling): the scan has no cross-rank exchange on this path.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

--impl reference times the fp64 CPU oracle on the host cores (a bounded
sample of the same workload per step) and prints the same metric.

Other lines (not the benchmark's headline): --block times the whole Mamba-1
block forward + backward on the block workload; --decode times single-token
decode (conv1d+SiLU step + scan step of 48 layers from carried states,
replayed from a CUDA graph) on the decode workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Mamba-1 selective scan fwd+bwd Mtokens/s; achieved % of HBM/SFU roofline"
E2E_SETS = 3   # device buffer sets of the end-to-end leg (uploads / compute / read-backs in flight)
E2E_WINDOWS = 3   # timed windows of the end-to-end leg (their median is reported)
WORKLOAD = "mamba1p4b_scan_bf16"
BLOCK_WORKLOAD = "mamba_block_fp32"
SM_COUNT = 152
PIPE_RATES = os.path.join(ROOT, "profiles", "pipe_rates_gb300.json")
# Used only when the committed pipe-rate measurement is absent (then labelled
# "assumed" in the line): MUFU ex2 and fp32 FFMA lanes per clock per SM.
EX2_PER_CLK_PER_SM_ASSUMED = 32.0
FP32_LANES_PER_CLK_PER_SM_ASSUMED = 128.0
CLOCK_WINDOW_S = 0.6             # minimum span of clock samples around a timed region


def parse():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline leg")
    p.add_argument("--seqlen", type=int, default=None,
                   help="run the workload's generator at this sequence length instead "
                        "(smaller cases for profiler captures; not the benchmark line)")
    p.add_argument("--batch", type=int, default=None,
                   help="batch override, like --seqlen (profiler captures only)")
    p.add_argument("--block", action="store_true",
                   help="time the whole Mamba-1 block (ssm_block_fwd + ssm_block_bwd) on the "
                        "block workload instead of the scan step")
    p.add_argument("--decode", action="store_true",
                   help="time single-token decode (conv1d+SiLU step + scan step per layer) on "
                        "the decode workload instead of the scan step")
    p.add_argument("--conv", action="store_true",
                   help="time the causal depthwise conv1d + SiLU (forward + backward) on the "
                        "block workload's shape instead of the scan step")
    p.add_argument("--measure-pipes", metavar="OUT_JSON", default=None,
                   help="measure the MUFU ex2 and fp32 FFMA / FFMA2 rates of the GPU with the "
                        "library's probe kernels (CUDA events + sampled SM clock), write them "
                        "to OUT_JSON and print them")
    p.add_argument("--measure-gemm-ref", metavar="OUT_JSON", default=None,
                   help="time the block's projection GEMMs through ssm_linear_fwd (3xTF32) beside "
                        "the vendor library's single TF32, BF16 and FP32 GEMMs of the same shapes "
                        "(context for the GEMM's tensor-core rate), write them to OUT_JSON")
    return p.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(ms, ws, device):
    """Slowest rank's time: every rank's work counts only once all are done."""
    if ws <= 1:
        return ms
    import torch
    import torch.distributed as dist
    tt = torch.tensor([float(ms)], device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_rate(tokens_per_rank, ws, ms):
    """Mtokens/s of the whole job: all ranks' tokens over the slowest rank's time."""
    return ws * tokens_per_rank / (ms * 1e-3) / 1e6


def pipe_rates():
    """Per-SM, per-clock MUFU ex2 and fp32 FFMA lane rates: the committed
    measurement (bench.py --measure-pipes) if present, else the assumed values."""
    try:
        with open(PIPE_RATES) as f:
            rec = json.load(f)
        fp32 = max(float(rec["ffma_lanes_per_clk_per_sm"]),
                   float(rec.get("ffma2_lanes_per_clk_per_sm", 0.0)))
        return (float(rec["ex2_per_clk_per_sm"]), fp32,
                f"measured ({os.path.relpath(PIPE_RATES, ROOT)})")
    except (OSError, ValueError, KeyError):
        return EX2_PER_CLK_PER_SM_ASSUMED, FP32_LANES_PER_CLK_PER_SM_ASSUMED, "assumed"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# ----------------------------------------------------------------- algorithmic work

def algorithmic(cfg):
    """Bytes and exponentials of one forward and one backward pass (the
    method's own data, not the implementation's checkpoints)."""
    M, D, N = cfg["batch"] * cfg["seqlen"], cfg["dinner"], cfg["dstate"]
    s = 2 if cfg["dtype"] == "bf16" else 4
    small = D * N * 4 + D * 4
    fwd_bytes = 4 * M * D * s + 2 * M * N * s + small          # u, delta_raw, z in; out; B, C
    bwd_bytes = 7 * M * D * s + 4 * M * N * s + 2 * small      # u, dr, z, dout in; du, ddr, dz out;
    #                                                             B, C in; dB, dC out; A_log/D, dA_log/dD
    exps = M * D * N                                           # exp(delta A) per pass
    return fwd_bytes, bwd_bytes, exps


# fp32 lane-operations per (step, channel, state) element that the
# recurrences need at the least (Euler B): forward delta*A, delta*u*B, the
# h update and the C.h readout (4); backward h recomputed (4: delta*A, a*h,
# + delta*u*B, dC) and the reverse pass (8: C*dy, the g update, g*a*h, the
# sums over states into ddelta and over time into dA, g*B, dB, delta*A).
FP32_OPS_FWD, FP32_OPS_BWD = 4, 12


def alu_roofline(cfg, t_fwd, t_bwd, lanes_per_clk, sm_mhz, rate_kind):
    """The same step against the fp32 pipe: the recurrences' minimal fp32
    lane-operations per element over the measured FFMA lane rate."""
    el = cfg["batch"] * cfg["seqlen"] * cfg["dinner"] * cfg["dstate"]
    peak = lanes_per_clk * SM_COUNT * sm_mhz * 1e6              # lane-ops / s
    f, b = FP32_OPS_FWD * el, FP32_OPS_BWD * el
    return {"unit": "Tlane-op/s", "peak": round(peak / 1e12, 3),
            "peak_source": f"{rate_kind} {lanes_per_clk:.1f} fp32 lanes/clk/SM x {SM_COUNT} SMs x "
                           f"{sm_mhz:.0f} MHz",
            "ops_per_element": {"fwd": FP32_OPS_FWD, "bwd": FP32_OPS_BWD},
            "fwd_frac": round(f / peak / (t_fwd * 1e-3), 4),
            "bwd_frac": round(b / peak / (t_bwd * 1e-3), 4),
            "step_frac": round((f + b) / peak / ((t_fwd + t_bwd) * 1e-3), 4)}


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def window(self, t0, t1, timed=None):
        """Keep only the samples read between host times t0 and t1; `timed`
        (a, b) is the timed region inside it, whose samples are also counted."""
        self.t0, self.t1 = t0, t1
        self.timed = timed

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        t0, t1 = getattr(self, "t0", -math.inf), getattr(self, "t1", math.inf)
        timed = getattr(self, "timed", None)
        n_timed = 0
        for ts, ln in self.lines:
            if not t0 <= ts <= t1:
                continue
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            if timed and timed[0] <= ts <= timed[1]:
                n_timed += 1
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        res = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(smax) if smax else None,
               "reasons": sorted(reasons), "samples": len(sm)}
        if timed:
            res["samples_in_timed_region"] = n_timed
        return res


def graph_kernel_count(run, dev):
    """Kernel launches of one call sequence: `run(stream)` captured once into a
    CUDA graph (outside any timed region, never replayed) and the graph's
    kernel nodes counted through the driver API.  Returns (count, note); count
    is None when the capture or the count is not available."""
    import ctypes
    import torch
    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)
    except TypeError:
        return None, "this PyTorch cannot keep a captured graph"
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    try:
        with torch.cuda.graph(g, stream=s):
            run(s)
        torch.cuda.synchronize(dev)
        cu = ctypes.CDLL("libcuda.so.1")
        graph = ctypes.c_void_p(g.raw_cuda_graph())
        n = ctypes.c_size_t(0)
        if cu.cuGraphGetNodes(graph, None, ctypes.byref(n)) != 0:
            return None, "cuGraphGetNodes failed"
        nodes = (ctypes.c_void_p * max(n.value, 1))()
        if cu.cuGraphGetNodes(graph, nodes, ctypes.byref(n)) != 0:
            return None, "cuGraphGetNodes failed"
        kind = ctypes.c_int(-1)
        kernels = 0
        for i in range(n.value):
            if cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(kind)) != 0:
                return None, "cuGraphNodeGetType failed"
            kernels += kind.value == 0          # CU_GRAPH_NODE_TYPE_KERNEL
        return kernels, f"kernel nodes of one step captured in a CUDA graph ({n.value} nodes in all)"
    except Exception as e:                      # capture refused by a call of the step
        return None, f"capture failed: {type(e).__name__}"


def clock_soak(step, sync, t_start, min_span=CLOCK_WINDOW_S):
    """Repeat `step` (untimed) until at least min_span seconds have passed
    since t_start, so that a short timed region still gets clock samples of
    the same load right after it.  Returns the soak's end time."""
    n = 0
    while time.perf_counter() - t_start < min_span:
        step()
        n += 1
        if n % 8 == 0:
            sync()
    sync()
    return time.perf_counter()


# ----------------------------------------------------------------- traffic record

def source_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "selective_state_space_ssm_gb300", "csrc")
    for name in ("scan_bwd.cu", "scan_args.cuh", "ssm_common.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes (read + write) per backward launch from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "scan_bwd_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_digest") != source_digest():
        return None
    return rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------- CPU oracle leg

def oracle_slice_seconds(inp, L, nb, dsub, threads):
    """Seconds the fp64 oracle (scan fwd + bwd) takes on the first nb batch rows
    (all L steps) and the first dsub channels of the workload's inputs."""
    import numpy as np
    import oracle
    sl, rows = slice(0, dsub), slice(0, nb * L)
    u, dr, z, dout = (inp[k][rows, sl].astype(np.float64) for k in ("u", "delta_raw", "z", "dout"))
    B, C = inp["B"][rows].astype(np.float64), inp["C"][rows].astype(np.float64)
    Al, Dv = inp["A_log"][sl].astype(np.float64), inp["D"][sl].astype(np.float64)
    t0 = time.perf_counter()
    oracle.scan_fwd(u, dr, Al, B, C, Dv, z, 0, batch=nb, threads=threads)
    oracle.scan_bwd(u, dr, Al, B, C, Dv, z, dout, 0, batch=nb, threads=threads)
    return time.perf_counter() - t0


def oracle_slice(cfg, inp, target_s, threads):
    """The slice of the workload the oracle covers in about target_s: grown
    from one batch row and a few channels (channels first, then batch rows).
    Returns (nb, dsub, seconds of the last run)."""
    import oracle
    oracle.build()
    L, D = cfg["seqlen"], cfg["dinner"]
    Bn = min(cfg["batch"], inp["u"].shape[0] // L)   # batch rows the inputs hold
    nb, dsub = 1, min(D, max(16, 8 * threads))
    t = oracle_slice_seconds(inp, L, nb, dsub, threads)
    for _ in range(4):
        if t >= 0.7 * target_s or (dsub >= D and nb >= Bn):
            break
        scale = target_s / max(t, 1e-3)
        if dsub < D:
            dsub = max(8, int(min(D, max(dsub + 8, dsub * scale))) // 8 * 8)
        else:
            nb = int(min(Bn, max(nb + 1, math.floor(nb * scale))))
        t = oracle_slice_seconds(inp, L, nb, dsub, threads)
    return nb, dsub, t


def oracle_rate(cfg, nb, dsub, t):
    """Mtokens/s of the full-width problem that a slice timed at t seconds is
    worth, and the slice's description."""
    L, D = cfg["seqlen"], cfg["dinner"]
    tokens = nb * L * dsub / D       # rows of the full-width problem this slice is worth
    return tokens / t / 1e6, f"batch rows [0, {nb}), {L} steps, channels [0, {dsub}) of {D}"


def cpu_oracle_sample(cfg, inp, target_s=12.0, threads=1):
    """Time the fp64 oracle (scan fwd + bwd) on a slice of the workload: the
    first `nb` batch rows, all seqlen steps, the first `dsub` channels, grown
    until it takes about target_s.  dB/dC/dA_log/dD over the slice are part of
    the work.  threads > 1 runs the oracle's chains on that many host threads
    (channel blocks).  Returns (Mtokens/s, sample text, seconds)."""
    nb, dsub, t = oracle_slice(cfg, inp, target_s, threads)
    v, sample = oracle_rate(cfg, nb, dsub, t)
    return v, sample, t


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def config_dict(cfg, ws):
    return {"workload": f"{WORKLOAD}: batch {cfg['batch']}, seqlen {cfg['seqlen']}, "
                        f"dinner {cfg['dinner']}, dstate {cfg['dstate']}, "
                        "bf16 activations, fp32 A_log/D and state, Euler B, SiLU gate",
            "global_batch": cfg["batch"] * ws, "seq_len": cfg["seqlen"],
            "dinner": cfg["dinner"], "dstate": cfg["dstate"],
            "parallelism": f"replicas x{ws}",
            "l2": "inputs larger than L2 (805 MB of activations per step), no flush"}


# ----------------------------------------------------------------- GPU leg

def run_gb300(args):
    import numpy as np
    import torch
    import torch.distributed as dist
    import selective_state_space_ssm_gb300 as ssm
    from selective_state_space_ssm_gb300 import build as ssm_build, workloads

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group(backend="nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssm_build.build()
    ssm.load()

    cfg = dict(workloads.SCAN_WORKLOADS[WORKLOAD])
    if args.seqlen or args.batch:
        cfg["seqlen"] = args.seqlen or cfg["seqlen"]
        cfg["batch"] = args.batch or cfg["batch"]
        inp = workloads.scan_inputs(**cfg)
    else:
        inp = workloads.named_scan_inputs(WORKLOAD)
    bt = torch.bfloat16 if cfg["dtype"] == "bf16" else torch.float32
    host = {k: torch.from_numpy(inp[k]) for k in ("u", "delta_raw", "z", "B", "C", "dout")}
    host = {k: v.to(bt) for k, v in host.items()}
    host["A_log"] = torch.from_numpy(inp["A_log"])
    host["D"] = torch.from_numpy(inp["D"])
    t = {k: v.to(dev) for k, v in host.items()}
    Bn = cfg["batch"]
    out = torch.empty_like(t["u"])
    du, ddr, dz = (torch.empty_like(t["u"]) for _ in range(3))
    dB, dC = torch.empty_like(t["B"]), torch.empty_like(t["C"])
    dA = torch.empty_like(t["A_log"])
    dD = torch.empty_like(t["D"])
    desc = ssm.scan_desc(t["u"], t["delta_raw"], t["A_log"], t["B"], t["C"], t["z"], batch=Bn,
                         out=out, dout=t["dout"], du=du, ddelta=ddr, dz=dz, dB=dB, dC=dC)
    ctx = torch.empty(ssm.ssm_scan_ctx_bytes(desc), dtype=torch.uint8, device=dev)
    wsb = torch.empty(ssm.ssm_scan_bwd_workspace_bytes(desc), dtype=torch.uint8, device=dev)
    nfw = ssm.ssm_scan_fwd_workspace_bytes(desc)
    wsf = torch.empty(nfw, dtype=torch.uint8, device=dev) if nfw else None
    stream = torch.cuda.current_stream()

    def fwd():
        ssm.ssm_scan_fwd(desc, t["u"], t["delta_raw"], t["A_log"], t["B"], t["C"], t["D"], t["z"],
                         out, ctx, wsf, stream)

    def bwd():
        ssm.ssm_scan_bwd(desc, t["u"], t["delta_raw"], t["A_log"], t["B"], t["C"], t["D"], t["z"],
                         t["dout"], ctx, du, ddr, dA, dB, dC, dD, dz, wsb, stream)

    def barrier():
        if ws > 1:
            dist.barrier()

    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    if ssm.ssm_device_faults():
        raise RuntimeError("kernel wait timeout during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    h0 = time.perf_counter()
    start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    h1 = time.perf_counter()

    def step_untimed():
        fwd()
        bwd()

    h2 = clock_soak(step_untimed, torch.cuda.synchronize, h0)
    clocks.window(h0, h2, timed=(h0, h1))
    clk = clocks.stop()
    clk["window"] = (f"nvidia-smi every 50 ms over the timed region ({h1 - h0:.3f} s) and an "
                     f"untimed repeat of the same step right after it, {h2 - h0:.3f} s in all")
    barrier()
    ms_total = start.elapsed_time(end)
    t_fwd = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    t_bwd = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    if ssm.ssm_device_faults():
        raise RuntimeError("kernel wait timeout in the timed region")
    ms_step = max_over_ranks(ms_total / K, ws, dev)
    M = cfg["batch"] * cfg["seqlen"]
    value = whole_job_rate(M, ws, ms_step)

    # ---- roofline (spec definition: max(bytes / HBM, exps / SFU) per pass)
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    ex2_clk, ffma_clk, rate_kind = pipe_rates()
    clock_known = bool(clk.get("sm_mhz"))
    sm_mhz = clk["sm_mhz"] if clock_known else float(peaks.get("sm_max_mhz", 2070.0))
    sfu_rate = ex2_clk * SM_COUNT * sm_mhz * 1e6                 # ex2 / s
    fwd_b, bwd_b, exps = algorithmic(cfg)
    bound_fwd = max(fwd_b / (hbm * 1e9), exps / sfu_rate)
    bound_bwd = max(bwd_b / (hbm * 1e9), exps / sfu_rate)
    bwd_hbm_bound = bwd_b / (hbm * 1e9) >= exps / sfu_rate
    achieved_bwd = (bwd_b / (t_bwd * 1e-3) / 1e9) if bwd_hbm_bound else exps / (t_bwd * 1e-3) / 1e12
    peak_bwd = hbm if bwd_hbm_bound else sfu_rate / 1e12
    traffic = recorded_traffic()
    roofline = {
        "kernel": "ssm_scan_bwd (scan_bwd_kernel + scan_reduce_kernel)",
        "bound": "hbm" if bwd_hbm_bound else "sfu",
        "achieved": round(achieved_bwd, 3),
        "peak": round(peak_bwd, 3),
        "unit": "GB/s" if bwd_hbm_bound else "Tex2/s",
        "frac": round(achieved_bwd / peak_bwd, 4),
        "traffic": traffic,
        "peak_source": f"{peak_kind} hbm_gbs" if bwd_hbm_bound else
                       f"{rate_kind} {ex2_clk:.1f} ex2/clk/SM x {SM_COUNT} SMs x {sm_mhz:.0f} MHz",
        "sfu_rate": {"ex2_per_clk_per_sm": ex2_clk, "source": rate_kind, "sm_mhz": sm_mhz,
                     "clock": "median sampled" if clock_known else
                              "NOT SAMPLED: max clock assumed, SFU terms invalid"},
        "valid": clock_known,
        "step_ms_x_mhz": round((t_fwd + t_bwd) * sm_mhz, 1),
        "alu": alu_roofline(cfg, t_fwd, t_bwd, ffma_clk, sm_mhz, rate_kind),
        "step_frac": round((bound_fwd + bound_bwd) / ((t_fwd + t_bwd) * 1e-3), 4),
        "fwd_ms": round(t_fwd, 4), "bwd_ms": round(t_bwd, 4),
        "fwd_frac": round(bound_fwd / (t_fwd * 1e-3), 4),
        "bwd_frac": round(bound_bwd / (t_bwd * 1e-3), 4),
    }

    # ---- end to end: host buffers, copies inside the timed region.  E2E_SETS
    # device buffer sets: step i uses set i % E2E_SETS, so the uploads of the
    # next steps and the read-backs of the previous ones run on their own
    # streams while step i computes.
    e2e = None
    if not args.no_e2e:
        pin = {k: v.pin_memory() for k, v in host.items()}
        outs = {"out": out, "du": du, "ddelta": ddr, "dz": dz, "dB": dB, "dC": dC, "dA_log": dA,
                "dD": dD}
        ins = [t] + [{k: torch.empty_like(v) for k, v in t.items()} for _ in range(E2E_SETS - 1)]
        osets = [outs] + [{k: torch.empty_like(v) for k, v in outs.items()}
                          for _ in range(E2E_SETS - 1)]
        hout = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
                for _ in range(E2E_SETS)]
        h2d = sum(v.numel() * v.element_size() for v in pin.values())
        d2h = sum(v.numel() * v.element_size() for v in hout[0].values())
        K2 = max(E2E_SETS, min(K, 20))
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        in_ready = [torch.cuda.Event() for _ in range(E2E_SETS)]
        computed = [torch.cuda.Event() for _ in range(E2E_SETS)]
        read_back = [torch.cuda.Event() for _ in range(E2E_SETS)]

        def e2e_step(i):
            j = i % E2E_SETS
            T, O = ins[j], osets[j]
            s_in.wait_event(computed[j])            # set j's inputs no longer read
            with torch.cuda.stream(s_in):
                for k, v in pin.items():
                    T[k].copy_(v, non_blocking=True)
                in_ready[j].record(s_in)
            stream.wait_event(in_ready[j])
            stream.wait_event(read_back[j])         # set j's outputs already read back
            ssm.ssm_scan_fwd(desc, T["u"], T["delta_raw"], T["A_log"], T["B"], T["C"], T["D"],
                             T["z"], O["out"], ctx, wsf, stream)
            ssm.ssm_scan_bwd(desc, T["u"], T["delta_raw"], T["A_log"], T["B"], T["C"], T["D"],
                             T["z"], T["dout"], ctx, O["du"], O["ddelta"], O["dA_log"], O["dB"],
                             O["dC"], O["dD"], O["dz"], wsb, stream)
            computed[j].record(stream)
            s_out.wait_event(computed[j])
            with torch.cuda.stream(s_out):
                for k, v in O.items():
                    hout[j][k].copy_(v, non_blocking=True)
                read_back[j].record(s_out)

        for i in range(E2E_SETS):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        # E2E_WINDOWS timed windows of K2 steps each; the median window is the
        # figure (the host link is shared with the machine's other GPUs)
        windows = []
        for _ in range(E2E_WINDOWS):
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(s_in)
            for i in range(K2):
                e2e_step(i)
            s_in.wait_stream(s_out)
            s1.record(s_in)
            torch.cuda.synchronize()
            windows.append(s0.elapsed_time(s1) / K2)
        if ssm.ssm_device_faults():
            raise RuntimeError("kernel wait timeout in the end-to-end leg")
        ms_e2e = max_over_ranks(statistics.median(windows), ws, dev)
        e2e = {"value": round(whole_job_rate(M, ws, ms_e2e), 4), "unit": "Mtokens/s",
               "ms_per_step": round(ms_e2e, 4), "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": K2, "windows": E2E_WINDOWS,
               "ms_per_step_windows": [round(w, 4) for w in windows],
               "overlap": f"uploads and read-backs on their own streams, {E2E_SETS} device buffer "
                          "sets, overlapping the compute of the neighbouring steps"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        ncores = host_cores()
        v, sample, secs = cpu_oracle_sample(cfg, inp, threads=ncores)
        v1, sample1, secs1 = cpu_oracle_sample(cfg, inp, target_s=6.0)
        cpu = {"value": round(v, 6), "unit": "Mtokens/s", "cores": ncores, "kind": "oracle",
               "sample": sample, "seconds": round(secs, 2),
               "threading": "the oracle's scan chains of disjoint channel blocks on one host "
                            "thread each (dB, dC added in thread order)",
               "single_core": {"value": round(v1, 6), "sample": sample1,
                               "seconds": round(secs1, 2)}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 4), "unit": "Mtokens/s", "n_gpus": ws,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; the workload's distributions)",
            "config": config_dict(cfg, ws),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 3 * K,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------- block leg

BLOCK_METRIC = "Mamba-1 block fwd+bwd Mtokens/s; achieved % of the TF32 tensor roofline"


def block_flops(dims):
    """fp32 multiply-add flops of the block's four projections, forward and
    backward (dX and dW each repeat the forward product)."""
    M = dims["batch"] * dims["seqlen"]
    dm, D, R, N = dims["dmodel"], dims["dinner"], dims["dtrank"], dims["dstate"]
    P = R + 2 * N
    fwd = 2 * M * (dm * 2 * D + D * P + R * D + D * dm)
    return fwd, 2 * fwd


def run_block(args):
    import numpy as np
    import torch
    import selective_state_space_ssm_gb300 as ssm
    from selective_state_space_ssm_gb300 import build as ssm_build, workloads

    ws, rank, local = dist_env()
    if ws > 1:
        raise SystemExit("--block runs on one GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssm_build.build()
    ssm.load()
    cfg = dict(workloads.BLOCK_WORKLOADS[BLOCK_WORKLOAD])
    seed = cfg.pop("seed")
    if args.seqlen:
        cfg["seqlen"] = args.seqlen
    if args.batch:
        cfg["batch"] = args.batch
    inp = workloads.block_inputs(**cfg, seed=seed)
    dims = inp["dims"]
    x = torch.from_numpy(inp["x"]).to(dev)
    dout = torch.from_numpy(inp["dout"]).to(dev)
    w = {k: torch.from_numpy(v).to(dev) for k, v in inp["weights"].items()}
    desc = ssm.block_desc(dims)
    out = torch.empty_like(x)
    dx = torch.empty_like(x)
    grads = {k: torch.empty_like(v) for k, v in w.items()}
    ctx = torch.empty(ssm.ssm_block_ctx_bytes(desc), dtype=torch.uint8, device=dev)
    wsb = torch.empty(ssm.ssm_block_workspace_bytes(desc), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def fwd():
        ssm.ssm_block_fwd(desc, x, w, out, ctx, wsb, stream)

    def bwd():
        ssm.ssm_block_bwd(desc, x, w, dout, ctx, dx, grads, wsb, stream)

    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    if ssm.ssm_device_faults():
        raise RuntimeError("kernel wait timeout during warm-up")
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    h0 = time.perf_counter()
    for i in range(K):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    h1 = time.perf_counter()

    def step_untimed():
        fwd()
        bwd()

    h2 = clock_soak(step_untimed, torch.cuda.synchronize, h0)
    clocks.window(h0, h2, timed=(h0, h1))
    clk = clocks.stop()
    if ssm.ssm_device_faults():
        raise RuntimeError("kernel wait timeout in the timed region")
    t_fwd = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    t_bwd = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    ms_step = t_fwd + t_bwd

    def step_on(s):
        ssm.ssm_block_fwd(desc, x, w, out, ctx, wsb, s)
        ssm.ssm_block_bwd(desc, x, w, dout, ctx, dx, grads, wsb, s)

    per_step, launch_note = graph_kernel_count(step_on, dev)
    M = dims["batch"] * dims["seqlen"]
    f_fwd, f_bwd = block_flops(dims)
    peaks, peak_kind = measured_peaks()
    # TF32 dense peak: the measured bf16 rate x the nominal tf32 / bf16 ratio (1.1 / 2.25)
    tf32_peak = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])) * 1.1 / 2.25
    achieved = (f_fwd + f_bwd) / (ms_step * 1e-3) / 1e12
    line = {
        "metric": BLOCK_METRIC, "value": round(M / (ms_step * 1e-3) / 1e6, 4), "unit": "Mtokens/s",
        "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; the workload's distributions)",
        "config": {"workload": "mamba_block_fp32: dmodel {dmodel}, dinner {dinner}, dtrank {dtrank}, "
                               "dstate {dstate}, dconv {dconv}, batch {batch}, seqlen {seqlen}, "
                               "fp32".format(**dims),
                   "global_batch": dims["batch"], "seq_len": dims["seqlen"]},
        "roofline": {"kernel": "whole block step (projection GEMMs dominate the flops)",
                     "bound": "tensor", "achieved": round(achieved, 2),
                     "peak": round(tf32_peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / tf32_peak, 4), "traffic": None,
                     "peak_source": f"{peak_kind} bf16_tflops_sustained x 1.1/2.25 (tf32/bf16)",
                     "flops_per_step": f_fwd + f_bwd,
                     "note": "fp32 products as three TF32 passes: the tensor cores run 3x these "
                             "flops, so 1/3 is this figure's ceiling",
                     "fwd_ms": round(t_fwd, 4), "bwd_ms": round(t_bwd, 4)},
        "gpu_launches": None if per_step is None else per_step * K,
        "gpu_launches_per_step": per_step, "gpu_launches_source": launch_note, "clocks": clk,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- decode leg

CONV_METRIC = "Mamba-1 conv1d+SiLU fwd+bwd Mtokens/s; achieved % of the HBM roofline"


def conv_bytes(M, D, K):
    """Algorithmic HBM bytes of the conv, fp32: forward x in, out out (plus
    the taps and bias); backward x and dout in, dx out (plus taps and bias
    in, dw and dbias out)."""
    params = D * (K + 1) * 4
    return M * D * 8 + params, M * D * 12 + 2 * params


def conv_cpu_sample(x, w, bias, dout, batch, target_s=8.0):
    """The fp64 oracle's conv forward + backward on the first dsub channels,
    grown until it takes about target_s; scaled to Mtokens/s of the full
    width."""
    import oracle
    oracle.build()
    D = x.shape[1]
    M = x.shape[0]
    dsub = 8
    while True:
        sl = slice(0, dsub)
        t0 = time.perf_counter()
        oracle.conv1d_silu_fwd(x[:, sl], w[sl], bias[sl], batch=batch)
        oracle.conv1d_silu_bwd(x[:, sl], w[sl], bias[sl], dout[:, sl], batch=batch)
        t = time.perf_counter() - t0
        if t >= 0.5 * target_s or dsub >= D:
            break
        dsub = int(min(D, max(2 * dsub, dsub * target_s / max(t, 1e-3))))
    return M * dsub / D / t / 1e6, f"all {M} rows, channels [0, {dsub}) of {D}", t


def run_conv(args):
    """The causal depthwise conv1d + SiLU on the block workload's shape (its x
    a column view of the in_proj output, as in the block), forward and
    backward, each against the measured HBM bandwidth."""
    import numpy as np
    import torch
    import selective_state_space_ssm_gb300 as ssm
    from selective_state_space_ssm_gb300 import build as ssm_build, workloads

    ws, rank, local = dist_env()
    if ws > 1:
        raise SystemExit("--conv runs on one GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssm_build.build()
    ssm.load()
    bcfg = workloads.BLOCK_WORKLOADS[BLOCK_WORKLOAD]
    Bn, L, D, K = bcfg["batch"], bcfg["seqlen"], bcfg["dinner"], bcfg["dconv"]
    if args.batch:
        Bn = args.batch
    if args.seqlen:
        L = args.seqlen
    M = Bn * L
    inp = workloads.conv_inputs(Bn, L, D, K, seed=bcfg["seed"])
    xz = torch.zeros((M, 2 * D), dtype=torch.float32, device=dev)
    xz[:, :D] = torch.from_numpy(inp["x"]).to(dev)
    x = xz[:, :D]                                   # the in_proj output's x half
    w = torch.from_numpy(inp["w"]).to(dev)
    b = torch.from_numpy(inp["bias"]).to(dev)
    dout = torch.from_numpy(inp["dout"]).to(dev)
    out = torch.empty((M, D), dtype=torch.float32, device=dev)
    dxz = torch.empty((M, 2 * D), dtype=torch.float32, device=dev)
    dx = dxz[:, :D]
    dw, db = torch.empty_like(w), torch.empty_like(b)
    wsb = torch.empty(ssm.ssm_conv1d_silu_bwd_workspace_bytes(Bn, L, D, K), dtype=torch.uint8,
                      device=dev)
    stream = torch.cuda.current_stream()

    def fwd():
        ssm.ssm_conv1d_silu(Bn, x, w, b, out, stream)

    def bwd():
        ssm.ssm_conv1d_silu_bwd(Bn, x, w, b, dout, dx, dw, db, wsb, stream)

    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    K2 = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K2)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    h0 = time.perf_counter()
    for i in range(K2):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    h1 = time.perf_counter()

    def step_untimed():
        fwd()
        bwd()

    h2 = clock_soak(step_untimed, torch.cuda.synchronize, h0)
    clocks.window(h0, h2, timed=(h0, h1))
    clk = clocks.stop()
    t_fwd = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    t_bwd = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    ms_step = t_fwd + t_bwd
    by_f, by_b = conv_bytes(M, D, K)
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    ach_f = by_f / (t_fwd * 1e-3) / 1e9
    ach_b = by_b / (t_bwd * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu:
        v, sample, secs = conv_cpu_sample(inp["x"], inp["w"], inp["bias"], inp["dout"], Bn)
        cpu = {"value": round(v, 6), "unit": "Mtokens/s", "cores": 1, "kind": "oracle",
               "sample": sample, "seconds": round(secs, 2)}
    line = {
        "metric": CONV_METRIC, "value": round(M / (ms_step * 1e-3) / 1e6, 4), "unit": "Mtokens/s",
        "n_gpus": 1, "steps": K2, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; the workload's distributions)",
        "config": {"workload": f"mamba_block_fp32 conv: batch {Bn}, seqlen {L}, dinner {D}, "
                               f"kconv {K}, fp32, x and dx column views of (M, 2 dinner)",
                   "global_batch": Bn, "seq_len": L,
                   "l2": "inputs larger than L2 (2 x 100 MB per pass), no flush"},
        "roofline": {"kernel": "conv1d_silu_bwd_kernel + conv1d_reduce_kernel (ssm_conv1d_silu_bwd)",
                     "bound": "hbm", "achieved": round(ach_b, 1), "peak": round(hbm, 1),
                     "unit": "GB/s", "frac": round(ach_b / hbm, 4), "traffic": None,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "bytes_per_launch": by_b, "fwd_bytes": by_f,
                     "fwd_ms": round(t_fwd, 4), "bwd_ms": round(t_bwd, 4),
                     "fwd_frac": round(ach_f / hbm, 4), "bwd_frac": round(ach_b / hbm, 4)},
        "cpu_baseline": cpu, "e2e": None,
        "e2e_note": "inside the block the conv's input and output stay on the device",
        "gpu_launches": 3 * K2, "clocks": clk,
    }
    print(json.dumps(line), flush=True)


DECODE_WORKLOAD = "mamba1p4b_decode_fp32"
DECODE_METRIC = ("Mamba-1 decode (conv1d+SiLU step + scan step per layer) tokens/s; "
                 "achieved % of the HBM roofline")


def decode_bytes(cfg):
    """Algorithmic HBM bytes of one scan step and one conv step of one layer
    (fp32): the states are read and written, each activation read or written once."""
    Bn, D, N, K = cfg["batch"], cfg["dinner"], cfg["dstate"], cfg["dconv"]
    scan = 2 * Bn * N * D * 4 + 4 * Bn * D * 4 + 2 * Bn * N * 4 + D * N * 4 + D * 4
    conv = Bn * D * 4 * (1 + 2 * (K - 1) + 1) + D * K * 4 + D * 4   # x, state in + out, out
    return scan, conv


def decode_cpu_sample(layer_inp, cfg, target_s=10.0):
    """The fp64 oracle's conv step + scan step on the workload's layers, one
    after another until about target_s; scaled to tokens/s of the full step."""
    import oracle
    oracle.build()
    Bn, NL = cfg["batch"], cfg["layers"]
    t0 = time.perf_counter()
    done = 0
    while done < NL and time.perf_counter() - t0 < target_s:
        li = layer_inp[done % len(layer_inp)]
        u, _ = oracle.conv1d_silu_step(li["conv_state"], li["x"], li["w"], li["bias"])
        oracle.scan_step(li["h"], u, li["delta_raw"], li["A_log"], li["B"], li["C"], li["D"],
                         li["z"], 0)
        done += 1
    secs = time.perf_counter() - t0
    per_layer = secs / done
    return Bn / (per_layer * NL), f"{done} of {NL} layers of one step, batch {Bn}", secs


def run_decode(args):
    import ctypes
    import numpy as np
    import torch
    import selective_state_space_ssm_gb300 as ssm
    from selective_state_space_ssm_gb300 import build as ssm_build, workloads

    ws, rank, local = dist_env()
    if ws > 1:
        raise SystemExit("--decode runs on one GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssm_build.build()
    lib = ssm.load()
    cfg = dict(workloads.DECODE_WORKLOADS[DECODE_WORKLOAD])
    if args.batch:
        cfg["batch"] = args.batch
    Bn, D, N, K, NL, seed = (cfg[k] for k in ("batch", "dinner", "dstate", "dconv", "layers", "seed"))

    # per layer: parameters (A_log, D, conv w/bias), the token's inputs, the carried states
    layers, host_sample = [], []
    for l in range(NL):
        si = workloads.scan_inputs(Bn, 1, D, N, seed=seed * 1000 + l, A_log_noise=0.5,
                                   clamp_frac=0.02)
        ci = workloads.conv_inputs(Bn, 1, D, K, seed=seed * 1000 + 500 + l)
        li = dict(x=ci["x"], w=ci["w"], bias=ci["bias"], delta_raw=si["delta_raw"], B=si["B"],
                  C=si["C"], z=si["z"], A_log=si["A_log"], D=si["D"],
                  h=workloads.state_inputs(Bn, N, D, seed=seed * 1000 + 800 + l, scale=0.1),
                  conv_state=workloads.state_inputs(Bn, K - 1, D, seed=seed * 1000 + 900 + l))
        if l < 2:
            host_sample.append(li)
        t = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in li.items()}
        t["u"] = torch.empty((Bn, D), dtype=torch.float32, device=dev)
        t["out"] = torch.empty((Bn, D), dtype=torch.float32, device=dev)
        layers.append(t)
    stream = torch.cuda.Stream(device=dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    P = lambda x: ctypes.c_void_p(x.data_ptr())
    descs = [ssm.ScanDesc(batch=Bn, seqlen=1, dinner=D, dstate=N, dtype=ssm.SSM_F32,
                          disc=ssm.SSM_DISC_EULER) for _ in range(NL)]
    conv_args = [(Bn, D, K, P(t["x"]), D, P(t["w"]), P(t["bias"]), P(t["conv_state"]), P(t["u"]),
                  D, sp) for t in layers]
    scan_args = [(ctypes.byref(descs[l]), P(t["u"]), P(t["delta_raw"]), P(t["A_log"]), P(t["B"]),
                  P(t["C"]), P(t["D"]), P(t["z"]), P(t["h"]), P(t["out"]), sp)
                 for l, t in enumerate(layers)]
    conv_fn, scan_fn = lib.ssm_conv1d_silu_step, lib.ssm_scan_step

    def step():
        bad = 0
        for l in range(NL):
            bad |= conv_fn(*conv_args[l])
            bad |= scan_fn(*scan_args[l])
        if bad:
            raise RuntimeError(f"decode step failed with status {bad}")

    def scans_only():
        for l in range(NL):
            scan_fn(*scan_args[l])

    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    Kst = args.steps
    # the ABI calls captured once into CUDA graphs (no position argument: the
    # captured step is the step at every position), then replayed
    g_step, g_scan = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        step()
    with torch.cuda.graph(g_scan, stream=stream):
        scans_only()
    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            g_step.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    h0 = time.perf_counter()
    ms_step = timed(g_step.replay, Kst)
    ms_scans = timed(g_scan.replay, Kst)
    ms_eager = timed(step, max(1, Kst // 5))
    clocks.window(h0, time.perf_counter())
    clk = clocks.stop()
    ms_scan_launch = ms_scans / NL
    value = Bn / (ms_step * 1e-3)

    peaks, peak_kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    scan_b, conv_b = decode_bytes(cfg)
    achieved = scan_b / (ms_scan_launch * 1e-3) / 1e9
    step_bytes = NL * (scan_b + conv_b)
    cpu = None
    if not args.no_cpu:
        v, sample, secs = decode_cpu_sample(host_sample, cfg)
        cpu = {"value": round(v, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": sample, "seconds": round(secs, 2)}
    line = {
        "metric": DECODE_METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": 1,
        "steps": Kst, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; the workload's distributions)",
        "config": {"workload": f"{DECODE_WORKLOAD}: batch {Bn}, dinner {D}, dstate {N}, dconv {K}, "
                               f"{NL} layers (one token per sequence through every layer's "
                               "conv1d+SiLU step and scan step), fp32",
                   "global_batch": Bn, "seq_len": 1,
                   "launch": "the step's 2 x layers ABI calls captured in one CUDA graph, replayed",
                   "l2": f"{NL} layers' states ({NL * Bn * N * D * 4 / 1e6:.0f} MB) exceed L2, no flush"},
        "roofline": {"kernel": "scan_step_kernel (ssm_scan_step)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": round(hbm, 1), "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": None,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "bytes_per_launch": scan_b, "us_per_launch": round(ms_scan_launch * 1e3, 3),
                     "step_frac": round(step_bytes / (hbm * 1e9) / (ms_step * 1e-3), 4)},
        "eager_ms_per_step": round(ms_eager, 4),
        "cpu_baseline": cpu, "e2e": None,
        "e2e_note": "decode inputs come from the previous layer on the device; no host copies",
        "gpu_launches": 2 * NL * Kst, "clocks": clk,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- pipe rates

def run_measure_pipes(args):
    """MUFU ex2, fp32 FFMA and packed FFMA2 lane-operations per clock per SM,
    from the library's probe kernels (ssm_probe_pipe): each kind launched
    repeatedly for about half a second, timed with CUDA events, divided by the
    SM count and the median SM clock sampled meanwhile."""
    import torch
    import selective_state_space_ssm_gb300 as ssm
    from selective_state_space_ssm_gb300 import build as ssm_build

    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssm_build.build()
    ssm.load()
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks = nsm * 8                       # 8 CTAs of 256 threads: 64 warps per SM
    sink = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    res = {"gpu_name": torch.cuda.get_device_name(dev), "sm_count": nsm}
    for kind, name, iters in ((0, "ex2", 4096), (1, "ffma", 16384), (2, "ffma2", 16384)):
        for _ in range(3):
            ssm.ssm_probe_pipe(kind, blocks, iters, sink, stream)
        torch.cuda.synchronize()
        clocks = ClockSampler(local)
        clocks.start()
        time.sleep(0.3)
        times = []
        h0 = time.perf_counter()
        while time.perf_counter() - h0 < 0.6:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ssm.ssm_probe_pipe(kind, blocks, iters, sink, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        clocks.window(h0, time.perf_counter())
        clk = clocks.stop()
        ops = blocks * 256 * iters * 8
        ms = statistics.median(times)
        mhz = clk["sm_mhz"]
        per_clk = ops / (ms * 1e-3) / (mhz * 1e6) / nsm if mhz else None
        res[name] = {"lane_ops_per_launch": ops, "median_ms": round(ms, 4), "launches": len(times),
                     "per_s": ops / (ms * 1e-3), "sm_mhz_median": mhz,
                     "per_clk_per_sm": round(per_clk, 2) if per_clk else None,
                     "clock_reasons": clk["reasons"], "clock_samples": clk["samples"]}
    res["ex2_per_clk_per_sm"] = res["ex2"]["per_clk_per_sm"]
    res["ffma_lanes_per_clk_per_sm"] = res["ffma"]["per_clk_per_sm"]
    res["ffma2_lanes_per_clk_per_sm"] = res["ffma2"]["per_clk_per_sm"]
    res["how"] = ("ssm_probe_pipe: CTAs of 256 threads (8 per SM), each thread 8 independent "
                  "chains (ex2: x <- 2^-x; ffma: x <- a x + b; ffma2: the same on 4 packed pairs); "
                  "median CUDA-event time per launch over about 0.6 s, divided by the SM count and "
                  "the median SM clock nvidia-smi read meanwhile")
    res["command"] = "python bench.py --measure-pipes OUT_JSON"
    if args.measure_pipes:
        with open(args.measure_pipes, "w") as f:
            json.dump(res, f, indent=1)
    print(json.dumps(res), flush=True)


def run_measure_gemm_ref(args):
    """The block workload's forward projection GEMMs (M = batch*seqlen rows)
    through ssm_linear_fwd (three TF32 products, fp32 in and out) and, for
    context, the vendor library's GEMM of the same shape in TF32 (one
    product), BF16 and plain FP32, each timed with CUDA events around 20
    back-to-back launches (median of 5 such runs, after 3 warm-ups).  TFLOP/s
    count 2*M*N*K once."""
    import torch
    import selective_state_space_ssm_gb300 as ssm
    from selective_state_space_ssm_gb300 import build as ssm_build, workloads

    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssm_build.build()
    ssm.load()
    cfg = workloads.BLOCK_WORKLOADS[BLOCK_WORKLOAD]
    M = cfg["batch"] * cfg["seqlen"]
    dm, di, r, n = cfg["dmodel"], cfg["dinner"], cfg["dtrank"], cfg["dstate"]
    shapes = {"in_proj": (M, 2 * di, dm), "x_proj": (M, r + 2 * n, di), "dt_proj": (M, di, r),
              "out_proj": (M, dm, di)}

    def timed(fn, n=20):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n):
                fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / n)
        return statistics.median(ts)

    res = {"gpu_name": torch.cuda.get_device_name(dev), "workload": BLOCK_WORKLOAD, "shapes": {}}
    old_tf32 = torch.backends.cuda.matmul.allow_tf32
    try:
        for name, (m, nn, k) in shapes.items():
            g = torch.Generator(device=dev).manual_seed(5)
            X = torch.randn(m, k, device=dev, generator=g)
            W = torch.randn(nn, k, device=dev, generator=g) / k ** 0.5
            flop = 2.0 * m * nn * k
            row = {"M": m, "N": nn, "K": k}
            ms = timed(lambda: ssm.linear(X, W))
            row["ssm_linear_3xtf32"] = {"ms": round(ms, 4), "tflops": round(flop / ms / 1e9, 1)}
            for label, dt, tf32 in (("vendor_tf32", torch.float32, True), ("vendor_bf16", torch.bfloat16, False),
                                    ("vendor_fp32", torch.float32, False)):
                torch.backends.cuda.matmul.allow_tf32 = tf32
                Xd, Wd = X.to(dt), W.to(dt)
                ms = timed(lambda: Xd @ Wd.t())
                row[label] = {"ms": round(ms, 4), "tflops": round(flop / ms / 1e9, 1)}
            res["shapes"][name] = row
    finally:
        torch.backends.cuda.matmul.allow_tf32 = old_tf32
    res["how"] = ("CUDA events around 20 back-to-back calls, median of 5 (ssm.linear includes its "
                  "output and workspace allocation from the caching allocator); the vendor rows are "
                  "torch.matmul")
    res["command"] = "python bench.py --measure-gemm-ref OUT_JSON"
    if args.measure_gemm_ref:
        with open(args.measure_gemm_ref, "w") as f:
            json.dump(res, f, indent=1)
    print(json.dumps(res), flush=True)


# ----------------------------------------------------------------- reference leg

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from selective_state_space_ssm_gb300 import workloads
    cfg = dict(workloads.SCAN_WORKLOADS[WORKLOAD])
    inp = workloads.named_scan_inputs(WORKLOAD)
    # the slice is sized once (about 60 s of oracle work over all steps), then
    # every warm-up and timed step runs that same slice
    per_step = max(0.25, 60.0 / max(1, args.steps + args.warmup))
    ncores = host_cores()
    nb, dsub, _ = oracle_slice(cfg, inp, per_step, ncores)
    vals, secs = [], []
    sample = ""
    for i in range(args.warmup + args.steps):
        s = oracle_slice_seconds(inp, cfg["seqlen"], nb, dsub, ncores)
        v, sample = oracle_rate(cfg, nb, dsub, s)
        if i >= args.warmup:
            vals.append(v)
            secs.append(s)
    value = statistics.mean(vals)
    ms = statistics.mean(secs) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "Mtokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; the workload's distributions)",
        "config": config_dict(cfg, ws),
        "cpu_baseline": {"value": round(value, 6), "unit": "Mtokens/s", "cores": ncores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "Mtokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.measure_pipes:
        run_measure_pipes(args)
    elif args.measure_gemm_ref:
        run_measure_gemm_ref(args)
    elif args.block:
        run_block(args)
    elif args.decode:
        run_decode(args)
    elif args.conv:
        run_conv(args)
    else:
        run_gb300(args)


if __name__ == "__main__":
    main()
