"""Benchmark of the fused linear-attention forward + backward on GB300.

One step = la_fwd followed by la_bwd over one batch of the workload (every kernel of the
path), inputs resident in HBM.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun with one process per GPU.  The operation has no exchange step
between (batch, kv head) groups, so ranks run independent replicas of the workload (weak
scaling, no data-path collective); the timing is max-over-ranks, and ``value`` counts the
tokens of all ranks.  ``--impl reference`` times the float64 CPU oracle (the only other
implementation of the method here) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from efficient_transformer_gb300 import inputs as gen  # noqa: E402

METRIC = "linear-attn fwd+bwd tokens/s and TFLOP/s at 1 GB300; % of roofline"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024
NOMINAL_CHUNK = 64          # chunk length of the nominal FLOP count
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# CUDA-core float32 peak: 152 SMs x 128 FP32 lanes x 2 flop per FMA x 2.07 GHz max clock.
ALU_F32_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


# ---------------------------------------------------------------------------------------
# Work counts

def tensor_bytes(w: gen.Workload):
    el = 4 if w.dtype == "f32" else 2
    qb = w.B * w.Hq * w.N * w.D * el
    kvb = w.B * w.Hkv * w.N * w.D * el
    return qb, kvb


def path_bytes(w: gen.Workload) -> int:
    """Compulsory bytes of fwd + bwd: fwd reads q, k, v and writes out; bwd reads q, k, v,
    grad_out and writes dq, dk, dv; position weights are read once per pass."""
    qb, kvb = tensor_bytes(w)
    wb = 2 * 4 * w.N if w.weights else 0
    return (2 * qb + 2 * kvb + wb) + (3 * qb + 4 * kvb + wb)


def path_flops(w: gen.Workload) -> float:
    """Nominal FLOPs of fwd + bwd, counted per query head with chunk length 64 and full
    intra-chunk tiles; P is the number of (S, z) state pairs."""
    P = 2 if w.weights else 1
    D = Dv = w.D
    rows = w.B * w.Hq * w.N
    if w.causal:
        f = rows * (4 * P * D * Dv + 2 * NOMINAL_CHUNK * (D + Dv))
        b = rows * (10 * P * D * Dv + 2 * NOMINAL_CHUNK * (3 * D + 2 * Dv))
    else:
        f = rows * 4 * D * Dv * P
        b = rows * 10 * D * Dv * P
    return float(f + b)


def kernel_work(name: str, w: gen.Workload):
    """(bound, algorithmic units per launch, unit) for one kernel of the path.

    CUDA-core kernels are bounded by float32 FMA throughput: their units are the FLOPs of
    the arithmetic they must do (state updates 2 P D (D+1) per key token; per query row
    the readout 2 P D (D+1) plus, causal, the 16-token intra-chunk tile).  Kernels that
    stream tensors are bounded by HBM: their units are the bytes they must move once."""
    P = 2 if w.weights else 1
    D = w.D
    qb, kvb = tensor_bytes(w)
    kv_rows = w.B * w.Hkv * w.N
    q_rows = w.B * w.Hq * w.N
    st = 2 * P * D * (D + 1)
    intra = (2 * 16 * P * D + 2 * 16 * (D + 1)) if w.causal else 0
    table = {
        "simt_seg_state": ("alu", kv_rows * st),
        "scan": ("hbm", None),
        "simt_fwd": ("alu", q_rows * (st + intra) + (kv_rows * st if w.causal else 0)),
        "simt_bwd_dq": ("alu", q_rows * (2 * st + 2 * intra) + (kv_rows * st if w.causal else 0)),
        "simt_seg_rstate": ("alu", q_rows * st),
        "simt_bwd_dkdv": ("alu", kv_rows * 2 * st + ((q_rows * (2 * intra + st)) if w.causal else 0)),
        # tensor-core kernels stream tensors: bytes each must move once
        "tc_seg_state": ("hbm", 2 * kvb),                        # k, v
        "tc_fwd_causal": ("hbm", 2 * qb + 2 * kvb),              # q, k, v -> out
        "tc_fwd_bidir": ("hbm", 2 * qb),                         # q -> out
        "tc_bwd_dq_causal": ("hbm", 3 * qb + 2 * kvb),           # q, g, k, v -> dq
        "tc_bwd_dq_bidir": ("hbm", 3 * qb),                      # q, g -> dq
        "tc_bwd_dkdv_causal": ("hbm", 2 * qb + 4 * kvb),         # q, g, k, v -> dk, dv
        "tc_bwd_dkdv_bidir": ("hbm", 4 * kvb),                   # k, v -> dk, dv
    }
    bound, units = table.get(name, ("hbm", None))
    return bound, units, ("TFLOP/s" if bound == "alu" else "GB/s")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------------------
# Clock sampling (nvidia-smi, during the timed region)

def nvsmi_id(dev, local: int) -> str:
    """nvidia-smi --id for this CUDA device (its UUID when torch exposes it)."""
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except (AttributeError, RuntimeError):
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x.strip() for x in vis.split(",") if x.strip()]
    return ids[local] if local < len(ids) else str(local)


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((ts, float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return None
        window = [r for r in rows if t0 <= r[0] <= t1]
        used = window if len(window) >= 3 else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in used for i, v in enumerate(r[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in used),
                "sm_max_mhz": max(r[2] for r in used),
                "power_w_max": max(r[3] for r in used),
                "reasons": reasons, "samples": len(used),
                "window": "timed region" if used is window else "whole run"}


# ---------------------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)

def oracle_sample(w: gen.Workload, tokens: int):
    """Inputs for the first ``tokens`` positions of every (batch, head) of ``w``."""
    ws = w.with_(N=tokens)
    inp = gen.make_inputs(ws, seed=0)
    return ws, inp


def time_oracle(w: gen.Workload, tokens: int):
    import oracle
    ws, inp = oracle_sample(w, tokens)
    kw = dict(is_causal=ws.causal, phi=ws.phi, eps=ws.eps, cos_weight=inp["cos_weight"],
              sin_weight=inp["sin_weight"])
    t0 = time.perf_counter()
    oracle.fwd(inp["q"], inp["k"], inp["v"], **kw)
    oracle.bwd(inp["q"], inp["k"], inp["v"], inp["grad_out"], **kw)
    return time.perf_counter() - t0


def oracle_tokens_for(w: gen.Workload, seconds: float) -> int:
    """Sample length (tokens per sequence) whose oracle fwd+bwd takes about ``seconds``."""
    probe = min(w.N, 128)
    t = max(time_oracle(w, probe), 1e-4)
    tokens = int(probe * seconds / t)
    return max(16, min(w.N, tokens))


def cpu_cores():
    import oracle
    return oracle.num_threads()


# ---------------------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the dominant kernels
# on the benchmark workload, from one ncu capture of the current kernels; a kernel changed
# since its capture must be removed from this table (its traffic is then reported as null).
MEASURED_TRAFFIC = {
    "tc_bwd_dq_causal": (1361156181 + 1041062826, "ncu one-pass capture of the current kernels (commit c663517)"),
    "tc_bwd_dkdv_causal": (1361027157 + 249435050, "ncu one-pass capture of the current kernels (commit c663517)"),
    "tc_fwd_causal": (815492352 + 498729642, "ncu one-pass capture of the current kernels (commit c663517)"),
}


def workload_of(args) -> gen.Workload:
    w = gen.WORKLOADS[args.workload]
    if args.seq_len:
        w = w.with_(name=f"{w.name}@n{args.seq_len}", N=args.seq_len)
    return w


def config_of(w: gen.Workload, world: int):
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "D": w.D,
            "causal": w.causal, "phi": w.phi, "eps": w.eps, "cos_sin_weights": w.weights,
            "input_scale": w.scale, "global_batch": w.B * world, "seq_len": w.N,
            "parallelism": f"replicas{world}",
            "step": "la_fwd, then la_bwd_from_fwd (the backward reads the forward's segment states)",
            "l2": f"no explicit flush: inputs larger than L2 ({path_bytes(w) / 2**20:.0f} MiB moved "
                  f"per step vs {L2_BYTES / 2**20:.0f} MiB L2); the per-workload table flushes L2 "
                  f"before each step of workloads that fit in it"}


def run_reference(args, world, rank):
    """Reference arm: the float64 oracle as it stands, on the host cores, rank 0 only."""
    if rank != 0:
        return 0
    w = workload_of(args)
    budget = 150.0 / max(1, args.steps + args.warmup)   # seconds per step, whole run ~2.5 min
    tokens = oracle_tokens_for(w, min(10.0, budget))
    for _ in range(args.warmup):
        time_oracle(w, tokens)
    times = [time_oracle(w, tokens) for _ in range(args.steps)]
    t = statistics.mean(times)
    value = w.B * tokens / t
    sample = (f"first {tokens} of {w.N} positions of every (batch, head), fwd+bwd, float64 oracle; "
              f"tokens/s = B*{tokens} / mean seconds per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) inputs)", "config": config_of(w, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# The HBM bandwidth of the operation's stated roofline (the slower of the tensor-core peak and
# HBM bytes at 8 TB/s); the measured copy bandwidth gives a second, stricter-looking fraction.
ROOFLINE_HBM_GBS = 8000.0
FLUSH_BYTES = 512 * 2**20   # written between timed steps of workloads that fit in L2


def path_roofline(w: gen.Workload, peaks: dict, ms_step: float, peak_src: str):
    nbytes, flops = path_bytes(w), path_flops(w)
    t_tc = flops / (peaks["bf16_tflops_sustained"] * 1e12)
    t_8 = max(nbytes / (ROOFLINE_HBM_GBS * 1e9), t_tc)
    t_m = max(nbytes / (peaks["hbm_gbs"] * 1e9), t_tc)
    return {"bytes_per_step": nbytes, "flops_per_step": flops,
            "t_roofline_ms": t_8 * 1e3, "frac": t_8 * 1e3 / ms_step,
            "basis": f"max(bytes / {ROOFLINE_HBM_GBS:.0f} GB/s, flops / {peak_src} bf16 sustained "
                     f"{peaks['bf16_tflops_sustained']} TFLOP/s)",
            "t_roofline_measured_hbm_ms": t_m * 1e3, "frac_measured_hbm": t_m * 1e3 / ms_step,
            "measured_hbm_gbs": peaks["hbm_gbs"]}


class Problem:
    """Device inputs, outputs and workspaces of one workload, and its step: la_fwd, then
    la_bwd_from_fwd on the forward's workspace."""

    def __init__(self, la, w: gen.Workload, dev, seed: int = 0, host=None):
        self.la, self.w = la, w
        host = host if host is not None else gen.make_inputs(w, seed=seed)
        self.d = {n: (t.to(dev) if t is not None else None) for n, t in host.items()}
        d = self.d
        self.out = torch.empty_like(d["q"])
        self.dq, self.dk, self.dv = torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"])
        has_w = d["cos_weight"] is not None
        self.ws_f = torch.empty(max(1, la.workspace_size(w.B, w.Hq, w.Hkv, w.N, w.D, d["q"].dtype, w.causal, has_w,
                                                         False)), dtype=torch.uint8, device=dev)
        self.ws_b = torch.empty(max(1, la.workspace_size(w.B, w.Hq, w.Hkv, w.N, w.D, d["q"].dtype, w.causal, has_w,
                                                         True)), dtype=torch.uint8, device=dev)

    def step(self, stream, x=None):
        la, w = self.la, self.w
        x = x or self.d
        la.fwd(x["q"], x["k"], x["v"], w.causal, w.phi, w.eps, x["cos_weight"], x["sin_weight"],
               out=self.out, workspace=self.ws_f, stream=stream)
        la.bwd(x["q"], x["k"], x["v"], x["grad_out"], w.causal, w.phi, w.eps, x["cos_weight"],
               x["sin_weight"], dq=self.dq, dk=self.dk, dv=self.dv, workspace=self.ws_b, stream=stream,
               fwd_workspace=self.ws_f)

    def paths(self):
        la, w = self.la, self.w
        names = {la.LA_PATH_SIMT: "simt", la.LA_PATH_TCGEN05: "tcgen05"}
        return {p: names[la.kernel_path(w.B, w.Hq, w.Hkv, w.N, w.D, w.torch_dtype, w.causal, w.weights, p == "bwd")]
                for p in ("fwd", "bwd")}


def time_blocks(step, dev, stream, steps: int, repeats: int, world: int):
    """`repeats` blocks of exactly `steps` steps; each block between two events on the
    stream, with a barrier and a synchronisation on both sides.  Returns ms per step of
    each block (max over ranks)."""
    per = []
    for _ in range(repeats):
        barrier(world)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        per.append(e0.elapsed_time(e1) / steps)
    barrier(world)
    return [max_over_ranks(x, world) for x in per]


def time_flushed(run, dev, stream, steps: int, flush: torch.Tensor):
    """`steps` single steps, L2 flushed (a 512 MiB write) before each; ms of each step."""
    per = []
    for _ in range(steps):
        with torch.cuda.stream(stream):
            flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        per.append(e0.elapsed_time(e1))
    return per


def summary_ms(per):
    return {"ms_per_step": statistics.median(per), "ms_min": min(per), "ms_max": max(per),
            "samples": len(per)}


def measure_config(la, w: gen.Workload, dev, steps: int, warmup: int, peaks, peak_src, flush):
    """One row of the per-workload table: the workload's step timed on its own."""
    pr = Problem(la, w, dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, warmup)):
        pr.step(stream)
    la.get_status(stream)
    small = path_bytes(w) < 4 * L2_BYTES
    row = {"workload": w.name, "paths": pr.paths()}
    if small:
        # launch-bound sizes: one step captured in a CUDA graph and replayed, L2 flushed first
        run, how = (lambda: pr.step(stream)), "library calls"
        try:
            g = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            with torch.cuda.graph(g, stream=cap):
                pr.step(torch.cuda.current_stream(dev))
            stream.wait_stream(cap)
            torch.cuda.synchronize(dev)
            run, how = g.replay, "one step captured in a CUDA graph, replayed"
        except RuntimeError as e:   # capture refused: time the plain calls
            how = f"library calls (graph capture failed: {str(e)[:80]})"
        run()
        torch.cuda.synchronize(dev)
        per = time_flushed(run, dev, stream, max(steps, 20), flush)
        row["timing"] = f"{how}; L2 flushed ({FLUSH_BYTES >> 20} MiB write) before each timed step"
    else:
        per = time_blocks(lambda: pr.step(stream), dev, stream, steps, 5, 1)
        row["timing"] = f"5 blocks of {steps} steps; inputs larger than L2"
    la.get_status(stream)
    row.update(summary_ms(per))
    ms = row["ms_per_step"]
    row["tokens_per_s"] = w.tokens / (ms / 1e3)
    row["tflops"] = path_flops(w) / (ms / 1e3) / 1e12
    rl = path_roofline(w, peaks, ms, peak_src)
    row["roofline_frac"] = rl["frac"]
    row["roofline_frac_measured_hbm"] = rl["frac_measured_hbm"]
    row["t_roofline_ms"] = rl["t_roofline_ms"]
    if w.dtype == "f32":
        row["note"] = "float32, 0.6 MiB per step: launch-bound, reported only"
    del pr
    torch.cuda.empty_cache()
    return row


def lowrank_counts(w: gen.LowRankWorkload):
    """(bytes, flops) of one low-rank forward and of one forward + backward: compulsory bytes
    (every input read once, every output written once) and the 2 m n k flops of the products
    the operation needs (the forward's two; the backward's dt, dx, dU, dV: t is the forward's)."""
    el = 2
    x_b, y_b = w.M * w.K_in * el, w.M * w.K_out * el
    wts = (w.K_in + w.K_out) * w.r * el + (w.K_out * el if w.bias else 0)
    f_fwd = 2.0 * w.M * w.r * (w.K_in + w.K_out)
    f_bwd = 2.0 * w.M * w.r * (2 * w.K_in + 2 * w.K_out)   # dt, dU (K_out); dx, dV (K_in)
    b_fwd = x_b + y_b + wts
    b_bwd = x_b + y_b + x_b + 2 * wts                      # x, g in; dx, dU, dV, dbias out
    return (b_fwd, f_fwd), (b_fwd + b_bwd, f_fwd + f_bwd)


def measure_lowrank(la, w: gen.LowRankWorkload, dev, steps: int, warmup: int, peaks, peak_src):
    """One row of the per-workload table for the low-rank projection: forward alone and
    forward + backward, each as blocks of `steps` calls between CUDA events.  The step's
    forward keeps the bottleneck t for its backward (la_lowrank_fwd_t / la_lowrank_bwd_t),
    as a training step that keeps its forward's context does."""
    host = gen.make_lowrank_inputs(w)
    d = {n: (t.to(dev) if t is not None else None) for n, t in host.items()}
    y = torch.empty((w.M, w.K_out), dtype=d["x"].dtype, device=dev)
    t = torch.empty((w.M, w.r), dtype=d["x"].dtype, device=dev)
    ws = torch.empty(max(1, la.load().la_lowrank_workspace_size(w.M, w.K_in, w.r, w.K_out, la.LA_BF16, 1)),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        la.lowrank_fwd(d["x"], d["U"], d["V"], d["bias"], out=y, stream=stream)

    def step():
        la.lowrank_fwd(d["x"], d["U"], d["V"], d["bias"], out=y, t_out=t, stream=stream)
        la.lowrank_bwd(d["x"], d["U"], d["V"], d["grad_out"], d["bias"], workspace=ws, t=t, stream=stream)

    for _ in range(max(3, warmup)):
        step()
    la.get_status(stream)
    per_f = time_blocks(fwd, dev, stream, steps, 5, 1)
    per = time_blocks(step, dev, stream, steps, 5, 1)
    la.get_status(stream)
    (bf, ff), (bs, fs) = lowrank_counts(w)
    row = {"workload": w.name, "paths": {"fwd": "tcgen05", "bwd": "tcgen05"},
           "timing": f"5 blocks of {steps} steps; inputs larger than L2", "metric": "TFLOP/s"}
    row.update(summary_ms(per))
    ms, ms_f = row["ms_per_step"], statistics.median(per_f)
    tc_peak = peaks["bf16_tflops_sustained"] * 1e12

    def frac(nbytes, flops, t_ms):
        t_roof = max(nbytes / (ROOFLINE_HBM_GBS * 1e9), flops / tc_peak)
        return t_roof * 1e3 / t_ms, ("tensor" if flops / tc_peak >= nbytes / (ROOFLINE_HBM_GBS * 1e9) else "hbm")

    row["tflops"] = fs / (ms / 1e3) / 1e12
    row["roofline_frac"], row["bound"] = frac(bs, fs, ms)
    row["fwd"] = {"ms": ms_f, "tflops": ff / (ms_f / 1e3) / 1e12, "roofline_frac": frac(bf, ff, ms_f)[0]}
    row["tokens_per_s"] = w.M / (ms / 1e3)
    row["roofline_basis"] = (f"max(bytes / {ROOFLINE_HBM_GBS:.0f} GB/s, flops / {peak_src} bf16 sustained "
                             f"{peaks['bf16_tflops_sustained']} TFLOP/s)")
    del d, y, t, ws
    torch.cuda.empty_cache()
    return row


def run_lowrank_only(args, local):
    """The low-rank projection's step alone, at --lowrank-rows rows: one JSON line with its
    forward and forward + backward times (the per-workload table's row)."""
    from efficient_transformer_gb300 import la

    la.load()
    base = next(iter(gen.LOWRANK_WORKLOADS.values()))
    wl = gen.LowRankWorkload(f"lowrank_m{args.lowrank_rows}_kin{base.K_in}_r{base.r}_kout{base.K_out}_bf16",
                             args.lowrank_rows, base.K_in, base.r, base.K_out)
    peaks, peak_src = load_peaks()
    row = measure_lowrank(la, wl, torch.device("cuda", local), args.steps, args.warmup, peaks, peak_src)
    print(json.dumps(row))
    return 0


def run_ours(args, world, rank, local):
    from efficient_transformer_gb300 import build as la_build
    from efficient_transformer_gb300 import la

    if rank == 0 and not os.path.exists(la.LIB_PATH):
        la_build.build()
    barrier(world)
    la.load()
    w = workload_of(args)
    dev = torch.device("cuda", local)
    host = gen.make_inputs(w, seed=rank)
    pinned = {n: (t.pin_memory() if t is not None else None) for n, t in host.items()}
    pr = Problem(la, w, dev, host=host)
    del host
    d = pr.d
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()

    clocks = ClockSampler(nvsmi_id(dev, local))
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        pr.step(stream)
    la.get_status(stream)

    # Device-timed region: inputs resident in HBM.  Blocks of exactly K steps, each between
    # two events on the launching stream; repeated for a few seconds of sustained load, the
    # reported step time being the median block.
    first = time_blocks(lambda: pr.step(stream), dev, stream, args.steps, 1, world)[0]
    repeats = args.repeats or max(5, min(200, int(math.ceil(3000.0 / max(first * args.steps, 1e-3)))))
    t_wall0 = time.time()
    per = time_blocks(lambda: pr.step(stream), dev, stream, args.steps, repeats, world)
    t_wall1 = time.time()
    la.get_status(stream)
    ms_step = statistics.median(per)
    # The same K steps again with every library launch bracketed by events (per-kernel shares
    # and the dominant kernel's launch time); kept apart so the events cost the timing nothing.
    barrier(world)
    torch.cuda.synchronize(dev)
    la.trace_start()
    for _ in range(args.steps):
        pr.step(stream)
    torch.cuda.synchronize(dev)
    kernels = la.trace_stop()
    barrier(world)
    la.get_status(stream)
    clocks.stop()
    clk = clocks.summary(t_wall0, t_wall1)

    # End to end: pinned host inputs -> device, fwd + bwd, every output back to pinned host.
    # Every step copies its own inputs in and all of its outputs out inside the timed region;
    # the copies run on their own streams with two device (and host-output) buffer sets, so
    # step i's input copy and step i-1's output copy overlap step i's kernels.
    e2e = None
    if not args.no_e2e:
        outs = (("out", pr.out), ("dq", pr.dq), ("dk", pr.dk), ("dv", pr.dv))
        h2d = sum(t.numel() * t.element_size() for t in pinned.values() if t is not None)
        d2h = sum(t.numel() * t.element_size() for _, t in outs)
        e2e_steps = max(2, min(args.steps, 10))
        sets = []
        for _ in range(2):
            sets.append({
                "x": {n: (torch.empty_like(t) if t is not None else None) for n, t in d.items()},
                "o": {n: torch.empty_like(t) for n, t in outs},
                "h": {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in outs},
                "wf": torch.empty_like(pr.ws_f), "wb": torch.empty_like(pr.ws_b)})
        s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))

        def e2e_run(nsteps, e_start=None, e_end=None):
            ev_cmp, ev_out = [None, None], [None, None]
            if e_start is not None:
                e_start.record(s_in)
            for i in range(nsteps):
                st = sets[i % 2]
                x, o = st["x"], st["o"]
                if ev_cmp[i % 2] is not None:   # the set's previous kernels have read its inputs
                    s_in.wait_event(ev_cmp[i % 2])
                with torch.cuda.stream(s_in):
                    for n, t in pinned.items():
                        if t is not None:
                            x[n].copy_(t, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
                s_cmp.wait_event(ev_in)
                if ev_out[i % 2] is not None:   # the set's previous outputs are copied out
                    s_cmp.wait_event(ev_out[i % 2])
                la.fwd(x["q"], x["k"], x["v"], w.causal, w.phi, w.eps, x["cos_weight"], x["sin_weight"],
                       out=o["out"], workspace=st["wf"], stream=s_cmp)
                la.bwd(x["q"], x["k"], x["v"], x["grad_out"], w.causal, w.phi, w.eps, x["cos_weight"],
                       x["sin_weight"], dq=o["dq"], dk=o["dk"], dv=o["dv"], workspace=st["wb"], stream=s_cmp,
                       fwd_workspace=st["wf"])
                ev_cmp[i % 2] = torch.cuda.Event()
                ev_cmp[i % 2].record(s_cmp)
                s_out.wait_event(ev_cmp[i % 2])
                with torch.cuda.stream(s_out):
                    for n, _ in outs:
                        st["h"][n].copy_(o[n], non_blocking=True)
                ev_out[i % 2] = torch.cuda.Event()
                ev_out[i % 2].record(s_out)
            if e_end is not None:   # the last output copy waits on everything before it
                e_end.record(s_out)

        e2e_run(2)
        torch.cuda.synchronize(dev)
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_run(e2e_steps, e0, e1)
        torch.cuda.synchronize(dev)
        barrier(world)
        la.get_status(s_cmp)
        e_ms = max_over_ranks(e0.elapsed_time(e1), world) / e2e_steps
        e2e = {"value": world * w.tokens / (e_ms / 1e3), "unit": UNIT, "ms_per_step": e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "overlap": "input copy, kernels and output copy on three streams, two buffer sets"}
        del sets

    # Per-workload table (one GPU): every workload's step timed on its own.
    table = None
    if world == 1 and not args.no_configs and not args.seq_len:
        del pinned
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        table = []
        for name, wc in gen.WORKLOADS.items():
            if name == w.name:
                continue
            table.append(measure_config(la, wc, dev, args.steps, args.warmup, peaks, peak_src, flush))
        del flush
        for wl in gen.LOWRANK_WORKLOADS.values():
            table.append(measure_lowrank(la, wl, dev, args.steps, args.warmup, peaks, peak_src))

    if rank != 0:
        return 0

    tokens_per_s = world * w.tokens / (ms_step / 1e3)
    flops = path_flops(w)

    # Dominant kernel: the one with the largest share of traced device time.
    launches = sum(n for n, _ in kernels.values())
    total_ms = sum(ms for _, ms in kernels.values())
    top = max(kernels.items(), key=lambda kv: kv[1][1])
    top_name, (top_n, top_ms) = top
    bound, units, unit = kernel_work(top_name, w)
    per_launch_s = top_ms / top_n / 1e3
    launches_per_step = top_n / args.steps
    if bound == "alu":
        achieved = units / launches_per_step / per_launch_s / 1e12
        peak = ALU_F32_TFLOPS
        peak_note = "derived: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz"
    elif bound == "tensor":
        achieved = units / launches_per_step / per_launch_s / 1e12
        peak = peaks["bf16_tflops_sustained"]
        peak_note = f"{peak_src} bf16_tflops_sustained"
    else:
        achieved = (units or 0) / launches_per_step / per_launch_s / 1e9
        peak = peaks["hbm_gbs"]
        peak_note = f"{peak_src} hbm_gbs"
    traffic = MEASURED_TRAFFIC.get(top_name) if w.name == gen.BENCH_WORKLOAD else None
    roofline = {"bound": bound, "kernel": top_name,
                "scope": "the dominant kernel alone (largest share of traced device time)",
                "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": traffic[0] if traffic else None,
                "traffic_source": traffic[1] if traffic else None, "peak_source": peak_note,
                "launch_ms": per_launch_s * 1e3,
                "share_of_traced_time": top_ms / total_ms if total_ms else None}

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        tokens = oracle_tokens_for(w, args.cpu_seconds)
        t = time_oracle(w, tokens)
        cpu = {"value": w.B * tokens / t, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"first {tokens} of {w.N} positions of every (batch, head), one fwd+bwd "
                         f"({t:.1f} s); tokens/s = B*{tokens} / seconds"}

    cfg = config_of(w, world)
    cfg["timing"] = (f"median of {repeats} blocks of {args.steps} steps (each block between two CUDA events, "
                     f"synchronised on both sides)")
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) inputs, scale per workload)",
        "config": cfg,
        "ms_spread": {"min": min(per), "max": max(per), "blocks": len(per)},
        "tflops": world * flops / (ms_step / 1e3) / 1e12,
        "path_roofline": path_roofline(w, peaks, ms_step, peak_src),
        "roofline": roofline,
        "kernels": {k: {"launches": n, "ms_per_launch": ms / n, "share": ms / total_ms if total_ms else None}
                    for k, (n, ms) in sorted(kernels.items(), key=lambda kv: -kv[1][1])},
        "gpu_launches": launches,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clk,
        "workloads": table,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=gen.BENCH_WORKLOAD, choices=sorted(gen.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="approximate length of the CPU-oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload table (every workload's step timed on its own)")
    ap.add_argument("--repeats", type=int, default=0,
                    help="timed blocks of --steps steps (default: enough for about 3 s)")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="run the workload at this sequence length instead (small cases for profilers)")
    ap.add_argument("--lowrank-rows", type=int, default=0,
                    help="time only the low-rank projection's step (forward + backward) at this many "
                         "rows, with the low-rank workload's other sizes (for profilers)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps; the number is not a valid measurement",
              file=sys.stderr)
    world, rank, local = dist_setup()
    if world != args.gpus and rank == 0:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        if args.lowrank_rows:
            return run_lowrank_only(args, local)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
