#!/usr/bin/env python3
"""Benchmark of the Gated DeltaNet core on one B300 (or N replicas).

Timed step: one gdn_prefill over the grouped-head prefill workload (B=1,
16 query/key heads shared by 32 value heads, T=65536, d=128, bf16 q/k/v,
fp32 gates and state, S0 ~ N(0, 0.02^2)).  Inputs are resident in HBM and
larger than L2 (1.6 GB per step), so no flush is needed between steps.
The same run also times the decode workload (B=256 sequences, 32 value heads
over 16 key heads, d=128, 128 single-token steps, fp32 state updated in place)
and reports it under "decode", and the layer steps around the recurrence
(fused prologue: short convolution, SiLU, L2Norm, gates; fused epilogue:
sigmoid gate times zero-centred RMSNorm) on the prefill shape under "layer",
and the backward pass (gradients of the recurrence) on the training-shape
workload (B=2, H=16, T=4096, d=128, bf16) under "backward": the chunked
tensor-core path, with the fp32 token-sequential path beside it.  The other
prefill workloads are timed beside it: the training shape ("prefill_train"),
the long-context prefill (B=1, H=16, T=2^20, "prefill_long") and the grouped
shape with gates that barely decay ("prefill_weak_decay") and the grouped
shape with the channel-wise decay gate ("prefill_channelwise"), each with its
rooflines and an oracle sample.  The line ends with "summary", the headline
number of every section.

Printed: one JSON line (rank 0).  `value` is prefill tokens/s summed over all
ranks; `e2e` is the same metric through the C ABI with host buffers
(gdn_prefill_host: pinned host -> device copies of the inputs and device ->
host copies of y and S_T inside the timed region, overlapped with the
prefill piece by piece); `roofline` is the prefill kernel against measured
HBM bandwidth (its binding roof) with its tensor-core fraction beside it;
`cpu_baseline` is the fp64 oracle timed on a bounded sample on the host cores;
the decode, layer and backward sections carry their own oracle timing the same
way (a bounded sample, its rate scaled to the section's workload).

`--impl reference` times the fp64 oracle instead (the only reference
implementation there is), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN prefill tokens/s at H=32,T=64K,d=128 (% TC peak); decode steps/s (% HBM BW)"
PREFILL_WORKLOAD = "grouped"
DECODE_WORKLOAD = "decode"
CHUNK = 64  # chunk length of the useful-FLOP convention


# ----------------------------------------------------------------- accounting
def useful_flops_per_token_head(d: int, group: int, chunk: int = CHUNK) -> float:
    """Algorithmic FLOPs per (token, value head) of the chunked prefill.

    Three d x d products per token (W S, Q S, K~^T U) plus the chunk-local
    terms (T K, T V, P U per value head; K K^T and Q K^T per key head, shared
    by `group` value heads), causal triangles counted as halves.
    """
    return 2.0 * (3 * d * d + (chunk / 2) * (d + 2 * d) + (chunk / 2) * (2 * d) / group)


def prefill_bytes(w: dict, esz: int = 2, channelwise: bool = False) -> int:
    """Algorithmic HBM bytes of one prefill: q, k, v, y, alpha, beta, S0 and S_T once each
    (alpha [B, T, Hv, d] with the channel-wise gate)."""
    B, T, Hqk, Hv, d = w["B"], w["T"], w["Hqk"], w["Hv"], w["d"]
    io = (2 * B * T * Hqk * d + 2 * B * T * Hv * d) * esz
    gates = (d + 1 if channelwise else 2) * B * T * Hv * 4
    state = (2 if w.get("s0_std", 0) > 0 else 1) * B * Hv * d * d * 4
    return io + gates + state


def decode_bytes(w: dict, esz: int = 2) -> int:
    """Algorithmic HBM bytes of one decode step: the state read and written once, plus q, k, v, y, gates."""
    B, Hqk, Hv, d = w["B"], w["Hqk"], w["Hv"], w["d"]
    return 2 * B * Hv * d * d * 4 + (2 * B * Hqk * d + 2 * B * Hv * d) * esz + 2 * B * Hv * 4


# DRAM bytes per launch measured by ncu (dram__bytes_read.sum + dram__bytes_write.sum,
# summaries under profiles/), valid only for the kernel sources they were taken on
# (or sources that differ from them in comments only): a changed source reports null.
MEASURED_TRAFFIC = {
    "prefill": {"sources": ("csrc/chunked_tc.cu", "csrc/tc_ptx.cuh"), "sha256_16": "444d1a1c7f1030ab", "bytes": 1.652684e9},
    "decode": {"sources": ("csrc/recurrent.cu",), "sha256_16": "a3dc266465d55bf7", "bytes": 1.021420e9},
}


def measured_traffic(kind: str):
    import hashlib

    rec = MEASURED_TRAFFIC[kind]
    h = hashlib.sha256()
    for rel in rec["sources"]:
        with open(os.path.join(ROOT, "linear_attention_recurrence_14_b300", rel), "rb") as f:
            h.update(f.read())
    return rec["bytes"] if h.hexdigest()[:16] == rec["sha256_16"] else None


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return {"hbm_gbs": m["hbm_gbs"], "bf16_tflops": m["bf16_tflops"],
                "bf16_tflops_sustained": m.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while a region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for name, flag in zip(names, f[3:7]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- distributed
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist

        import torch

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def whole_job_rate(units_per_rank: float, local_ms: float, ws: int, device) -> tuple[float, float]:
    """Aggregate throughput of a weak-scaled run: every rank processed
    `units_per_rank` in `local_ms`; the job took the slowest rank's time.
    Returns (units per second over all ranks, max milliseconds)."""
    ms = max_over_ranks(local_ms, ws, device)
    return units_per_rank * ws / (ms * 1e-3), ms


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- oracle timing
def time_oracle_prefill(w: dict, seed: int, target_s: float, device="cpu", label: str = PREFILL_WORKLOAD,
                        channelwise: bool = False):
    """Time the fp64 oracle on the first T_s tokens of the workload (all heads).

    Returns (tokens/s, sample description, threads).  T_s is grown until one
    run takes about target_s seconds (bounded by the workload's T).
    """
    import oracle
    from linear_attention_recurrence_14_b300.inputs import make_channelwise_alpha, make_prefill_inputs

    oracle.build()
    threads = os.cpu_count() or 1
    Ts = 256
    while True:
        x = make_prefill_inputs(w["B"], Ts, w["Hqk"], w["Hv"], w["d"], w["dtype"], w["decay_scale"], w["s0_std"],
                                seed=seed, device=device)
        if channelwise:
            x.alpha = make_channelwise_alpha(w["B"], Ts, w["Hv"], w["d"], w["decay_scale"], seed=seed, device=device)
        t0 = time.perf_counter()
        oracle.recurrence(x.q, x.k, x.v, x.alpha, x.beta, x.S0, threads=threads)
        dt = time.perf_counter() - t0
        if dt >= target_s * 0.5 or Ts >= w["T"]:
            break
        Ts = min(w["T"], int(Ts * min(16.0, max(2.0, target_s / max(dt, 1e-3)))))
    tokens = w["B"] * Ts
    sample = (f"oracle fp64 on B={w['B']} x T={Ts} tokens x {w['Hv']} value heads of the "
              f"{label} workload ({dt:.2f} s)")
    return tokens / dt, sample, threads, dt


def _oracle_timed(fn, what: str) -> dict:
    """A bounded oracle timing beside a GPU section; a failure is reported in the line, not raised."""
    try:
        return fn()
    except Exception as exc:  # noqa: BLE001
        return {"kind": "oracle", "error": f"{what}: {type(exc).__name__}: {exc}"}


def _grow(n: int, dt: float, target_s: float, cap: int) -> int:
    return min(cap, int(n * min(16.0, max(2.0, target_s / max(dt, 1e-3)))))


def time_oracle_decode(w: dict, seed: int, target_s: float, sample_b: int = 16) -> dict:
    """The fp64 oracle stepping sample_b of the decode workload's sequences (all heads, state carried);
    the rate is scaled to the whole batch: steps/s of the full workload."""
    import oracle
    from linear_attention_recurrence_14_b300.inputs import make_decode_inputs

    oracle.build()
    threads = os.cpu_count() or 1
    Bs = min(sample_b, w["B"])
    steps = 1
    while True:
        d = make_decode_inputs(Bs, steps, w["Hqk"], w["Hv"], w["d"], w["dtype"], w["decay_scale"], w["s0_std"],
                               seed=seed, device="cpu")
        S = d.S0
        t0 = time.perf_counter()
        for i in range(steps):
            _, S = oracle.recurrence(d.q[i], d.k[i], d.v[i], d.alpha[i], d.beta[i], S, threads=threads)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * target_s or steps >= w["steps"]:
            break
        steps = _grow(steps, dt, target_s, w["steps"])
    return {"value": steps / dt * Bs / w["B"], "unit": "steps/s", "cores": threads, "kind": "oracle",
            "sample": f"oracle fp64, {steps} decode step(s) of {Bs} of the {w['B']} sequences x {w['Hv']} value "
                      f"heads ({dt:.2f} s); rate scaled to the whole batch"}


def time_oracle_layer(B, Hqk, Hv, d, K, T_full, seed: int, target_s: float) -> dict:
    """The numpy fp64 layer steps (prologue, then epilogue) on the first T_s tokens: tokens/s of both."""
    import oracle.layer as olayer
    from linear_attention_recurrence_14_b300.inputs import make_layer_inputs

    Ts = 64
    while True:
        x = make_layer_inputs(B, Ts, Hqk, Hv, d, K, seed=seed, device="cpu", with_state=True)
        t0 = time.perf_counter()
        olayer.prologue(x.xq, x.xk, x.xv, x.wq, x.wk, x.wv, x.a_raw, x.b_raw, x.A, x.b_alpha,
                        x.state_q, x.state_k, x.state_v)
        olayer.epilogue(x.y, x.z, x.norm_w, 1e-6)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * target_s or Ts >= T_full:
            break
        Ts = _grow(Ts, dt, target_s, T_full)
    return {"value": B * Ts / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"numpy fp64 prologue + epilogue on B={B} x T={Ts} tokens, all heads ({dt:.2f} s)"}


def time_oracle_backward(x, g, seed: int, target_s: float) -> dict:
    """The fp64 backward oracle on one (batch, value head) over the first T_s tokens; the rate is scaled
    to all value heads (the oracle runs heads one after another): tokens/s of the whole shape."""
    import oracle.backward as obw

    B, T, Hqk, d = x.q.shape
    Hv = x.v.shape[2]
    group = Hv // Hqk
    cpu = lambda t, n: t[:1, :n].detach().cpu()  # noqa: E731
    Ts = 64
    while True:
        q, k = cpu(x.q, Ts)[:, :, :1], cpu(x.k, Ts)[:, :, :1]
        v, a, b, dy = (cpu(t, Ts)[:, :, :1] for t in (x.v, x.alpha, x.beta, g.dy))
        dST = None if g.dS_T is None else g.dS_T[:1, :1].detach().cpu()
        t0 = time.perf_counter()
        obw.recurrence_grad(q, k, v, a, b, None, dy, dST)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * target_s or Ts >= T:
            break
        Ts = _grow(Ts, dt, target_s, T)
    return {"value": Ts / (dt * Hv), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"numpy fp64 backward of one value head (of {Hv}, group {group}) over T={Ts} tokens "
                      f"({dt:.2f} s); rate divided by the head count"}


# ----------------------------------------------------------------- main arms
def run_reference(args, ws, rank):
    if rank != 0:
        return
    from linear_attention_recurrence_14_b300.inputs import WORKLOADS

    w = dict(WORKLOADS[PREFILL_WORKLOAD])
    target = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    # size the sample once, then time K steps of it
    v, sample, threads, dt = time_oracle_prefill(w, args.seed, target)
    Ts = None
    for tok in sample.split():
        if tok.startswith("T="):
            Ts = int(tok[2:])
    import oracle
    from linear_attention_recurrence_14_b300.inputs import make_prefill_inputs

    x = make_prefill_inputs(w["B"], Ts, w["Hqk"], w["Hv"], w["d"], w["dtype"], w["decay_scale"], w["s0_std"],
                            seed=args.seed)
    for _ in range(args.warmup):
        oracle.recurrence(x.q, x.k, x.v, x.alpha, x.beta, x.S0, threads=threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.recurrence(x.q, x.k, x.v, x.alpha, x.beta, x.S0, threads=threads)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = w["B"] * Ts * args.steps / tot
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{PREFILL_WORKLOAD} prefill (B=1, Hqk=16, Hv=32, T=65536, d=128) sampled to T={Ts}",
                   "l2": "n/a (host)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"B={w['B']} x T={Ts} tokens x {w['Hv']} value heads per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_ours(args, ws, rank, local):
    import torch

    from linear_attention_recurrence_14_b300 import gdn
    from linear_attention_recurrence_14_b300.inputs import WORKLOADS, make_decode_inputs, make_prefill_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    gdn.lib()
    peaks = load_peaks()
    seed = args.seed + rank

    # ------------------------------------------------------------- prefill
    w = dict(WORKLOADS[PREFILL_WORKLOAD])
    x = make_prefill_inputs(w["B"], w["T"], w["Hqk"], w["Hv"], w["d"], w["dtype"], w["decay_scale"], w["s0_std"],
                            seed=seed, device=dev)
    shape = gdn.shape_of(x.q, x.v)
    y = torch.empty_like(x.v)
    S_T = torch.empty((w["B"], w["Hv"], w["d"], w["d"]), dtype=torch.float32, device=dev)
    ws_buf = gdn.new_workspace(shape, dev)
    launches = gdn.prefill_launches(shape, algorithm=args.algorithm, segments=args.segments)

    def prefill_once():
        gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, x.S0, y=y, S_T=S_T, workspace=ws_buf,
                    algorithm=args.algorithm, segments=args.segments)

    for _ in range(args.warmup):
        prefill_once()
    torch.cuda.synchronize()
    status = gdn.read_device_status(ws_buf)
    if status != 0:
        raise SystemExit(f"device status {status} after warm-up")

    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_all0 = torch.cuda.Event(enable_timing=True)
        t_all1 = torch.cuda.Event(enable_timing=True)
        t_all0.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            prefill_once()
            ev[i][1].record(stream)
        t_all1.record(stream)
        torch.cuda.synchronize()
    barrier(ws)
    status = gdn.read_device_status(ws_buf)
    if status != 0:
        raise SystemExit(f"device status {status} in the timed region")
    per_launch_ms = [a.elapsed_time(b) for a, b in ev]
    tokens = w["B"] * w["T"]
    value, total_ms = whole_job_rate(tokens * args.steps, t_all0.elapsed_time(t_all1), ws, dev)
    ms_per_step = total_ms / args.steps
    clocks = clk.summary()

    kern_s = statistics.mean(per_launch_ms) * 1e-3
    pbytes = prefill_bytes(w)
    flops = useful_flops_per_token_head(w["d"], w["Hv"] // w["Hqk"]) * w["B"] * w["T"] * w["Hv"]
    achieved_gbs = pbytes / kern_s / 1e9
    achieved_tflops = flops / kern_s / 1e12
    roofline = {
        "bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
        "frac": achieved_gbs / peaks["hbm_gbs"],
        "traffic": args.traffic if args.traffic is not None else measured_traffic("prefill"),
        "peak_source": peaks["source"], "bytes_per_launch": pbytes, "launch_ms": kern_s * 1e3,
        "tensor": {"achieved": achieved_tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                   "frac": achieved_tflops / peaks["bf16_tflops"],
                   "frac_sustained": achieved_tflops / peaks["bf16_tflops_sustained"]
                   if peaks.get("bf16_tflops_sustained") else None,
                   "flops_per_launch": flops},
    }

    # correctness spot check of this very run: sampled heads against the oracle
    check = None
    if args.check and rank == 0:
        check = spot_check(x, y, S_T, w)

    # ------------------------------------------------------------- e2e (host buffers)
    e2e = None
    if not args.no_e2e:
        e2e = time_e2e(args, x, shape, w, dev, ws)

    del ws_buf
    x = None
    torch.cuda.empty_cache()

    # ------------------------------------------------------------- the other prefill workloads
    prefills = {}
    if not args.no_prefill_configs:
        for name, nlaunch in (("train", 20), ("weak", 5), ("long", 3)):
            prefills[name] = time_prefill_section(args, peaks, seed, dev, ws, local, name, nlaunch)
        prefills["channelwise"] = time_prefill_section(args, peaks, seed, dev, ws, local, "grouped", 5,
                                                       channelwise=True)

    # ------------------------------------------------------------- decode
    dec = dec_cw = None
    if not args.no_decode:
        dec = time_decode(args, peaks, seed, dev, ws, local)
        dec_cw = time_decode(args, peaks, seed, dev, ws, local, channelwise=True)

    # ------------------------------------------------------------- layer prologue / epilogue
    layer = None
    if not args.no_layer:
        layer = time_layer(args, peaks, seed, dev, ws, local)
        torch.cuda.empty_cache()

    # ------------------------------------------------------------- backward
    bwd = None
    if not args.no_backward:
        bwd = time_backward(args, peaks, seed, dev, ws, local)
        torch.cuda.empty_cache()

    # ------------------------------------------------------------- cpu baseline
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, sample, threads, _ = time_oracle_prefill(w, seed, args.cpu_seconds)
        cpu = {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample}

    gpu_launches = launches * args.steps
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "grouped-head prefill: B=1, Hqk=16, Hv=32, T=65536, dk=dv=128, bf16 q/k/v, "
                               "fp32 alpha/beta/state, S0~N(0,0.02^2)",
                   "l2": "inputs larger than L2 (1.6 GB per step), no flush",
                   "algorithm": gdn.ALGO_NAMES[args.algorithm], "segments": args.segments,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": roofline, "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": gpu_launches,
        "check": check, "layer": layer, "backward": bwd,
        "prefill_train": prefills.get("train"), "prefill_long": prefills.get("long"),
        "prefill_weak_decay": prefills.get("weak"), "prefill_channelwise": prefills.get("channelwise"),
        "decode": dec, "decode_channelwise": dec_cw,
    }
    # Last, so that a reader of the line's tail sees every section: its headline numbers.
    line["summary"] = summarize(line)
    if rank == 0:
        print(json.dumps(line), flush=True)


def time_prefill_section(args, peaks, seed, dev, ws, local, name: str, launches_timed: int = 10,
                         channelwise: bool = False) -> dict:
    """gdn_prefill on another prefill workload (name in WORKLOADS): the median of `launches_timed`
    launches (CUDA events on the launching stream), its HBM and tensor-core rooflines, clocks, and
    the oracle on a bounded prefix of the same workload.  channelwise: the same workload with the
    channel-wise decay gate (alpha [B, T, Hv, d], same gate scale) through gdn_prefill_cw_ex."""
    import torch

    from linear_attention_recurrence_14_b300 import gdn
    from linear_attention_recurrence_14_b300.inputs import WORKLOADS, make_channelwise_alpha, make_prefill_inputs

    w = dict(WORKLOADS[name])
    x = make_prefill_inputs(w["B"], w["T"], w["Hqk"], w["Hv"], w["d"], w["dtype"], w["decay_scale"], w["s0_std"],
                            seed=seed, device=dev)
    shape = gdn.shape_of(x.q, x.v)
    y = torch.empty_like(x.v)
    S_T = torch.empty((w["B"], w["Hv"], w["d"], w["d"]), dtype=torch.float32, device=dev)
    if channelwise:
        x.alpha = make_channelwise_alpha(w["B"], w["T"], w["Hv"], w["d"], w["decay_scale"], seed=seed, device=dev)
        wsb = gdn.new_cw_workspace(shape, dev)
        wstat = gdn.new_workspace(shape, dev)   # status word only: read for uniformity with the scalar path

        def fn():
            gdn.prefill_cw(x.q, x.k, x.v, x.alpha, x.beta, x.S0, y=y, S_T=S_T, workspace=wsb)
    else:
        wsb = wstat = gdn.new_workspace(shape, dev)

        def fn():
            gdn.prefill(x.q, x.k, x.v, x.alpha, x.beta, x.S0, y=y, S_T=S_T, workspace=wsb)

    for _ in range(max(3, args.warmup)):
        fn()
    torch.cuda.synchronize()
    if gdn.read_device_status(wstat) != 0:
        raise SystemExit(f"device status error in the {name} prefill")
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(launches_timed)]
    barrier(ws)
    with ClockSampler(local) as clk:
        for a, b in evs:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
    if gdn.read_device_status(wstat) != 0:
        raise SystemExit(f"device status error in the {name} prefill")
    ms = max_over_ranks(statistics.median(a.elapsed_time(b) for a, b in evs), ws, dev)
    nbytes = prefill_bytes(w, channelwise=channelwise)
    # channel-wise: every value head forms its own gated keys, so no Gram product is shared
    flops = useful_flops_per_token_head(w["d"], 1 if channelwise else w["Hv"] // w["Hqk"]) * w["B"] * w["T"] * w["Hv"]
    gbs = nbytes / (ms * 1e-3) / 1e9
    tf = flops / (ms * 1e-3) / 1e12
    out = {
        "workload": f"{name}: B={w['B']}, T={w['T']}, Hqk={w['Hqk']}, Hv={w['Hv']}, d={w['d']}, {w['dtype']} q/k/v, "
                    f"{'channel-wise ' if channelwise else ''}gate scale {w['decay_scale']}, S0 std {w['s0_std']}",
        "ms": ms, "tokens_per_s": w["B"] * w["T"] * ws / (ms * 1e-3),
        "gpu_launches": (2 if channelwise else gdn.prefill_launches(shape)) * launches_timed,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None, "bytes_per_launch": nbytes,
                     "peak_source": peaks["source"],
                     "tensor": {"achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                "frac": tf / peaks["bf16_tflops"], "flops_per_launch": flops}},
        "clocks": clk.summary(),
        "l2": f"inputs {nbytes / 1e9:.2f} GB per launch" + (" (larger than L2, no flush)" if nbytes > 126e6 else
                                                            " (fit in L2: timed back to back)"),
    }
    if channelwise:
        out["kernels"] = "cw_prepass_kernel (per chunk) + cw_chain_kernel (per head and segment); roofline over both"
    del x, y, S_T, wsb, wstat
    torch.cuda.empty_cache()
    if local == 0 and not args.no_cpu_baseline:
        def oracle_rate():
            v, sample, threads, _ = time_oracle_prefill(w, seed, args.oracle_seconds, label=name,
                                                        channelwise=channelwise)
            return {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample}
        out["cpu_baseline"] = _oracle_timed(oracle_rate, f"{name} oracle")
    return out


def summarize(line: dict) -> dict:
    """Headline numbers of every section of the line, rounded: times (ms), rates, and the
    fraction of the binding roof (HBM, or the fp32 FMA peak for the backward)."""
    def g(d, *path):
        for k in path:
            if not isinstance(d, dict) or d.get(k) is None:
                return None
            d = d[k]
        return float(f"{d:.4g}") if isinstance(d, (int, float)) else d
    out = {"grouped_ms": g(line, "roofline", "launch_ms"), "grouped_hbm": g(line, "roofline", "frac"),
           "grouped_tc": g(line, "roofline", "tensor", "frac"), "e2e_ms": g(line, "e2e", "ms_per_step"),
           "e2e_of_link_floor": g(line, "e2e", "link", "frac_of_floor"),
           "check_err": g(line, "check", "max_rel_err_y")}
    for key, short in (("prefill_train", "train"), ("prefill_long", "long"), ("prefill_weak_decay", "weak"),
                       ("prefill_channelwise", "cw")):
        out[f"{short}_ms"] = g(line, key, "ms")
        out[f"{short}_hbm"] = g(line, key, "roofline", "frac")
    out["decode_steps_s"] = g(line, "decode", "value")
    out["decode_hbm"] = g(line, "decode", "roofline", "frac")
    out["decode_cw_steps_s"] = g(line, "decode_channelwise", "value")
    out["decode_cw_hbm"] = g(line, "decode_channelwise", "roofline", "frac")
    out["prologue_hbm"] = g(line, "layer", "prologue", "roofline", "frac")
    out["epilogue_hbm"] = g(line, "layer", "epilogue", "roofline", "frac")
    out["backward_ms"] = g(line, "backward", "ms")
    out["backward_tc"] = g(line, "backward", "roofline", "frac")
    out["backward_fp32_ms"] = g(line, "backward", "sequential_fp32", "ms")
    return {k: v for k, v in out.items() if v is not None}


def spot_check(x, y, S_T, w):
    """Compare two sampled value heads over the first tokens with the oracle."""
    import numpy as np

    import oracle

    Tcheck = min(w["T"], 8192)
    errs = []
    for hv in (0, w["Hv"] - 1):
        yo, so = oracle.recurrence_head(x.q, x.k, x.v, x.alpha, x.beta, x.S0, 0, hv, T=Tcheck)
        yg = y[0, :Tcheck, hv].double().cpu().numpy()
        errs.append(float(np.abs(yg - yo).max() / max(np.abs(yo).max(), 1e-30)))
    return {"heads": [0, w["Hv"] - 1], "tokens": Tcheck, "max_rel_err_y": max(errs)}


def time_e2e(args, x, shape, w, dev, ws):
    """Prefill from host buffers through gdn_prefill_host (the public entry point for host memory):
    the host-to-device copy of the inputs and the device-to-host copy of y and S_T are inside the
    timed region, overlapped with the prefill piece by piece (pieces of T/8 tokens)."""
    import torch

    from linear_attention_recurrence_14_b300 import gdn

    host = {n: getattr(x, n).cpu().pin_memory() for n in ("q", "k", "v", "alpha", "beta")}
    host["S0"] = x.S0.cpu().pin_memory() if x.S0 is not None else None
    y_host = torch.empty_like(host["v"]).pin_memory()
    S_host = torch.empty((w["B"], w["Hv"], w["d"], w["d"]), dtype=torch.float32).pin_memory()
    wsb = gdn.new_host_workspace(shape, dev)
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = y_host.numel() * y_host.element_size() + S_host.numel() * 4

    def step():
        gdn.prefill_host(host["q"], host["k"], host["v"], host["alpha"], host["beta"], host["S0"], y=y_host,
                         S_T=S_host, workspace=wsb, device=dev)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 5))
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    value = w["B"] * w["T"] * ws * steps / (ms * 1e-3)
    link = measure_link(dev, h2d, d2h)
    floor_ms = link["both_ms"]
    link.update({"floor_ms_per_step": floor_ms, "frac_of_floor": floor_ms / (ms / steps),
                 "floor": "the step's two copies issued together on two streams (measured), i.e. the "
                          "host link with nothing else to do"})
    return {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "ms_per_step": ms / steps, "api": "gdn_prefill_host (pinned host buffers)",
            "link": link}


def measure_link(dev, h2d: int, d2h: int) -> dict:
    """Host link rates: one pinned host -> device copy of h2d bytes and one device -> host copy of
    d2h bytes, each timed alone with CUDA events (best of 3), and both issued together on two
    streams (host clock around a synchronised pair, best of 3)."""
    import torch

    a = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    b = torch.empty(h2d, dtype=torch.uint8, device=dev)
    c = torch.empty(d2h, dtype=torch.uint8, device=dev)
    e = torch.empty(d2h, dtype=torch.uint8).pin_memory()

    def best(fn, n):
        t = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            t.append(e0.elapsed_time(e1))
        return n / (min(t) * 1e-3) / 1e9

    out = {"h2d_gbs": best(lambda: b.copy_(a, non_blocking=True), h2d),
           "d2h_gbs": best(lambda: e.copy_(c, non_blocking=True), d2h)}
    # both directions at once (two streams): what the host link sustains for one e2e step
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    t = []
    for _ in range(3):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(s1):
            b.copy_(a, non_blocking=True)
        with torch.cuda.stream(s2):
            e.copy_(c, non_blocking=True)
        torch.cuda.synchronize()
        t.append((time.perf_counter() - t0) * 1e3)
    out["both_ms"] = min(t)
    del a, b, c, e
    torch.cuda.empty_cache()
    return out


def layer_bytes(B, T, Hqk, Hv, d, kconv=4) -> tuple[int, int]:
    """Algorithmic HBM bytes of the layer prologue and epilogue: every input read once and
    every output written once (bf16 features, fp32 gates; taps and states negligible)."""
    rows_qk, rows_v = B * T * Hqk, B * T * Hv
    pro = 2 * (2 * rows_qk + rows_v) * d * 2 + 4 * rows_v * 4
    epi = 3 * rows_v * d * 2
    return pro, epi


def time_layer(args, peaks, seed, dev, ws, local):
    """The layer prologue and epilogue on the prefill shape (B=1, T=65536, Hqk=16, Hv=32, d=128,
    four convolution taps); each against measured HBM bandwidth."""
    import torch

    from linear_attention_recurrence_14_b300 import gdn
    from linear_attention_recurrence_14_b300.inputs import make_layer_inputs

    B, T, Hqk, Hv, d, K = 1, 65536, 16, 32, 128, 4
    x = make_layer_inputs(B, T, Hqk, Hv, d, K, seed=seed, device=dev, with_state=True)
    out = gdn.layer_prologue(x.xq, x.xk, x.xv, x.wq, x.wk, x.wv, x.a_raw, x.b_raw, x.A, x.b_alpha,
                             state_q=x.state_q, state_k=x.state_k, state_v=x.state_v, state_out=True)
    o = torch.empty_like(x.y)
    stream = torch.cuda.current_stream()

    def pro():
        gdn.layer_prologue(x.xq, x.xk, x.xv, x.wq, x.wk, x.wv, x.a_raw, x.b_raw, x.A, x.b_alpha,
                           state_q=x.state_q, state_k=x.state_k, state_v=x.state_v, state_out=True, out=out)

    def epi():
        gdn.layer_epilogue(x.y, x.z, x.norm_w, 1e-6, o=o)

    res = {}
    pb, eb = layer_bytes(B, T, Hqk, Hv, d, K)
    with ClockSampler(local) as clk:
        for name, fn, nbytes in (("prologue", pro, pb), ("epilogue", epi, eb)):
            for _ in range(max(3, args.warmup)):
                fn()
            torch.cuda.synchronize()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
            barrier(ws)
            for a, b in evs:
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize()
            ms = max_over_ranks(statistics.median(a.elapsed_time(b) for a, b in evs), ws, dev)
            gbs = nbytes / (ms * 1e-3) / 1e9
            res[name] = {"ms": ms, "tokens_per_s": B * T * ws / (ms * 1e-3),
                         "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                      "frac": gbs / peaks["hbm_gbs"], "traffic": None, "bytes_per_launch": nbytes,
                                      "peak_source": peaks["source"]},
                         "gpu_launches": 1}
    if local == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = _oracle_timed(
            lambda: time_oracle_layer(B, Hqk, Hv, d, K, T, seed, args.oracle_seconds), "layer oracle")
    res["config"] = "B=1, T=65536, Hqk=16, Hv=32, d=128, 4 taps, bf16 features, fp32 gates; median of 20 launches"
    res["l2"] = "inputs larger than L2 (2.2 GB prologue, 1.6 GB epilogue), no flush"
    res["clocks"] = clk.summary()
    return res


def backward_flops_per_token_head(d: int) -> float:
    """Useful fp32 FLOPs of one backward token per (token, value head): eight d x d passes of two FLOPs
    per element -- S dy, G += q dy^T, G^T k, G e, S~ de, G -= k de^T, and the forward rebuild's S^T k
    and state update."""
    return 8 * 2.0 * d * d


def fp32_alu_peak_tflops(sm_mhz: float, sms: int = 148) -> float:
    """FP32 FMA peak: 128 FMA lanes per SM, 2 FLOPs per FMA, at the given SM clock."""
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


def backward_chunked_flops_per_chunk(d: int = 128, chunk: int = 64) -> float:
    """Tensor-core FLOPs of the chunked backward per (chunk, value head), products as executed
    (block-triangular operands skip their zero blocks): the pre-pass, the forward chain (no y),
    the reverse chain and the per-chunk gradient kernel."""
    C, blocks = chunk, chunk // 16
    tri = sum(range(1, blocks + 1)) / blocks ** 2        # fraction of 16 x 16 blocks on or below the diagonal
    full_cd = C * d * d            # a 64 x d x d product
    cc_d = C * C * d               # a 64 x 64 x d product
    prepass = 2 * cc_d * tri + 2 * C * C * d * tri       # A and P by row block; W and U~ from block-lower T
    fwd_chain = 2 * full_cd                              # U = U~ - W S, S' = gamma S + Kl^T U
    rev_chain = cc_d * tri + 3 * full_cd                 # P^T dY, Kl dS', Qp^T dY, W^T dU
    grad = (2 * cc_d                                     # K K^T, Q K^T
            + 2 * cc_d * tri + full_cd                   # W, U~; W S
            + full_cd + cc_d * tri                       # K dS'; P^T dY
            + 3 * full_cd + cc_d                         # U dS'^T, dY S^T, Q S; dY U^T
            + 2 * cc_d * tri + full_cd                   # dQK K, dQK^T Q; dU S^T
            + 2 * cc_d * tri + 2 * cc_d                  # T^T dU, T^T dW; dW K^T, dU V^T
            + C * C * C * tri + C * C * C                # T^T dT; X T^T
            + 2 * cc_d * tri)                            # (dKK + dKK^T) K
    return 2.0 * (prepass + fwd_chain + rev_chain + grad)


def time_backward(args, peaks, seed, dev, ws, local):
    """gdn_backward_chunked (tensor cores) and gdn_backward (fp32, token by token) on the
    training-shape workload (B=2, H=16, T=4096, d=128, bf16 inputs, dy ~ N(0,1), dS_T ~ N(0,1));
    median of 10 calls each."""
    import torch

    from linear_attention_recurrence_14_b300 import gdn
    from linear_attention_recurrence_14_b300.inputs import make_backward_grads, workload_inputs

    x = workload_inputs("train", seed=seed, device=dev)
    B, T, Hqk, d = x.q.shape
    Hv = x.v.shape[2]
    g = make_backward_grads(B, T, Hv, d, "bf16", ds_std=1.0, seed=seed, device=dev)
    shape = gdn.shape_of(x.q, x.v)
    stream = torch.cuda.current_stream()
    # algorithmic HBM bytes: inputs (q, k, v, dy bf16; alpha, beta fp32), outputs (dq, dk, dv fp32,
    # dlog_alpha, dbeta fp32), dS_T in and dS0 out
    nbytes = (2 * B * T * Hqk * d * 2 + 2 * B * T * Hv * d * 2 + 2 * B * T * Hv * 4
              + 2 * B * T * Hqk * d * 4 + B * T * Hv * d * 4 + 2 * B * T * Hv * 4 + 2 * B * Hv * d * d * 4)

    def timed(algorithm):
        chunked = algorithm == gdn.ALGO_CHUNKED
        wsb = gdn.new_backward_workspace(shape, dev, chunked=chunked)
        out = gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, g.dS_T, workspace=wsb, algorithm=algorithm)

        def fn():
            gdn.backward(x.q, x.k, x.v, x.alpha, x.beta, x.S0, g.dy, g.dS_T, out=out, workspace=wsb,
                         algorithm=algorithm)

        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
        barrier(ws)
        with ClockSampler(local) as clk:
            for a, b in evs:
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize()
        ms = max_over_ranks(statistics.median(a.elapsed_time(b) for a, b in evs), ws, dev)
        del wsb, out
        torch.cuda.empty_cache()
        return ms, clk.summary()

    hbm = lambda ms: {"bytes_per_call": nbytes, "achieved_gbs": nbytes / (ms * 1e-3) / 1e9,  # noqa: E731
                      "frac": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}
    # chunked, tensor cores: against the bf16 tensor peak
    ms, clocks = timed(gdn.ALGO_CHUNKED)
    nchunks = (T + 63) // 64
    flops = backward_chunked_flops_per_chunk(d) * B * nchunks * Hv
    tf = flops / (ms * 1e-3) / 1e12
    # fp32 token-sequential: against the fp32 FMA peak
    ms_s, clocks_s = timed(gdn.ALGO_SEQUENTIAL)
    flops_s = backward_flops_per_token_head(d) * B * T * Hv
    tf_s = flops_s / (ms_s * 1e-3) / 1e12
    peak_s = fp32_alu_peak_tflops(clocks_s.get("sm_max_mhz") or 2032)
    return {"ms": ms, "tokens_per_s": B * T * ws / (ms * 1e-3),
            "path": "gdn_backward_chunked: pre-pass, forward chain, reverse chain, per-chunk gradients "
                    "(warp-level bf16 MMAs, fp32 accumulation)",
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16_tflops"], "traffic": None, "flops_per_call": flops,
                         "flops_convention": "MMA products as executed, zero blocks of triangular operands skipped",
                         "peak_source": peaks["source"], "hbm": hbm(ms)},
            "gpu_launches": 4 * 10,
            "sequential_fp32": {"ms": ms_s, "tokens_per_s": B * T * ws / (ms_s * 1e-3),
                                "roofline": {"bound": "alu", "achieved": tf_s, "peak": peak_s, "unit": "TFLOP/s",
                                             "frac": tf_s / peak_s, "flops_per_call": flops_s,
                                             "peak_source": "fp32 FMA: 148 SMs x 128 lanes x 2 FLOPs at the "
                                                            "sampled max SM clock", "hbm": hbm(ms_s)},
                                "gpu_launches": gdn.backward_launches(shape) * 10, "clocks": clocks_s},
            "config": "training-shape backward: B=2, H=16, T=4096, d=128, bf16 q/k/v/dy, fp32 gates, state and "
                      "gradients; median of 10 calls",
            "l2": "inputs and workspace larger than L2, no flush", "clocks": clocks,
            "cpu_baseline": _oracle_timed(lambda: time_oracle_backward(x, g, seed, args.oracle_seconds),
                                          "backward oracle") if local == 0 and not args.no_cpu_baseline else None}


def time_decode(args, peaks, seed, dev, ws, local, channelwise=False):
    """128 decode steps of the decode workload, state in place; returns steps/s and its HBM roofline.
    channelwise: the per-key-channel decay gate (gdn_decode_step_cw, alpha [B, 1, Hv, dk])."""
    import torch

    from linear_attention_recurrence_14_b300 import gdn
    from linear_attention_recurrence_14_b300.inputs import WORKLOADS, make_channelwise_alpha, make_decode_inputs

    w = dict(WORKLOADS[DECODE_WORKLOAD])
    nsteps = args.decode_steps
    d = make_decode_inputs(w["B"], nsteps, w["Hqk"], w["Hv"], w["d"], w["dtype"], w["decay_scale"], w["s0_std"],
                           seed=seed, device=dev)
    S = d.S0.clone()
    ys = torch.empty((nsteps,) + tuple(d.v.shape[1:]), dtype=d.v.dtype, device=dev)
    if channelwise:
        acw = make_channelwise_alpha(nsteps * w["B"], 1, w["Hv"], w["d"], w["decay_scale"], seed=seed, device=dev)
        acw = acw.reshape(nsteps, w["B"], 1, w["Hv"], w["d"])

    def one(s):
        if channelwise:
            gdn.decode_step_cw(d.q[s], d.k[s], d.v[s], acw[s], d.beta[s], S, y=ys[s])
        else:
            gdn.decode_step(d.q[s], d.k[s], d.v[s], d.alpha[s], d.beta[s], S, y=ys[s])

    def run_all():
        for s in range(nsteps):
            one(s)

    for _ in range(max(1, args.warmup)):
        S.copy_(d.S0)
        run_all()
    torch.cuda.synchronize()
    S.copy_(d.S0)
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nsteps)]
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for s in range(nsteps):
            evs[s][0].record(stream)
            one(s)
            evs[s][1].record(stream)
        a1.record(stream)
        torch.cuda.synchronize()
    total_ms = max_over_ranks(a0.elapsed_time(a1), ws, dev)
    per = [a.elapsed_time(b) for a, b in evs]
    kern_s = statistics.mean(per) * 1e-3
    nbytes = decode_bytes(w) + (w["B"] * w["Hv"] * (w["d"] - 1) * 4 if channelwise else 0)
    gbs = nbytes / kern_s / 1e9
    return {
        "metric": "decode steps/s (B=256, Hv=32, Hqk=16, d=128, fp32 state in place, bf16 q/k/v"
                  + (", channel-wise decay gate)" if channelwise else ")"),
        "value": nsteps * ws / (total_ms * 1e-3), "unit": "steps/s", "steps": nsteps, "ms_per_step": total_ms / nsteps,
        "gpu_launches": nsteps,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"],
                     "traffic": None if channelwise else (
                         args.decode_traffic if args.decode_traffic is not None else measured_traffic("decode")),
                     "bytes_per_launch": nbytes,
                     "launch_ms": kern_s * 1e3, "peak_source": peaks["source"]},
        "clocks": clk.summary(),
        "l2": "state 512 MiB > L2, no flush",
        "cpu_baseline": _oracle_timed(lambda: time_oracle_decode(w, seed, args.oracle_seconds), "decode oracle")
        if local == 0 and not args.no_cpu_baseline and not channelwise else None,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--algorithm", type=int, default=0, help="0 auto, 1 chunked, 2 sequential")
    ap.add_argument("--segments", type=int, default=0, help="0 = chosen by the library")
    ap.add_argument("--decode-steps", type=int, default=128)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--oracle-seconds", type=float, default=3.0,
                    help="target time of each oracle sample beside the decode, layer and backward sections")
    ap.add_argument("--traffic", type=float, default=None, help="ncu dram bytes per prefill launch, if measured")
    ap.add_argument("--decode-traffic", type=float, default=None, help="ncu dram bytes per decode launch")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-layer", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-prefill-configs", action="store_true",
                    help="skip the training-shape, long-context and weak-decay prefill sections")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-check", dest="check", action="store_false")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
