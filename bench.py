"""Benchmark: CSR SpMM / SDDMM useful throughput on GB300.

One step = one pass of the whole hot path over the Transformer-FFN workload
of "Sparse GPU Kernels for Deep Learning" (Gale et al., SC 2020) as
configured here: sparse weights A of 4096x1024 and 1024x4096 at 70/80/90/95%
sparsity, each used by the SpMM forward (C = A·B, B K x 2048) and the SDDMM
weight gradient (mask(A) ⊙ X·Yᵀ with X M x 2048, Y K x 2048), in fp32 and in
bf16-in/fp32-accumulate: 32 launches of the library per step.  The row
swizzles are built once per sparsity pattern before timing (set-up, like the
pattern itself).

Metric: useful GFLOP/s = Σ 2·nnz·N over the step's products ÷ time.
Output: one JSON line (rank 0).  --impl reference times the CPU oracle on the
host cores instead (bounded row samples of the same workload).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

N_FFN = 2048
FP32_LANES_PER_SM = 128
SM_MAX_MHZ_DEFAULT = 2070.0  # GB300's maximum SM clock, when nothing better is known
# On-chip operand delivery: every useful FMA reads one dense-operand element
# from shared memory that no other FMA of its lane reuses, and shared memory
# delivers 128 B/clk/SM to 32-, 64- and 128-bit loads at random staged rows
# (measured on GB300 with clock64() in every CTA: profiles/operand_bound.md):
# at most 128/4 fp32 (128/2 bf16) FMAs per clock per SM.
SMEM_BYTES_PER_CLK = 128.0


class Device:
    """The SM count and maximum SM clock the roofline figures use: read from
    the device (and MEASURED_PEAKS.json's sm_max_mhz) when a GPU is present."""
    sms = 152
    sm_max_mhz = SM_MAX_MHZ_DEFAULT

    @classmethod
    def probe(cls, index=0):
        import torch
        cls.sms = torch.cuda.get_device_properties(index).multi_processor_count
        cls.sm_max_mhz = float((measured_peaks() or {}).get("sm_max_mhz", SM_MAX_MHZ_DEFAULT))


def fp32_peak_tflops():
    """FP32 CUDA-core peak: SMs x 128 FMA lanes x 2 flop x the maximum SM clock."""
    return Device.sms * FP32_LANES_PER_SM * 2 * Device.sm_max_mhz * 1e6 / 1e12


def operand_bound_tflops(elem_bytes):
    return Device.sms * SMEM_BYTES_PER_CLK / elem_bytes * 2 * Device.sm_max_mhz * 1e6 / 1e12
WORKLOAD = ("transformer_ffn: A 4096x1024 and 1024x4096 at 70/80/90/95% sparsity (row lengths "
            "N(mu, (0.1mu)^2), uniform columns, values N(0,0.02)); SpMM forward with B Kx2048 and "
            "SDDMM weight-gradient with X Mx2048, Y Kx2048, N(0,1); fp32 and bf16-in/fp32-acc")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except OSError:
        return None


# ---------------------------------------------------------------------------
# Work list
# ---------------------------------------------------------------------------
def tag_of(dtype, M, K, s):
    return f"{dtype}_{M}x{K}_s{s}"


WORKLOADS = {
    "ffn": "the hot path: SpMM forward + SDDMM weight-gradient per FFN problem (the bench line)",
    "ffn_train": "the sparse layer's training step per FFN problem: forward SpMM, weight-gradient SDDMM "
                 "(X = dC, Y = B), weights permuted into Aᵀ order, input-gradient SpMM on Aᵀ",
    "attention": "sparse attention, 8 heads x 4096, bf16: SDDMM scores, then the SpMM with V with the row softmax "
                 "fused into it (csr_spmm_row_softmax)",
    "attention_unfused": "sparse attention, 8 heads x 4096, bf16: SDDMM scores, row softmax to bf16, SpMM with V "
                         "(three calls)",
    "lstm": "LSTM-sized sweep, fp32: A 8192x4096 at 50/60/70/80/90/95/98%, B 4096x128, SpMM only",
    "dense_masks": "denser masks, fp32 SpMM only: the FFN shapes (A 4096x1024 and 1024x4096, B Kx2048) at "
                   "20/30/40/50% sparsity and the LSTM shape (A 8192x4096, B 4096x128) at 10/20/30/40% (masks at "
                   "least 55% set run the row-group kernel)",
    "resnet": "ResNet-50-like 1x1 conv, fp32: A 512x2048 at 80%, B 2048x3136 SpMM and SDDMM weight-gradient "
              "(X 512x3136, Y 2048x3136); L2 flushed before every step",
    "tiny": "tiny parity config, fp32: A 256x256 at 90%, B/X/Y 256x64, SpMM and SDDMM; launch-bound, so each "
            "call is timed as a CUDA graph of 100 calls (warm L2: the whole problem is 0.2 MB)",
}
DENSE_FFN_SPARSITIES = (20, 30, 40, 50)
DENSE_LSTM_SPARSITIES = (10, 20, 30, 40)
GRAPH_CALLS = 100  # calls per CUDA graph for the launch-bound workloads
GRAPHED = {"tiny"}
# Workloads whose operands fit in L2: a 256 MB buffer is written before every
# step and throughput comes from the launches' own events.
FLUSH_L2 = {"resnet"}


def problems(only=None, workload="ffn"):
    """Problems of one step.  `only` keeps the problems whose tag contains
    that substring."""
    if workload.startswith("attention"):
        return [W.attention()]
    keep = lambda p: not only or only.split(":")[-1] in tag_of(p.dtype, p.csr.M, p.csr.K, p.meta["sparsity"])
    if workload == "lstm":
        return [p for p in (W.lstm(s) for s in W.LSTM_SPARSITIES) if keep(p)]
    if workload == "resnet":
        return [p for p in [W.resnet()] if keep(p)]
    if workload == "tiny":
        return [W.tiny()]
    if workload == "dense_masks":
        ffn = [W.ffn(M, K, s, "f32", N=N_FFN, with_sddmm=False) for (M, K) in W.FFN_SHAPES
               for s in DENSE_FFN_SPARSITIES if not only or only.split(":")[-1] in tag_of("f32", M, K, s)]
        lstm = [W.lstm(s) for s in DENSE_LSTM_SPARSITIES
                if not only or only.split(":")[-1] in tag_of("f32", 8192, 4096, s)]
        return ffn + lstm
    out = []
    for dtype in ("f32", "bf16"):
        for (M, K) in W.FFN_SHAPES:
            for s in W.FFN_SPARSITIES:
                if only and only.split(":")[-1] not in tag_of(dtype, M, K, s):
                    continue
                out.append(W.ffn(M, K, s, dtype, N=N_FFN))
    return out


def ops_of(only, workload="ffn"):
    """Launches per problem; --only spmm:<tag> / sddmm:<tag> restricts the
    operation too."""
    if only and ":" in only:
        return (only.split(":")[0],)
    if workload == "ffn_train":
        return ("spmm", "sddmm_w", "permute", "spmm_t")
    if workload == "attention":
        return ("sddmm", "spmm_softmax")
    if workload == "attention_unfused":
        return ("sddmm", "softmax", "spmm")
    if workload in ("lstm", "dense_masks"):
        return ("spmm",)
    return ("spmm", "sddmm")


def width_of(p):
    return p.meta.get("N", N_FFN)


def flops_of(p, op):
    """Useful flops: 2·nnz·N for every product; the permutation and the
    softmax are not counted (their time is)."""
    if op in ("permute", "softmax"):
        return 0.0
    return 2.0 * p.csr.nnz * width_of(p)


def alg_bytes(p, op):
    """Bytes the operation must move at minimum (each operand once)."""
    es = 2 if p.dtype == "bf16" else 4
    M, K, nnz, N = p.csr.M, p.csr.K, p.csr.nnz, width_of(p)
    if op == "spmm":
        return nnz * (es + 4) + 4 * (M + 1) + K * N * es + 4 * M * N
    if op == "spmm_softmax":  # fp32 scores as values
        return nnz * (4 + 4) + 4 * (M + 1) + K * N * es + 4 * M * N
    if op == "spmm_t":  # Aᵀ (K x M) · dC (M x N) -> K x N
        return nnz * (es + 4) + 4 * (K + 1) + M * N * es + 4 * K * N
    if op == "permute":
        return nnz * (4 + 2 * es)
    if op == "softmax":
        return nnz * (4 + es) + 4 * (M + 1)
    return nnz * (4 + 4) + 4 * (M + 1) + (M + K) * N * es  # SDDMM variants, fp32 out


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, f in enumerate(flags) if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# Replicas over ranks (one GPU each; no data exchange)
# ---------------------------------------------------------------------------
def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (the job's time is its slowest
    replica's).  Uses the default process group; the tensor lives on
    `device` (the rank's GPU under NCCL, CPU under gloo)."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job rate: the units all ranks processed over the slowest rank's
    time (weak scaling: every replica runs the same step)."""
    return units_per_rank_step * steps * world / (max_ms * 1e-3)


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import torch
    import unstructured_sparse_matmul_gb300 as usm

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    Device.probe(local_rank)
    FP32_PEAK_TFLOPS = fp32_peak_tflops()
    usm.load()
    stream = torch.cuda.current_stream()

    def to_dev(x, dtype):
        if dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)

    wl = args.workload
    probs = problems(args.only, wl)
    if not probs:
        raise SystemExit(f"--only {args.only!r} matches no launch")
    lib = usm.load()
    items = []
    for p in probs:
        csr = p.csr
        N = width_of(p)
        bf = p.dtype == "bf16"
        d = {"p": p, "ro": to_dev(csr.row_offsets, "i32"), "ci": to_dev(csr.col_indices, "i32")}
        seg = p.meta.get("seq", 0) if wl.startswith("attention") else 0
        d["perm"] = usm.row_swizzle(d["ro"], csr.K, seg_rows=seg)
        d["seg"] = seg
        if wl.startswith("attention"):
            d["X"], d["Y"], d["V"] = to_dev(p.X, "bf16"), to_dev(p.Y, "bf16"), to_dev(p.V, "bf16")
            d["S"] = torch.empty(csr.nnz, dtype=torch.float32, device=dev)
            d["P"] = torch.empty(csr.nnz, dtype=torch.bfloat16, device=dev)
            d["C"] = torch.empty((csr.M, N), dtype=torch.float32, device=dev)
            ws_bytes = 0
        else:
            d["vals"] = to_dev(csr.values, p.dtype)
            d["B"] = to_dev(p.B, p.dtype)
            d["C"] = torch.empty((csr.M, N), dtype=torch.float32, device=dev)
            d["out"] = torch.empty(csr.nnz, dtype=torch.float32, device=dev)
            if wl == "ffn_train":
                d["dC"] = to_dev(W.dense(W.rng_for(9, p.meta["sparsity"], 6), csr.M, N, 1.0, p.dtype), p.dtype)
                d["ro_t"], d["ci_t"], d["v_t"], d["tperm"] = usm.csr_transpose(d["ro"], d["ci"], d["vals"], csr.K,
                                                                               with_perm=True)
                d["perm_t"] = usm.row_swizzle(d["ro_t"], csr.M)
                d["dB"] = torch.empty((csr.K, N), dtype=torch.float32, device=dev)
            elif p.X is not None:
                d["X"], d["Y"] = to_dev(p.X, p.dtype), to_dev(p.Y, p.dtype)
            ws_bytes = (lib.csr_sddmm_workspace_bytes(csr.M, csr.K, N, csr.nnz, 1 if bf else 0)
                        if any(op.startswith("sddmm") for op in ops_of(args.only, wl)) else 0)
        d["ws"] = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        d["nk_sddmm"] = 2 if ws_bytes > 0 else 1
        items.append(d)
    torch.cuda.synchronize()

    # Set-up cost, off the timed loop: the row swizzle of every pattern
    # (mean of 5 builds each, CUDA events).
    swz_ms = 0.0
    for d in items:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(5):
            usm.row_swizzle(d["ro"], d["p"].csr.K, seg_rows=d["seg"], out=d["perm"])
        e1.record(stream)
        torch.cuda.synchronize()
        swz_ms += e0.elapsed_time(e1) / 5

    # Launch list of one step: (label, op, item)
    launches = []
    for d in items:
        p = d["p"]
        tag = "bf16_8x4096_h64" if wl.startswith("attention") else tag_of(p.dtype, p.csr.M, p.csr.K, p.meta["sparsity"])
        for op in ops_of(args.only, wl):
            launches.append((f"{op}_{tag}", op, d))
    kernels_per_launch = {label: (d["nk_sddmm"] if op.startswith("sddmm") else 1) for label, op, d in launches}

    def run_one(op, d):
        K = d["p"].csr.K
        if wl.startswith("attention"):
            seg = d["p"].meta["seq"]
            if op == "sddmm":
                usm.sddmm(d["ro"], d["ci"], d["X"], d["Y"], row_swizzle=d["perm"], out=d["S"], seg_rows=seg)
            elif op == "spmm_softmax":
                usm.spmm_row_softmax(d["ro"], d["ci"], d["S"], d["V"], K=K, row_swizzle=d["perm"], out=d["C"],
                                     seg_rows=seg)
            elif op == "softmax":
                usm.row_softmax(d["ro"], d["S"], out=d["P"])
            else:
                usm.spmm(d["ro"], d["ci"], d["P"], d["V"], K=K, row_swizzle=d["perm"], out=d["C"], seg_rows=seg)
        elif op == "spmm":
            usm.spmm(d["ro"], d["ci"], d["vals"], d["B"], K=K, row_swizzle=d["perm"], out=d["C"])
        elif op == "sddmm":
            usm.sddmm(d["ro"], d["ci"], d["X"], d["Y"], row_swizzle=d["perm"], out=d["out"], workspace=d["ws"])
        elif op == "sddmm_w":
            usm.sddmm(d["ro"], d["ci"], d["dC"], d["B"], row_swizzle=d["perm"], out=d["out"], workspace=d["ws"])
        elif op == "permute":
            usm.csr_permute_values(d["tperm"], d["vals"], out=d["v_t"])
        elif op == "spmm_t":
            usm.spmm(d["ro_t"], d["ci_t"], d["v_t"], d["dC"], K=d["p"].csr.M, row_swizzle=d["perm_t"], out=d["dB"])

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if wl in FLUSH_L2 else None

    def step(events=None):
        """One pass over the launch list on one stream, optionally with
        events around every call."""
        if flush is not None:
            flush.zero_()
        for i, (label, op, d) in enumerate(launches):
            if events is not None:
                events[i][0].record(stream)
            run_one(op, d)
            if events is not None:
                events[i][1].record(stream)

    # The step's problems are independent (own outputs and workspaces): they
    # are dealt round-robin over `streams` compute streams, each problem's
    # calls in order on its stream, so one call's last wave of CTAs overlaps
    # the next problem's first.
    groups = []
    for label, op, d in launches:
        if not groups or groups[-1][0] is not d:
            groups.append((d, []))
        groups[-1][1].append(op)
    n_streams = max(1, min(args.streams, len(groups)))
    concurrent = n_streams > 1 and flush is None and wl not in GRAPHED
    cstreams = [torch.cuda.Stream(device=dev) for _ in range(n_streams)] if concurrent else []
    fork = torch.cuda.Event()
    joins = [torch.cuda.Event() for _ in cstreams]

    def step_streams():
        fork.record(stream)
        for cs in cstreams:
            cs.wait_event(fork)
        for j, (d, ops) in enumerate(groups):
            with torch.cuda.stream(cstreams[j % n_streams]):
                for op in ops:
                    run_one(op, d)
        for cs, e in zip(cstreams, joins):
            e.record(cs)
            stream.wait_event(e)

    for _ in range(args.warmup):
        step()
        if concurrent:
            step_streams()
    torch.cuda.synchronize()
    if usm.poll_status() != 0:
        raise RuntimeError("device status word set during warm-up")

    # Timed regions: (1) K steps on the compute streams (the step's time);
    # (2) K steps on one stream with events around every call (per-launch
    # durations and the roofline, free of overlap).  Clocks sampled across both.
    ev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in launches]
          for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    if concurrent:
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for k in range(args.steps):
            step_streams()
        c1.record(stream)
        torch.cuda.synchronize()
    start.record(stream)
    for k in range(args.steps):
        step(ev[k])
    stop.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    one_stream_ms = start.elapsed_time(stop)
    elapsed_ms = c0.elapsed_time(c1) if concurrent else one_stream_ms
    if usm.poll_status() != 0:
        raise RuntimeError("device status word set during the timed region")
    per_launch_ms = {label: statistics.mean(ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(args.steps))
                     for i, (label, _, _) in enumerate(launches)}

    if wl in GRAPHED:
        # Launch-bound: each call's time from a CUDA graph of GRAPH_CALLS calls
        # replayed `steps` times, so launch gaps do not count.
        side = torch.cuda.Stream(device=dev)
        for label, op, d in launches:
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                for _ in range(3):
                    run_one(op, d)
            stream.wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(GRAPH_CALLS):
                    run_one(op, d)
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            graph.replay()
            g0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            g1.record(stream)
            torch.cuda.synchronize()
            per_launch_ms[label] = g0.elapsed_time(g1) / (args.steps * GRAPH_CALLS)
        if usm.poll_status() != 0:
            raise RuntimeError("device status word set during the graph replays")
    if flush is not None or wl in GRAPHED:  # time the launches alone
        elapsed_ms = sum(per_launch_ms.values()) * args.steps
        one_stream_ms = elapsed_ms
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    one_stream_ms = max_over_ranks(one_stream_ms, world, dev)

    step_flops = sum(flops_of(d["p"], op) for _, op, d in launches)
    step_bytes = sum(alg_bytes(d["p"], op) for _, op, d in launches)
    value = job_throughput(step_flops, args.steps, world, elapsed_ms) / 1e9
    hbm = (measured_peaks() or {}).get("hbm_gbs", 6800.0)

    # Dominant launch (largest time) and its roofline.
    rows = []
    for label, op, d in launches:
        t = per_launch_ms[label] * 1e-3
        fl, by = flops_of(d["p"], op), alg_bytes(d["p"], op)
        # Launch roofline: min of the FP32 peak and HBM at the launch's
        # arithmetic intensity (algorithmic bytes).
        roof = min(FP32_PEAK_TFLOPS, hbm * 1e9 * fl / by / 1e12) if fl > 0 else 0.0
        opb = operand_bound_tflops(2 if d["p"].dtype == "bf16" else 4)
        rows.append({"launch": label, "ms": round(t * 1e3, 4), "tflops": round(fl / t / 1e12, 2),
                     "alg_gbs": round(by / t / 1e9, 1),
                     "frac_fp32": round(fl / t / 1e12 / FP32_PEAK_TFLOPS, 4),
                     "roofline_tflops": round(roof, 2),
                     "frac_roofline": round(fl / t / 1e12 / roof, 4) if roof > 0 else None,
                     "frac_operand_bound": round(fl / t / 1e12 / opb, 4) if fl > 0 else None})
    dom = max(rows, key=lambda r: r["ms"])
    dom_label = dom["launch"]
    traffic = recorded_traffic(dom_label)

    # End to end through the public API with host buffers.
    e2e = run_e2e(args, usm, torch, dev, launches, step_flops, n_streams) if not args.no_e2e and wl == "ffn" else None

    result = {
        "metric": "SpMM/SDDMM useful GFLOP/s (2·nnz·N), HBM GB/s, % of roofline on 1 GB300",
        "value": round(value, 1),
        "unit": "GFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 4),
        "ms_per_step_one_stream": round(one_stream_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("f32 + bf16-in/fp32-acc" if len({d["p"].dtype for d in items}) > 1
                  else "f32" if items[0]["p"].dtype == "f32" else "bf16-in/fp32-acc"),
        "data": "synthetic (seeded, shaped like the pages' " + ("Transformer-FFN weights)" if wl.startswith("ffn")
                                                                else f"{wl} workload)"),
        "config": {"workload": (WORKLOAD if wl == "ffn" else f"{wl}: {WORKLOADS[wl]}")
                   + (f" [only {args.only}]" if args.only else ""),
                   "launches_per_step": len(launches),
                   "l2": ("L2 flushed (256 MB written) before every step; value from the launches' events"
                          if flush is not None else
                          f"warm L2 (0.2 MB problem); each call timed in a CUDA graph of {GRAPH_CALLS} calls"
                          if wl in GRAPHED else "inputs larger than L2: each step's operands exceed 129 MB"),
                   "swizzle": "row swizzle built once per pattern before timing",
                   "streams": (f"{n_streams} compute streams, problems dealt round-robin, each problem's calls "
                               "in order on its stream; per-launch table and roofline from a second timed pass "
                               "on one stream with events around every call" if concurrent
                               else "one stream, events around every call"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "hbm_alg_gbs": round(step_bytes * args.steps * world / (elapsed_ms * 1e-3) / 1e9, 1),
        "roofline_frac_step": round(value / 1e3 / (FP32_PEAK_TFLOPS * world), 4),
        "roofline": {"bound": "alu", "achieved": dom["tflops"], "peak": round(FP32_PEAK_TFLOPS, 2),
                     "unit": "TFLOP/s", "frac": round(dom["tflops"] / FP32_PEAK_TFLOPS, 4),
                     "traffic": traffic, "kernel": dom_label,
                     "peak_source": f"derived: {Device.sms} SMs x 128 FP32 lanes x 2 flop x "
                                    f"{Device.sm_max_mhz / 1e3:.3g} GHz",
                     "operand_bound": {"peak": round(operand_bound_tflops(2 if "bf16" in dom_label else 4), 2),
                                       "frac": dom["frac_operand_bound"],
                                       "source": "shared-memory delivery 128 B/clk/SM (profiles/operand_bound.md), "
                                                 "one dense element per useful FMA"}},
        "setup": {"row_swizzle_ms_all_patterns": round(swz_ms, 4), "patterns": len(items)},
        # Measured character of every generated matrix (sparsity within its
        # diagonal block, mean row length, row-length CoV).
        "matrices": [dict({"name": d["p"].name, "dtype": d["p"].dtype},
                          **{k: (round(v, 4) if isinstance(v, float) else v) for k, v in W.stats(d["p"].csr).items()})
                     for d in items],
        "per_launch": rows,
        "gpu_launches": sum(kernels_per_launch[label] for label, _, _ in launches) * args.steps
                        * (GRAPH_CALLS if wl in GRAPHED else 1),
        "clocks": clocks,
    }
    if e2e is not None:
        result["e2e"] = e2e
    if rank == 0 and world == 1 and not args.no_cpu_baseline and wl == "ffn":
        result["cpu_baseline"] = cpu_baseline(args.cpu_sample, args.only)
    return result


# Source files that fix each timed operation's kernels and launch shapes (the
# grid decides how often staged tiles are re-read, so a launch-model change
# retires a capture as surely as a kernel change).
KERNEL_SOURCES = {
    "spmm": ("usm_spmm_kernel.cuh", "usm_spmm_group.cuh", "usm_spmm.cu", "usm_device.cuh", "usm_args.h",
             "usm_internal.h"),
    "sddmm": ("usm_sddmm_kernel.cuh", "usm_sddmm.cu", "usm_device.cuh", "usm_args.h", "usm_internal.h"),
}


def kernel_source_hash(op):
    """Hash of those sources (comments and whitespace removed, so only a
    change to the code itself retires a recorded capture)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES["spmm" if op.startswith("spmm") else "sddmm"]:
        with open(os.path.join(ROOT, "unstructured_sparse_matmul_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(label):
    """DRAM bytes per launch from the committed ncu summary for this launch,
    if it was captured on the current sources of its kernels (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash(label.split("_")[0])
    for line in open(path):
        parts = line.split()  # launch, bytes, [algorithmic bytes,] source hash
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == label and parts[-1] == src:
            return int(parts[1])
    return None


def run_e2e(args, usm, torch, dev, launches, step_flops, n_streams=1):
    """Same metric through the API with host buffers: every step copies the
    step's inputs from pinned host memory and reads the results back.

    The copies are pipelined against the kernels the way a caller feeding the
    library from host memory would: uploads on one stream, the library calls
    on the compute streams (problems dealt round-robin, as in the device-side
    step), downloads on another, problem by problem, with events so that
    problem i's kernels start once its own inputs have landed and a step never
    overwrites buffers the previous step still reads."""
    main = torch.cuda.current_stream()
    comps = [torch.cuda.Stream(device=dev) for _ in range(max(1, n_streams))]
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    order, per = [], {}
    for label, op, d in launches:
        key = id(d)
        if key not in per:
            order.append(key)
            ins = [(d[name].cpu().pin_memory(), d[name]) for name in ("ro", "ci", "vals", "B", "X", "Y", "perm")]
            per[key] = {"d": d, "in": ins, "out": [], "ops": []}
        out_t = d["C"] if op == "spmm" else d["out"]
        per[key]["out"].append((torch.empty(out_t.shape, dtype=out_t.dtype).pin_memory(), out_t))
        per[key]["ops"].append(op)
    h2d = sum(h.numel() * h.element_size() for k in order for h, _ in per[k]["in"])
    d2h = sum(h.numel() * h.element_size() for k in order for h, _ in per[k]["out"])
    ev = {k: {n: torch.cuda.Event() for n in ("in", "comp", "out")} for k in order}

    def e2e_step(serial=False):
        for j, k in enumerate(order):
            item, e = per[k], ev[k]
            comp = comps[0] if serial else comps[j % len(comps)]
            if serial:  # no overlap: each upload waits for the previous download
                comp.wait_stream(down)
                up.wait_stream(comp)
            d = item["d"]
            up.wait_event(e["comp"])  # the previous step's kernels are done with these inputs
            with torch.cuda.stream(up):
                for h, dv in item["in"]:
                    dv.copy_(h, non_blocking=True)
            e["in"].record(up)
            comp.wait_event(e["in"])
            comp.wait_event(e["out"])  # the previous step's results have been read back
            for op in item["ops"]:
                if op == "spmm":
                    usm.spmm(d["ro"], d["ci"], d["vals"], d["B"], K=d["p"].csr.K, row_swizzle=d["perm"],
                             out=d["C"], stream=comp)
                else:
                    usm.sddmm(d["ro"], d["ci"], d["X"], d["Y"], row_swizzle=d["perm"], out=d["out"],
                              workspace=d["ws"], stream=comp)
            e["comp"].record(comp)
            down.wait_event(e["comp"])
            with torch.cuda.stream(down):
                for h, dv in item["out"]:
                    h.copy_(dv, non_blocking=True)
            e["out"].record(down)

    steps = max(2, min(args.steps, 10))

    def timed(serial):
        for _ in range(2):
            e2e_step(serial)
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(main)
        for st in comps + [up, down]:
            st.wait_event(s0)
        for _ in range(steps):
            e2e_step(serial)
        for st in comps + [up, down]:
            main.wait_stream(st)
        s1.record(main)
        torch.cuda.synchronize()
        return step_flops * steps / (s0.elapsed_time(s1) * 1e-3) / 1e9

    value = timed(False)
    serial = timed(True)
    return {"value": round(value, 1), "unit": "GFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "overlap": f"uploads, kernels ({len(comps)} compute streams) and downloads pipelined problem by problem",
            "serial_value": round(serial, 1)}


# ---------------------------------------------------------------------------
# CPU oracle arm (cpu_baseline / --impl reference)
# ---------------------------------------------------------------------------
def oracle_sample_pass(probs, frac, nthreads=0):
    """Run the oracle on a row sample of every launch of one step on
    `nthreads` host threads (0: all); returns (flops done, seconds)."""
    import oracle
    flops, secs = 0.0, 0.0
    for p in probs:
        csr = p.csr
        nrows = max(1, int(round(csr.M * frac)))
        rows = np.arange(0, csr.M, max(1, csr.M // nrows))[:nrows]
        ro, ci, pos = oracle.select_rows(csr.row_offsets, csr.col_indices, rows)
        vals = oracle.widen(csr.values, p.dtype)[pos]
        B = oracle.widen(p.B, p.dtype)
        X = oracle.widen(p.X, p.dtype)[rows]
        Y = oracle.widen(p.Y, p.dtype)
        t0 = time.perf_counter()
        oracle.spmm(rows.size, csr.K, ro, ci, vals, B, nthreads)
        oracle.sddmm(rows.size, csr.K, ro, ci, X, Y, nthreads)
        secs += time.perf_counter() - t0
        flops += 2 * 2.0 * pos.size * N_FFN
    return flops, secs


def cpu_baseline(frac, only=None, passes=6):
    """The oracle timed on the host cores over `passes` passes of a row
    sample of every launch of one step (~10 s of CPU work on 16 cores at the
    defaults, where the sample is every row)."""
    import oracle
    probs = problems(only)
    flops, secs = 0.0, 0.0
    for _ in range(passes):
        f, t = oracle_sample_pass(probs, frac)
        flops += f
        secs += t
    # The same on one core, on a sample 1/16 the size (about as long).
    f1, t1 = oracle_sample_pass(probs, frac / 16, nthreads=1)
    return {"value": round(flops / secs / 1e9, 3), "unit": "GFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{passes} passes over every launch of one step, "
                      + ("all rows" if frac >= 1 else f"a {frac:.4g} row sample (rows evenly spaced)")
                      + f": {flops / 1e9:.1f} GFLOP in {secs:.1f} s",
            "value_1core": round(f1 / t1 / 1e9, 3),
            "sample_1core": f"one pass on a {frac / 16:.4g} row sample: {f1 / 1e9:.1f} GFLOP in {t1:.1f} s"}


def run_reference(args, rank, world):
    import oracle
    if rank != 0:
        return None
    probs = problems()
    frac = args.ref_sample
    for _ in range(args.warmup):
        oracle_sample_pass(probs, frac / 4)
    tot_f, tot_s = 0.0, 0.0
    for _ in range(args.steps):
        f, s = oracle_sample_pass(probs, frac)
        tot_f += f
        tot_s += s
    value = tot_f / tot_s / 1e9
    return {
        "impl": "reference",
        "metric": "SpMM/SDDMM useful GFLOP/s (2·nnz·N), HBM GB/s, % of roofline on 1 GB300",
        "value": round(value, 3), "unit": "GFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot_s * 1e3 / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": f"{frac:.4g} of the rows of every launch per step"},
        "cpu_baseline": {"value": round(value, 3), "unit": "GFLOP/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": f"{frac:.4g} row sample of every launch, per step"},
        "e2e": {"value": round(value, 3), "unit": "GFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def relaunch_under_torchrun(n):
    """Run this script again as n ranks on this node (127.0.0.1, a free
    port); returns the launcher's exit status."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd, env=dict(os.environ, MASTER_ADDR="127.0.0.1"))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample", type=float, default=1.0,
                    help="row fraction of each launch the cpu_baseline oracle computes (6 passes)")
    ap.add_argument("--ref-sample", type=float, default=0.25,
                    help="row fraction of each launch per step of the --impl reference arm")
    ap.add_argument("--streams", type=int, default=3,
                    help="compute streams the step's independent problems are dealt over (1: one stream)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="ffn", choices=sorted(WORKLOADS),
                    help="ffn (default, the bench line) or a measurement of the next rows")
    ap.add_argument("--only", default=None,
                    help="restrict to launches whose tag contains this (e.g. spmm:f32_4096x1024_s70); "
                         "for profiling a single kernel, not a bench line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.gpus < 1:
        raise SystemExit("--gpus must be at least 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # One process per GPU: start the N ranks under torch.distributed.run
        # (the same launch the multi-GPU runs use) and pass its status on.
        raise SystemExit(relaunch_under_torchrun(args.gpus))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch one rank per GPU")

    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res))
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
