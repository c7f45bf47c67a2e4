#!/usr/bin/env python3
"""Benchmark of the outer-product associative-memory layers on one GPU per rank.

Default run (N=1): the Tensor Cache bf16 prefill workload (B=4, H=8, T=4096,
d=64, W=512) as the headline step -- one tc_layer_forward over the batch --
captured once into a CUDA graph and replayed, each replay timed with CUDA
events after warm-up and an L2 flush (256 MiB write) between timed steps (the
same step as eager Python calls is reported under "eager"), plus:
  * roofline of the dominant kernel, timed live through the library's
    profiling events, against MEASURED_PEAKS.json;
  * e2e: the same step through the public binding from pinned host buffers,
    host<->device copies inside the timed region (per-sequence chunks on two
    streams, so uploads, compute and downloads overlap);
  * cpu_baseline: the float64 oracle on the host cores;
  * the other workloads (long-context prefill, 64-sequence decode, DeltaNet,
    BDH sparse) under "workloads", each with its own roofline;
  * SM clocks / throttle reasons sampled with nvidia-smi during timing.
``--impl reference`` times the oracle instead (the reference arm).
Multi-GPU (torchrun): each rank runs an independent batch (weak scaling, no
collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "memory-layer tokens/s (prefill, decode) and % of HBM/tensor-core roofline"
HEADLINE = "tc_bf16_B4_H8_T4096_d64_W512"
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ----------------------------------------------------------------- peaks
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- algorithmic work
def tc_pairs(T, W):
    """Number of (query, key) pairs inside the causal window of W, per head."""
    if T <= W:
        return T * (T + 1) // 2
    return W * (W + 1) // 2 + (T - W) * W


def tc_prefill_work(B, H, T, d_k, d_v, W, elem, l2=True):
    """Algorithmic flops / bytes of the prefill: QK^T and PV over the window;
    with the L2 memory, per token with an eviction the write of k v^T into A
    (2 d_k d_v) and the read q A (2 d_k d_v); q, k, v read once, y written
    once."""
    BH = B * H
    soft = 2 * (d_k + d_v) * tc_pairs(T, W) * BH
    l2_rw = 4 * d_k * d_v * max(0, T - W) * BH if l2 else 0
    flops = soft + l2_rw
    bytes_ = BH * T * (2 * d_k + 2 * d_v) * elem
    return flops, bytes_


def tc_decode_work(S, H, d_k, d_v, W, elem):
    """Per decode step: the ring (W keys + W values) streamed once, A read and
    written once (fp32), q/k/v in and y out."""
    SH = S * H
    flops = SH * (2 * W * (d_k + d_v) + 4 * d_k * d_v)
    bytes_ = SH * (W * (d_k + d_v) * elem + 2 * d_k * d_v * 4 + (2 * d_k + 2 * d_v) * elem)
    return flops, bytes_


def delta_work(B, H, T, d_k, d_v, elem, C=64):
    """Chunked form: per token 2C(d_k + d_v) (intra-chunk products) plus
    6 d_k d_v (state read, correction, write); q, k, v, beta read, y written."""
    BH = B * H
    flops = BH * T * (4 * C * (d_k + d_v) // 2 + 6 * d_k * d_v)
    bytes_ = BH * T * ((2 * d_k + 2 * d_v) * elem + 4)
    return flops, bytes_


def delta_decode_work(S, H, d_k, d_v, elem):
    """Per decode step: the fp32 state read and written once (two dot products
    and a rank-1 update, 6 d_k d_v flops), q/k/v and beta in, y out."""
    SH = S * H
    flops = SH * 6 * d_k * d_v
    bytes_ = SH * (2 * d_k * d_v * 4 + (2 * d_k + 2 * d_v) * elem + 4)
    return flops, bytes_


def tc_backward_work(B, H, T, d_k, d_v, W, elem, split=False):
    """Backward of the prefill: the window part recomputes S = QK^T and the
    statistics (2 d_k per pair), y_loc (2 d_v), then dP = dy V^T (2 d_v),
    dQ, dK (2 d_k each) and dV (2 d_v) per (query, key) pair in the window;
    the L2 part is four d_k x d_v contractions per evicted token (dq, dk',
    dv', and the state write it replays), plus the same for the lambda
    derivative.  Bytes: q, k, v, dy read once; dq, dk, dv written once.
    With split=True the flops come back as (window, L2) separately."""
    BH = B * H
    pairs = tc_pairs(T, W) * BH
    window = pairs * (2 * d_k + 2 * d_v + 2 * d_v + 2 * d_k + 2 * d_k + 2 * d_v)
    l2 = 10 * d_k * d_v * max(0, T - W) * BH
    bytes_ = BH * T * (3 * d_k + 3 * d_v) * elem
    if split:
        return window, l2, bytes_
    return window + l2, bytes_


def mixed_roofline(fl_tc, fl_alu, bytes_, seconds, peaks, scope):
    """Roofline of work split between the tensor cores (fl_tc at the bf16
    burst peak) and the CUDA cores (fl_alu at the FP32 FMA rate): the ideal
    time is the sum of the two, and the peak reported is the effective rate
    (all flops over that time), so frac = ideal time / measured time."""
    t_tc = fl_tc / (peaks["bf16_tflops"] * 1e12)
    t_alu = fl_alu / (peaks["fp32_tflops"] * 1e12)
    fl = fl_tc + fl_alu
    ach = fl / seconds / 1e12
    peak = fl / (t_tc + t_alu) / 1e12
    return {"bound": "alu" if t_alu >= t_tc else "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
            "frac": ach / peak, "traffic": None, "algorithmic_bytes": bytes_, "algorithmic_flops": fl,
            "scope": scope, "peak_kind": "mixed: bf16_tflops for the window products, fp32_tflops for the L2 part",
            "ideal_us": {"tensor": t_tc * 1e6, "alu": t_alu * 1e6}}


def delta_backward_work(B, H, T, d_k, d_v, elem):
    """Per token-head: the forward replay (S k and the rank-1 write, 4 d_k d_v)
    and the reverse step (S^T do, dS update, dS k, the state reversal, dk and
    the dS write-back: 12 d_k d_v).  Bytes: q, k, v, dy read, dq, dk, dv
    written, beta and dbeta (fp32)."""
    BH = B * H
    flops = BH * T * 16 * d_k * d_v
    bytes_ = BH * T * ((3 * d_k + 3 * d_v) * elem + 8)
    return flops, bytes_


def sparse_keygen_work(B, H, T, R, N, d_v, density):
    """The sparse attention's fp32 work (4 nnz d_v flops per token-head, as in
    sparse_work) and the bytes: x (bf16) for q and k, U once per head (bf16),
    v read and y written (fp32).  The key generation's own 2 R N flops per
    token-head for q and for k run on the tensor cores in bf16; they are
    returned third so that they are rated against the tensor peak, not the
    FP32 rate."""
    BH = B * H
    flops = BH * T * 4 * density * N * d_v
    bytes_ = BH * T * (2 * R * 2 + 2 * d_v * 4) + H * R * N * 2
    gemm_flops = BH * T * 4 * R * N
    return flops, bytes_, gemm_flops


def sparse_work(B, H, T, N, d_v, density):
    """Sparse write + read: 4 nnz d_v flops per token; dense q, k, v read, y written."""
    BH = B * H
    nnz = density * N
    flops = BH * T * 4 * nnz * d_v
    bytes_ = BH * T * (2 * N + 2 * d_v) * 4
    return flops, bytes_


def roofline(flops, bytes_, seconds, peaks, peak_kind, traffic=None, scope="kernel"):
    """peak_kind: "burst" / "sustained" bf16 tensor peak for the bf16 paths,
    "fp32" for the float32 paths (the measured FP32 FMA rate, bound "alu")."""
    tf_key = {"burst": "bf16_tflops", "sustained": "bf16_tflops_sustained", "fp32": "fp32_tflops"}[peak_kind]
    t_mem = bytes_ / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks[tf_key] * 1e12)
    if t_mem >= t_tc:
        ach = bytes_ / seconds / 1e9
        out = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        ach = flops / seconds / 1e12
        out = {"bound": "alu" if peak_kind == "fp32" else "tensor", "achieved": ach, "peak": peaks[tf_key],
               "unit": "TFLOP/s"}
    out["frac"] = out["achieved"] / out["peak"]
    out["traffic"] = traffic
    out["algorithmic_bytes"] = bytes_
    out["algorithmic_flops"] = flops
    out["scope"] = scope
    out["peak_kind"] = tf_key
    return out


def fp32_peak(torch, binding):
    """FP32 FMA rate of this GPU, from the library's probe kernel: 8 waves of
    CTAs (256 threads, 8 FMA chains each), timed with CUDA events, best of 5."""
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    blocks, iters = sms * 8 * 8, 4096
    out = torch.empty(blocks * 256, dtype=torch.float32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    binding.fp32_fma_probe(out, blocks, iters)
    best = None
    for _ in range(5):
        e0.record()
        fl = binding.fp32_fma_probe(out, blocks, iters)
        e1.record()
        torch.cuda.synchronize()
        rate = fl / (e0.elapsed_time(e1) / 1e3) / 1e12
        best = rate if best is None else max(best, rate)
    return best


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = [r for t, r in self.rows if t0 - 0.25 <= t <= t1 + 0.25] or [r for _, r in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Max of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank, seconds_per_rank, world):
    """Whole-job throughput: units all ranks processed / slowest rank's time."""
    return units_per_rank * world / max_over_ranks(seconds_per_rank, world)


# ----------------------------------------------------------------- timing helpers
def timed_steps(step, K, flush, torch, prof=True, binding=None):
    """K steps, each bracketed by events; L2 flushed before each (untimed).
    Returns (per-step ms list, dominant-kernel ms list or None)."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    kd = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in ev + kd:   # torch creates the CUDA event on first record
        a.record()
        b.record()
    torch.cuda.synchronize()
    for i in range(K):
        if flush is not None:
            flush.zero_()
        if prof and binding is not None:
            binding.profile_events(kd[i][0], kd[i][1])
        ev[i][0].record()
        step()
        ev[i][1].record()
    if binding is not None:
        binding.profile_events(None, None)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    dom_ms = [a.elapsed_time(b) for a, b in kd] if prof and binding is not None else None
    return step_ms, dom_ms


def load_traffic(kernel):
    """ncu DRAM bytes per launch recorded for `kernel`, if the kernel source is
    unchanged since the capture (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    import hashlib
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d:
        return None
    src = os.path.join(ROOT, "outer_product_associative_chunked_b300", "csrc", d["source"])
    if not os.path.exists(src):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return d["dram_bytes_per_launch"] if h == d["source_sha256_16"] else None


def timed_graph_steps(step, K, flush, torch, binding):
    """The step captured once into a CUDA graph (without profiling events, so
    kernels launched as programmatic dependents keep their overlap), then K
    replays, each after an L2 flush (untimed) and each timed with CUDA events
    on the replay stream.  Returns (per-step ms, kernels per step)."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for ev in (e0, e1):   # torch creates the CUDA event on first record
        ev.record()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    binding.profile_events(None, None)
    l0 = binding.kernel_launches()
    with torch.cuda.graph(graph):
        step()
    per_step = binding.kernel_launches() - l0
    graph.replay()
    torch.cuda.synchronize()
    step_ms = []
    for _ in range(K):
        flush.zero_()
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        step_ms.append(e0.elapsed_time(e1))
    return step_ms, per_step


# ----------------------------------------------------------------- our arm
def tc_prefill_setup(name, rank, torch, binding, synth):
    w = synth.WORKLOADS[name]
    d = w.dims
    inp = synth.tc_inputs(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], d["W"], dtype=d["dtype"],
                          seed=w.seed + 1000 * rank, lam=d.get("lam"), eta=d.get("eta"), gate=d.get("gate"))
    return w, d, inp


def bench_headline(args, rank, world, torch, binding, synth, peaks, peak_src, flush):
    w, d, inp = tc_prefill_setup(args.workload, rank, torch, binding, synth)
    q, k, v, lam, eta, gate = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)]
    y = torch.empty(d["B"], d["H"], d["T"], d["d_v"], dtype=q.dtype, device="cuda")
    ws = torch.empty(binding.tc_layer_forward_workspace_size(d["B"], d["H"], d["T"], d["d_k"], d["d_v"],
                                                             d["W"], q.dtype), dtype=torch.uint8, device="cuda")

    def step():
        binding.tc_layer_forward(q, k, v, lam, eta, gate, d["W"], out=y, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    # Eager calls first (host enqueue included; the dominant kernel is timed
    # here, on its own, between the library's events), then the same step
    # replayed from a CUDA graph; the graph replay is the reported step.
    eager_ms, dom_ms = timed_steps(step, args.steps, flush, torch, prof=True, binding=binding)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    step_ms, per_step = timed_graph_steps(step, args.steps, flush, torch, binding)
    t1 = time.time()
    launches = per_step * args.steps
    barrier(world)
    if sampler:
        time.sleep(0.3)
        sampler.stop()
    tokens = d["B"] * d["T"]
    total_s = sum(step_ms) / 1e3
    value = aggregate_throughput(tokens * args.steps, total_s, world)
    ms_per_step = max_over_ranks(total_s, world) * 1e3 / args.steps
    elem = 2 if d["dtype"] == "bf16" else 4
    fl, by = tc_prefill_work(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], d["W"], elem)
    dom_s = statistics.mean(dom_ms) / 1e3
    roof = roofline(fl, by, dom_s, peaks, "burst", traffic=load_traffic("tc_fwd"), scope="kernel")
    roof["kernel"] = "tc_fwd (fused window softmax + L2 read + gate)"
    roof["kernel_ms"] = dom_s * 1e3
    # The same kernel against the tensor-core peaks as well (its arithmetic
    # intensity sits near the ridge): achieved TFLOP/s over burst and sustained.
    roof["tensor_tflops"] = fl / dom_s / 1e12
    roof["tensor_frac_burst"] = roof["tensor_tflops"] / peaks["bf16_tflops"]
    roof["tensor_frac_sustained"] = roof["tensor_tflops"] / peaks["bf16_tflops_sustained"]
    roof["peak_source"] = f"of {peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "of fallback"
    eager = {"ms_per_step": statistics.mean(eager_ms),
             "value": tokens / (statistics.mean(eager_ms) / 1e3),
             "note": "same step as eager calls from Python; host enqueue time is included"}
    clocks = sampler.summary(t0, t1) if sampler else None

    # e2e through the public binding from pinned host memory
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (x.pin_memory() for x in (inp.q, inp.k, inp.v))
        hl, he, hg = (x.pin_memory() for x in (inp.lam, inp.eta, inp.gate))
        hy = torch.empty(tuple(y.shape), dtype=y.dtype).pin_memory()
        dq, dk_, dv_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        dl, de, dg = torch.empty_like(lam), torch.empty_like(eta), torch.empty_like(gate)

        # The batch goes through in per-sequence chunks on two streams, so each
        # chunk's upload overlaps the previous chunk's compute and download
        # (the copy engines run both directions at once).  Each stream has its
        # own workspace, since calls that share one must not overlap.
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        ws1 = binding.tc_layer_forward_workspace_size(1, d["H"], d["T"], d["d_k"], d["d_v"], d["W"], q.dtype)
        wss = [torch.empty(ws1, dtype=torch.uint8, device="cuda") for _ in streams]

        def e2e_step():
            main = torch.cuda.current_stream()
            for dst, src in ((dl, hl), (de, he), (dg, hg)):
                dst.copy_(src, non_blocking=True)
            ready = main.record_event()
            for b in range(d["B"]):
                s = streams[b % 2]
                s.wait_event(ready)
                with torch.cuda.stream(s):
                    for dst, src in ((dq, hq), (dk_, hk), (dv_, hv)):
                        dst[b].copy_(src[b], non_blocking=True)
                    binding.tc_layer_forward(dq[b:b + 1], dk_[b:b + 1], dv_[b:b + 1], dl, de, dg, d["W"],
                                             out=y[b:b + 1], workspace=wss[b % 2], stream=s)
                    hy[b].copy_(y[b], non_blocking=True)
            for s in streams:
                main.wait_stream(s)

        # The same step as one call: the whole batch up, one tc_layer_forward
        # (the launch the device-timed value measures), the whole y down.
        ws_all = torch.empty(binding.tc_layer_forward_workspace_size(d["B"], d["H"], d["T"], d["d_k"], d["d_v"],
                                                                     d["W"], q.dtype), dtype=torch.uint8,
                             device="cuda")

        def e2e_single():
            for dst, src in ((dq, hq), (dk_, hk), (dv_, hv), (dl, hl), (de, he), (dg, hg)):
                dst.copy_(src, non_blocking=True)
            binding.tc_layer_forward(dq, dk_, dv_, dl, de, dg, d["W"], out=y, workspace=ws_all)
            hy.copy_(y, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
            e2e_single()
        barrier(world)
        e_ms, _ = timed_steps(e2e_step, args.steps, None, torch, prof=False)
        s_ms, _ = timed_steps(e2e_single, args.steps, None, torch, prof=False)
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hl, he, hg))
        d2h = hy.numel() * hy.element_size()
        e2e = {"value": aggregate_throughput(tokens * args.steps, sum(e_ms) / 1e3, world), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": statistics.mean(e_ms),
               "how": "per-sequence chunks on two streams, uploads and downloads overlapping compute",
               "single_call": {"value": aggregate_throughput(tokens * args.steps, sum(s_ms) / 1e3, world),
                               "ms_per_step": statistics.mean(s_ms),
                               "how": "whole batch up, one tc_layer_forward, whole y down, in order"}}
        del ws_all
    del ws
    return {"value": value, "ms_per_step": ms_per_step, "roofline": roof, "clocks": clocks,
            "e2e": e2e, "gpu_launches": launches, "tokens_per_step": tokens, "dims": d, "inp": inp,
            "eager": eager}


def bench_extras(args, torch, binding, synth, peaks, flush):
    """The other workloads, each timed with CUDA events (L2 flushed between
    steps); roofline on the whole step's algorithmic work."""
    out = {}
    K, Wm = args.extra_steps, 2

    def summarize(name, tokens, ms, fl, by, peak_kind, kernel, dom):
        r = roofline(fl, by, statistics.mean(ms) / 1e3, peaks, peak_kind, scope="step")
        entry = {"value": tokens / (statistics.mean(ms) / 1e3), "unit": "tokens/s",
                 "ms_per_step": statistics.mean(ms), "roofline": r, "dominant_kernel": kernel}
        if dom:
            entry["dominant_kernel_ms"] = statistics.mean(dom)
            entry["dominant_roofline"] = roofline(fl, by, statistics.mean(dom) / 1e3, peaks, peak_kind,
                                                  scope="kernel")
        out[name] = entry

    # The float32 Tensor Cache workload (B=H=1, T=256, d=32, W=32), replayed
    # from a CUDA graph like the headline: it is launch-latency bound.
    name = "tc_fp32_T256_d32_W32"
    w, d, inp = tc_prefill_setup(name, 0, torch, binding, synth)
    q, k, v, lam, eta, gate = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)]
    y = torch.empty(d["B"], d["H"], d["T"], d["d_v"], dtype=q.dtype, device="cuda")
    ws = torch.empty(binding.tc_layer_forward_workspace_size(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], d["W"],
                                                             q.dtype), dtype=torch.uint8, device="cuda")
    step = lambda: binding.tc_layer_forward(q, k, v, lam, eta, gate, d["W"], out=y, workspace=ws)  # noqa: E731
    for _ in range(Wm):
        step()
    ms, per_step = timed_graph_steps(step, 4 * K, flush, torch, binding)
    fl, by = tc_prefill_work(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], d["W"], 4)
    summarize(name, d["B"] * d["T"], ms, fl, by, "fp32", "tc_fwd_simt (CUDA cores)", None)
    out[name].update({"launch": "step captured once into a CUDA graph and replayed",
                      "kernels_per_step": per_step,
                      "note": "2 MFLOP and 131 KB per step: bound by launch latency, not by either roof"})
    del q, k, v, y, ws

    # Window-only variant against the full layer on the headline inputs, both
    # replayed from CUDA graphs back to back: the ratio is the cost of the L2
    # memory (the pages compare the layer with pure sliding-window attention).
    name = "tc_window_bf16_B4_H8_T4096_d64_W512"
    w, d, inp = tc_prefill_setup("tc_bf16_B4_H8_T4096_d64_W512", 0, torch, binding, synth)
    q, k, v, lam, eta, gate = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)]
    y = torch.empty(d["B"], d["H"], d["T"], d["d_v"], dtype=q.dtype, device="cuda")
    ws = torch.empty(binding.tc_layer_forward_workspace_size(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], d["W"],
                                                             q.dtype), dtype=torch.uint8, device="cuda")
    wsw = torch.empty(binding.STATUS_BYTES, dtype=torch.uint8, device="cuda")
    win = lambda: binding.tc_window_forward(q, k, v, d["W"], out=y, workspace=wsw)  # noqa: E731
    layer = lambda: binding.tc_layer_forward(q, k, v, lam, eta, gate, d["W"], out=y, workspace=ws)  # noqa: E731
    for _ in range(Wm):
        win()
        layer()
    win_ms, _ = timed_graph_steps(win, 4 * K, flush, torch, binding)
    layer_ms, _ = timed_graph_steps(layer, 4 * K, flush, torch, binding)
    fl, by = tc_prefill_work(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], d["W"], 2, l2=False)
    summarize(name, d["B"] * d["T"], win_ms, fl, by, "burst", "tc_fwd (window only)", None)
    ring = d["W"] * (d["d_k"] + d["d_v"]) * 2
    out[name].update({
        "launch": "step captured once into a CUDA graph and replayed",
        "layer_ms_per_step": statistics.mean(layer_ms),
        "l2_overhead": statistics.mean(layer_ms) / statistics.mean(win_ms) - 1.0,
        "state_bytes_per_head": {"window_only": ring, "tensor_cache": ring + d["d_k"] * d["d_v"] * 4},
    })
    del q, k, v, y, ws

    # Long-context prefill, then the 64-sequence decode continuing from it.
    # The prefill kernel runs about a millisecond on its own, so it is rated
    # against the burst tensor peak.
    name = "tc_bf16_B1_H16_T32768_d128_W2048"
    w, d, inp = tc_prefill_setup(name, 0, torch, binding, synth)
    q, k, v, lam, eta, gate = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)]
    y = torch.empty(d["B"], d["H"], d["T"], d["d_v"], dtype=q.dtype, device="cuda")
    ws = torch.empty(binding.tc_layer_forward_workspace_size(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], d["W"],
                                                             q.dtype), dtype=torch.uint8, device="cuda")
    st1 = binding.TCState(d["B"], d["H"], d["W"], d["d_k"], d["d_v"], dtype=q.dtype)
    step = lambda: binding.tc_layer_forward(q, k, v, lam, eta, gate, d["W"], out=y, workspace=ws)  # noqa: E731
    for _ in range(Wm):
        step()
    ms, dom = timed_steps(step, K, flush, torch, prof=True, binding=binding)
    fl, by = tc_prefill_work(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], d["W"], 2)
    summarize(name, d["B"] * d["T"], ms, fl, by, "burst", "tc_fwd", dom)
    binding.tc_layer_forward(q, k, v, lam, eta, gate, d["W"], out=y, workspace=ws, state=st1)
    del ws, y, q, k, v

    dname = "tc_decode_bf16_S64_H16_d128_W2048_steps256"
    dd = synth.WORKLOADS[dname].dims
    S, steps = dd["S"], dd["steps"]
    dec = synth.tc_decode_inputs(steps, S, dd["H"], dd["d_k"], dd["d_v"], dtype="bf16",
                                 seed=synth.WORKLOADS[dname].seed)
    dq, dk_, dv_ = dec.q.cuda(), dec.k.cuda(), dec.v.cuda()
    st = binding.TCState(S, dd["H"], dd["W"], dd["d_k"], dd["d_v"], dtype=torch.bfloat16)
    st.ring_k.copy_(st1.ring_k.expand(S, -1, -1, -1))
    st.ring_v.copy_(st1.ring_v.expand(S, -1, -1, -1))
    st.A.copy_(st1.A.expand(S, -1, -1, -1))
    st.pos.fill_(d["T"])
    yd = torch.empty(S, dd["H"], dd["d_v"], dtype=torch.bfloat16, device="cuda")
    wsd = torch.empty(binding.tc_decode_step_workspace_size(st), dtype=torch.uint8, device="cuda")
    counter = [0]

    def dstep():
        i = counter[0] % steps
        binding.tc_decode_step(st, dq[i], dk_[i], dv_[i], lam, eta, gate, out=yd, workspace=wsd)
        counter[0] += 1

    for _ in range(Wm):
        dstep()
    # One timed "step" of this workload = 256 decode steps; the working set
    # (ring 1 GiB + A 64 MiB) is far above L2, so no flush is needed.
    ms, dom = timed_steps(dstep, steps, None, torch, prof=True, binding=binding)
    fl, by = tc_decode_work(S, dd["H"], dd["d_k"], dd["d_v"], dd["W"], 2)
    summarize(dname, S, ms, fl, by, "sustained", "tc_decode_partial", dom)
    out[dname]["note"] = "value = decoded tokens/s (64 sequences x 1 token per step, averaged over 256 steps)"
    del st, st1, dq, dk_, dv_, wsd

    name = "delta_bf16_B8_H16_T8192_d128_C64"
    d = synth.WORKLOADS[name].dims
    inp = synth.delta_inputs(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], dtype="bf16",
                             seed=synth.WORKLOADS[name].seed)
    q, k, v, beta = inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.beta.cuda()
    y = torch.empty_like(v)
    ws = torch.empty(binding.delta_rule_forward_workspace_size(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], 64,
                                                               torch.bfloat16), dtype=torch.uint8, device="cuda")
    step = lambda: binding.delta_rule_forward(q, k, v, beta, chunk=64, out=y, workspace=ws)  # noqa: E731
    for _ in range(Wm):
        step()
    ms, dom = timed_steps(step, K, flush, torch, prof=True, binding=binding)
    fl, by = delta_work(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], 2)
    summarize(name, d["B"] * d["T"], ms, fl, by, "burst", "delta_fused", dom)
    del q, k, v, beta, y, ws

    dname = "delta_decode_bf16_S256_H16_d128_steps64"
    dd = synth.WORKLOADS[dname].dims
    S, steps = dd["S"], dd["steps"]
    dec = synth.delta_decode_inputs(steps, S, dd["H"], dd["d_k"], dd["d_v"], dtype="bf16",
                                    seed=synth.WORKLOADS[dname].seed)
    dq, dk_, dv_, db = dec.q.cuda(), dec.k.cuda(), dec.v.cuda(), dec.beta.cuda()
    Sd = dec.S0.cuda()
    yd = torch.empty(S, dd["H"], dd["d_v"], dtype=torch.bfloat16, device="cuda")
    counter = [0]

    def ddstep():
        i = counter[0] % steps
        binding.delta_decode_step(Sd, dq[i], dk_[i], dv_[i], db[i], out=yd)
        counter[0] += 1

    for _ in range(Wm):
        ddstep()
    # One timed "step" of this workload = 64 decode steps; the state (256 MiB)
    # is above L2, so no flush is needed.
    ms, dom = timed_steps(ddstep, steps, None, torch, prof=True, binding=binding)
    fl, by = delta_decode_work(S, dd["H"], dd["d_k"], dd["d_v"], 2)
    summarize(dname, S, ms, fl, by, "sustained", "delta_decode", dom)
    out[dname]["note"] = "value = decoded tokens/s (256 sequences x 1 token per step, averaged over 64 steps)"
    del dq, dk_, dv_, db, Sd, yd, dec

    # Backward of the headline prefill (fp32 arithmetic on the CUDA cores).
    name = "tc_backward_bf16_B4_H8_T4096_d64_W512"
    w, d, inp = tc_prefill_setup("tc_bf16_B4_H8_T4096_d64_W512", 0, torch, binding, synth)
    q, k, v, lam, eta, gate = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)]
    dy = torch.randn(q.shape[:-1] + (d["d_v"],), generator=torch.Generator().manual_seed(9)).to(q.dtype).cuda()
    outs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(lam),
            torch.empty_like(eta), torch.empty_like(gate))
    ws = torch.empty(binding.tc_layer_backward_workspace_size(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], d["W"],
                                                              q.dtype), dtype=torch.uint8, device="cuda")
    step = lambda: binding.tc_layer_backward(q, k, v, lam, eta, gate, d["W"], dy, out=outs, workspace=ws)  # noqa: E731
    for _ in range(Wm):
        step()
    ms, dom = timed_steps(step, K, flush, torch, prof=True, binding=binding)
    fl_w, fl_l2, by = tc_backward_work(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], d["W"], 2, split=True)
    summarize(name, d["B"] * d["T"], ms, fl_w + fl_l2, by, "fp32", "tcb_window_dq_tc .. tcb_finalize (all five)",
              dom)
    out[name]["roofline"] = mixed_roofline(fl_w, fl_l2, by, statistics.mean(ms) / 1e3, peaks, "step")
    if dom:
        out[name]["dominant_roofline"] = mixed_roofline(fl_w, fl_l2, by, statistics.mean(dom) / 1e3, peaks,
                                                        "kernel")
    out[name]["note"] = ("value = tokens/s of the backward pass; the window products on the tensor cores (bf16 "
                         "operands, fp32 accumulation), the L2 part in fp32 on the CUDA cores")
    del q, k, v, dy, outs, ws

    # Backward of the delta rule at the DeltaNet workload's shape.
    name = "delta_backward_bf16_B8_H16_T8192_d128"
    d = synth.WORKLOADS["delta_bf16_B8_H16_T8192_d128_C64"].dims
    inp = synth.delta_inputs(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], dtype="bf16", seed=2)
    q, k, v, beta = inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.beta.cuda()
    dy = torch.randn(v.shape, generator=torch.Generator().manual_seed(10)).to(v.dtype).cuda()
    outs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(beta), None)
    ws = torch.empty(binding.delta_rule_backward_workspace_size(d["B"], d["H"], d["T"], d["d_k"], d["d_v"],
                                                                torch.bfloat16), dtype=torch.uint8, device="cuda")
    step = lambda: binding.delta_rule_backward(q, k, v, beta, dy, out=outs, workspace=ws)  # noqa: E731
    step()
    ms, dom = timed_steps(step, max(1, K // 2), flush, torch, prof=True, binding=binding)
    fl, by = delta_backward_work(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], 2)
    summarize(name, d["B"] * d["T"], ms, fl, by, "fp32", "delta_backward", dom)
    out[name]["note"] = ("value = tokens/s of the backward pass; per-token reverse recurrence on the CUDA cores, "
                         "one CTA per (batch, head)")
    del q, k, v, beta, dy, outs, ws

    # BDH attention with keys and queries generated on the GPU.
    name = "bdh_keygen_B2_H4_T2048_R256_N16384_dv256"
    d = synth.WORKLOADS[name].dims
    kg = synth.sparse_keygen_inputs(d["B"], d["H"], d["T"], d["N"], d["d_v"], seed=synth.WORKLOADS[name].seed,
                                    rank=d["R"])
    xq, xk, U, v = kg.xq.cuda(), kg.xk.cuda(), kg.U.cuda(), kg.v.cuda()
    y = torch.empty_like(v)
    ws = torch.empty(binding.sparse_linattn_keygen_forward_workspace_size(d["B"], d["H"], d["T"], d["R"], d["N"],
                                                                          d["d_v"]), dtype=torch.uint8, device="cuda")
    step = lambda: binding.sparse_linattn_keygen_forward(xq, xk, U, kg.theta, v, out=y, workspace=ws)  # noqa: E731
    for _ in range(Wm):
        step()
    ms, dom = timed_steps(step, K, flush, torch, prof=True, binding=binding)
    fl, by, gemm = sparse_keygen_work(d["B"], d["H"], d["T"], d["R"], d["N"], d["d_v"], 0.05)
    summarize(name, d["B"] * d["T"], ms, fl, by, "fp32", "pair_tile", dom)
    out[name]["keygen_gemm"] = {"flops": gemm, "floor_ms": gemm / (peaks["bf16_tflops"] * 1e12) * 1e3,
                                "note": "x U_h for q and k on the tensor cores (bf16); its time at the burst peak"}
    out[name]["note"] = "keys and queries generated on chip (bf16 x U, fp32 accumulation); attention in fp32"
    del xq, xk, U, v, y, ws

    name = "bdh_fp32_B2_H4_T2048_N16384_dv256"
    d = synth.WORKLOADS[name].dims
    inp = synth.sparse_inputs(d["B"], d["H"], d["T"], d["N"], d["d_v"], seed=synth.WORKLOADS[name].seed)
    dens = float((inp.k > 0).float().mean())
    q, k, v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
    y = torch.empty_like(v)
    ws = torch.empty(binding.sparse_linattn_forward_workspace_size(d["B"], d["H"], d["T"], d["N"], d["d_v"]),
                     dtype=torch.uint8, device="cuda")
    step = lambda: binding.sparse_linattn_forward(q, k, v, out=y, workspace=ws)  # noqa: E731
    for _ in range(Wm):
        step()
    ms, dom = timed_steps(step, K, flush, torch, prof=True, binding=binding)
    fl, by = sparse_work(d["B"], d["H"], d["T"], d["N"], d["d_v"], dens)
    summarize(name, d["B"] * d["T"], ms, fl, by, "fp32", "pair_tile", dom)
    out[name]["density"] = dens
    del q, k, v, y, ws
    return out


# ----------------------------------------------------------------- oracle on the host cores
def _oracle_rate(oracle, fn, tokens, threads):
    """Run fn() with `threads` OpenMP threads, once untimed (first-touch page
    faults of the oracle's fresh buffers) and once timed; returns (tokens/s,
    seconds)."""
    oracle.set_threads(threads)
    fn()
    t0 = time.perf_counter()
    fn()
    dt = time.perf_counter() - t0
    return tokens / dt, dt


def cpu_baseline_headline(inp, d):
    """The float64 oracle on the host cores on the headline batch: every
    (batch, head) unit, all threads (the same sample the reference arm
    times per step), plus one unit on one thread."""
    from oracle import oracle
    oracle.build()
    threads = oracle.get_threads()
    B, H, T, W = d["B"], d["H"], d["T"], d["W"]
    allv, dt = _oracle_rate(oracle, lambda: oracle.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, W),
                            B * T, threads)
    one, dt1 = _oracle_rate(oracle, lambda: oracle.tc_prefill(inp.q[:1, :1], inp.k[:1, :1], inp.v[:1, :1],
                                                              inp.lam[:1], inp.eta[:1], inp.gate[:1], W),
                            T / H, 1)
    oracle.set_threads(threads)
    return {"value": allv, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"the whole batch: {B} sequences x {H} heads x {T} tokens (float64, OpenMP over the "
                      f"{B * H} units), {dt:.2f} s",
            "single_thread": {"value": one, "cores": 1,
                              "sample": f"1 unit (1 head x {T} tokens) on one thread, {dt1:.2f} s; value in "
                                        f"tokens of all {H} heads per second"}}


def _f64(inputs):
    """The same inputs as float64 numpy arrays (exact), so that the timed
    oracle calls do not include the conversion."""
    import dataclasses
    from oracle import oracle
    return dataclasses.replace(inputs, **{f.name: oracle.f64(getattr(inputs, f.name))
                                          for f in dataclasses.fields(inputs)
                                          if hasattr(getattr(inputs, f.name), "shape")})


def cpu_baselines(synth):
    """The float64 oracle as it stands, timed on the host cores on a bounded
    sample of each extra workload: all threads over the sample's units, and
    one unit on one thread.  Values are in the workload's own unit (tokens of
    all heads per second; decoded tokens per second for decode)."""
    import numpy as np
    from oracle import oracle
    oracle.build()
    threads = oracle.get_threads()
    res = {}

    def record(name, allv, dt, sample, one, dt1, sample1):
        res[name] = {"value": allv, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                     "sample": f"{sample}, {dt:.2f} s",
                     "single_thread": {"value": one, "cores": 1, "sample": f"{sample1}, {dt1:.2f} s"}}

    # fp32 T=256: the whole workload (one unit), repeated for a measurable time
    d = synth.WORKLOADS["tc_fp32_T256_d32_W32"].dims
    inp = _f64(synth.tc_inputs(1, 1, 256, 32, 32, 32, dtype="f32", seed=0, lam=d["lam"], eta=d["eta"],
                               gate=d["gate"]))
    reps = 200
    f = lambda: [oracle.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, 32) for _ in range(reps)]  # noqa: E731
    v1, dt1 = _oracle_rate(oracle, f, reps * 256, 1)
    record("tc_fp32_T256_d32_W32", v1, dt1, f"the whole workload x {reps} (one unit: one thread is all it uses)",
           v1, dt1, f"the whole workload x {reps}")

    # window only: the layer with eta = 0, one sequence (8 heads) / one unit
    w = synth.WORKLOADS["tc_bf16_B4_H8_T4096_d64_W512"]
    d = w.dims
    inp = _f64(synth.tc_inputs(1, d["H"], d["T"], 64, 64, d["W"], dtype="bf16", seed=w.seed))
    z = np.zeros(d["H"])
    allv, dt = _oracle_rate(oracle, lambda: oracle.tc_prefill(inp.q, inp.k, inp.v, inp.lam, z, inp.gate, d["W"]),
                            d["T"], threads)
    one, dt1 = _oracle_rate(oracle, lambda: oracle.tc_prefill(inp.q[:, :1], inp.k[:, :1], inp.v[:, :1],
                                                              inp.lam[:1], z[:1], inp.gate[:1], d["W"]),
                            d["T"] / d["H"], 1)
    record("tc_window_bf16_B4_H8_T4096_d64_W512", allv, dt,
           f"1 of 4 sequences ({d['H']} heads x {d['T']} tokens) with eta = 0", one, dt1, "1 head of it")

    # long prefill: a prefix of 3W tokens of every head (the per-token cost is
    # flat once the window is full)
    w = synth.WORKLOADS["tc_bf16_B1_H16_T32768_d128_W2048"]
    d = w.dims
    Tp = 3 * d["W"]
    inp = _f64(synth.tc_inputs(1, d["H"], Tp, 128, 128, d["W"], dtype="bf16", seed=w.seed))
    allv, dt = _oracle_rate(oracle, lambda: oracle.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate,
                                                              d["W"]), Tp, threads)
    one, dt1 = _oracle_rate(oracle, lambda: oracle.tc_prefill(inp.q[:, :1], inp.k[:, :1], inp.v[:, :1],
                                                              inp.lam[:1], inp.eta[:1], inp.gate[:1], d["W"]),
                            Tp / d["H"], 1)
    record("tc_bf16_B1_H16_T32768_d128_W2048", allv, dt,
           f"the first {Tp} of {d['T']} tokens, all {d['H']} heads", one, dt1, f"1 head, first {Tp} tokens")

    # decode: a full ring and state (seeded), a few steps of all 64 sequences
    w = synth.WORKLOADS["tc_decode_bf16_S64_H16_d128_W2048_steps256"]
    d = w.dims
    Ss = 16
    st = {k_: oracle.f64(v_) if k_ != "pos" else v_.numpy()
          for k_, v_ in synth.tc_decode_state(Ss, d["H"], d["W"], 128, 128, pos=32768, dtype="bf16",
                                              seed=w.seed + 1).items()}
    dec = _f64(synth.tc_decode_inputs(8, Ss, d["H"], 128, 128, dtype="bf16", seed=w.seed))
    lam = np.full(d["H"], 0.95)
    allv, dt = _oracle_rate(oracle, lambda: oracle.tc_decode(st, dec.q, dec.k, dec.v, lam, lam, lam),
                            8 * Ss, threads)
    st1 = {k_: v_[:1] for k_, v_ in st.items()}
    one, dt1 = _oracle_rate(oracle, lambda: oracle.tc_decode(st1, dec.q[:, :1], dec.k[:, :1], dec.v[:, :1], lam,
                                                             lam, lam), 8, 1)
    record("tc_decode_bf16_S64_H16_d128_W2048_steps256", allv, dt,
           f"8 steps of {Ss} of the {d['S']} sequences x {d['H']} heads from a seeded full state (W = "
           f"{d['W']}, d = 128)", one, dt1, "8 steps of 1 sequence")

    # DeltaNet: the first 1024 tokens of every head
    w = synth.WORKLOADS["delta_bf16_B8_H16_T8192_d128_C64"]
    d = w.dims
    Tp = 1024
    inp = _f64(synth.delta_inputs(d["B"], d["H"], Tp, 128, 128, dtype="bf16", seed=w.seed))
    allv, dt = _oracle_rate(oracle, lambda: oracle.delta(inp.q, inp.k, inp.v, inp.beta), d["B"] * Tp, threads)
    one, dt1 = _oracle_rate(oracle, lambda: oracle.delta(inp.q[:1, :1], inp.k[:1, :1], inp.v[:1, :1],
                                                         inp.beta[:1, :1]), Tp / d["H"], 1)
    record("delta_bf16_B8_H16_T8192_d128_C64", allv, dt,
           f"the first {Tp} of {d['T']} tokens of all {d['B']}x{d['H']} units", one, dt1, f"1 unit, {Tp} tokens")

    # DeltaNet decode: 4 steps of all 256 sequences
    w = synth.WORKLOADS["delta_decode_bf16_S256_H16_d128_steps64"]
    d = w.dims
    dd = _f64(synth.delta_decode_inputs(4, d["S"], d["H"], 128, 128, dtype="bf16", seed=w.seed))
    mv = lambda t: np.ascontiguousarray(np.moveaxis(t, 0, 2))  # noqa: E731  [steps,S,H,..] -> [S,H,steps,..]
    allv, dt = _oracle_rate(oracle, lambda: oracle.delta(mv(dd.q), mv(dd.k), mv(dd.v), mv(dd.beta), S0=dd.S0),
                            4 * d["S"], threads)
    one, dt1 = _oracle_rate(oracle, lambda: oracle.delta(mv(dd.q)[:1], mv(dd.k)[:1], mv(dd.v)[:1],
                                                         mv(dd.beta)[:1], S0=dd.S0[:1]), 4, 1)
    record("delta_decode_bf16_S256_H16_d128_steps64", allv, dt,
           f"4 steps of all {d['S']} sequences x {d['H']} heads", one, dt1, "4 steps of 1 sequence")

    # BDH: the first 128 tokens of every unit (the dense oracle streams the
    # whole N x d_v state per token)
    w = synth.WORKLOADS["bdh_fp32_B2_H4_T2048_N16384_dv256"]
    d = w.dims
    Tp = 128
    sp = _f64(synth.sparse_inputs(d["B"], d["H"], Tp, d["N"], d["d_v"], seed=w.seed))
    allv, dt = _oracle_rate(oracle, lambda: oracle.sparse_linattn(sp.q, sp.k, sp.v), d["B"] * Tp, threads)
    one, dt1 = _oracle_rate(oracle, lambda: oracle.sparse_linattn(sp.q[:1, :1, :32], sp.k[:1, :1, :32],
                                                                  sp.v[:1, :1, :32]), 32 / d["H"], 1)
    record("bdh_fp32_B2_H4_T2048_N16384_dv256", allv, dt,
           f"the first {Tp} of {d['T']} tokens of all {d['B']}x{d['H']} units (at most 8 threads busy)",
           one, dt1, "1 unit, 32 tokens")

    # Tensor Cache backward: one whole sequence (8 heads x 4096 tokens), the
    # same inputs and output gradient as the GPU line
    import torch
    w = synth.WORKLOADS["tc_bf16_B4_H8_T4096_d64_W512"]
    d = w.dims
    inp = synth.tc_inputs(d["B"], d["H"], d["T"], 64, 64, d["W"], dtype="bf16", seed=w.seed)
    dy = torch.randn(inp.q.shape[:-1] + (64,), generator=torch.Generator().manual_seed(9)).to(inp.q.dtype)
    a = [oracle.f64(x[:1]) for x in (inp.q, inp.k, inp.v, dy)]
    s = [oracle.f64(x) for x in (inp.lam, inp.eta, inp.gate)]
    allv, dt = _oracle_rate(oracle, lambda: oracle.tc_backward(a[0], a[1], a[2], s[0], s[1], s[2], d["W"], a[3]),
                            d["T"], threads)
    one, dt1 = _oracle_rate(oracle, lambda: oracle.tc_backward(a[0][:, :1], a[1][:, :1], a[2][:, :1], s[0][:1],
                                                               s[1][:1], s[2][:1], d["W"], a[3][:, :1]),
                            d["T"] / d["H"], 1)
    record("tc_backward_bf16_B4_H8_T4096_d64_W512", allv, dt,
           f"1 of {d['B']} sequences ({d['H']} heads x {d['T']} tokens), float64 reverse pass", one, dt1,
           "1 head of it")

    # delta-rule backward: the first 512 tokens of every unit
    d = synth.WORKLOADS["delta_bf16_B8_H16_T8192_d128_C64"].dims
    Tp = 512
    inp = synth.delta_inputs(d["B"], d["H"], Tp, 128, 128, dtype="bf16", seed=2)
    dy = torch.randn(inp.v.shape, generator=torch.Generator().manual_seed(10)).to(inp.v.dtype)
    a = [oracle.f64(x) for x in (inp.q, inp.k, inp.v, inp.beta, dy)]
    allv, dt = _oracle_rate(oracle, lambda: oracle.delta_backward(*a), d["B"] * Tp, threads)
    one, dt1 = _oracle_rate(oracle, lambda: oracle.delta_backward(*[x[:1, :1] for x in a]), Tp / d["H"], 1)
    record("delta_backward_bf16_B8_H16_T8192_d128", allv, dt,
           f"the first {Tp} of {d['T']} tokens of all {d['B']}x{d['H']} units", one, dt1, f"1 unit, {Tp} tokens")

    # BDH with generated keys: keys and queries by the oracle's max(0, x U - theta),
    # then its attention, on the first 64 tokens of every unit
    name = "bdh_keygen_B2_H4_T2048_R256_N16384_dv256"
    d = synth.WORKLOADS[name].dims
    Tp = 64
    kg = synth.sparse_keygen_inputs(d["B"], d["H"], Tp, d["N"], d["d_v"], seed=synth.WORKLOADS[name].seed,
                                    rank=d["R"])
    xq, xk, U, vv = (oracle.f64(x) for x in (kg.xq, kg.xk, kg.U, kg.v))

    def keygen_attn(b, h):
        qk = oracle.bdh_keys(xq[:b, :h], U[:h], kg.theta)
        kk = oracle.bdh_keys(xk[:b, :h], U[:h], kg.theta)
        return oracle.sparse_linattn(qk, kk, vv[:b, :h])

    allv, dt = _oracle_rate(oracle, lambda: keygen_attn(d["B"], d["H"]), d["B"] * Tp, threads)
    one, dt1 = _oracle_rate(oracle, lambda: keygen_attn(1, 1), Tp / d["H"], 1)
    record(name, allv, dt, f"the first {Tp} of {d['T']} tokens of all {d['B']}x{d['H']} units (keys generated "
           f"by the oracle, then its attention)", one, dt1, f"1 unit, {Tp} tokens")
    oracle.set_threads(threads)
    return res


# ----------------------------------------------------------------- reference arm
def bench_reference(args, rank, world):
    """The oracle as the reference arm: each step is the whole headline batch
    (every (batch, head) unit) on all host cores -- the same sample as our
    arm's cpu_baseline."""
    if rank != 0:
        return None
    import torch  # noqa: F401
    from outer_product_associative_chunked_b300 import synth
    from oracle import oracle
    oracle.build()
    w = synth.WORKLOADS[args.workload]
    d = w.dims
    inp = synth.tc_inputs(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], d["W"], dtype=d["dtype"], seed=w.seed,
                          lam=d.get("lam"), eta=d.get("eta"), gate=d.get("gate"))
    threads = oracle.get_threads()
    sample = lambda: oracle.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, d["W"])  # noqa: E731
    for _ in range(args.warmup):
        sample()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sample()
    dt = time.perf_counter() - t0
    value = d["B"] * d["T"] * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generator)",
            "config": {"workload": args.workload, **{k: v for k, v in d.items() if k != "dtype"},
                       "input_dtype": d["dtype"]},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"each step: the whole batch, {d['B']} sequences x {d['H']} heads x "
                                       f"{d['T']} tokens, OpenMP over the {d['B'] * d['H']} units"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return line


# ----------------------------------------------------------------- main
def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--extra-steps", type=int, default=5)
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_setup()

    if args.impl == "reference":
        line = bench_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    from outer_product_associative_chunked_b300 import binding, build, synth
    build.build()
    peaks, peak_src = load_peaks()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    peaks["fp32_tflops"] = fp32_peak(torch, binding)
    res = bench_headline(args, rank, world, torch, binding, synth, peaks, peak_src, flush)
    extras = None
    if rank == 0 and world == 1 and not args.no_extras:
        extras = bench_extras(args, torch, binding, synth, peaks, flush)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_headline(res["inp"], res["dims"])
        if extras is not None:
            for name, cb in cpu_baselines(synth).items():
                if name in extras:
                    extras[name]["cpu_baseline"] = cb
    if rank == 0:
        d = res["dims"]
        line = {"metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if d["dtype"] == "bf16" else "f32",
                "data": "synthetic (seeded generator, page workload shapes)",
                "config": {"workload": args.workload, **{k: v for k, v in d.items() if k != "dtype"},
                           "input_dtype": d["dtype"], "accumulate": "f32",
                           "tokens_per_step": res["tokens_per_step"],
                           "l2": "256 MiB buffer written between timed steps (untimed)",
                           "launch": "step captured once into a CUDA graph and replayed",
                           "parallelism": f"replicas x{world} (independent batch per GPU)"},
                "roofline": res["roofline"], "cpu_baseline": cpu, "e2e": res["e2e"],
                "peaks": {k: peaks[k] for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained", "fp32_tflops")},
                "peak_sources": {"hbm_gbs": peak_src, "bf16_tflops": peak_src, "bf16_tflops_sustained": peak_src,
                                 "fp32_tflops": "measured in this run (library FP32 FMA probe, best of 5)"},
                "gpu_launches": res["gpu_launches"], "clocks": res["clocks"], "eager": res["eager"]}
        if extras is not None:
            line["workloads"] = extras
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
