"""Benchmark of the MFA decode step on GB300 (one JSON line on rank 0).

A step is one pass of the whole hot path -- decode kernel plus log-sum-exp
combine -- over one batch of synthetic decode inputs.  The headline workload is
the largest one that fits a GPU: B=128 sequences of 1,024-8,192 tokens (seeded,
uniform), bf16 KV with 1% of the key elements x20, 64 query heads of width 256
over one shared K/V head in 64-token pages whose physical order is a seeded
permutation.  Every other target workload (4K and 64K+ contexts in bf16 and
e4m3, multi-token decode, the tiny case) is measured on the same run and
reported under "workloads" with its own value, roofline and e2e.

value      : KV-cache bytes read per second over the timed steps (GB/s), inputs
             resident in HBM; several input copies rotate so that each step reads
             KV that is not in L2.
e2e        : the same metric through the C ABI's host-buffer step (mfa_decode_run_host):
             each step's inputs (q, block table, lengths) are copied from pinned host
             memory and its outputs (out, lse) copied back, inside the timed region, with
             three streams in rotation so that copies overlap the other steps' kernels; the
             KV cache stays resident (it is the attention instance's state).
roofline   : the decode kernel alone, algorithmic bytes per launch / its mean
             CUDA-event duration, against the measured HBM copy bandwidth.
cpu_baseline: the fp64 CPU oracle on a bounded sample of the same workload.
kv_append  : the KV-cache append kernel for the same batch (each sequence's new key
             and value row, quantised for an e4m3 or MXFP4 cache), alone; the decode step
             with the append chained in front of it; and the same step through
             mfa_decode_append_run, which appends inside the decode kernel for one new token
             per sequence.

--impl reference times the oracle itself (the reference arm) on the same
workload, each step a bounded sample.
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
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "ragged_b128_l1024_8192_bf16"
# The other target workloads, measured on the same run and reported under "workloads" (the
# comparison attention shapes and the 4-bit cache last).
SIDE_WORKLOADS = ("tiny_b1_l512_bf16", "b32_l4096_bf16", "b128_l4096_fp8", "long_b4_l131072_bf16",
                  "b32_l4096_fp8", "long_b4_l131072_fp8", "mtp2_b32_l4096_bf16", "mtp2_b32_l4096_fp8",
                  "gqa_b32_l4096_bf16", "mla_b32_l4096_bf16", "b128_l4096_mxfp4", "b32_l4096_mxfp4")
# the arithmetic each cache format's path computes in
PATH_DTYPE = {"bf16": "bf16", "fp8_e4m3": "e4m3", "mxfp4": "mxfp4 KV, e4m3 MMA"}


def shape_args(w) -> dict:
    """Accounting arguments of a workload's attention shape."""
    return dict(H=w.num_q_heads, d=w.head_dim, row=w.head_dim * w.num_kv_heads, shared=w.kv_shared)
SIDE_STEPS = 100
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ------------------------------------------------------------------ accounting

def row_bytes(kv_dtype: str, row: int = 256) -> int:
    """Bytes of one stored row of `row` elements: bf16; e4m3 codes + one fp32 scale; or MXFP4
    code pairs + one E8M0 byte per 32 elements."""
    if kv_dtype == "bf16":
        return 2 * row
    if kv_dtype == "mxfp4":
        return row // 2 + row // 32
    return row + 4


def kv_bytes_per_token(kv_dtype: str, row: int = 256, shared: bool = False) -> int:
    """Cached rows of one token: K and V rows of `row` elements (all key/value heads), or one
    row when a latent serves as both."""
    return (1 if shared else 2) * row_bytes(kv_dtype, row)


def algorithmic_bytes(lens, kv_dtype: str, H: int = 64, d: int = 256, page: int = 64, T: int = 1,
                      row: int = 256, shared: bool = False) -> dict:
    """HBM bytes one decode step must move: every cached K/V row once (shared by a sequence's
    T new query tokens), q, out and lse once per query token, the used block-table entries
    and the lengths."""
    tokens = int(sum(lens))
    pages = int(sum((L + page - 1) // page for L in lens))
    B = len(lens)
    kv = tokens * kv_bytes_per_token(kv_dtype, row, shared)
    other = B * T * (H * d * 2) * 2 + pages * 4 + B * 4 + B * T * H * 4
    return {"kv": kv, "total": kv + other}


def append_bytes(batch: int, kv_dtype: str, d: int = 256, T: int = 1) -> int:
    """Algorithmic bytes of one KV append: per sequence its position in, and per new token
    (T of them) the bf16 K and V rows and the page id in, and the stored rows out."""
    out_row = row_bytes(kv_dtype, d)
    return batch * (4 + T * (2 * 2 * d + 4 + 2 * out_row))


def algorithmic_flops(lens, H: int = 64, d: int = 256, T: int = 1) -> int:
    """2*H*d for q.K^T plus 2*H*d for P.V per (query token, visible cached token) pair
    (softmax not counted); query token i of T sees L - T + 1 + i tokens."""
    pairs = sum(max(0, int(L) - (T - 1 - i)) for L in lens for i in range(T))
    return int(pairs) * 4 * H * d


def intensity_per_token(kv_dtype: str, H: int = 64, d: int = 256, kv_heads_bytes: float = None) -> float:
    """FLOPs per KV byte of the decode step, per token (8-bit KV without scales: 4Hd/2d = 2H)."""
    b = kv_bytes_per_token(kv_dtype) if kv_heads_bytes is None else kv_heads_bytes
    return 4 * H * d / b


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# GB300's nominal HBM3e bandwidth (the measured copy bandwidth is the roofline's peak; the
# fraction of this nominal figure is reported beside it)
NOMINAL_HBM_GBS = 7900.0

# Streams of the end-to-end leg: with two, a step's copies are not fully hidden (35.4 against
# 32.1 us per step at bf16 4K); with three they are; with four, concurrent steps also fill the
# SMs that one step's tail leaves idle, and e2e exceeds the single-stream device number.
E2E_LANES = 3


def source_digest() -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "decode_attention_02_gb300", "csrc")
    for name in sorted(os.listdir(d)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(d, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"mfa_decode_kernel_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_digest") != source_digest():
        return None
    try:
        return int(float(vals["dram_bytes_per_launch_full_workload"]))
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, windows):
        samples = []
        for t, line in self.lines:
            if not any(a <= t <= b for a, b in windows):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                samples.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                    reasons={"hw_slowdown": parts[5], "hw_thermal_slowdown": parts[6],
                                             "sw_thermal_slowdown": parts[7], "sw_power_cap": parts[8]}))
            except ValueError:
                continue
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({k for s in samples for k, v in s["reasons"].items() if v.lower() == "active"})
        return {"sm_mhz": statistics.median(s["sm"] for s in samples),
                "sm_max_mhz": max(s["smax"] for s in samples), "reasons": reasons, "samples": len(samples)}


# ------------------------------------------------------------------ arms

def cpu_oracle_sample(case, target_s: float = 10.0, nthreads: int = 0):
    """Time the oracle on a bounded sample of the workload (about target_s seconds of work).

    The sample is the first k sequences of the batch, repeated r times when the
    whole batch takes less than target_s; returns (GB/s, seconds, k, r).
    """
    import oracle
    lens = case.seq_lens.tolist()
    T = case.workload.tokens_per_seq   # the oracle's rows are (sequence, query token) pairs
    order = [b for b in range(len(lens)) if lens[b] > 0]
    t0 = time.perf_counter()
    oracle.decode(case, batch_slice=slice(order[0] * T, (order[0] + 1) * T), nthreads=nthreads)
    t1 = time.perf_counter() - t0
    k = max(1, min(len(lens), int(target_s / max(t1, 1e-3))))
    t0 = time.perf_counter()
    oracle.decode(case, batch_slice=slice(0, k * T), nthreads=nthreads)
    once = time.perf_counter() - t0
    reps = max(1, int(target_s / max(once, 1e-3)))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.decode(case, batch_slice=slice(0, k * T), nthreads=nthreads)
    dt = time.perf_counter() - t0
    kv = algorithmic_bytes(lens[:k], case.workload.kv_dtype, **shape_args(case.workload))["kv"] * reps
    return kv / dt / 1e9, dt, k, reps


def run_reference(args, case, rank: int, world: int):
    import oracle
    if rank != 0:
        return None
    oracle.build()
    cores = oracle.num_cpus()
    lens = case.seq_lens.tolist()
    T = case.workload.tokens_per_seq   # the oracle's rows are (sequence, query token) pairs
    # bounded sample per step: enough sequences for ~1-3 s of oracle work on all cores
    t0 = time.perf_counter()
    oracle.decode(case, batch_slice=slice(0, T))
    t1 = time.perf_counter() - t0
    k = max(1, min(len(lens), int(2.0 / max(t1, 1e-3))))
    for _ in range(args.warmup):
        oracle.decode(case, batch_slice=slice(0, T))
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.decode(case, batch_slice=slice(0, k * T))
        times.append(time.perf_counter() - t0)
    kv = algorithmic_bytes(lens[:k], case.workload.kv_dtype, **shape_args(case.workload))["kv"]
    total = sum(times)
    value = kv * args.steps / total / 1e9
    sample = f"{k} of {len(lens)} sequences per step ({sum(lens[:k])} tokens), fp64, all {cores} cores"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(case),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


METRIC = "MFA decode-attention KV GB/s and TFLOP/s at 1 GB300; % of HBM/tensor roofline"


def workload_config(case, extra=None):
    w = case.workload
    lens = case.seq_lens.tolist()
    cfg = {"workload": w.name, "batch": len(lens), "total_tokens": int(sum(lens)),
           "min_len": int(min(lens)), "max_len": int(max(lens)), "num_q_heads": w.num_q_heads,
           "head_dim": w.head_dim, "kv_heads": w.num_kv_heads, "kv_shared": w.kv_shared,
           "page_size": w.page_size, "kv_dtype": w.kv_dtype,
           "softmax_scale": w.scale(), "parallelism": "replica per GPU",
           "new_tokens_per_seq": w.tokens_per_seq}
    if extra:
        cfg.update(extra)
    return cfg


def rank_workload(w, rank: int):
    """The shard of a multi-GPU run that rank ``rank`` decodes: the same workload
    shape with its own sequences (the seed moves with the rank).  Ranks share no
    data, so the timed steps have no collective; whole-job throughput is
    world x one rank's bytes over the slowest rank's time (weak scaling)."""
    if rank == 0:
        return w
    import dataclasses
    return dataclasses.replace(w, seed=w.seed + 7919 * rank)


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of one float over all ranks (the value itself on one rank)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank: int, world: int, ms: float) -> float:
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


class _Timer:
    """Device timing helpers shared by the workloads: CUDA events on the launching stream,
    barrier + synchronize on both sides of every timed region, max over ranks."""

    def __init__(self, dev, dist, windows):
        import torch
        self.torch = torch
        self.dev = dev
        self.dist = dist
        self.windows = windows
        self.stream = torch.cuda.current_stream(dev)

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()
        self.torch.cuda.synchronize()

    def graph_ms(self, fn, steps):
        """Mean ms per call of fn(i), i < steps, replayed from one CUDA graph of exactly
        `steps` calls (the first replay, which uploads the graph, is untimed)."""
        torch = self.torch
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(steps):
                fn(i)
        graph.replay()
        self.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_start = time.time()
        e0.record(self.stream)
        graph.replay()
        e1.record(self.stream)
        self.barrier()
        self.windows.append((t_start, time.time()))
        return max_over_ranks(e0.elapsed_time(e1), self.dist, self.dev) / steps, graph

    def per_launch_ms(self, fn, n):
        """Mean ms of fn(i) alone: per-launch events, queued behind a GPU sleep so that the
        launches run back to back whatever the host-side cost of enqueueing them."""
        torch = self.torch
        for i in range(3):
            fn(i)
        self.barrier()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        t_start = time.time()
        torch.cuda._sleep(int(2e7))
        for i in range(n):
            evs[i][0].record(self.stream)
            fn(i)
            evs[i][1].record(self.stream)
        self.barrier()
        self.windows.append((t_start, time.time()))
        return max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / n, self.dist, self.dev)


def measure_workload(args, case, tm, world: int, steps: int, headline: bool):
    """Time one workload: the whole step (decode + combine) from a CUDA graph, the decode
    kernel alone, and the step end to end through the host-buffer C ABI call.  The headline
    workload also gets the step without early metadata, each kernel alone and the KV append."""
    import torch
    import decode_attention_02_gb300 as mfa
    from decode_attention_02_gb300 import inputs

    dev = tm.dev
    w = case.workload
    lens = case.seq_lens.tolist()
    kv = mfa.KV_DTYPES[w.kv_dtype]
    B = len(lens)
    T = w.tokens_per_seq
    sa = shape_args(w)
    acct = algorithmic_bytes(lens, w.kv_dtype, T=T, **sa)
    flops = algorithmic_flops(lens, H=sa["H"], d=sa["d"], T=T)
    H, dq = w.num_q_heads, w.head_dim

    # rotating input copies: consecutive steps never find their KV in L2
    set_bytes = case.k_cache.numel() * case.k_cache.element_size() * (1 if w.kv_shared else 2)
    nsets = 1 + max(1, math.ceil(2 * L2_BYTES / max(set_bytes, 1)))
    sets = []
    for _ in range(nsets):
        k_dev = case.k_cache.to(dev)
        sets.append(dict(
            q=case.q.to(dev), k=k_dev, v=k_dev if w.kv_shared else case.v_cache.to(dev),
            ks=None if case.k_scale is None else case.k_scale.to(dev),
            vs=None if case.v_scale is None else case.v_scale.to(dev),
            table=case.block_table.to(dev), lens=case.seq_lens.to(dev)))
    out = torch.empty(B * T, H, dq, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B * T, H, dtype=torch.float32, device=dev)

    def decoder(flags):
        return mfa.Decoder(B, case.max_pages, case.num_blocks, kv_dtype=kv, softmax_scale=w.scale(),
                           host_seq_lens=lens, flags=flags, device=dev, tokens_per_seq=T,
                           shape=(w.num_q_heads, w.head_dim, w.num_kv_heads, w.kv_shared))

    # the timed steps are back-to-back decode steps whose lengths and block table are
    # filled once, before the loop: each step's decode may therefore read them while the
    # previous step's combine is still running (q, K, V and all outputs stay ordered)
    dec = decoder(mfa.MFA_PLAN_EARLY_METADATA)
    # the decode kernel alone, in the configuration the timed steps launch it with
    dec_only = decoder(mfa.MFA_PLAN_NO_COMBINE | mfa.MFA_PLAN_EARLY_METADATA)
    G = dec.plan.num_ctas
    launches_per_step = 1 + (1 if G > 1 else 0)

    def step(i, d=dec):
        s = sets[i % nsets]
        mfa.mfa_decode_run(d.plan, d.problem, s["q"], s["k"], s["v"], s["ks"], s["vs"], s["table"], s["lens"],
                           out, lse, d.workspace, None)

    # the status word of this exact launch configuration must stay clear
    step(0)
    torch.cuda.synchronize()
    status = mfa.mfa_read_device_status(dec.workspace)
    if status != 0:
        raise RuntimeError(f"decode step set device status bits {status:#x} on {w.name}")

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    ms_step, graph = tm.graph_ms(step, steps)
    kern_mean_ms = tm.per_launch_ms(lambda i: step(i, dec_only), max(min(steps, 400), 50))

    # end to end through the C ABI with host buffers (mfa_decode_run_host): every step
    # copies its pinned host inputs (q, block table, lengths) in and its outputs (out, lse)
    # back inside the timed region.  Three streams rotate, each with its own device buffers
    # and workspace, so that one step's copies overlap the other steps' kernels.
    q_h = case.q.pin_memory()
    table_h = case.block_table.pin_memory()
    lens_h = case.seq_lens.pin_memory()
    lanes = []
    for _ in range(E2E_LANES):
        lanes.append((decoder(mfa.MFA_PLAN_EARLY_METADATA), torch.cuda.Stream(dev),
                      torch.empty(B * T, H, dq, dtype=torch.bfloat16).pin_memory(),
                      torch.empty(B * T, H, dtype=torch.float32).pin_memory()))
    h2d = sum(t.numel() * t.element_size() for t in (q_h, table_h, lens_h))
    d2h = sum(t.numel() * t.element_size() for t in lanes[0][2:])

    def e2e_step(i):
        d_k, st_k, o_h, l_h = lanes[i % len(lanes)]
        s = sets[i % nsets]
        d_k.run_host(q_h, table_h, lens_h, o_h, l_h, s["k"], s["v"], s["ks"], s["vs"], stream=st_k)

    def join_lanes():
        for _, st_k, _, _ in lanes:
            ev = torch.cuda.Event()
            ev.record(st_k)
            tm.stream.wait_event(ev)

    for i in range(args.warmup):
        e2e_step(i)
    join_lanes()
    tm.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start = time.time()
    e0.record(tm.stream)
    for _, st_k, _, _ in lanes:
        st_k.wait_event(e0)
    t_enq = time.perf_counter()
    for i in range(steps):
        e2e_step(i)
    enqueue_ms = (time.perf_counter() - t_enq) * 1e3 / steps   # host time to issue one step
    join_lanes()
    e1.record(tm.stream)
    tm.barrier()
    tm.windows.append((t_start, time.time()))
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), tm.dist, dev) / steps

    hbm_peak, bf16_peak, _, peak_src = load_peaks()
    achieved = acct["total"] / (kern_mean_ms * 1e-3) / 1e9
    res = {
        "value": whole_job_gbs(acct["kv"], world, ms_step), "unit": "GB/s", "ms_per_step": ms_step,
        "tflops": flops * world / (ms_step * 1e-3) / 1e12,
        "hbm_roofline_frac": (acct["total"] / (hbm_peak * 1e9)) / (ms_step * 1e-3),
        "tensor_roofline_frac": (flops / (bf16_peak * 1e12)) / (ms_step * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": profiled_traffic(w.name),
                     "kernel": "mfa_decode_kernel", "mean_launch_ms": kern_mean_ms,
                     "algorithmic_bytes_per_launch": acct["total"], "peak_source": f"{peak_src} hbm_gbs",
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS},
        "e2e": {"value": whole_job_gbs(acct["kv"], world, e2e_ms), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "path": f"mfa_decode_run_host (pinned host buffers in and out), {E2E_LANES} streams in rotation",
                "host_enqueue_ms_per_step": enqueue_ms},
        "config": workload_config(case, {"l2": f"{nsets} rotating input copies ({nsets * set_bytes / 1e6:.0f} MB "
                                               f"of KV) so no step reads KV left in L2 by the previous one",
                                         "num_ctas": G, "timing": "K steps replayed from one CUDA graph",
                                         "flags": "MFA_PLAN_EARLY_METADATA"}),
        "steps": steps,
        "gpu_launches": launches_per_step * steps,
        "device_status": status,
    }
    if not headline:
        del sets, lanes, graph
        return res

    # --- the same K steps without the early-metadata overlap (every read after the previous step)
    dec_strict = decoder(0)
    res["ms_per_step_without_early_metadata"], _ = tm.graph_ms(lambda i: step(i, dec_strict), steps)

    # --- the combine kernel alone, on the partials the last decode-only launch left in the
    #     workspace, so that one step's kernel shares can be set beside the ncu launch list's
    comb_lens = sets[0]["lens"]
    step(0, dec_only)
    comb_mean_ms = tm.per_launch_ms(
        lambda i: mfa.mfa_combine(dec_only.plan, dec_only.problem, dec_only.workspace, comb_lens, out, lse),
        max(min(steps, 400), 50))

    if (w.num_q_heads, w.head_dim, w.num_kv_heads) != (64, 256, 1):
        # the append writes MFA cache rows only
        res["kernels_live"] = {"mean_launch_ms": {"mfa_decode_kernel": kern_mean_ms, "mfa_combine_kernel": comb_mean_ms}}
        res["kv_append"] = None
        return res

    # --- the KV append of the same batch (each sequence's T new rows at its last T positions),
    #     alone and chained in front of the decode step (append -> decode -> combine)
    k_new = inputs.new_token_rows(B * T, seed=w.seed + 101, kinds=("normal",)).to(dev)
    v_new = inputs.new_token_rows(B * T, seed=w.seed + 102, kinds=("normal",)).to(dev)
    positions = (case.seq_lens.to(torch.int32) - T).to(dev)

    def append(i):
        s = sets[i % nsets]
        mfa.mfa_kv_append(dec.problem, k_new, v_new, positions, s["table"], s["k"], s["v"], s["ks"], s["vs"],
                          device_status=dec.workspace)

    app_mean_ms = tm.per_launch_ms(append, max(min(steps, 400), 50))

    def append_and_step(i):
        append(i)
        step(i)

    ms_step_append, _ = tm.graph_ms(append_and_step, steps)

    # the same step through mfa_decode_append_run: one kernel launch for one new token per
    # sequence (the CTA that reads a sequence's last page writes its new rows first)
    def fused_step(i):
        s = sets[i % nsets]
        mfa.mfa_decode_append_run(dec.plan, dec.problem, s["q"], s["k"], s["v"], s["ks"], s["vs"], s["table"],
                                  s["lens"], k_new, v_new, positions, out, lse, dec.workspace, None)

    ms_step_fused, _ = tm.graph_ms(fused_step, steps)
    app_status = mfa.mfa_read_device_status(dec.workspace)
    if app_status != 0:
        raise RuntimeError(f"append + decode steps set device status bits {app_status:#x} on {w.name}")
    app_bytes = append_bytes(B, w.kv_dtype, T=T)
    res["kernels_live"] = {
        "mean_launch_ms": {"mfa_decode_kernel": kern_mean_ms, "mfa_combine_kernel": comb_mean_ms,
                           "mfa_kv_append_kernel": app_mean_ms},
        "share_of_one_step": {k: v / (kern_mean_ms + comb_mean_ms + app_mean_ms) for k, v in
                              (("mfa_decode_kernel", kern_mean_ms), ("mfa_combine_kernel", comb_mean_ms),
                               ("mfa_kv_append_kernel", app_mean_ms))},
        "timing": "each kernel alone, per-launch events behind a GPU sleep (launch latency included)"}
    res["kv_append"] = {
        "kernel": "mfa_kv_append_kernel", "mean_launch_ms": app_mean_ms,
        "algorithmic_bytes_per_launch": app_bytes,
        "achieved_gbs": app_bytes / (app_mean_ms * 1e-3) / 1e9,
        "frac_of_hbm": app_bytes / (app_mean_ms * 1e-3) / 1e9 / hbm_peak,
        "bound": "latency: one dependent load chain (position, page id, row) per row",
        "ms_per_step_with_append": ms_step_append,
        "added_ms_per_step": ms_step_append - ms_step,
        "ms_per_step_with_fused_append": ms_step_fused,
        "added_ms_per_step_fused": ms_step_fused - ms_step,
        "fused": "mfa_decode_append_run: " + ("one kernel (the append inside the decode)" if T == 1
                                              else "the append kernel, then the decode"),
        "timing": "append alone: per-launch events behind a GPU sleep; with append: "
                  "K steps of append + decode + combine from one CUDA graph",
        "device_status": app_status}
    return res


def run_native(args, case, rank: int, world: int, side_names=()):
    import torch
    from decode_attention_02_gb300 import build, inputs

    build.build_library()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
    windows = []
    tm = _Timer(dev, dist, windows)
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.2)

    head = measure_workload(args, case, tm, world, args.steps, headline=True)
    side = {}
    for name in side_names:
        c = inputs.generate(rank_workload(inputs.WORKLOADS[name], rank))
        r = measure_workload(args, c, tm, world, min(args.steps, SIDE_STEPS), headline=False)
        side[name] = {k: r[k] for k in ("value", "unit", "ms_per_step", "tflops", "hbm_roofline_frac", "roofline",
                                        "e2e", "steps", "device_status")}
        side[name]["config"] = {k: r["config"][k] for k in ("batch", "total_tokens", "kv_dtype", "num_ctas",
                                                             "new_tokens_per_seq", "num_q_heads", "head_dim",
                                                             "kv_heads", "kv_shared")}
        del c, r
        torch.cuda.empty_cache()

    # keep sampling clocks until the windows hold enough samples
    clocks = sampler.summary(windows)
    if clocks["samples"] < 5:
        t_start = time.time()
        while time.time() - t_start < 0.6:
            tm.barrier()
            time.sleep(0.01)
        windows.append((t_start, time.time()))
        time.sleep(0.1)
        clocks = sampler.summary(windows)
        clocks["window"] = "timed regions plus 0.6 s idle"
    sampler.stop()

    w = case.workload
    result = {
        "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": PATH_DTYPE[w.kv_dtype],
        "data": "synthetic", "config": head["config"],
    }
    for k in ("tflops", "ms_per_step_without_early_metadata", "hbm_roofline_frac", "tensor_roofline_frac",
              "roofline", "e2e", "gpu_launches", "device_status", "kernels_live", "kv_append"):
        result[k] = head[k]
    result["clocks"] = clocks
    if side:
        result["workloads"] = side
    return result


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workloads", default="all",
                    help="side workloads measured after the headline: all, none, or a comma list")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from decode_attention_02_gb300 import inputs
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    case = inputs.generate(rank_workload(inputs.WORKLOADS[args.workload], rank))

    if args.impl == "reference":
        res = run_reference(args, case, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    if args.workloads == "all":
        side_names = [n for n in SIDE_WORKLOADS if n != args.workload]
    elif args.workloads == "none":
        side_names = []
    else:
        side_names = [n for n in args.workloads.split(",") if n]
    res = run_native(args, case, rank, world, side_names)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            import oracle
            oracle.build()
            v, dt, k, reps = cpu_oracle_sample(case)
            v1, dt1, k1, reps1 = cpu_oracle_sample(case, target_s=4.0, nthreads=1)
            res["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": oracle.num_cpus(), "kind": "oracle",
                                   "sample": f"{k} of {len(case.seq_lens)} sequences x {reps} passes, "
                                             f"fp64, {dt:.1f} s",
                                   "single_thread": {"value": v1, "unit": "GB/s", "cores": 1,
                                                     "sample": f"{k1} sequences x {reps1} passes, {dt1:.1f} s"}}
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
