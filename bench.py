"""Benchmark of the KDA library on one GB300 (or N replicas under torchrun).

Default workload: batched prefill B4 H32 T4096 d128 (inputs larger than L2,
resident in HBM).  One step = one kda_chunk_fwd call over the whole batch
(every hot-path stage: decay scan, intra-chunk matrices, UT transform, state
hand-off, segment split when chosen).  The batched decode workload (256
sequences x 32 heads, d128, fresh inputs each step) is measured in the same
run and reported under "decode".

Prints one JSON line on rank 0.  `--impl reference` times the fp64 CPU
oracle on the host cores instead (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

CHUNK = 64
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=1, choices=[1, 2, 3])
    ap.add_argument("--decode-steps", type=int, default=64)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-fused", action="store_true")
    ap.add_argument("--no-checkpoints", action="store_true")
    ap.add_argument("--no-long", action="store_true",
                    help="skip the long-context legs (workloads 2 and 3)")
    ap.add_argument("--soak-s", type=float, default=1.0,
                    help="untimed seconds of the headline step with the clock sampler running")
    return ap.parse_args()


# ---------------------------------------------------------------- algorithmic work

def prefill_bytes(n_token_heads, n_seq_heads, d, has_s0):
    """q, k, v (bf16), log_alpha (f32), beta (f32) read, out (bf16) written per
    token-head; S0 read (if given) and S_final written per sequence-head."""
    per_th = 3 * 2 * d + 4 * d + 4 + 2 * d
    per_sh = 4 * d * d * (2 if has_s0 else 1)
    return n_token_heads * per_th + n_seq_heads * per_sh


def prefill_bytes_fused(n_token_heads, n_seq_heads, d, has_s0):
    """The fused entry point: raw q, k, v and the gate logits (all bf16), beta
    (f32) read, out (bf16) written per token-head; the state as above."""
    per_th = 4 * 2 * d + 4 + 2 * d
    per_sh = 4 * d * d * (2 if has_s0 else 1)
    return n_token_heads * per_th + n_seq_heads * per_sh


def prefill_flops(n_token_heads, d, C=CHUNK):
    """Fixed convention, triangular-aware: 6 d^2 (W S, Q S, K'^T U) plus
    C(3 dk + 2 dv) for the intra-chunk products, per token-head."""
    return n_token_heads * (6 * d * d + 5 * C * d)


def decode_bytes(n_seq_heads, d):
    """State read + write (f32) plus q, k, v, out (bf16), log_alpha (f32), beta."""
    return n_seq_heads * (8 * d * d + 12 * d + 4)


def decode_flops(n_seq_heads, d):
    return n_seq_heads * 7 * d * d


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_sha(path):
    with open(path, "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()[:16]


def recorded_traffic(kernel, src_file):
    """DRAM bytes per launch from the committed ncu summary of `kernel`, or None
    when absent or taken on a different version of the kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)[kernel]
    except (OSError, KeyError, ValueError):
        return None
    src = os.path.join(ROOT, "gated_delta_rule_48_gb300", "csrc", src_file)
    if not os.path.exists(src) or rec.get("source_sha") != source_sha(src):
        return None
    return float(rec["bytes_per_launch"])


def recorded_traffic_leg(kernel, workload_idx, segment_tokens=None):
    """DRAM bytes per launch of `kernel` on a long-context workload, from the
    committed ncu summary, or None (absent, another version of the kernel
    sources, or another segment length than the one this run splits at)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)[f"{kernel}@w{workload_idx}"]
    except (OSError, KeyError, ValueError):
        return None
    if "segment_tokens" in rec and rec["segment_tokens"] != segment_tokens:
        return None
    srcs = rec.get("sources", {})
    for f, sha in srcs.items():
        path = os.path.join(ROOT, "gated_delta_rule_48_gb300", "csrc", f)
        if not os.path.exists(path) or source_sha(path) != sha:
            return None
    return float(rec["bytes_per_launch"]) if srcs else None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=self.file, stderr=subprocess.DEVNULL)
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
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        with open(self.file.name) as fh:
            rows = [r.strip().split(", ") for r in fh if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- ranks

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
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- GPU arm

def _device_inputs(p):
    cu = None if p.uniform else torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda()
    return dict(q=p.q.cuda(), k=p.k.cuda(), v=p.v.cuda(), log_alpha=p.log_alpha.cuda(),
                beta=p.beta.cuda(), S0=None if p.S0 is None else p.S0.cuda(), cu_seqlens=cu)


def time_prefill(kb, p, steps, warmup, world, soak_s=0.0, d=None):
    """Device-resident inputs; K timed kda_chunk_fwd calls bracketed by a
    barrier and a synchronize.  Before them, ``soak_s`` seconds of the same
    call run untimed with the clock sampler already on, so the clock record
    covers a sustained load and not only the (short) timed region.  Returns
    (ms per step, per-kernel tracing, clocks, per-step statistics)."""
    if d is None:
        d = _device_inputs(p)
    out = torch.empty((p.total_T, p.H, p.dv), dtype=torch.bfloat16, device="cuda")
    S = torch.empty((p.n_seqs, p.H, p.dk, p.dv), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        kb.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"],
                         d["cu_seqlens"], out=out, S_final=S, n_seqs=p.n_seqs, stream=stream)

    for _ in range(warmup):
        step()
    if kb.kda_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    kb.profile_read()  # drop anything recorded so far
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with ClockSampler(torch.cuda.current_device()) as clocks:
        if soak_s > 0:
            torch.cuda.synchronize()
            t_end = time.perf_counter() + soak_s
            while time.perf_counter() < t_end:
                for _ in range(8):
                    step()
                torch.cuda.synchronize()
        kb.profile_enable(True)
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(steps):
            marks[i].record(stream)
            step()
        marks[steps].record(stream)
        stop.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    kb.profile_enable(False)
    kernels = kb.profile_read()
    ms = start.elapsed_time(stop) / steps
    per = sorted(marks[i].elapsed_time(marks[i + 1]) for i in range(steps))
    stats = {"median": per[len(per) // 2], "min": per[0], "max": per[-1]}
    return ms, kernels, clocks.summary(), stats


def long_leg(kb, idx, steps, warmup, world, peaks, peak_src):
    """One long-context prefill workload (2 or 3) timed like the headline: the
    whole kda_chunk_fwd call per step (planner, summary, scan and replay when
    the library splits the sequences).  Inputs are drawn on the device with
    the workload's recipe.  The roofline is that of the whole path: the
    step's algorithmic bytes over the summed event time of the library's
    kernels in one step."""
    from gated_delta_rule_48_gb300 import inputs as kin
    p = kin.workload_device(idx)
    d = dict(q=p.q, k=p.k, v=p.v, log_alpha=p.log_alpha, beta=p.beta, S0=p.S0,
             cu_seqlens=None if p.uniform else
             torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda())
    th, sh, dd = p.total_T * p.H, p.n_seqs * p.H, p.dk
    alg_bytes = prefill_bytes(th, sh, dd, p.S0 is not None)
    alg_flops = prefill_flops(th, dd)
    ms, kernels, clocks, stats = time_prefill(kb, p, steps, warmup, world, d=d)
    ms = max_over_ranks(ms, world)
    path_ms = sum(t for _, t in kernels.values()) / steps
    achieved = alg_bytes / (path_ms * 1e-3) / 1e9
    top_name, (top_n, top_ms) = max(kernels.items(), key=lambda kv: kv[1][1])
    tflops = alg_flops / (ms * 1e-3) / 1e12
    attainable = min(peaks["bf16_tflops"], alg_flops / alg_bytes * peaks["hbm_gbs"] / 1e3)
    # DRAM bytes per step from the committed ncu records of each kernel; the
    # planner reads at most cu_seqlens and writes the segment list (a few KB),
    # so it counts as zero
    traffic = None
    seg = kb.kda_auto_segment_tokens(p.total_T, p.n_seqs, p.H,
                                     torch.cuda.get_device_properties(0).multi_processor_count,
                                     p.uniform)
    recs = [0.0 if name == "kda_plan" else recorded_traffic_leg(name, idx, seg) for name in kernels]
    if kernels and all(r is not None for r in recs):
        traffic = sum(r * (n / steps) for r, (n, _) in zip(recs, kernels.values()))
    leg = {
        "workload": kin.WORKLOADS[idx], "value": p.total_T / (ms * 1e-3) / 1e6,
        "unit": "Mtok/s", "ms_per_step": ms, "step_ms": stats,
        "config": workload_config(p, idx),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": "whole path: " + ", ".join(sorted(kernels)),
                     "dominant_kernel": top_name, "peak_source": peak_src,
                     "algorithmic_bytes_per_step": alg_bytes},
        "tensor": {"tflops": tflops, "frac_of_bf16_peak": tflops / peaks["bf16_tflops"],
                   "attainable_tflops": attainable, "frac_of_attainable": tflops / attainable},
        "kernels": {k: {"launches_per_step": n / steps, "avg_ms": t / n,
                        "share": t / max(1e-12, sum(tt for _, tt in kernels.values()))}
                    for k, (n, t) in kernels.items()},
        "gpu_launches": sum(n for n, _ in kernels.values()),
        "clocks": clocks,
        "data": "synthetic, drawn on the device (same recipe and lengths, other values)",
    }
    return leg, p


def time_prefill_fused(kb, r, steps, warmup):
    """Device-resident raw inputs; K timed kda_chunk_fwd_fused calls.  Returns
    (ms per step, per-kernel tracing)."""
    q, k, v, g = r.q_raw.cuda(), r.k_raw.cuda(), r.v.cuda(), r.gate.cuda()
    b = r.beta.cuda()
    S0 = None if r.S0 is None else r.S0.cuda()
    out = torch.empty((r.total_T, r.H, r.dv), dtype=torch.bfloat16, device="cuda")
    S = torch.empty((r.n_seqs, r.H, r.dk, r.dv), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        kb.kda_chunk_fwd_fused(q, k, v, g, b, S0, None, out=out, S_final=S, n_seqs=r.n_seqs,
                               stream=stream)

    for _ in range(warmup):
        step()
    if kb.kda_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    kb.profile_read()
    kb.profile_enable(True)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    kb.profile_enable(False)
    return start.elapsed_time(stop) / steps, kb.profile_read()


def time_prefill_checkpoints(kb, p, interval, steps, warmup):
    """kda_chunk_fwd_checkpoints on device-resident inputs; returns (ms per step,
    checkpoints per step)."""
    d = _device_inputs(p)
    cu = d["cu_seqlens"]
    if cu is None:
        cu = torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda()
    lens = np.diff(p.cu_seqlens)
    n_ck = int(np.sum(lens // interval))
    stream = torch.cuda.current_stream()

    def step():
        return kb.kda_chunk_fwd_checkpoints(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                            d["S0"], cu, interval=interval,
                                            max_checkpoints=n_ck, stream=stream)

    for _ in range(warmup):
        step()
    if kb.kda_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(stop) / steps, n_ck


def time_prefill_e2e_host(kb, p, steps, warmup):
    """The public host-memory entry point (kda_chunk_fwd_host) on pinned HOST
    buffers: every step moves that step's inputs host->device and out +
    S_final back, pipelined with the prefill in 512-token slices."""
    pin = lambda t: None if t is None else t.contiguous().pin_memory()
    q, k, v, la, b, S0 = (pin(t) for t in (p.q, p.k, p.v, p.log_alpha, p.beta, p.S0))
    out_h = torch.empty((p.total_T, p.H, p.dv), dtype=torch.bfloat16).pin_memory()
    S_h = torch.empty((p.n_seqs, p.H, p.dk, p.dv), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v, la, b, S0) if t is not None)
    d2h = out_h.numel() * out_h.element_size() + S_h.numel() * S_h.element_size()

    def step():
        kb.kda_chunk_fwd_host(q, k, v, la, b, S0, out_h, S_h, n_seqs=p.n_seqs, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(stop) / steps, h2d, d2h


def time_prefill_e2e(kb, p, steps, warmup):
    """Same calls through the public API from pinned HOST buffers: every step
    copies that step's inputs host->device and reads out + S_final back."""
    host = dict(q=p.q.pin_memory(), k=p.k.pin_memory(), v=p.v.pin_memory(),
                log_alpha=p.log_alpha.pin_memory(), beta=p.beta.pin_memory(),
                S0=None if p.S0 is None else p.S0.pin_memory())
    dev = {k: (None if v is None else torch.empty_like(v, device="cuda"))
           for k, v in host.items()}
    cu = None if p.uniform else torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda()
    out = torch.empty((p.total_T, p.H, p.dv), dtype=torch.bfloat16, device="cuda")
    S = torch.empty((p.n_seqs, p.H, p.dk, p.dv), dtype=torch.float32, device="cuda")
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    S_h = torch.empty(S.shape, dtype=S.dtype).pin_memory()
    stream = torch.cuda.current_stream()
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = out_h.numel() * out_h.element_size() + S_h.numel() * S_h.element_size()

    def step():
        for k, v in host.items():
            if v is not None:
                dev[k].copy_(v, non_blocking=True)
        kb.kda_chunk_fwd(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["beta"],
                         dev["S0"], cu, out=out, S_final=S, n_seqs=p.n_seqs, stream=stream)
        out_h.copy_(out, non_blocking=True)
        S_h.copy_(S, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(stop) / steps, h2d, d2h


def time_decode(kb, dec, steps_per_run, warmup, runs=3):
    """Batched decode: `steps_per_run` consecutive in-place steps with fresh
    inputs per step (all resident on the device); the state (512 MiB for the
    default workload) exceeds L2, so no flush is needed."""
    q, k, v = dec.q.cuda(), dec.k.cuda(), dec.v.cuda()
    la, b = dec.log_alpha.cuda(), dec.beta.cuda()
    S = dec.S.cuda()
    N, H, dk = dec.q.shape[1:4]
    out = torch.empty((N, H, dec.v.shape[3]), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    n_in = q.shape[0]
    for i in range(warmup):
        kb.kda_decode_step(q[i % n_in], k[i % n_in], v[i % n_in], la[i % n_in], b[i % n_in],
                           S, out, stream=stream)
    torch.cuda.synchronize()
    kb.profile_read()
    kb.profile_enable(True)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(runs):
        for i in range(steps_per_run):
            j = i % n_in
            kb.kda_decode_step(q[j], k[j], v[j], la[j], b[j], S, out, stream=stream)
    stop.record(stream)
    torch.cuda.synchronize()
    kb.profile_enable(False)
    kernels = kb.profile_read()
    return start.elapsed_time(stop) / (runs * steps_per_run), kernels


def time_decode_tokens(kb, dec, calls, warmup):
    """kda_decode_tokens with all of a call's tokens committed: [N, K, ...]
    inputs resident on the device, `calls` timed calls in a row."""
    f = lambda t: t.transpose(0, 1).contiguous().cuda()
    q, k, v, la, b = f(dec.q), f(dec.k), f(dec.v), f(dec.log_alpha), f(dec.beta)
    S = dec.S.cuda()
    out = torch.empty(tuple(v.shape), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        kb.kda_decode_tokens(q, k, v, la, b, S, None, out, stream=stream)
    torch.cuda.synchronize()
    kb.profile_read()
    kb.profile_enable(True)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(calls):
        kb.kda_decode_tokens(q, k, v, la, b, S, None, out, stream=stream)
    stop.record(stream)
    torch.cuda.synchronize()
    kb.profile_enable(False)
    return start.elapsed_time(stop) / calls, kb.profile_read()


# ---------------------------------------------------------------- CPU oracle

def cpu_sample(p, n_seqs, max_tokens=None):
    """The first `n_seqs` sequences of a workload (all heads); with
    `max_tokens`, only the first tokens of the first sequence."""
    from gated_delta_rule_48_gb300 import inputs as kin
    t1 = int(p.cu_seqlens[n_seqs])
    cu = p.cu_seqlens[:n_seqs + 1].copy()
    if max_tokens is not None:
        t1 = min(int(p.cu_seqlens[1]), int(max_tokens))
        cu = np.array([0, t1], dtype=np.int64)
        n_seqs = 1
    return dict(q=kin.bf16_bits(p.q[:t1]), k=kin.bf16_bits(p.k[:t1]), v=kin.bf16_bits(p.v[:t1]),
                log_alpha=p.log_alpha[:t1].numpy(), beta=p.beta[:t1].numpy(),
                S0=None if p.S0 is None else p.S0[:n_seqs].numpy(),
                cu=cu, tokens=t1)


def long_cpu_baseline(p, heads=(0, 2), max_tokens=65536):
    """The oracle on heads 0-1 of the million-token workload, bounded to the
    first `max_tokens` tokens of each sequence (16 independent chains)."""
    import oracle
    from gated_delta_rule_48_gb300 import inputs as kin
    oracle.build()
    threads = oracle.default_threads()
    cu = p.cu_seqlens
    rows, lens = [], []
    for n in range(p.n_seqs):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        t1 = min(t1, t0 + max_tokens)
        rows.append(torch.arange(t0, t1))
        lens.append(t1 - t0)
    idx = torch.cat(rows)
    h0, h1 = heads
    take = lambda t: t.index_select(0, idx.to(t.device))[:, h0:h1].contiguous().cpu()
    q, k, v = take(p.q), take(p.k), take(p.v)
    la, b = take(p.log_alpha), take(p.beta)
    S0 = None if p.S0 is None else p.S0[:, h0:h1].contiguous().cpu().numpy()
    cu_s = np.zeros(len(lens) + 1, dtype=np.int64)
    cu_s[1:] = np.cumsum(lens)
    sample = dict(q=kin.bf16_bits(q), k=kin.bf16_bits(k), v=kin.bf16_bits(v),
                  log_alpha=la.numpy(), beta=b.numpy(), S0=S0, cu=cu_s, tokens=int(cu_s[-1]))
    sec = time_oracle(sample, threads)
    th = sample["tokens"] * (h1 - h0)
    return {"value": th / sec / 1e6, "unit": "M token-heads/s", "cores": threads,
            "kind": "oracle", "cpu": cpu_model(), "seconds": sec,
            "sample": f"heads {h0}-{h1 - 1}, first {max_tokens} tokens of each of the "
                      f"{p.n_seqs} sequences ({sample['tokens']} tokens, {th} token-heads), "
                      "fp64 token-by-token recurrence"}


def time_oracle(sample, threads):
    import oracle
    t0 = time.perf_counter()
    oracle.forward(sample["q"], sample["k"], sample["v"], sample["log_alpha"], sample["beta"],
                   sample["S0"], sample["cu"], threads=threads)
    return time.perf_counter() - t0


def cpu_model():
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def workload_config(p, idx):
    from gated_delta_rule_48_gb300 import inputs as kin
    lens = np.diff(p.cu_seqlens)
    return {"workload": kin.WORKLOADS[idx], "n_seqs": p.n_seqs, "heads": p.H, "dk": p.dk,
            "dv": p.dv, "tokens": p.total_T, "seq_len": int(lens.max()) if lens.size else 0,
            "chunk": CHUNK, "l2": "inputs larger than L2 (no flush)"}


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle, as it stands, on the host cores.

    Each of the K timed steps evaluates the oracle on a bounded sample of the
    workload -- the first L tokens of sequence 0, all heads -- with L chosen
    from a short calibration so the whole run takes about a minute.  Under
    torchrun only rank 0 works and prints; the other ranks exit without work.
    """
    from gated_delta_rule_48_gb300 import inputs as kin
    import oracle
    if rank != 0:
        return
    oracle.build()
    p = kin.workload(args.workload)
    threads = oracle.default_threads()
    calib = cpu_sample(p, 1, max_tokens=128)
    t_cal = max(time_oracle(calib, threads), 1e-3)
    rate = calib["tokens"] / t_cal                       # tokens per second, all heads
    budget = 45.0                                        # seconds for the timed steps
    L = int(max(64, min(int(p.cu_seqlens[1]), rate * budget / max(1, args.steps))))
    sample = cpu_sample(p, 1, max_tokens=L)
    warm = cpu_sample(p, 1, max_tokens=64)
    for _ in range(args.warmup):
        time_oracle(warm, threads)
    per = [time_oracle(sample, threads) for _ in range(args.steps)]
    sec = statistics.mean(per)
    value = sample["tokens"] / sec / 1e6
    desc = (f"first {sample['tokens']} tokens of sequence 0 x {p.H} heads per step, fp64 "
            "token-by-token recurrence")
    line = {"impl": "reference", "metric": "KDA prefill throughput", "value": value,
            "unit": "Mtok/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(p, args.workload),
            "cpu_baseline": {"value": value, "unit": "Mtok/s", "cores": threads,
                             "kind": "oracle", "sample": desc, "cpu": cpu_model()},
            "e2e": {"value": value, "unit": "Mtok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
        barrier(world)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for the library arm")

    import gated_delta_rule_48_gb300 as kda
    from gated_delta_rule_48_gb300 import binding as kb
    from gated_delta_rule_48_gb300 import inputs as kin

    kda.build()
    peaks, peak_src = load_peaks()
    p = kin.workload(args.workload)
    d = p.dk
    th = p.total_T * p.H
    sh = p.n_seqs * p.H
    alg_bytes = prefill_bytes(th, sh, d, p.S0 is not None)
    alg_flops = prefill_flops(th, d)

    ms, kernels, clocks, step_stats = time_prefill(kb, p, args.steps, args.warmup, world,
                                                   soak_s=args.soak_s)
    ms = max_over_ranks(ms, world)
    tokens_all = sum_over_ranks(p.total_T, world)
    value = tokens_all / (ms * 1e-3) / 1e6  # Mtok/s over all ranks

    # dominant kernel: the one with the largest summed time in the timed region
    launches = sum(n for n, _ in kernels.values())
    top_name, (top_n, top_ms) = max(kernels.items(), key=lambda kv: kv[1][1])
    top_avg_ms = top_ms / top_n
    if len(kernels) == 1:
        # one kernel per step (the batched workload): its launch covers the
        # whole batch once, so the step's algorithmic bytes are its own
        per_launch_bytes = alg_bytes * (args.steps / top_n)
        achieved_gbs = per_launch_bytes / (top_avg_ms * 1e-3) / 1e9
    else:
        # several kernels per step (a split workload): the roofline of the
        # whole path, the step's bytes over the summed kernel time per step
        per_launch_bytes = alg_bytes
        achieved_gbs = alg_bytes / (sum(t for _, t in kernels.values()) / args.steps * 1e-3) / 1e9
        top_name = "whole path: " + ", ".join(sorted(kernels))
    tflops = alg_flops / (ms * 1e-3) / 1e12
    traffic = recorded_traffic(top_name, "kda_prefill_tc.cu")

    line = {
        "metric": "KDA prefill throughput", "value": value, "unit": "Mtok/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(p, args.workload),
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved_gbs / peaks["hbm_gbs"],
                     "traffic": traffic, "kernel": top_name, "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": per_launch_bytes},
        "tensor": {"tflops": tflops, "bf16_peak": peaks["bf16_tflops"],
                   "frac_of_bf16_peak": tflops / peaks["bf16_tflops"],
                   # attainable = min(tensor peak, arithmetic intensity x HBM bandwidth)
                   "attainable_tflops": min(peaks["bf16_tflops"],
                                            alg_flops / alg_bytes * peaks["hbm_gbs"] / 1e3),
                   "frac_of_attainable": tflops / min(peaks["bf16_tflops"],
                                                      alg_flops / alg_bytes * peaks["hbm_gbs"] / 1e3),
                   "algorithmic_flops_per_step": alg_flops,
                   "dense_tile_flops_per_step": th * (6 * d * d + 10 * CHUNK * d),
                   "peak_source": peak_src},
        "step_ms": step_stats,
        "kernels": {k: {"launches": n, "avg_ms": t / n} for k, (n, t) in kernels.items()},
        "gpu_launches": launches,
        "clocks": clocks,
    }

    if not args.no_long:
        # the long-context workloads: 65,536-token sequences and the packed
        # million-token batch, both split across SMs by the library
        for idx in (2, 3):
            if idx == args.workload:
                continue
            leg, lp = long_leg(kb, idx, max(3, min(args.steps, 20)), max(3, args.warmup),
                               world, peaks, peak_src)
            line[f"prefill_w{idx}"] = leg
            if rank == 0 and world == 1 and not args.no_cpu_baseline and idx == 3:
                leg["cpu_baseline"] = long_cpu_baseline(lp)
            del lp
            torch.cuda.empty_cache()

    if not args.no_e2e:
        e2e_fn = time_prefill_e2e_host if p.uniform else time_prefill_e2e
        e2e_ms, h2d, d2h = e2e_fn(kb, p, max(3, min(args.steps, 20)), 2)
        e2e_ms = max_over_ranks(e2e_ms, world)
        line["e2e"] = {"value": tokens_all / (e2e_ms * 1e-3) / 1e6, "unit": "Mtok/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e2e_ms,
                       "api": "kda_chunk_fwd_host" if p.uniform else "kda_chunk_fwd + copies"}

    if not args.no_fused and p.uniform:
        # the same batch shape through the entry point that prepares its inputs on
        # load (raw q, k projections, bf16 gate logits)
        T_b = p.total_T // p.n_seqs
        r = kin.make_prefill_raw([T_b] * p.n_seqs, p.H, d, seed=100 + args.workload,
                                 s0_std=0.02 if p.S0 is not None else 0.0)
        fms, fk = time_prefill_fused(kb, r, max(3, min(args.steps, 50)), args.warmup)
        fbytes = prefill_bytes_fused(th, sh, d, r.S0 is not None)
        fn, ft = fk["kda_prefill_replay"]
        f_gbs = fbytes * (max(3, min(args.steps, 50)) / fn) / (ft / fn * 1e-3) / 1e9
        line["fused_prep"] = {
            "workload": workload_config(p, args.workload)["workload"]
                        + ", raw projections (unnormalised q, k; bf16 gate logits)",
            "value": p.total_T / (fms * 1e-3) / 1e6, "unit": "Mtok/s", "ms_per_step": fms,
            "roofline": {"bound": "hbm", "achieved": f_gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": f_gbs / peaks["hbm_gbs"],
                         "traffic": recorded_traffic("kda_prefill_replay_fused", "kda_prefill_tc.cu"),
                         "kernel": "kda_prefill_replay", "peak_source": peak_src,
                         "algorithmic_bytes_per_launch": fbytes}}
        line["gpu_launches_fused"] = sum(n for n, _ in fk.values())
        del r

    if not args.no_checkpoints:
        # the same prefill, also emitting the state every 1024 tokens of each sequence
        cms, n_ck = time_prefill_checkpoints(kb, p, 1024, max(3, min(args.steps, 50)),
                                             args.warmup)
        line["checkpoints"] = {
            "workload": workload_config(p, args.workload)["workload"]
                        + ", state checkpoint every 1024 tokens",
            "value": p.total_T / (cms * 1e-3) / 1e6, "unit": "Mtok/s", "ms_per_step": cms,
            "checkpoints_per_step": n_ck * p.H,
            "checkpoint_bytes_per_step": n_ck * p.H * d * d * 4}

    if not args.no_decode:
        dec = kin.decode_workload(steps=args.decode_steps)
        n_sh = dec.q.shape[1] * dec.q.shape[2]
        dms, dk_kernels = time_decode(kb, dec, args.decode_steps, args.warmup)
        dbytes = decode_bytes(n_sh, dec.q.shape[3])
        dn, dt = dk_kernels["kda_decode_step"]
        kern_gbs = dbytes / (dt / dn * 1e-3) / 1e9
        line["decode"] = {
            "workload": kin.WORKLOADS[4], "value": dbytes / (dms * 1e-3) / 1e9, "unit": "GB/s",
            "ms_per_step": dms, "ms_per_64_steps": 64 * dms,
            "tokens_per_s": n_sh / dec.q.shape[2] / (dms * 1e-3),
            "roofline": {"bound": "hbm", "achieved": kern_gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": kern_gbs / peaks["hbm_gbs"],
                         "traffic": recorded_traffic("kda_decode_step", "kda_decode.cu"),
                         "kernel": "kda_decode_step", "peak_source": peak_src,
                         "algorithmic_bytes_per_launch": dbytes}}
        del dec
        # several tokens per call (speculative drafts): 8 tokens of each of the
        # same 256 x 32 sequence-heads, all committed
        K = 8
        decK = kin.make_decode(256, 32, 128, steps=K, seed=4)
        tms, tk = time_decode_tokens(kb, decK, 20, args.warmup)
        n_sh = 256 * 32
        tbytes = n_sh * (8 * 128 * 128 + K * (12 * 128 + 4))
        tn, tt = tk["kda_decode_tokens"]
        t_gbs = tbytes / (tt / tn * 1e-3) / 1e9
        line["decode_tokens"] = {
            "workload": f"batched decode 256 seqs H32 d128, {K} tokens per call, all committed",
            "value": 256 * K / (tms * 1e-3), "unit": "tokens/s", "ms_per_call": tms,
            "roofline": {"bound": "hbm", "achieved": t_gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": t_gbs / peaks["hbm_gbs"],
                         "traffic": recorded_traffic("kda_decode_tokens", "kda_decode_tokens.cu"),
                         "kernel": "kda_decode_tokens", "peak_source": peak_src,
                         "algorithmic_bytes_per_launch": tbytes}}
        del decK

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        threads = oracle.default_threads()
        sample = cpu_sample(p, min(p.n_seqs, 4))
        sec = time_oracle(sample, threads)
        line["cpu_baseline"] = {
            "value": sample["tokens"] / sec / 1e6, "unit": "Mtok/s", "cores": threads,
            "kind": "oracle", "cpu": cpu_model(), "seconds": sec,
            "sample": f"first {min(p.n_seqs, 4)} sequences of the workload ({sample['tokens']} "
                      f"tokens x {p.H} heads), fp64 token-by-token recurrence"}
        # the same oracle on one thread, on the tiny workload (token-heads per second)
        p0 = kin.workload(0)
        s0 = cpu_sample(p0, p0.n_seqs)
        sec0 = min(time_oracle(s0, 1) for _ in range(3))
        line["cpu_baseline"]["single_thread"] = {
            "value": s0["tokens"] * p0.H / sec0, "unit": "token-heads/s", "cores": 1,
            "sample": kin.WORKLOADS[0]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier(world)


if __name__ == "__main__":
    main()
