#!/usr/bin/env python
"""Benchmark: Jagged Flash Attention forward + backward on one GB300.

One step = one pass of the whole hot path over one batch: the host tile
schedules, the forward kernel (O, LSE), the backward pre-pass (Delta) and the
backward kernel (dQ summed over the batch, dK, dV), all through the C ABI.

Workload (the headline metric's configuration): jagged broadcast-Q attention in
the ads shape, B=512 sequences with lognormal KV lengths (median 256,
sigma 1, clipped to [8, 4096]), one dense Q [256, 4, 128] shared by every
sequence, bf16 N(0,1) inputs and upstream gradient, non-causal.  Inputs are
synthetic and seeded (jfa_inputs).  K+V alone (~390 MB) exceed the 129 MB
L2, so no explicit L2 flush is done between steps.

Metric: useful TFLOPS of forward + backward (4*D*H*pairs for the forward,
2.5x that for the backward; no padding is counted).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on a bounded sample of the same workload instead.
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

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import jfa_inputs  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOAD = "ads_bwd"  # default: the configuration the headline metric is quoted on
WORKLOAD_DESC = ("jagged broadcast-Q attention fwd+bwd, ads shape: B=512, KV lengths lognormal(median 256, "
                 "sigma 1) clipped to [8,4096], Q [256,4,128] shared, packed K/V [N,4,128], bf16, non-causal")


def workload_desc(name):
    """One-line description of a workload (the ads step keeps its fixed wording)."""
    if name == WORKLOAD:
        return WORKLOAD_DESC
    w = jfa_inputs.WORKLOADS[name]
    mode = (f"broadcast Q [{w.Lq},{w.H},{w.D}] shared" if w.broadcast_q else f"per-sequence Q [N,{w.H},{w.D}]")
    return (f"jagged attention {'fwd+bwd' if w.backward else 'fwd only'}, {name}: B={w.B}, KV lengths {w.lengths}, "
            f"{mode}, packed K/V [N,{w.H},{w.D}], bf16, {'causal' if w.causal else 'non-causal'}")


def metric_name(name, backward, sparse=None):
    what = "fwd+bwd" if backward else "fwd"
    tail = f", block-sparse (selection ratio {sparse})" if sparse is not None else ""
    if name == WORKLOAD:
        return f"{what} TFLOPS (bf16, 1 GB300) on jagged broadcast-Q{tail}"
    return f"{what} TFLOPS (bf16, 1 GB300) on {name}{tail}"


# ----------------------------------------------------------------------------
# FLOP / byte accounting (useful work only)
# ----------------------------------------------------------------------------
def pair_count(offsets, Lq, broadcast_q, causal, first=None):
    L = (offsets[1:] - offsets[:-1]).to(torch.int64)
    if first is not None:
        L = L[:first]
    if broadcast_q:
        return int(Lq * L.sum())
    if causal:
        return int((L * (L + 1) // 2).sum())
    return int((L * L).sum())


def accounting(x):
    B, Lq, H, D, N = x["B"], x["Lq"], x["H"], x["D"], x["N"]
    pairs = pair_count(x["offsets"], Lq, x["broadcast_q"], x["causal"])
    f_fwd = 4.0 * D * H * pairs
    f_bwd = 2.5 * f_fwd
    q_rows = Lq if x["broadcast_q"] else N
    o_rows = B * Lq if x["broadcast_q"] else N
    e = H * D
    q_b, kv_b, o_b = 2 * q_rows * e, 2 * N * e, 2 * o_rows * e
    stat_b = 4 * o_rows * H
    bytes_fwd = q_b + 2 * kv_b + o_b + stat_b                       # Q, K, V in; O, LSE out
    bytes_pre = 2 * o_b + stat_b                                     # O, dO in; Delta out
    bytes_bwd = q_b + 2 * kv_b + o_b + 2 * stat_b + 2 * kv_b + 2 * q_b  # Q,K,V,dO,LSE,Delta in; dK,dV,dQ(fp32) out
    return dict(pairs=pairs, flops_fwd=f_fwd, flops_bwd=f_bwd, bytes_fwd=bytes_fwd, bytes_pre=bytes_pre,
                bytes_bwd=bytes_bwd, flops_pre=2.0 * o_rows * e)


def selected_keys(offsets, mask):
    """Block-sparse: keys selected per (sequence, head), int64 [B, H]."""
    lens = (offsets[1:] - offsets[:-1]).tolist()
    out = torch.zeros(len(lens), mask.shape[1], dtype=torch.int64)
    g = 0
    for b, L in enumerate(lens):
        n = (L + 127) // 128
        if n:
            sizes = torch.tensor([min(128, L - 128 * i) for i in range(n)], dtype=torch.int64)
            out[b] = (mask[g:g + n].to(torch.int64) * sizes[:, None]).sum(0)
        g += n
    return out


def accounting_sparse(x, mask):
    """Useful work of the block-sparse step: only (query, key) pairs of selected blocks count, and
    only selected K/V rows are read; dK/dV of unselected rows are written as zeros (their own kernel)."""
    acc = accounting(x)
    sel = selected_keys(x["offsets"], mask)                      # [B, H]
    lens = (x["offsets"][1:] - x["offsets"][:-1]).to(torch.int64)
    rows = torch.full_like(lens, x["Lq"]) if x["broadcast_q"] else lens
    pairs_total = int((rows[:, None] * sel).sum())                # over heads
    H, D = x["H"], x["D"]
    f_fwd = 4.0 * D * pairs_total
    kv_sel = 2 * D * int(sel.sum())                               # bytes of K (or V) rows read
    kv_all = 2 * x["N"] * H * D
    q_rows = x["Lq"] if x["broadcast_q"] else x["N"]
    o_rows = x["B"] * x["Lq"] if x["broadcast_q"] else x["N"]
    q_b, o_b, stat_b = 2 * q_rows * H * D, 2 * o_rows * H * D, 4 * o_rows * H
    acc.update(pairs=pairs_total / H, flops_fwd=f_fwd, flops_bwd=2.5 * f_fwd,
               bytes_fwd=q_b + 2 * kv_sel + o_b + stat_b,
               bytes_bwd=q_b + 2 * kv_sel + o_b + 2 * stat_b + 2 * kv_sel + 2 * q_b,
               bytes_zero=2 * (kv_all - kv_sel), selected_fraction=int(sel.sum()) / max(1, x["N"] * H))
    return acc


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


def make_inputs(args, backward=None):
    """The workload's synthetic inputs; with --lengths, its shapes with those KV lengths
    (e.g. "131072,512x31": one 131072-key sequence and 31 of 512 keys)."""
    if not args.lengths:
        return jfa_inputs.make(args.workload) if backward is None else jfa_inputs.make(args.workload, backward=backward)
    w = jfa_inputs.WORKLOADS[args.workload]
    lens = []
    for part in args.lengths.split(","):
        n, _, rep_ = part.partition("x")
        lens += [int(n)] * (int(rep_) if rep_ else 1)
    x = jfa_inputs.custom(len(lens), w.Lq, w.H, w.D, lens, w.broadcast_q, w.causal, seed=1,
                          backward=w.backward if backward is None else backward)
    x["workload"] = f"{args.workload} with lengths {args.lengths}"
    return x


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("fwd.cu", "bwd.cu", "ptx.cuh", "kernels.h"):
        with open(os.path.join(ROOT, "bwd_jagged_flashattention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic():
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return {}
    with open(p) as f:
        d = json.load(f)
    if d.get("source_sha") != kernel_source_hash():
        return {}
    return d.get("kernels", {})


# ----------------------------------------------------------------------------
# Clock sampling during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == 0:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l for (t, l) in self.lines if self.t0 is not None and self.t0 - 0.05 <= t <= (self.t1 or t) + 0.15]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2]))
                smax.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[6:10]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_smi_id(dev) -> str:
    """nvidia-smi's identifier for this CUDA device (its UUID when torch exposes it)."""
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    return str(dev.index or 0)


# ----------------------------------------------------------------------------
# Distributed plumbing (independent replicas; no data-path collective)
# ----------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float, device) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# CPU oracle baseline (bounded sample of the same workload)
# ----------------------------------------------------------------------------
def oracle_sample(x, nseq, mask=None):
    import oracle
    off = x["offsets"][: nseq + 1].clone()
    N = int(off[-1])
    sub = dict(x, B=nseq, offsets=off, N=N, k=x["k"][:N], v=x["v"][:N])
    sub["do"] = x["do"][:nseq] if x["broadcast_q"] else x["do"][:N]
    sub["q"] = x["q"] if x["broadcast_q"] else x["q"][:N]
    m = None
    if mask is None:
        flops = 3.5 * 4.0 * x["D"] * x["H"] * pair_count(off, x["Lq"], x["broadcast_q"], x["causal"])
    else:
        m = mask[: jfa_inputs.num_kv_blocks(off)]
        flops = 3.5 * accounting_sparse(sub, m)["flops_fwd"]
    t0 = time.perf_counter()
    oracle.fwd(sub["q"], sub["k"], sub["v"], off, x["Lq"], x["broadcast_q"], x["causal"], x["scale"],
               kv_block_mask=m)
    oracle.bwd(sub["q"], sub["k"], sub["v"], sub["do"], off, x["Lq"], x["broadcast_q"], x["causal"], x["scale"],
               kv_block_mask=m)
    return flops, time.perf_counter() - t0


def size_oracle_sample(x, budget_s, mask=None):
    """Number of leading sequences whose oracle fwd+bwd takes about budget_s."""
    f1, t1 = oracle_sample(x, 2, mask)
    rate = f1 / max(t1, 1e-6)
    total = (3.5 * 4.0 * x["D"] * x["H"] * pair_count(x["offsets"], x["Lq"], x["broadcast_q"], x["causal"])
             if mask is None else 3.5 * accounting_sparse(x, mask)["flops_fwd"])
    return max(1, min(x["B"], int(budget_s * rate / (total / x["B"]))))


def cpu_baseline(x, budget_s=12.0, mask=None):
    """The oracle as it stands on the host cores: repeated passes over the first n sequences
    until about budget_s seconds of CPU work have been timed."""
    import oracle
    n = size_oracle_sample(x, budget_s, mask)
    flops = secs = 0.0
    reps = 0
    while secs < budget_s * 0.8 and reps < 8:
        f, t = oracle_sample(x, n, mask)
        flops, secs, reps = flops + f, secs + t, reps + 1
    return {"value": flops / secs / 1e12, "unit": "TFLOPS", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd, {reps} pass(es) over the first {n} of {x['B']} sequences of the "
                      f"same inputs ({flops / 1e9:.1f} GFLOP useful, {secs:.1f} s)"}


def first_sequences(x, n):
    """The same workload restricted to its first n sequences (for small profiling runs)."""
    off = x["offsets"][: n + 1].clone()
    N = int(off[-1])
    y = dict(x, B=n, offsets=off, N=N, k=x["k"][:N].contiguous(), v=x["v"][:N].contiguous())
    if "do" in x:
        y["do"] = (x["do"][:n] if x["broadcast_q"] else x["do"][:N]).contiguous()
    if not x["broadcast_q"]:
        y["q"] = x["q"][:N].contiguous()
    return y


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    x = jfa_inputs.make(args.workload)
    mask = (jfa_inputs.kv_block_mask(x["offsets"], x["H"], args.block_sparse, seed=1)
            if args.block_sparse is not None else None)
    budget = max(0.05, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    n = size_oracle_sample(x, budget, mask)
    for _ in range(args.warmup):
        oracle_sample(x, n, mask)
    tot_f, tot_t = 0.0, 0.0
    for _ in range(args.steps):
        f, t = oracle_sample(x, n, mask)
        tot_f += f
        tot_t += t
    value = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": metric_name(args.workload, True, args.block_sparse),
            "value": value, "unit": "TFLOPS", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_t / max(1, args.steps), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(args.workload), "sample": f"first {n} of {x['B']} sequences per step"},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"fp64 oracle fwd+bwd on the first {n} of {x['B']} sequences, per step"},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------
# The GPU arm
# ----------------------------------------------------------------------------
def run_mxfp8(args, world, rank):
    """The MXFP8 forward (P V in block-scaled E4M3, Q K^T bf16) on the workload's forward, V quantized once
    before timing (the forward's input, resident like the bf16 forward's bf16 V); the bf16 forward on the same
    inputs and the quantizer are timed beside it.  Not the headline line."""
    import bwd_jagged_flashattention_gb300 as jfa
    import oracle
    jfa.lib()
    dev = torch.device("cuda", 0 if world == 1 else int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    x = make_inputs(args, backward=False)
    if args.batch:
        x = first_sequences(x, args.batch)
    acc = accounting(x)
    B, Lq, H, D, N = x["B"], x["Lq"], x["H"], x["D"], x["N"]
    bq, causal = x["broadcast_q"], x["causal"]
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    off_h, off_d = x["offsets"], x["offsets"].to(dev)
    o = torch.empty((B, Lq, H, D) if bq else (N, H, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, Lq) if bq else (H, N), dtype=torch.float32, device=dev)
    ws = jfa.new_workspace(B, N, Lq if bq else 0, H, D, bq, causal, dev)
    v8, vs = jfa.quantize_v_mxfp8(v, off_d, offsets_host=off_h, workspace=ws)
    stream = torch.cuda.current_stream(dev)

    def mx_step(q_=q, k_=k, v8_=v8, vs_=vs, off_=off_d, o_=o, lse_=lse):
        jfa.fwd_mxfp8(q_, k_, v8_, vs_, off_, broadcast_q=bq, causal=causal, scale=x["scale"], offsets_host=off_h,
                      workspace=ws, out=o_, lse=lse_)

    def bf16_step():
        jfa.fwd(q, k, v, off_d, broadcast_q=bq, causal=causal, scale=x["scale"], offsets_host=off_h, workspace=ws,
                out=o, lse=lse)

    def quant_step():
        jfa.quantize_v_mxfp8(v, off_d, offsets_host=off_h, workspace=ws, v8=v8, v_scale=vs)

    def timed(fn, n):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        jfa.profile_enable(True)
        jfa.profile_read()
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        prof = jfa.profile_read()
        jfa.profile_enable(False)
        return max_over_ranks(world, a.elapsed_time(b), dev) / n, prof

    sampler = ClockSampler(gpu_smi_id(dev))
    sampler.start()
    sampler.mark(0)
    ms, prof = timed(mx_step, args.steps)
    sampler.mark(1)
    clocks = sampler.stop()
    assert jfa.device_status(ws) == 0, "kernel status word reports a timeout"
    bf16_ms, bf16_prof = timed(bf16_step, min(args.steps, 200))
    quant_ms, quant_prof = timed(quant_step, min(args.steps, 200))
    value = world * acc["flops_fwd"] / (ms * 1e-3) / 1e12
    peaks = load_peaks()
    # half the FLOPs (Q K^T) run at the bf16 rate, half (P V) at the E4M3 rate, twice the bf16 one
    # (2.25 vs 4.5 PFLOP/s dense nominal): the mix's peak is 4/3 of the bf16 peak.
    peak_mix = peaks["bf16_tflops"] * 4.0 / 3.0
    fwd_ms, nf = prof["fwd"]
    fwd_avg = fwd_ms / max(nf, 1)
    v_bytes = N * H * D + N * H * D // 32
    bytes_fwd = acc["bytes_fwd"] - 2 * N * H * D + v_bytes
    achieved = acc["flops_fwd"] / (fwd_avg * 1e-3) / 1e12
    traffic = load_traffic().get("fwd_mxfp8")
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak_mix, "unit": "TFLOP/s", "frac": achieved / peak_mix,
            "traffic": traffic, "kernel": "jfa_fwd_kernel<D, dense, mxfp8>", "peak_source": peaks["source"],
            "peak_note": "4/3 x bf16 peak: half the FLOPs bf16 (Q K^T), half E4M3 at twice the rate (P V)",
            "algorithmic_per_launch": acc["flops_fwd"], "algorithmic_bytes_per_launch": bytes_fwd}
    # End to end: inputs (Q, K, MXFP8 V and its scales, offsets) from pinned host memory, the forward, the
    # outputs (O, LSE) back to pinned host memory, every step.
    host_in = {"q": x["q"].pin_memory(), "k": x["k"].pin_memory(), "v8": v8.cpu().pin_memory(),
               "vs": vs.cpu().pin_memory(), "off": off_h.pin_memory()}
    dev_in = {n_: torch.empty_like(t_, device=dev) for n_, t_ in host_in.items()}
    host_out = {"o": torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                "lse": torch.empty(lse.shape, dtype=lse.dtype).pin_memory()}
    h2d = sum(t_.numel() * t_.element_size() for t_ in host_in.values())
    d2h = sum(t_.numel() * t_.element_size() for t_ in host_out.values())

    def e2e_step():
        for n_, t_ in host_in.items():
            dev_in[n_].copy_(t_, non_blocking=True)
        mx_step(dev_in["q"], dev_in["k"], dev_in["v8"], dev_in["vs"], dev_in["off"])
        host_out["o"].copy_(o, non_blocking=True)
        host_out["lse"].copy_(lse, non_blocking=True)

    e2e_ms, _ = timed(e2e_step, args.e2e_steps)
    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        nseq, t_cpu = 1, 0.0
        while True:  # grow the sample until the oracle takes a few seconds
            sub = first_sequences(x, nseq)
            r8, rs = oracle.quantize_v_mxfp8(sub["v"], sub["offsets"])
            t0 = time.perf_counter()
            oracle.fwd_mxfp8(sub["q"], sub["k"], r8, rs, sub["offsets"], Lq, bq, causal, x["scale"])
            t_cpu = time.perf_counter() - t0
            if t_cpu > 3.0 or nseq >= B:
                break
            nseq = min(B, nseq * 4)
        cpu = {"value": accounting(sub)["flops_fwd"] / t_cpu / 1e12, "unit": "TFLOPS",
               "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"oracle fwd_mxfp8 on the first {nseq} sequences ({t_cpu:.1f} s)"}
    line = {
        "metric": f"fwd TFLOPS (MXFP8 P V, bf16 Q K^T, 1 GB300) on {args.workload}",
        "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 (P V, E8M0 scales) + bf16 (Q K^T)", "data": "synthetic",
        "config": {"workload": workload_desc(args.workload) + "; forward only, V in MXFP8"
                   + (f"; sequence lengths replaced by {args.lengths}" if args.lengths else ""),
                   "B": B, "Lq": Lq, "H": H, "D": D, "N": N, "pairs": acc["pairs"],
                   "l2": "no flush: Q, K, V inputs exceed the 129 MB L2" if 3 * N * H * D > 129e6 else "no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "bf16_fwd": {"ms_per_step": bf16_ms, "tflops": world * acc["flops_fwd"] / (bf16_ms * 1e-3) / 1e12,
                     "speedup_of_mxfp8": bf16_ms / ms},
        "quantize_v": {"ms": quant_prof["quant_v"][0] / max(quant_prof["quant_v"][1], 1),
                       "algorithmic_bytes": 2 * N * H * D + v_bytes},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": world * acc["flops_fwd"] / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": int(prof["fwd"][1] + prof["fwd_merge"][1]),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="use only the first BATCH sequences (small profiling case; not a bench line)")
    ap.add_argument("--workload", default=WORKLOAD, choices=list(jfa_inputs.WORKLOAD_ORDER),
                    help="synthetic workload (default: the ads fwd+bwd step the headline metric is quoted on)")
    ap.add_argument("--lengths", default=None, metavar="SPEC",
                    help="explicit sequence lengths instead of the workload's recipe, e.g. 131072,512x31 "
                         "(Lq, H, D and mode stay the workload's; a skew case, not a bench line)")
    ap.add_argument("--block-sparse", type=float, default=None, metavar="RATIO",
                    help="block-sparse variant: each (128-key block, head) selected with this probability "
                         "(seeded); also times the dense step on the same inputs (not a bench line)")
    ap.add_argument("--mxfp8", action="store_true",
                    help="MXFP8 variant of the forward (P V in E4M3 with E8M0 scales), forward only, with the bf16 "
                         "forward timed beside it (not the headline line)")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.mxfp8:
        assert args.warmup >= 3, "at least 3 warm-up steps"
        return run_mxfp8(args, world, rank)
    assert args.warmup >= 3, "at least 3 warm-up steps"

    import bwd_jagged_flashattention_gb300 as jfa
    jfa.lib()  # raises if the CUDA library is missing: no fallback
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = make_inputs(args)
    backward = "do" in x
    if args.batch:
        x = first_sequences(x, args.batch)
    sparse = args.block_sparse is not None
    mask_h = None
    if sparse:
        assert not x["causal"], "the block-sparse variant is not defined with causal masking"
        assert 0.0 < args.block_sparse <= 1.0
        mask_h = jfa_inputs.kv_block_mask(x["offsets"], x["H"], args.block_sparse, seed=1)
    acc = accounting_sparse(x, mask_h) if sparse else accounting(x)
    if not backward:
        acc.update(flops_bwd=0.0, bytes_bwd=0, flops_pre=0.0, bytes_pre=0)
    B, Lq, H, D, N = x["B"], x["Lq"], x["H"], x["D"], x["N"]
    bq, causal = x["broadcast_q"], x["causal"]
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    do = x["do"].to(dev) if backward else None
    off_h = x["offsets"]
    off_d = off_h.to(dev)
    o = torch.empty((B, Lq, H, D) if bq else (N, H, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, Lq) if bq else (H, N), dtype=torch.float32, device=dev)
    dq = torch.empty((Lq, H, D) if bq else (N, H, D), dtype=torch.float32, device=dev)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ws = jfa.new_workspace(B, N, Lq if bq else 0, H, D, bq, causal, dev)
    stream = torch.cuda.current_stream(dev)

    bufs0 = dict(q=q, k=k, v=v, do=do, off=off_d, o=o, lse=lse, dq=dq, dk=dk, dv=dv)

    def fwd_pass(b=bufs0):
        if sparse:
            jfa.fwd_block_sparse(b["q"], b["k"], b["v"], b["off"], mask_h, broadcast_q=bq, scale=x["scale"],
                                 offsets_host=off_h, workspace=ws, out=b["o"], lse=b["lse"])
        else:
            jfa.fwd(b["q"], b["k"], b["v"], b["off"], broadcast_q=bq, causal=causal, scale=x["scale"],
                    offsets_host=off_h, workspace=ws, out=b["o"], lse=b["lse"])

    def bwd_pass(b=bufs0):
        if not backward:
            return
        if sparse:
            jfa.bwd_block_sparse(b["q"], b["k"], b["v"], b["o"], b["lse"], b["do"], b["off"], mask_h,
                                 broadcast_q=bq, scale=x["scale"], offsets_host=off_h, workspace=ws, dq=b["dq"],
                                 dk=b["dk"], dv=b["dv"])
        else:
            jfa.bwd(b["q"], b["k"], b["v"], b["o"], b["lse"], b["do"], b["off"], broadcast_q=bq, causal=causal,
                    scale=x["scale"], offsets_host=off_h, workspace=ws, dq=b["dq"], dk=b["dk"], dv=b["dv"])

    def step(b=bufs0):
        fwd_pass(b)
        bwd_pass(b)

    def dense_step():
        jfa.fwd(q, k, v, off_d, broadcast_q=bq, causal=causal, scale=x["scale"], offsets_host=off_h, workspace=ws,
                out=o, lse=lse)
        if backward:
            jfa.bwd(q, k, v, o, lse, do, off_d, broadcast_q=bq, causal=causal, scale=x["scale"], offsets_host=off_h,
                    workspace=ws, dq=dq, dk=dk, dv=dv)

    def timed_steps(n):
        """n steps with events around each pass on the launching stream: (total ms, fwd-pass ms list,
        bwd-pass ms list, host seconds spent issuing the steps)."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_start.record(stream)
        h0 = time.perf_counter()
        for i in range(n):
            evs[i][0].record(stream)
            fwd_pass()
            evs[i][1].record(stream)
            bwd_pass()
            evs[i][2].record(stream)
        host_s = time.perf_counter() - h0
        e_end.record(stream)
        torch.cuda.synchronize()
        return (e_start.elapsed_time(e_end), [e[0].elapsed_time(e[1]) for e in evs],
                [e[1].elapsed_time(e[2]) for e in evs] if backward else [], host_s)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert jfa.device_status(ws) == 0, "kernel status word reports a timeout"

    # The headline region runs without the library's per-kernel events (an event between the
    # Delta pre-pass and the backward kernel would keep the latter from starting early); the
    # per-kernel durations come from a second region of the same K steps with them on.
    sampler = ClockSampler(gpu_smi_id(dev))
    sampler.start()
    for _ in range(3):
        step()
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark(0)
    total_ms, fwd_ms_list, bwd_ms_list, host_s = timed_steps(args.steps)
    sampler.mark(1)
    barrier(world)
    clocks = sampler.stop()
    jfa.profile_enable(True)
    jfa.profile_read()
    prof_total_ms, _, _, _ = timed_steps(args.steps)
    prof = jfa.profile_read()
    jfa.profile_enable(False)
    elapsed_ms = max_over_ranks(world, total_ms, dev)
    ms_per_step = elapsed_ms / args.steps
    step_flops = acc["flops_fwd"] + acc["flops_bwd"]
    value = world * step_flops / (ms_per_step * 1e-3) / 1e12
    assert jfa.device_status(ws) == 0, "kernel status word reports a timeout"
    fwd_pass_ms = statistics.mean(fwd_ms_list)
    bwd_pass_ms = statistics.mean(bwd_ms_list) if backward else None

    # Host-side cost of the schedules the calls above built (the pages call it negligible): the
    # forward and backward tile schedules, built alone on the host.
    P_ctas = jfa.num_ctas()
    host_sched = {}
    for name_, fn_ in (("fwd", lambda: jfa.host_schedule(off_h, Lq if bq else 0, H, bq, causal, False, P_ctas,
                                                          policy=jfa.SCHED_GREEDY)),
                       ("bwd", lambda: jfa.host_schedule(off_h, Lq if bq else 0, H, bq, causal, True, P_ctas,
                                                          policy=jfa.SCHED_ZIGZAG))):
        ts = []
        for _ in range(7):
            t0 = time.perf_counter()
            fn_()
            ts.append(time.perf_counter() - t0)
        host_sched[name_ + "_ms"] = 1e3 * statistics.median(ts)
    host_sched["host_issue_ms_per_step"] = 1e3 * host_s / args.steps
    host_sched["note"] = ("schedules built alone on the host (median of 7); host_issue_ms_per_step = host time to "
                          "issue one whole step (argument checks, schedules, copies, launches), overlapped with "
                          "the GPU's work")

    # Deal-policy ablation (the pages' longest-first sort + zigzag recovered ~20% of the forward):
    # the same step with each way of dealing the sorted items to the CTAs.
    ablation = None
    if not args.batch and world == 1:
        ablation = {}
        n_ab = max(20, min(args.steps, 100))
        for pol_name, fpol, bpol in (("lpt_greedy", jfa.SCHED_GREEDY, jfa.SCHED_GREEDY),
                                     ("lpt_zigzag", jfa.SCHED_ZIGZAG, jfa.SCHED_ZIGZAG),
                                     ("naive_round_robin", jfa.SCHED_NAIVE, jfa.SCHED_NAIVE),
                                     ("cluster_launch_control", jfa.SCHED_GREEDY, jfa.SCHED_CLC),
                                     ("per_head_queue", jfa.SCHED_GREEDY, jfa.SCHED_QUEUE)):
            jfa.set_schedule_policy(fpol, bpol)
            for _ in range(3):
                step()
            _, f_l, b_l, _ = timed_steps(n_ab)
            ablation[pol_name] = {"fwd_ms": statistics.mean(f_l), "bwd_ms": statistics.mean(b_l) if backward else None}
        jfa.set_schedule_policy()  # the library's defaults: greedy forward, zigzag backward
        ablation["note"] = (f"{n_ab} steps per policy, same inputs; the library deals the forward lpt_greedy and "
                            f"the backward lpt_zigzag; cluster_launch_control deals the backward at run time "
                            f"(one CTA per item, resident CTAs taking over those not started), per_head_queue "
                            f"too (one CTA per SM, each taking its head group's next longest item), forward "
                            f"lpt_greedy")

    # Per-kernel live timing -> rooflines.
    peaks = load_peaks()
    traffic = load_traffic()
    kernels = {}
    for name, flops, nbytes in (("fwd", acc["flops_fwd"], acc["bytes_fwd"]),
                                ("bwd_pre", acc["flops_pre"] if backward else 0.0, acc["bytes_pre"] if backward else 0),
                                ("bwd", acc["flops_bwd"], acc["bytes_bwd"]),
                                ("zero_tiles", 0.0, acc.get("bytes_zero", 0) if backward else 0),
                                ("fwd_merge", 0.0, 0)):
        ms, n = prof[name]
        avg = ms / max(n, 1)
        tflops = flops / (avg * 1e-3) / 1e12 if avg > 0 else 0.0
        gbs = nbytes / (avg * 1e-3) / 1e9 if avg > 0 else 0.0
        t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
        t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
        bound = "tensor" if (t_tensor >= t_hbm and name in ("fwd", "bwd")) else "hbm"
        kernels[name] = {"launches": n, "avg_ms": avg, "share": None, "tflops": tflops, "gbs": gbs,
                         "tensor_frac": tflops / peaks["bf16_tflops"], "hbm_frac": gbs / peaks["hbm_gbs"],
                         "model_bound": bound, "algorithmic_flops": flops, "algorithmic_bytes": nbytes,
                         # the committed DRAM counters were taken on the dense kernels
                         "traffic": None if (sparse and name in ("fwd", "bwd")) else traffic.get(name)}
    total_k = sum(k_["avg_ms"] * k_["launches"] for k_ in kernels.values())
    for k_ in kernels.values():
        k_["share"] = k_["avg_ms"] * k_["launches"] / total_k if total_k else None
    dom_name = max(kernels, key=lambda n_: kernels[n_]["avg_ms"] * kernels[n_]["launches"])
    dom = kernels[dom_name]
    if dom["model_bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": dom["tflops"], "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": dom["tflops"] / peaks["bf16_tflops"]}
    else:
        roof = {"bound": "hbm", "achieved": dom["gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": dom["gbs"] / peaks["hbm_gbs"]}
    roof.update(kernel=f"jfa_{dom_name}_kernel", traffic=dom["traffic"], peak_source=peaks["source"],
                algorithmic_per_launch=dom["algorithmic_bytes"] if roof["bound"] == "hbm" else dom["algorithmic_flops"])

    # Host link rates (pinned memory, 256 MiB copies), each direction alone and both at once: the
    # rates the end-to-end line's copies should be read against.
    link = None
    if world == 1:
        nb_ = 256 << 20
        hbuf, hbuf2 = torch.empty(nb_, dtype=torch.uint8).pin_memory(), torch.empty(nb_, dtype=torch.uint8).pin_memory()
        dbuf, dbuf2 = torch.empty(nb_, dtype=torch.uint8, device=dev), torch.empty(nb_, dtype=torch.uint8, device=dev)
        s2 = torch.cuda.Stream(dev)

        def copy_rate(h2d_, d2h_):
            dbuf.copy_(hbuf, non_blocking=True)
            torch.cuda.synchronize()
            ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ea.record(stream)
            s2.wait_stream(stream)
            for _ in range(3):
                if h2d_:
                    dbuf.copy_(hbuf, non_blocking=True)
                if d2h_:
                    with torch.cuda.stream(s2):
                        hbuf2.copy_(dbuf2, non_blocking=True)
            stream.wait_stream(s2)
            eb.record(stream)
            torch.cuda.synchronize()
            return 3 * nb_ * (int(h2d_) + int(d2h_)) / (ea.elapsed_time(eb) * 1e-3) / 1e9

        link = {"h2d_gbs": copy_rate(True, False), "d2h_gbs": copy_rate(False, True),
                "both_gbs": copy_rate(True, True), "how": "3 x 256 MiB pinned copies per direction, CUDA events"}
        del hbuf, hbuf2, dbuf, dbuf2

    # End to end: every step copies its inputs from pinned host memory to the device, runs both
    # passes through the library's API and copies all of its outputs (O, LSE, dQ, dK, dV) back to
    # pinned host memory.  Steps are pipelined the way a streaming caller would: two sets of device
    # buffers, the input copy of step i+1 on one stream and the output copy of step i-1 on another
    # while step i computes, with events ordering every reuse of a buffer.
    in_names = ["q", "k", "v"] + (["do"] if backward else [])
    out_names = ["o", "lse"] + (["dq", "dk", "dv"] if backward else [])
    host_in = {n_: x[n_].pin_memory() for n_ in in_names}
    host_in["off"] = off_h.pin_memory()
    sets = [bufs0, {n_: torch.empty_like(t_) for n_, t_ in bufs0.items() if t_ is not None}]
    host_out = [{n_: torch.empty(bufs0[n_].shape, dtype=bufs0[n_].dtype).pin_memory() for n_ in out_names}
                for _ in range(2)]
    h2d = sum(h.numel() * h.element_size() for h in host_in.values())
    d2h = sum(h.numel() * h.element_size() for h in host_out[0].values())
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_done = [ev(), ev()]      # inputs of set j landed
    comp_done = [ev(), ev()]    # step on set j finished (its inputs free, its outputs ready)
    out_done = [ev(), ev()]     # outputs of set j copied out (set j's output buffers free)
    started = [False, False]

    def e2e_steps(n_steps):
        for i in range(n_steps):
            j = i % 2
            b = sets[j]
            with torch.cuda.stream(s_in):
                if started[j]:
                    s_in.wait_event(comp_done[j])
                for n_ in list(in_names) + ["off"]:
                    b[n_].copy_(host_in[n_], non_blocking=True)
                in_done[j].record(s_in)
            stream.wait_event(in_done[j])
            if started[j]:
                stream.wait_event(out_done[j])
            step(b)
            comp_done[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[j])
                for n_ in out_names:
                    host_out[j][n_].copy_(b[n_], non_blocking=True)
                out_done[j].record(s_out)
            started[j] = True

    e2e_steps(3)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_stream(stream)
    e2e_steps(args.e2e_steps)
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(world, e0.elapsed_time(e1), dev) / args.e2e_steps
    # The pipelined steps computed what a plain step computes: the last one's copied-back
    # outputs against a fresh step on the first buffer set (dQ sums with atomics: tolerance).
    last = host_out[(args.e2e_steps - 1) % 2]
    step()
    torch.cuda.synchronize()
    for n_ in out_names:
        ref = bufs0[n_].cpu()
        if n_ == "dq":
            err = (last[n_].double() - ref.double()).norm() / max(ref.double().norm(), 1e-30)
            assert err <= 1e-4, f"e2e pipeline: dq differs from a plain step (rel {err})"
        else:
            assert torch.equal(last[n_], ref), f"e2e pipeline: {n_} differs from a plain step"
    e2e_value = world * step_flops / (e2e_ms * 1e-3) / 1e12

    # Block-sparse: the dense step on the same inputs, timed the same way, for the speedup.
    sparse_info = None
    if sparse:
        for _ in range(3):
            dense_step()
        torch.cuda.synchronize()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        nd = min(args.steps, 200)
        d0.record(stream)
        for _ in range(nd):
            dense_step()
        d1.record(stream)
        torch.cuda.synchronize()
        dense_ms = max_over_ranks(world, d0.elapsed_time(d1), dev) / nd
        sparse_info = {"ratio": args.block_sparse, "selected_fraction": acc["selected_fraction"],
                       "mask": "jfa_inputs.kv_block_mask(offsets, H, ratio, seed=1): uint8 [NB, H]",
                       "dense_ms_per_step": dense_ms, "speedup_vs_dense": dense_ms / ms_per_step}

    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(x, mask=mask_h) if backward else None
    line = {
        "metric": metric_name(args.workload, backward, args.block_sparse),
        "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": (workload_desc(args.workload) if not args.batch
                                else f"first {B} sequences of: " + workload_desc(args.workload))
                   + (f"; sequence lengths replaced by {args.lengths}" if args.lengths else ""),
                   "B": B, "Lq": Lq, "H": H, "D": D, "N": N, "pairs": acc["pairs"],
                   "l2": (f"no flush: K+V inputs (~{4 * N * H * D / 1e6:.0f} MB) exceed the 129 MB L2"
                          if 4 * N * H * D > 129e6 else
                          f"no flush; K+V inputs (~{4 * N * H * D / 1e6:.0f} MB) fit in the 129 MB L2"),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   **({"block_sparse": sparse_info} if sparse else {})},
        # Each pass timed on the launching stream from its first to its last operation: the forward
        # pass is its kernel (and a split-KV merge when one runs); the backward pass is the dQ memset,
        # the Delta pre-pass and the backward kernel.
        "fwd_ms": fwd_pass_ms, "bwd_ms": bwd_pass_ms,
        "fwd_tflops": acc["flops_fwd"] / (fwd_pass_ms * 1e-3) / 1e12,
        "bwd_tflops": acc["flops_bwd"] / (bwd_pass_ms * 1e-3) / 1e12 if backward else None,
        "tensor_peak_frac": {"fwd": acc["flops_fwd"] / (fwd_pass_ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                             "bwd": (acc["flops_bwd"] / (bwd_pass_ms * 1e-3) / 1e12 / peaks["bf16_tflops"]
                                     if backward else None),
                             "fwd_kernel": kernels["fwd"]["tensor_frac"],
                             "bwd_kernel": kernels["bwd"]["tensor_frac"] if backward else None,
                             "peak_tflops": peaks["bf16_tflops"], "peak_source": peaks["source"]},
        "roofline": roof,
        "kernels": kernels,
        "host_schedule": host_sched,
        "schedule_ablation": ablation,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOPS", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms,
                "pipeline": "double-buffered: H2D of step i+1 and D2H of step i-1 overlap step i (3 streams)",
                "host_link": link,
                "link_floor_ms": (max(h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9),
                                      (h2d + d2h) / (link["both_gbs"] * 1e9)) * 1e3 if link else None)},
        "gpu_launches": int(sum(k_["launches"] for k_ in kernels.values())),
        "kernel_timing": (f"per-kernel CUDA events on the launching stream over a second region of {args.steps} "
                          f"steps right after the headline one ({prof_total_ms / args.steps:.4f} ms per step "
                          f"with the events on)"),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
