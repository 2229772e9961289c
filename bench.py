#!/usr/bin/env python3
"""Benchmark of the chunkwise gated delta rule on one GB300 (or N replicas).

A step is one pass of the whole path over one batch: gdn_fwd (keeping the chunk
boundary states) followed by gdn_bwd, on the training shape B=8, T=4096, H=6,
K=V=128, chunk 64, bf16 inputs with float32 state.  The headline value is
fwd+bwd token*heads per second with every input resident in HBM; the forward
alone is reported beside it.  Inputs (about 200 MB) and workspace exceed the
129 MB L2, so no L2 flush is needed between steps.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun (N > 1) every rank runs its own batch on its own GPU (the (b,h)
streams are independent; no collective on the data path) and rank 0 prints the
whole-job throughput, timed as the max over ranks.

The float64 CPU oracle is timed on a bounded sample of the same workload
(cpu_baseline) and also gates the run: the GPU results on the sampled streams
must match it within the tolerances before anything is timed.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from gated_delta_rule_19_gb300.inputs import WORKLOADS, custom, make_inputs  # noqa: E402

METRIC = "gated-delta fwd & fwd+bwd tokens*heads/s at 1 GB300; % of bf16 TC roofline"
UNIT = "tokens*heads/s"
DEFAULT_WORKLOAD = "train_bf16_B8_T4096_H6_K128_V128"
FALLBACK_PEAKS = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0)


# ----------------------------------------------------------------- arguments

def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode-step, prologue, varlen, sequence-split and per-config lines")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if (args.impl == "gdn" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ oracle (CPU)

def sample_streams(w, n):
    """n (b, h) streams spread over the batch and the heads."""
    all_s = [(b, h) for b in range(w.B) for h in range(w.H)]
    if n >= len(all_s):
        return all_s
    idx = np.linspace(0, len(all_s) - 1, n).round().astype(int)
    return [all_s[i] for i in idx]


def oracle_step(oracle, np_in, streams, threads):
    from_s = lambda x: np.stack([x[b, :, h] for b, h in streams], axis=1)[None]  # noqa: E731
    st = lambda x: None if x is None else np.stack([x[b, h] for b, h in streams])[None]  # noqa
    q, k, v, a, be, do = (from_s(np_in[n]) for n in ("q", "k", "v", "alpha", "beta", "d_o"))
    s0, dsT = st(np_in["initial_state"]), st(np_in["d_final_state"])
    t0 = time.perf_counter()
    o, sT = oracle.gated_delta_fwd(q, k, v, a, be, s0, threads=threads)
    g = oracle.gated_delta_bwd(q, k, v, a, be, s0, do, dsT, threads=threads)
    dt = time.perf_counter() - t0
    return dt, dict(o=o, final_state=sT, **g)


def np_inputs(inp):
    return {n: (t.double().numpy() if t is not None else None) for n, t in inp.items()}


def n_sample_streams(w, threads):
    return max(1, min(w.B * w.H, threads))


def run_reference(args, world, rank):
    """The reference arm: the float64 CPU oracle, timed as it stands on the
    host cores, each step a bounded sample (as many full-length streams as
    there are cores) of the workload."""
    if rank != 0:
        return
    import oracle

    oracle.build()
    w = WORKLOADS[args.workload]
    threads = oracle.threads(0)
    streams = sample_streams(w, n_sample_streams(w, threads))
    np_in = np_inputs(make_inputs(w))
    for _ in range(args.warmup):
        oracle_step(oracle, np_in, streams, threads)
    total = 0.0
    for _ in range(args.steps):
        dt, _ = oracle_step(oracle, np_in, streams, threads)
        total += dt
    units = len(streams) * w.T
    value = units * args.steps / total
    sample = (f"{len(streams)} of {w.B * w.H} (b,h) streams, full T={w.T}, fwd+bwd, "
              "float64 token recurrence")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V,
                   "chunk": w.chunk, "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        uuid = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            pass
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if uuid:
            cmd += ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sms, maxs, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxs.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sms) if sms else None,
                "sm_max_mhz": max(maxs) if maxs else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sms), "reasons": sorted(reasons)}


# ------------------------------------------------------------- roofline

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return dict(hbm_gbs=float(pk["hbm_gbs"]), bf16_tflops=float(pk["bf16_tflops"]),
                    bf16_tflops_sustained=float(pk.get("bf16_tflops_sustained",
                                                       pk["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


def kernel_work(name, w):
    """Algorithmic flops and bytes per token*head of each kernel: the per-unit
    counts of the whole path (fwd flops 2C(3K+2V)+6KV, bwd flops
    14KV+10CV+18CK+4C^2; bytes = the path's own inputs and outputs in the run
    dtype) split by the step each kernel performs."""
    C, K, V = w.chunk, w.K, w.V
    es = 2 if w.dtype == "bf16" else 4
    read_inputs = es * (2 * K + V) + 2 * es
    table = {
        "prep_kernel(fwd)": (6 * C * K + 2 * C * V, read_inputs),
        "prep_fwd_tc": (6 * C * K + 2 * C * V, read_inputs),
        "scan_fwd_tc": (6 * K * V + 2 * C * V, es * V),
        "prep_fwd_tc(bwd)": (6 * C * K + 2 * C * V, read_inputs),
        "scan_fwd_tc(state-only)": (4 * K * V, 0),
        "scan_bwd_tc": (8 * K * V + 2 * C * V, es * V),
        "grad_qk_tc": (6 * K * V + 2 * C * V + 4 * C * K, es * K),
        "grad_wy_tc": (8 * C * K + 4 * C * V + 4 * C * C, es * (K + V) + 2 * es),
        "scan_fwd_kernel": (6 * K * V + 2 * C * V, es * V),
        "prep_kernel(bwd)": (6 * C * K + 2 * C * V, read_inputs),
        "scan_fwd_kernel(state-only)": (4 * K * V, 0),
        "scan_bwd_kernel": (8 * K * V + 2 * C * V, es * V),
        "grad_kernel": (6 * K * V + 6 * C * V + 12 * C * K + 4 * C * C, es * (2 * K + V) + 2 * es),
    }
    return table.get(name, (0, 0))


def path_roofline(w, peaks, ms, fwd_ms):
    """The whole path against its algorithmic bound: per token*head the forward
    does 2C(3K+2V)+6KV flops and moves 2(2K+2V)+4 bytes at bf16 (es(2K+2V)+2es in
    general); the backward 14KV+10CV+18CK+4C^2 flops and es(4K+3V)+4es bytes (reads
    q,k,v,dO,alpha,beta; writes dq,dk,dv,dalpha,dbeta).  The bound time is the larger
    of flops / burst bf16 peak and bytes / HBM copy bandwidth (the step is timed in
    windows of about 10 ms, not in a seconds-long loop, so the burst figure is the
    one that applies)."""
    C, K, V = w.chunk, w.K, w.V
    es = 2 if w.dtype == "bf16" else 4
    f_fwd = 2 * C * (3 * K + 2 * V) + 6 * K * V
    f_bwd = 14 * K * V + 10 * C * V + 18 * C * K + 4 * C * C
    b_fwd = es * (2 * K + 2 * V) + 2 * es
    b_bwd = es * (4 * K + 3 * V) + 4 * es
    n = w.token_heads
    def bound_ms(f, b):
        return 1e3 * max(f * n / (peaks["bf16_tflops"] * 1e12), b * n / (peaks["hbm_gbs"] * 1e9))
    step_ms = bound_ms(f_fwd + f_bwd, b_fwd + b_bwd)
    fwd_bound = bound_ms(f_fwd, b_fwd)
    return {"bound_ms": step_ms, "frac": step_ms / ms, "fwd_bound_ms": fwd_bound,
            "fwd_frac": fwd_bound / fwd_ms if fwd_ms else None,
            "tc_peak_frac": (f_fwd + f_bwd) * n / (ms / 1e3) / (peaks["bf16_tflops"] * 1e12),
            "per_token_head": {"fwd_flops": f_fwd, "bwd_flops": f_bwd, "fwd_bytes": b_fwd, "bwd_bytes": b_bwd}}


def traffic_for(name):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, if
    that summary was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except Exception:
        return None
    ent = t.get("kernels", {}).get(name)
    if not ent or ent.get("source_hash") != source_hash():
        return None
    return ent.get("dram_bytes_per_launch_full_workload")


def source_hash():
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_delta_rule_19_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, fn), "rb") as f:
                h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def roofline(summary, w, peaks):
    """One row per kernel: achieved = its algorithmic flops (or bytes) per launch
    / its average launch time, against the burst bf16 peak (each kernel is timed
    in windows of about 10 ms, not a seconds-long loop) or the HBM copy rate,
    whichever bound is larger for its counts.  traffic_ratio = the DRAM bytes ncu
    counted per launch / the kernel's algorithmic bytes per launch (its own
    inputs and outputs of the path); well above 1 means scratch and re-reads."""
    units = w.token_heads
    rows = []
    for name, (n, ms) in summary.items():
        flops, byts = kernel_work(name, w)
        avg_s = ms / n / 1e3
        t_f = flops * units / (peaks["bf16_tflops"] * 1e12)
        t_b = byts * units / (peaks["hbm_gbs"] * 1e9)
        if t_f >= t_b:
            ach = flops * units / avg_s / 1e12
            row = dict(bound="tensor", achieved=ach, peak=peaks["bf16_tflops"],
                       unit="TFLOP/s")
        else:
            ach = byts * units / avg_s / 1e9
            row = dict(bound="hbm", achieved=ach, peak=peaks["hbm_gbs"], unit="GB/s")
        traffic = traffic_for(name)
        alg_bytes = byts * units
        row.update(frac=row["achieved"] / row["peak"], kernel=name, launches=n,
                   avg_ms=ms / n, share=0.0, traffic=traffic, algorithmic_bytes=alg_bytes,
                   traffic_ratio=(traffic / alg_bytes) if (traffic and alg_bytes) else None,
                   peak_source=peaks["source"] + (" burst bf16" if row["bound"] == "tensor"
                                                  else " hbm copy"))
        rows.append(row)
    tot = sum(r["avg_ms"] * r["launches"] for r in rows) or 1.0
    for r in rows:
        r["share"] = r["avg_ms"] * r["launches"] / tot
    rows.sort(key=lambda r: -r["share"])
    return rows


# ------------------------------------------------------------------ GPU arm

def measure_prologue(gdn, dev, stream, args, world, w):
    """Times the fused prologue (q/k L2 normalisation and gate activations) and its
    backward on the training shape: both are elementwise passes bound by HBM
    traffic, taken against the measured HBM copy rate.  Property check: the
    normalised rows have unit length up to the 1e-6 epsilon."""
    from gated_delta_rule_19_gb300.inputs import make_prologue_inputs

    x = {n: t.to(dev) for n, t in make_prologue_inputs(w.B, w.T, w.H, w.K, w.dtype, seed=w.seed).items()}
    fwd_in = [x[n] for n in ("q_raw", "k_raw", "a_logit", "b_logit")]
    bwd_in = fwd_in + [x[n] for n in ("dq", "dk", "dalpha", "dbeta")]
    out_f = gdn.gdn_prologue_fwd(*fwd_in)
    out_b = gdn.gdn_prologue_bwd(*bwd_in)
    torch.cuda.synchronize(dev)
    norm_err = float((out_f[0].float().norm(dim=-1) - 1).abs().max())

    def timed(fn, n):
        for _ in range(max(3, args.warmup)):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return max_over_ranks(e0.elapsed_time(e1) / n, world, dev)

    n = max(20, args.steps)
    f_ms = timed(lambda: gdn.gdn_prologue_fwd(*fwd_in, out=out_f), n)
    b_ms = timed(lambda: gdn.gdn_prologue_bwd(*bwd_in, out=out_b), n)
    es = 2 if w.dtype == "bf16" else 4
    rows = w.B * w.T * w.H
    fb = rows * (4 * w.K + 4) * es
    bb = rows * (6 * w.K + 6) * es
    hbm = load_peaks()["hbm_gbs"]
    return {"workload": w.name, "fwd_us": f_ms * 1e3, "bwd_us": b_ms * 1e3,
            "fwd_bytes": fb, "bwd_bytes": bb,
            "fwd_GBs": fb / (f_ms / 1e3) / 1e9, "bwd_GBs": bb / (b_ms / 1e3) / 1e9,
            "fwd_frac_of_hbm": fb / (f_ms / 1e3) / 1e9 / hbm, "bwd_frac_of_hbm": bb / (b_ms / 1e3) / 1e9 / hbm,
            "max_unit_norm_error": norm_err}


def measure_raw(gdn, dev, stream, args, world, w):
    """The training step with its prologue on the training shape, two ways, from
    raw q/k rows and gate logits (q_raw, k_raw ~ N(0, 3^2), logits ~ N(0, 2^2)):
    folded into the kernels (gdn_fwd_raw(saved) + gdn_bwd_raw), and as separate
    passes (gdn_prologue_fwd, gdn_fwd(saved), gdn_bwd, gdn_prologue_bwd).  Both
    compute the same function; the check compares their outputs and raw-input
    gradients (relative L2, they differ only in where alpha and beta are
    rounded), and the oracle chain checks both in the tests."""
    from gated_delta_rule_19_gb300.inputs import make_prologue_inputs

    x = {n: t.to(dev) for n, t in make_prologue_inputs(w.B, w.T, w.H, w.K, w.dtype, seed=w.seed).items()}
    r = make_inputs(w)
    v, do = r["v"].to(dev), r["d_o"].to(dev)
    s0 = r["initial_state"].to(dev) if r["initial_state"] is not None else None
    dsT = r["d_final_state"].to(dev) if r["d_final_state"] is not None else None
    raw_in = (x["q_raw"], x["k_raw"], v, x["a_logit"], x["b_logit"], s0)
    p = gdn.make_problem(w.B, w.T, w.H, w.K, w.V, w.chunk, x["q_raw"].dtype)
    sv_raw = torch.empty(gdn.gdn_raw_saved_bytes(p), dtype=torch.uint8, device=dev)
    ws_raw = torch.empty(max(gdn.gdn_raw_fwd_workspace_bytes(p), gdn.gdn_raw_bwd_workspace_bytes(p)),
                         dtype=torch.uint8, device=dev)
    sv = torch.empty(gdn.gdn_saved_bytes(p), dtype=torch.uint8, device=dev)
    ws = torch.empty(max(gdn.gdn_fwd_workspace_bytes(p), gdn.gdn_bwd_workspace_bytes(p)), dtype=torch.uint8,
                     device=dev)
    o1 = torch.empty_like(v)
    g1 = tuple(torch.empty_like(t) for t in (x["q_raw"], x["k_raw"], v, x["a_logit"], x["b_logit"]))

    def folded():
        o, _, _ = gdn.gdn_fwd_raw(*raw_in, chunk=w.chunk, o=o1, final_state=False, saved=sv_raw, workspace=ws_raw)
        return (o,) + gdn.gdn_bwd_raw(*raw_in, do, dsT, saved=sv_raw, chunk=w.chunk, grads=g1,
                                      d_initial_state=False, workspace=ws_raw)[:5]

    pro_f = tuple(torch.empty_like(t) for t in (x["q_raw"], x["k_raw"], x["a_logit"], x["b_logit"]))
    pro_b = tuple(torch.empty_like(t) for t in (x["q_raw"], x["k_raw"], x["a_logit"], x["b_logit"]))
    o2 = torch.empty_like(v)
    g2 = tuple(torch.empty_like(t) for t in (x["q_raw"], x["k_raw"], v, x["a_logit"], x["b_logit"]))

    def separate():
        q, k, al, be = gdn.gdn_prologue_fwd(x["q_raw"], x["k_raw"], x["a_logit"], x["b_logit"], out=pro_f)
        o, _, _ = gdn.gdn_fwd(q, k, v, al, be, s0, chunk=w.chunk, o=o2, final_state=False, saved=sv, workspace=ws)
        dq, dk, dv, da, db, _ = gdn.gdn_bwd(q, k, v, al, be, s0, do, dsT, saved=sv, chunk=w.chunk, grads=g2,
                                            d_initial_state=False, workspace=ws)
        dqr, dkr, dar, dbr = gdn.gdn_prologue_bwd(x["q_raw"], x["k_raw"], x["a_logit"], x["b_logit"], dq, dk, da,
                                                  db, out=pro_b)
        return (o, dqr, dkr, dv, dar, dbr)

    a, b = folded(), separate()
    torch.cuda.synchronize(dev)
    rel = lambda u, t: float((u.float() - t.float()).norm() / t.float().norm())
    names = ("o", "dq_raw", "dk_raw", "dv", "da_logit", "db_logit")
    agree = {n: rel(u, t) for n, u, t in zip(names, a, b)}

    def timed(fn, n):
        for _ in range(max(3, args.warmup)):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return max_over_ranks(e0.elapsed_time(e1) / n, world, dev)

    n = max(20, args.steps)
    f_ms = timed(folded, n)
    s_ms = timed(separate, n)

    def split_of(fn, reps=5):  # the per-kernel split, outside the timed loops
        gdn.gdn_profiler_start(32 * reps + 32)
        for _ in range(reps):
            fn()
        torch.cuda.synchronize(dev)
        gdn.gdn_profiler_stop()
        return {k: round(t / reps * 1e3, 1) for k, (_, t) in gdn.gdn_profiler_summary().items()}

    f_split, s_split = split_of(folded), split_of(separate)
    return {"workload": w.name, "inputs": "raw q/k ~ N(0, 3^2), gate logits ~ N(0, 2^2)",
            "folded": {"step": "gdn_fwd_raw(saved) + gdn_bwd_raw", "ms_per_step": f_ms,
                       "token_heads_per_s": w.token_heads / (f_ms / 1e3), "us_per_step_by_kernel": f_split},
            "separate": {"step": "gdn_prologue_fwd + gdn_fwd(saved) + gdn_bwd + gdn_prologue_bwd",
                         "ms_per_step": s_ms, "token_heads_per_s": w.token_heads / (s_ms / 1e3),
                         "us_per_step_by_kernel": s_split},
            "speedup": s_ms / f_ms, "rel_l2_folded_vs_separate": agree}


def measure_decode(gdn, dev, stream, args, world):
    """Times gdn_decode on the decode workload (256 sequences x 16 heads, one
    token, K=V=128 bf16): its 256 MB fp32 state is read and written once per
    call, so the call is bound by that traffic; achieved bandwidth is taken
    against the measured HBM copy rate.  Before timing, one call is checked
    against the chunked forward (gdn_fwd) on the same token; the oracle checks
    the decode step in the tests."""
    from gated_delta_rule_19_gb300.inputs import DECODE_WORKLOADS

    w = DECODE_WORKLOADS["decode_bf16_B256_T1_H16_K128_V128"]
    inp = make_inputs(w)
    d = {n: (t.to(dev) if t is not None else None) for n, t in inp.items()}
    args_in = [d[n] for n in ("q", "k", "v", "alpha", "beta")]
    state = d["initial_state"].clone()
    o = torch.empty_like(d["v"])
    gdn.gdn_decode(*args_in, state, o=o)
    of, sf, _ = gdn.gdn_fwd(*args_in, d["initial_state"], chunk=w.chunk)
    torch.cuda.synchronize(dev)
    rel = lambda a, b: float((a.float() - b.float()).norm() / b.float().norm())
    consistency = {"o": rel(o, of), "state": rel(state, sf)}
    del of, sf
    for _ in range(max(3, args.warmup)):
        gdn.gdn_decode(*args_in, state, o=o)
    n = max(20, args.steps)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(n):
        gdn.gdn_decode(*args_in, state, o=o)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1) / n, world, dev)
    BH = w.B * w.H
    byts = BH * w.V * w.K * 4 * 2 + BH * w.T * (2 * w.K + 2 * w.V + 2) * 2
    peaks = load_peaks()
    return {"workload": w.name, "us_per_call": ms * 1e3,
            "token_heads_per_s": world * BH * w.T / (ms / 1e3),
            "bytes_per_call": byts, "achieved_GBs": byts / (ms / 1e3) / 1e9,
            "frac_of_hbm": byts / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
            "l2": "state 256 MB > L2 (no flush)", "rel_l2_vs_gdn_fwd": consistency}


def measure_varlen(gdn, dev, stream, args, world, dense_ms, dense_token_heads):
    """Times one training step (gdn_varlen_fwd with saved states + gdn_varlen_bwd)
    on a packed batch with the large training shape's 32768 tokens split into
    sequences of log-uniform lengths in [128, 8192].  Throughput counts the real
    tokens; every sequence starts a new chunk, so the kernels process
    sum(ceil(len / 64) * 64) token rows per head (rows_processed_per_token), and
    each scan walks its own sequence's chunks, so the longest sequence is the
    critical path.  Before timing, the error
    word is checked and one sequence's output is compared with gdn_fwd on that
    sequence alone; the oracle checks the varlen calls in the tests."""
    from gated_delta_rule_19_gb300.inputs import VARLEN_WORKLOADS, make_varlen_inputs, varlen_lengths

    name, spec = next(iter(VARLEN_WORKLOADS.items()))
    lengths = varlen_lengths(spec["total"], spec["lo"], spec["hi"], spec["seed"])
    inp = make_varlen_inputs(lengths, spec["H"], spec["K"], spec["V"], spec["dtype"], seed=spec["seed"])
    d = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in inp.items()}
    S, total, H = len(lengths), spec["total"], spec["H"]
    max_len = max(lengths)
    ins = [d[n] for n in ("q", "k", "v", "alpha", "beta")]
    p = gdn.make_problem(S, max_len, H, spec["K"], spec["V"], 64, d["q"].dtype)
    ws_f = torch.empty(gdn.gdn_varlen_fwd_workspace_bytes(p, total), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(gdn.gdn_varlen_bwd_workspace_bytes(p, total), dtype=torch.uint8, device=dev)
    saved = torch.empty(gdn.gdn_varlen_saved_bytes(p, total), dtype=torch.uint8, device=dev)
    o = torch.empty_like(d["v"])
    sT = torch.empty(S, H, spec["V"], spec["K"], dtype=torch.float32, device=dev)
    grads = tuple(torch.empty_like(t) for t in ins)
    ds0 = torch.empty_like(sT)

    def step(check=False):
        gdn.gdn_varlen_fwd(*ins, d["cu_seqlens"], max_len, None, o=o, final_state=sT, saved=saved,
                           workspace=ws_f, check=check)
        gdn.gdn_varlen_bwd(*ins, d["cu_seqlens"], max_len, None, d["d_o"], None, saved=saved, grads=grads,
                           d_initial_state=ds0, workspace=ws_b, check=check)

    step(check=True)
    s = max(range(S), key=lambda i: lengths[i])
    a, e = int(inp["cu_seqlens"][s]), int(inp["cu_seqlens"][s + 1])
    o1, _, _ = gdn.gdn_fwd(*(t[a:e].unsqueeze(0).clone() for t in ins), None)  # clone: 16-byte aligned
    torch.cuda.synchronize(dev)
    rel = float((o[a:e].float() - o1[0].float()).norm() / o1.float().norm())
    for _ in range(max(3, args.warmup)):
        step()
    n = max(10, args.steps)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1) / n, world, dev)
    gdn.gdn_profiler_start(32 * n + 32)  # the per-kernel split, outside the timed loop
    for _ in range(n):
        step()
    torch.cuda.synchronize(dev)
    gdn.gdn_profiler_stop()
    split = {k: round(t / n * 1e3, 1) for k, (_, t) in gdn.gdn_profiler_summary().items()}
    C = 64
    flat_rows = sum((L + C - 1) // C * C for L in lengths)
    return {"workload": name, "sequences": S, "tokens": total, "max_len": max_len,
            "layout": "flat chunk rows, each sequence starts a chunk",
            "rows_processed_per_token": flat_rows / total, "ms_per_step": ms,
            "token_heads_per_s": world * total * H / (ms / 1e3),
            "dense_same_tokens_token_heads_per_s": world * dense_token_heads / (dense_ms / 1e3),
            "step": "gdn_varlen_fwd(saved) + gdn_varlen_bwd", "us_per_step_by_kernel": split,
            "critical_path": f"the longest sequence's scan: {(max_len + C - 1) // C} chunks",
            "rel_l2_longest_seq_vs_gdn_fwd": rel}


def measure_split(gdn, dev, stream, args, world):
    """Times one training step (gdn_fwd with saved states + gdn_bwd) on a long
    context with few streams (B=1, T=65536, H=4, K=V=128 bf16: 4 streams, 1024
    chunks each) with the within-call sequence split off and automatic.  The
    unsplit scans run 1024 chunks in a row on 32 CTAs; the split cuts each
    stream into pieces that run side by side.  Before timing, the two results are
    compared (they differ by the fp32 rounding of the piece chain only)."""
    w = custom("long_bf16_B1_T65536_H4_K128_V128", B=1, T=65536, H=4, K=128, V=128, chunk=64, dtype="bf16",
               seed=7, init_std=0.1)
    d = {n: (t.to(dev) if t is not None else None) for n, t in make_inputs(w).items()}
    ins = [d[n] for n in ("q", "k", "v", "alpha", "beta")]
    p = gdn.make_problem(w.B, w.T, w.H, w.K, w.V, w.chunk, d["q"].dtype)
    res = {}
    outs = {}
    for name, policy in (("unsplit", 1), ("split", 0)):
        gdn.gdn_set_sequence_split(policy)
        ws_f = torch.empty(gdn.gdn_fwd_workspace_bytes(p), dtype=torch.uint8, device=dev)
        ws_b = torch.empty(gdn.gdn_bwd_workspace_bytes(p), dtype=torch.uint8, device=dev)
        saved = torch.empty(gdn.gdn_saved_bytes(p), dtype=torch.uint8, device=dev)
        o = torch.empty_like(d["v"])
        sT = torch.empty(w.B, w.H, w.V, w.K, dtype=torch.float32, device=dev)
        grads = tuple(torch.empty_like(t) for t in ins)

        def step():
            gdn.gdn_fwd(*ins, d["initial_state"], o=o, final_state=sT, saved=saved, workspace=ws_f)
            gdn.gdn_bwd(*ins, d["initial_state"], d["d_o"], None, saved=saved, grads=grads, workspace=ws_b)

        for _ in range(max(3, args.warmup)):
            step()
        n = max(5, args.steps)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(n):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = max_over_ranks(e0.elapsed_time(e1) / n, world, dev)
        gdn.gdn_profiler_start(64 * n + 64)  # the per-kernel split, outside the timed loop
        for _ in range(n):
            step()
        torch.cuda.synchronize(dev)
        gdn.gdn_profiler_stop()
        split = {k: round(t / n * 1e3, 1) for k, (_, t) in gdn.gdn_profiler_summary().items()}
        res[name] = {"ms_per_step": ms, "token_heads_per_s": world * w.token_heads / (ms / 1e3),
                     "us_per_step_by_kernel": split}
        outs[name] = (o.float().clone(), grads[0].float().clone())
    gdn.gdn_set_sequence_split(0)
    rel = lambda a, b: float((a - b).norm() / b.norm())
    return {"workload": w.name, "step": "gdn_fwd(saved) + gdn_bwd", **res,
            "speedup": res["unsplit"]["ms_per_step"] / res["split"]["ms_per_step"],
            "rel_l2_split_vs_unsplit": {"o": rel(outs["split"][0], outs["unsplit"][0]),
                                        "dq": rel(outs["split"][1], outs["unsplit"][1])}}


def measure_configs(gdn, dev, stream, args, world):
    """Throughput on every workload config at this N: the forward (a streaming
    config runs its calls in sequence, each passing its final state to the next)
    and, where the config trains, gdn_fwd(saved) + gdn_bwd; inputs resident, the
    median of three windows of K steps; fractions against path_roofline's bound."""
    peaks = load_peaks()
    res = {}
    for name, w in WORKLOADS.items():
        inp = make_inputs(w)
        d = {n: (t.to(dev) if t is not None else None) for n, t in inp.items()}
        Tc = w.T // w.calls
        if w.calls > 1 and w.B != 1:
            raise SystemExit(f"{name}: a streaming config runs with B = 1")

        def part(t, i):  # the i-th call's tokens (contiguous: B = 1 when calls > 1)
            return None if t is None else t[:, i * Tc:(i + 1) * Tc]

        p = gdn.make_problem(w.B, Tc, w.H, w.K, w.V, w.chunk, d["q"].dtype)
        ws_f = torch.empty(max(gdn.gdn_fwd_workspace_bytes(p), 1), dtype=torch.uint8, device=dev)
        ws_b = torch.empty(max(gdn.gdn_bwd_workspace_bytes(p), 1), dtype=torch.uint8, device=dev)
        saved = torch.empty(max(gdn.gdn_saved_bytes(p), 1), dtype=torch.uint8, device=dev)
        o = torch.empty_like(d["v"])
        states = [torch.empty(w.B, w.H, w.V, w.K, dtype=torch.float32, device=dev) for _ in range(2)]
        grads = (torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"]),
                 torch.empty_like(d["alpha"]), torch.empty_like(d["beta"]))
        ds0 = torch.empty_like(states[0])

        def fwd():
            s_in = d["initial_state"]
            for i in range(w.calls):
                out_state = states[i & 1]
                gdn.gdn_fwd(part(d["q"], i), part(d["k"], i), part(d["v"], i), part(d["alpha"], i),
                            part(d["beta"], i), s_in, chunk=w.chunk, o=part(o, i), final_state=out_state,
                            workspace=ws_f)
                s_in = out_state

        def train():
            a_in = (d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["initial_state"])
            gdn.gdn_fwd(*a_in, chunk=w.chunk, o=o, final_state=states[0], saved=saved, workspace=ws_f)
            gdn.gdn_bwd(*a_in, d["d_o"], d["d_final_state"], saved=saved, chunk=w.chunk, grads=grads,
                        d_initial_state=ds0, workspace=ws_b)

        def timed(fn):
            for _ in range(3):
                fn()
            wins = []
            for _ in range(3):
                barrier(world)
                torch.cuda.synchronize(dev)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(args.steps):
                    fn()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                wins.append(e0.elapsed_time(e1) / args.steps)
            return max_over_ranks(statistics.median(wins), world, dev)

        fwd_ms = timed(fwd)
        train_ms = timed(train) if (w.backward and w.calls == 1) else None
        rl = path_roofline(w, peaks, train_ms or fwd_ms, fwd_ms)
        entry = {"dtype": w.dtype, "calls": w.calls,
                 "fwd": {"ms_per_step": fwd_ms, "token_heads_per_s": world * w.token_heads / (fwd_ms / 1e3),
                         "frac_of_bound": rl["fwd_frac"]}}
        if train_ms is not None:
            entry["fwd_bwd"] = {"ms_per_step": train_ms,
                                "token_heads_per_s": world * w.token_heads / (train_ms / 1e3),
                                "frac_of_bound": rl["frac"], "tc_peak_frac": rl["tc_peak_frac"]}
        res[name] = entry
        del d, ws_f, ws_b, saved, o, states, grads, ds0
        torch.cuda.empty_cache()
    return res


def run_gdn(args, world, rank, local):
    from gated_delta_rule_19_gb300 import _build, gdn

    _build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    if w.calls != 1 or not w.backward:
        raise SystemExit(f"{w.name} is not a single-call training workload")
    inp_cpu = make_inputs(w.with_(seed=w.seed + 1000 * rank) if rank else w)
    d = {n: (t.to(dev) if t is not None else None) for n, t in inp_cpu.items()}
    p = gdn.make_problem(w.B, w.T, w.H, w.K, w.V, w.chunk, d["q"].dtype)
    ws_f = torch.empty(gdn.gdn_fwd_workspace_bytes(p), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(gdn.gdn_bwd_workspace_bytes(p), dtype=torch.uint8, device=dev)
    saved = torch.empty(gdn.gdn_saved_bytes(p), dtype=torch.uint8, device=dev)
    o = torch.empty_like(d["v"])
    sT = torch.empty(w.B, w.H, w.V, w.K, dtype=torch.float32, device=dev)
    grads = (torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"]),
             torch.empty_like(d["alpha"]), torch.empty_like(d["beta"]))
    ds0 = torch.empty_like(sT)
    args_in = (d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["initial_state"])

    def step():
        gdn.gdn_fwd(*args_in, chunk=w.chunk, o=o, final_state=sT, saved=saved, workspace=ws_f)
        gdn.gdn_bwd(*args_in, d["d_o"], d["d_final_state"], saved=saved, chunk=w.chunk,
                    grads=grads, d_initial_state=ds0, workspace=ws_b)

    def fwd_only():
        gdn.gdn_fwd(*args_in, chunk=w.chunk, o=o, final_state=sT, workspace=ws_f)

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize(dev)

    # correctness gate + cpu baseline (rank 0): the oracle on sampled streams
    cpu = None
    parity = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        threads = oracle.threads(0)
        streams = sample_streams(w, n_sample_streams(w, threads))
        np_in = np_inputs(inp_cpu)
        dt, ref = oracle_step(oracle, np_in, streams, threads)
        dt1, _ = oracle_step(oracle, np_in, streams[:1], 1)  # one stream on one thread
        got = dict(o=o, final_state=sT, dq=grads[0], dk=grads[1], dv=grads[2],
                   dalpha=grads[3], dbeta=grads[4], d_initial_state=ds0)
        parity = {}
        for n, t in got.items():
            x = t.detach().double().cpu().numpy()
            if n in ("final_state", "d_initial_state"):
                x = np.stack([x[b, h] for b, h in streams])[None]
            else:
                x = np.stack([x[b, :, h] for b, h in streams], axis=1)[None]
            r = ref[n]
            parity[n] = float(np.linalg.norm(x - r) / max(np.linalg.norm(r), 1e-300))
        tol = {"o": 2e-2, "final_state": 2e-2}
        bad = {n: e for n, e in parity.items() if not e <= tol.get(n, 3e-2)}
        if bad:
            print(json.dumps({"error": "parity gate failed", "parity": parity}), flush=True)
            raise SystemExit(3)
        cpu = {"value": len(streams) * w.T / dt, "unit": UNIT, "cores": threads,
               "kind": "oracle",
               "sample": f"{len(streams)} of {w.B * w.H} (b,h) streams at full T={w.T}, "
                         f"fwd+bwd float64, {dt:.2f} s",
               "single_thread": {"value": w.T / dt1, "unit": UNIT, "cores": 1,
                                 "sample": f"1 (b,h) stream at full T={w.T}, fwd+bwd float64, {dt1:.2f} s"}}

    # ---- timed region: windows of exactly K fwd+bwd steps, inputs resident in
    # HBM, each bracketed by a barrier and a synchronize; the value is the median
    # window (every window's clock samples fall inside timed work).  The library's
    # per-kernel event timer is off here: its two event records per launch cost
    # about 20 us per step.
    stream = torch.cuda.current_stream(dev)

    def timed_window():
        barrier(world)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / args.steps

    clocks = ClockSampler(dev)
    time.sleep(0.3)
    windows = [timed_window()]
    while sum(windows) * args.steps < 500.0 and len(windows) < 200:  # about 0.5 s of timed steps
        windows.append(timed_window())
    clk = clocks.stop()
    ms = statistics.median(windows)
    ms_max = max_over_ranks(ms, world, dev)
    barrier(world)
    # the per-kernel split: one more window of K steps with the event timer on
    torch.cuda.synchronize(dev)
    gdn.gdn_profiler_start(16 * args.steps + 16)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize(dev)
    gdn.gdn_profiler_stop()
    summary = gdn.gdn_profiler_summary()
    launches = sum(n for n, _ in summary.values())
    barrier(world)

    # ---- forward only
    torch.cuda.synchronize(dev)
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        fwd_only()
    f1.record(stream)
    torch.cuda.synchronize(dev)
    fwd_ms = max_over_ranks(f0.elapsed_time(f1) / args.steps, world, dev)

    # ---- end to end through the public API with host buffers.  Every step copies its
    # inputs from pinned host memory and its results back; uploads run on one copy
    # stream and downloads on another, so that adjacent steps' copies overlap this
    # step's compute (device inputs and outputs are double-buffered).
    e2e = None
    if not args.no_e2e:
        names_in = ("q", "k", "v", "alpha", "beta", "initial_state", "d_o", "d_final_state")
        host_in = {n: inp_cpu[n].pin_memory() for n in names_in if inp_cpu[n] is not None}
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        outs_dev = [o, sT] + list(grads) + [ds0]
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs_dev]
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        dev_in = [{n: torch.empty_like(t, device=dev) for n, t in host_in.items()} for _ in range(2)]
        dev_out = [outs_dev] + [[torch.empty_like(t) for t in outs_dev]]
        up = torch.cuda.Stream(dev)
        down = torch.cuda.Stream(dev)
        done_in = [None, None]   # compute of the step that last used input set j
        done_out = [None, None]  # download of the step that last used output set j

        def e2e_step(n):
            j = n & 1
            din, dout = dev_in[j], dev_out[j]
            fwd_names = ("q", "k", "v", "alpha", "beta", "initial_state")
            with torch.cuda.stream(up):
                if done_in[j] is not None:
                    up.wait_event(done_in[j])
                for nm in fwd_names:
                    if nm in din:
                        din[nm].copy_(host_in[nm], non_blocking=True)
                ev_fwd_in = torch.cuda.Event()
                ev_fwd_in.record(up)
                for nm in ("d_o", "d_final_state"):
                    if nm in din:
                        din[nm].copy_(host_in[nm], non_blocking=True)
                ev_bwd_in = torch.cuda.Event()
                ev_bwd_in.record(up)
            stream.wait_event(ev_fwd_in)
            if done_out[j] is not None:
                stream.wait_event(done_out[j])
            a_in = (din["q"], din["k"], din["v"], din["alpha"], din["beta"], din.get("initial_state"))
            gdn.gdn_fwd(*a_in, chunk=w.chunk, o=dout[0], final_state=dout[1], saved=saved, workspace=ws_f)
            ev_fwd = torch.cuda.Event()
            ev_fwd.record(stream)
            stream.wait_event(ev_bwd_in)
            gdn.gdn_bwd(*a_in, din["d_o"], din.get("d_final_state"), saved=saved, chunk=w.chunk,
                        grads=tuple(dout[2:7]), d_initial_state=dout[7], workspace=ws_b)
            ev_bwd = torch.cuda.Event()
            ev_bwd.record(stream)
            done_in[j] = ev_bwd
            with torch.cuda.stream(down):
                down.wait_event(ev_fwd)
                for src, dst in zip(dout[:2], host_out[:2]):
                    dst.copy_(src, non_blocking=True)
                down.wait_event(ev_bwd)
                for src, dst in zip(dout[2:], host_out[2:]):
                    dst.copy_(src, non_blocking=True)
                ev_out = torch.cuda.Event()
                ev_out.record(down)
            done_out[j] = ev_out

        for n in range(2):
            e2e_step(n)
        torch.cuda.synchronize(dev)
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        up.wait_event(g0)
        down.wait_event(g0)
        for n in range(args.steps):
            e2e_step(n)
        stream.wait_stream(up)
        stream.wait_stream(down)
        g1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(g0.elapsed_time(g1) / args.steps, world, dev)
        # every step's results arrived: compare the last step's with the resident run's
        ok_e2e = all(torch.equal(hst, dv.cpu()) for hst, dv in zip(host_out, outs_dev))
        e2e = {"value": world * w.token_heads / (e2e_ms / 1e3), "unit": UNIT,
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "pipeline": "uploads and downloads on two copy streams overlap adjacent steps' compute",
               "results_match_resident_run": ok_e2e}

    # ---- the decode step: one token per call, the state
    # carried in place between calls
    decode = None if args.no_decode else measure_decode(gdn, dev, stream, args, world)
    prologue = None if args.no_decode else measure_prologue(gdn, dev, stream, args, world, w)
    raw = None if args.no_decode else measure_raw(gdn, dev, stream, args, world, w)
    varlen = None if args.no_decode else measure_varlen(gdn, dev, stream, args, world, ms_max, w.token_heads)
    split = None if args.no_decode else measure_split(gdn, dev, stream, args, world)
    configs = None if args.no_decode else measure_configs(gdn, dev, stream, args, world)

    if rank != 0:
        return
    peaks = load_peaks()
    rows = roofline(summary, w, peaks)
    dom = rows[0]
    rl = {k: dom[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    rl.update(kernel=dom["kernel"], avg_ms=dom["avg_ms"], share=dom["share"],
              peak_source=dom["peak_source"], traffic_ratio=dom["traffic_ratio"])
    # the whole step's DRAM traffic (ncu, summed over its kernels) against the
    # bytes the path itself must move
    tr = [r["traffic"] for r in rows]
    pr_step = path_roofline(w, peaks, ms_max, fwd_ms)
    alg_step = (pr_step["per_token_head"]["fwd_bytes"] + pr_step["per_token_head"]["bwd_bytes"]) * w.token_heads
    step_traffic = sum(tr) if tr and all(t is not None for t in tr) else None
    pr_step["traffic"] = step_traffic
    pr_step["algorithmic_bytes"] = alg_step
    pr_step["traffic_ratio"] = (step_traffic / alg_step) if step_traffic else None
    value = world * w.token_heads / (ms_max / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "timing": {"windows": len(windows), "steps_per_window": args.steps, "value_from": "median window",
                   "ms_per_step_min": min(windows), "ms_per_step_max": max(windows),
                   "kernel_timer": "off in the timed windows; per-kernel split from one extra window"},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
        if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V,
                   "chunk": w.chunk, "state": "f32", "step": "gdn_fwd(saved) + gdn_bwd",
                   "l2": "inputs and workspace larger than L2 (no flush)",
                   "parallelism": f"replicas x{world}"},
        "fwd": {"value": world * w.token_heads / (fwd_ms / 1e3), "unit": UNIT,
                "ms_per_step": fwd_ms},
        "roofline": rl,
        "path_roofline": pr_step,
        "kernels": [{k: r[k] for k in ("kernel", "launches", "avg_ms", "share", "bound",
                                       "achieved", "unit", "frac", "traffic", "traffic_ratio")} for r in rows],
        "cpu_baseline": cpu,
        "parity_sampled": parity,
        "e2e": e2e,
        "decode": decode,
        "prologue": prologue,
        "prologue_folded": raw,
        "varlen": varlen,
        "sequence_split": split,
        "configs": configs,
        "gpu_launches": launches,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gdn(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
