#!/usr/bin/env python
"""Benchmark: chunked gated delta rule forward + backward on one GB300 per rank.

One step = gdn_chunk_fwd + gdn_chunk_bwd over the training-shape workload
(B=8, T=4096, H=6, Dk=Dv=128, bf16 inputs, fp32 state), inputs resident in HBM.
Prints ONE JSON line (rank 0). Under torchrun every rank runs its own replica
(weak scaling; the layer shards over (batch, head) with no exchange), timing
takes the max over ranks and `value` is the whole job's tokens/s.

--impl reference times the float64 CPU oracle (the only other implementation of
this method available here) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN fwd+bwd tokens/s at B8 T4096 H6 D128 bf16; % tensor peak; decode HBM GB/s"
WORKLOAD = "train_fwdbwd"
L2_BYTES = 129 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="skip decode, e2e and cpu baseline legs")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the batch size (small profiling cases only; the JSON line says so)")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed helpers
def dist_setup():
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest x over all ranks (the slowest rank's time bounds the job)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, ms_max: float) -> float:
    """Whole-job throughput: the tokens every rank processed over the slowest rank's time."""
    return world * tokens_per_rank / (ms_max / 1e3)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        for r in csv.reader(io.StringIO(open(self.path).read())):
            r = [x.strip() for x in r]
            if len(r) >= 9:
                rows.append(r)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1])]
        smax = [num(r[2]) for r in rows if num(r[2])]
        under_load = [s for s in sm if s and s > 0.5 * (max(smax) if smax else 1)] or sm
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for i, n in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(under_load) if under_load else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ------------------------------------------------------------------ roofline tables
def method_work(B, T, H, D, es=2):
    """The method's own work per fwd+bwd step, independent of this implementation.

    Bytes: every input read once and every output written once, forward (q, k, v,
    g, beta, h0 -> out, h_final) and backward (q, k, v, g, beta, dout, dh_final ->
    dq, dk, dv, dg, dbeta, dh0): the minimum. Plus the chunk-start states kept
    between the passes in fp32, written once and read once (one [Dk, Dv] state per
    64-token chunk and head): the plan's figure with residual states. FLOPs: the
    chunked form's dense products at Dk = Dv = 128, about 10 MFLOP forward and 21
    backward per 64-token chunk-head (2 FLOP per multiply-add), 31 MFLOP in all:
    95 GFLOP at B8 T4096 H6."""
    tok = B * T * H  # head-tokens
    io = tok * D * es  # one [B,T,H,D] tensor
    gate = tok * es    # one [B,T,H] tensor
    state = B * H * D * D * 4
    fwd = 4 * io + gate + state + io + state
    bwd = 4 * io + gate + io + state + 4 * io + gate + state
    chunks = B * H * (T // 64)
    states = 2 * chunks * D * D * 4
    flops = chunks * 31.0e6 if D == 128 else None
    return {"min_bytes": fwd + bwd, "bytes_with_states": fwd + bwd + states, "flops": flops}


def kernel_work(B, T, H, D, es=2):
    """Record bytes and tensor FLOPs per launch of each chunk-path kernel.

    Bytes are what this implementation's kernels move by their own contract: the
    inputs and inter-kernel records each reads once and writes once, per 64-token
    chunk and head, times the chunk-heads of one launch. They describe how close a
    kernel runs to HBM speed on its own traffic, not the method's minimum (see
    method_work). FLOPs are each kernel's dense products (2 per MAC)."""
    C = 64
    n = B * H * (T // C)
    CD, CC, DD = C * D * es, C * C * es, D * D * es
    gam = D * 4
    per = {
        # reads q, k, v, g, beta; writes scale*Aqk, T, -W, U', scale*Q-hat, K-tilde, gam
        "chunk_prep_kernel": (4 * CD + C * es + 2 * CC + 4 * CD + gam,
                              2 * C * C * D * 2 + 2 * C * C * D * 2),
        # reads -W, K-tilde, U', gam; writes the chunk-start state and U
        "chunk_scan_fwd_kernel": (3 * CD + gam + DD + CD, 2 * C * D * D * 2),
        # reads scale*Q-hat, scale*Aqk, state, U; writes out
        "chunk_out_kernel": (CD + CC + DD + CD + CD, C * D * D * 2 + C * C * D * 2),
        # reads dout, scale*Aqk, K-tilde, scale*Q-hat, -W, gam; writes dU, dS
        "chunk_scan_bwd_kernel": (CD + CC + 3 * CD + gam + CD + DD, C * C * D * 2 + 3 * C * D * D * 2),
        # reads dout, U, state; writes dQ-hat, dAqk (beside the reverse scan, on a second stream)
        "chunk_dqa_kernel": (2 * CD + DD + CD + CC, C * C * D * 2 + C * D * D * 2),
        # reads T, v, U, dU, state, dS, beta; writes dv, dBk, dK-tilde, dAkk, dgam, dbeta_v
        "chunk_dstate_kernel": (CC + 3 * CD + 2 * DD + C * es + 3 * CD + CC + gam + C * 4,
                                2 * C * C * D * 2 + 2 * C * D * D * 2),
        # reads q, k, g, beta, dQ-hat, dBk, dK-tilde, dAqk, dAkk, dgam; writes dq, dk, dg and partials
        "chunk_grads_kernel": (3 * CD + C * es + 3 * CD + 2 * CC + gam + 3 * CD + 2 * 2 * C * 4,
                               4 * C * C * D * 2),
        "chunk_bwd_finalize_kernel": (C * 4 + 2 * 2 * C * 4 + C * es, 0),
        # fused chunk gradients on tcgen05: reads T, dU, U, state, dS, dout, q, k, v, g, beta;
        # writes dq, dk, dv, dg, dbeta (no intermediate records)
        "chunk_bwd_tc_kernel": (CC + 3 * CD + 2 * DD + CD + 4 * CD + C * es + 4 * CD + C * es,
                                2 * D * C * C + 2 * 2 * C * D * D + 2 * D * D * 2 * C + 2 * D * C * D
                                + 2 * D * 2 * C * C + 2 * D * C * 2 * C),
    }
    # the tensor-core kernels keep the record contracts of the CUDA-core ones they replace
    per["chunk_prep_tc_kernel"] = per["chunk_prep_kernel"]
    per["chunk_scan_fwd_tc_kernel"] = per["chunk_scan_fwd_kernel"]
    per["chunk_scan_bwd_tc_kernel"] = per["chunk_scan_bwd_kernel"]
    out = {k: (b * n, f * n) for k, (b, f) in per.items()}
    # zeroes the single backward launch's counters: one 128-byte line per (batch, head) + one
    out["chunk_bwd_sync_zero_kernel"] = (B * H * 128 + 128, 0)
    return out


# the files the chunk kernels (the ones profiles/traffic.json covers) are compiled from
CHUNK_KERNEL_SOURCES = ("chunk_fwd.cu", "chunk_bwd.cu", "chunk_grads.cu", "chunk_scan_tc.cu",
                        "chunk_prep_tc.cu", "chunk_bwd_tc.cu", "chunk_prep.cuh", "chunk_dqa.cuh",
                        "chunk_out.cuh", "chunk_scan_tc.cuh", "common.cuh", "umma.cuh", "kernels.h")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_deltanet_gdn_gb300", "csrc")
    for f in CHUNK_KERNEL_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def load_traffic():
    """Per-launch DRAM bytes from the committed ncu capture, if the kernels are unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return {}
    d = json.load(open(p))
    if d.get("source_hash") != kernel_source_hash():
        return {}
    return d.get("per_launch_bytes", {})


# ------------------------------------------------------------------ the gdn arm
def run_gdn(args, world, rank, local):
    import torch

    import gated_deltanet_gdn_gb300 as gdn
    from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs

    gdn.load(build_if_needed=True)
    dev = torch.device("cuda", local)
    w = WORKLOADS[WORKLOAD]
    if args.batch:
        w = w.with_(B=args.batch)
    host = make_inputs(w)
    d = {k: (None if v is None else v.to(dev)) for k, v in host.items()}
    dims = gdn.make_dims(d["q"], d["v"], d["g"])
    res = torch.empty(gdn.gdn_chunk_residual_bytes(dims), dtype=torch.uint8, device=dev)
    ws = torch.empty(gdn.gdn_chunk_bwd_workspace_bytes(dims), dtype=torch.uint8, device=dev)
    out = torch.empty_like(d["v"])
    hT = torch.empty((w.B, w.H, w.Dk, w.Dv), dtype=torch.float32, device=dev)
    grads = {"dq": torch.empty_like(d["q"]), "dk": torch.empty_like(d["k"]), "dv": torch.empty_like(d["v"]),
             "dg": torch.empty_like(d["g"]), "dbeta": torch.empty_like(d["beta"]),
             "dh0": torch.empty_like(hT)}

    def step(src=d, dst=None):
        o = dst if dst is not None else dict(grads, out=out, h_final=hT)
        gdn.gdn_chunk_fwd(src["q"], src["k"], src["v"], src["g"], src["beta"], src["h0"], out=o["out"],
                          h_final=o["h_final"], residuals=res)
        gdn.gdn_chunk_bwd(src["q"], src["k"], src["v"], src["g"], src["beta"], src["h0"], res, src["dout"],
                          src["dh_final"], workspace=ws,
                          grads={k: o[k] for k in ("dq", "dk", "dv", "dg", "dbeta", "dh0")})

    # gate (before any timing): every result finite, and on rank 0 the sampled (batch, head)
    # pairs of the CPU-baseline leg, whose float64 oracle forward and reverse pass that leg
    # computes, agree with this step's out, h_final and gradients within the bf16 tolerance
    step()
    torch.cuda.synchronize()
    finite = all(bool(torch.isfinite(t.float()).all()) for t in list(grads.values()) + [out, hT])
    gate = {"finite": finite}
    baseline = None
    if rank == 0:
        baseline, ref = cpu_baseline(w, host)
        gate.update(oracle_gate(ref, dict(grads, out=out, h_final=hT)))
    barrier(world)
    if not (finite and gate.get("passed", True)):
        raise SystemExit(f"correctness gate failed: {json.dumps(gate)}")

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        barrier(world)
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(ms, world)
    tokens = w.B * w.T
    value = job_tokens_per_s(world, tokens, ms_max)

    # forward alone and backward alone (the backward re-reads one forward's residuals)
    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        for _ in range(n):
            fn()
        a1.record()
        torch.cuda.synchronize()
        return a0.elapsed_time(a1) / n

    def fwd_only():
        gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], out=out, h_final=hT, residuals=res)

    def bwd_only():
        gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], res, d["dout"], d["dh_final"],
                          workspace=ws, grads={k: grads[k] for k in ("dq", "dk", "dv", "dg", "dbeta", "dh0")})

    split_n = min(args.steps, 200)
    split = {"fwd_ms": round(timed(fwd_only, split_n), 4), "bwd_ms": round(timed(bwd_only, split_n), 4),
             "steps": split_n}

    # per-kernel launch durations: events on the launch stream around every kernel
    prof_steps = min(args.steps, 50)
    gdn.gdn_profile_enable(True)
    for _ in range(prof_steps):
        step()
    prof = gdn.gdn_profile_read()
    gdn.gdn_profile_enable(False)
    total = sum(v[0] for v in prof.values()) or 1.0
    work = kernel_work(w.B, w.T, w.H, w.Dk)
    if "chunk_scan_fwd_tc_kernel" in prof and "chunk_out_kernel" not in prof:
        # the forward scan's launch also formed the chunk outputs (output CTAs beside it)
        work["chunk_scan_fwd_tc_kernel"] = tuple(
            x + y for x, y in zip(work["chunk_scan_fwd_tc_kernel"], work["chunk_out_kernel"]))
    if "chunk_bwd_tc_kernel" in prof and "chunk_scan_bwd_tc_kernel" not in prof:
        # the gradient launch also ran the reverse scan (scan CTAs beside the gradient CTAs)
        work["chunk_bwd_tc_kernel"] = tuple(
            x + y for x, y in zip(work["chunk_bwd_tc_kernel"], work["chunk_scan_bwd_tc_kernel"]))
    peaks = load_peaks()
    traffic = load_traffic()
    kernels = {}
    for name, (tms, nl) in prof.items():
        avg = tms / nl
        b, f = work.get(name, (None, None))
        kernels[name] = {"launches_per_step": nl // prof_steps, "avg_ms": round(avg, 4),
                         "share": round(tms / total, 4)}
        if b:
            kernels[name]["gbs"] = round(b / (avg / 1e3) / 1e9, 1)
            kernels[name]["tflops"] = round(f / (avg / 1e3) / 1e12, 2)
    dom = max(prof, key=lambda k: prof[k][0])
    b, f = work.get(dom, (0, 0))
    avg = prof[dom][0] / prof[dom][1]
    # The roofline of the whole pass (the chunked fwd + bwd is HBM-bound as a whole): the
    # method's bytes per step with fp32 chunk-start states between the passes, over the
    # measured step time, against the measured HBM copy bandwidth. traffic: the DRAM bytes
    # of one step summed over its kernels from the committed ncu capture (null if the
    # kernels changed since).
    mw = method_work(w.B, w.T, w.H, w.Dk)
    step_s = ms / 1e3
    achieved = mw["bytes_with_states"] / step_s / 1e9
    ran = {k: prof[k][1] // prof_steps for k in prof if k in work}
    step_traffic = None
    if traffic and all(k in traffic for k in ran):
        step_traffic = int(sum(traffic[k] * n for k, n in ran.items()))
    roofline = {"bound": "hbm", "kernel": "whole fwd+bwd step (%d kernel launches)" % sum(ran.values()),
                "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": step_traffic,
                "method_bytes": mw["bytes_with_states"], "method_bytes_min": mw["min_bytes"],
                "frac_min_bytes": round(mw["min_bytes"] / step_s / 1e9 / peaks["hbm_gbs"], 4),
                "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)" if peaks["source"] == "measured"
                else peaks["source"],
                "dominant_kernel": {"name": dom, "avg_ms": round(avg, 4), "record_bytes": b,
                                    "record_gbs": round(b / (avg / 1e3) / 1e9, 1),
                                    "frac": round(b / (avg / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                                    "traffic": traffic.get(dom)}}
    tensor = {"method_flops": mw["flops"], "step_tflops": round(mw["flops"] / step_s / 1e12, 2),
              "frac_of_burst_bf16": round(mw["flops"] / step_s / 1e12 / peaks["bf16_tflops"], 4),
              "frac_of_sustained_bf16": round(mw["flops"] / step_s / 1e12 / peaks["bf16_tflops_sustained"], 4)}
    # this implementation's own record traffic, summed over the kernels that ran
    bytes_step = sum(work[k][0] * n for k, n in ran.items())
    hbm = {"step_record_bytes": int(bytes_step), "step_gbs": round(bytes_step / step_s / 1e9, 1),
           "frac_of_measured": round(bytes_step / step_s / 1e9 / peaks["hbm_gbs"], 4),
           "record_bytes_over_method_bytes": round(bytes_step / mw["bytes_with_states"], 3)}

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "chunked fwd+bwd, B%d T4096 H6 Dk=Dv=128, bf16 inputs / fp32 state, "
                               "per-channel decay, chunk 64" % w.B,
                   "B": w.B, "T": w.T, "H": w.H, "Dk": w.Dk, "Dv": w.Dv, "tokens_per_step_per_gpu": tokens,
                   "l2": "inputs larger than L2 (q,k,v,g,dout %.0f MB + residuals %.0f MB > 129 MB)" % (
                       5 * d["q"].numel() * 2 / 1e6, res.numel() / 1e6),
                   "parallelism": f"replicas x{world} (no collective)"},
        "gpu_launches": sum(ran.values()) * args.steps,
        "roofline": roofline,
        "tensor": tensor,
        "hbm_whole_step": hbm,
        "kernels": kernels,
        "fwd_bwd_split": split,
        "clocks": clk.summary(),
        "correctness_gate": gate,
        "variants": variants_leg(args, w, host, dev),
    }
    if not args.no_extras:
        outputs = dict(grads, out=out, h_final=hT)
        result["e2e"] = e2e_leg(args, host, d, step, outputs, world)
        if rank == 0:
            result["decode"] = decode_leg(dev)
        if rank == 0 and world == 1:
            result["cpu_baseline"] = baseline
    if rank == 0:
        print(json.dumps(result), flush=True)


def variants_leg(args, w, host, dev):
    """The same fwd+bwd step for the input variants the library also supports: q/k
    L2-normalised in the library (GDN_FLAG_QK_L2NORM, raw q and k of norm ~ sqrt(Dk)), one
    scalar decay per head (g [B,T,H]), fp32 operands (the CUDA-core kernel chain), and the
    long-context shape B1 T32768 H16 (16 scan chains of 512 chunks). CUDA events around N
    steps each."""
    import torch

    import gated_deltanet_gdn_gb300 as gdn
    from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs

    res = {}
    n = max(3, min(100, args.steps))
    for name, wv, flags in (("qk_l2norm", w.with_(normalize_qk=False), gdn.GDN_FLAG_QK_L2NORM),
                            ("scalar_decay", w.with_(g_per_channel=False, g_kind="logsigmoid", g_mu=2.0), 0),
                            ("fp32", w.with_(dtype="f32"), 0),
                            ("long_context", WORKLOADS["long_context"], 0)):
        d = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(wv).items()}
        dims = gdn.make_dims(d["q"], d["v"], d["g"], flags)
        res_buf = torch.empty(gdn.gdn_chunk_residual_bytes(dims), dtype=torch.uint8, device=dev)
        ws = torch.empty(gdn.gdn_chunk_bwd_workspace_bytes(dims), dtype=torch.uint8, device=dev)

        def step():
            gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], residuals=res_buf, flags=flags)
            gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], res_buf, d["dout"],
                              d["dh_final"], workspace=ws, flags=flags)

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            step()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        res[name] = {"ms_per_step": round(ms, 4), "tokens_per_s": round(wv.B * wv.T / (ms / 1e3), 1), "steps": n,
                     "workload": "B%d T%d H%d D%d %s, %s" % (
                         wv.B, wv.T, wv.H, wv.Dk, wv.dtype,
                         "raw q/k normalised in the library" if flags else
                         "fp32 operands" if name == "fp32" else
                         "long context, per-channel decay -softplus(N(-1,1)), nonzero h0" if name == "long_context"
                         else "scalar decay logsigmoid(N(2,1)) per head")}
        del d, res_buf, ws
    res["chunk128_forward"] = chunk128_leg(args, w, host, dev)
    return res


def chunk128_leg(args, w, host, dev):
    """The forward alone, and forward + backward, on the headline inputs with 64-token
    chunks (the step) and with 128-token chunks (GDN_FLAG_CHUNK128: the 64-token blocks'
    records from the same preparation, merged, then the CUDA-core scan and outputs over
    128-token chunks; the backward's reverse scan over 128-token chunks, the 64-token
    blocks' records across each block boundary, then the 64-token chunk gradients). CUDA
    events around N calls each, the per-kernel split of the 128-token forward and backward
    from the library's launch events, and the forward's bytes against HBM: q, k, v, g,
    beta and h0 read, out and h_final written, plus the chunk-start states (bf16, one per
    128-token chunk) written once."""
    import torch

    import gated_deltanet_gdn_gb300 as gdn

    d = {k: (None if v is None else v.to(dev)) for k, v in host.items()}
    n = max(3, min(100, args.steps))
    out = {}
    for name, flags in (("chunk64", 0), ("chunk128", gdn.GDN_FLAG_CHUNK128)):
        dims = gdn.make_dims(d["q"], d["v"], d["g"], flags)
        rbuf = torch.empty(gdn.gdn_chunk_residual_bytes(dims), dtype=torch.uint8, device=dev)

        def fwd():
            return gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], residuals=rbuf,
                                     flags=flags)

        for _ in range(3):
            fwd()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fwd()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        out[name] = {"ms": round(ms, 4), "tokens_per_s": round(w.B * w.T / (ms / 1e3), 1)}
        if flags:
            gdn.gdn_profile_enable(True)
            for _ in range(n):
                fwd()
            prof = gdn.gdn_profile_read()
            gdn.gdn_profile_enable(False)
            out[name]["kernels_ms"] = {k: round(v[0] / max(1, v[1]), 4) for k, v in prof.items()}
            BTH, D = w.B * w.T * w.H, w.Dk
            fwd_bytes = BTH * (4 * D * 2 + 2) + 2 * w.B * w.H * D * D * 4 + BTH * D * 2 \
                + (w.T // 128) * w.B * w.H * D * D * 2
            peaks = load_peaks()
            gbs = fwd_bytes / (ms / 1e3) / 1e9
            out[name]["roofline"] = {"bound": "hbm", "method_bytes": int(fwd_bytes), "achieved": round(gbs, 1),
                                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                     "frac": round(gbs / peaks["hbm_gbs"], 4)}
        ws = torch.empty(gdn.gdn_chunk_bwd_workspace_bytes(dims), dtype=torch.uint8, device=dev)

        def step():
            fwd()
            gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], rbuf, d["dout"],
                              d["dh_final"], workspace=ws, flags=flags)

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n):
            step()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        out[name]["fwd_bwd_ms"] = round(ms, 4)
        out[name]["fwd_bwd_tokens_per_s"] = round(w.B * w.T / (ms / 1e3), 1)
        if flags:
            gdn.gdn_profile_enable(True)
            for _ in range(n):
                step()
            prof = gdn.gdn_profile_read()
            gdn.gdn_profile_enable(False)
            out[name]["fwd_bwd_kernels_ms"] = {k: round(v[0] / n, 4) for k, v in prof.items()}
        del rbuf, ws
    out["workload"] = "forward, and forward + backward, B%d T%d H%d D%d bf16, per-channel decay" % (
        w.B, w.T, w.H, w.Dk)
    return out


def e2e_leg(args, host, d, step, outputs, world):
    """The same step through the public API with HOST buffers: each step copies its
    inputs host->device from pinned memory, runs forward + backward, and reads the
    output, final state and every gradient back into pinned host memory. As a data
    loader would, the copies run on their own streams (inputs on one, results on
    another) and overlap the neighbouring steps' compute: device inputs and outputs
    are double-buffered, and CUDA events order each copy against the compute that
    produces or consumes its buffer."""
    import torch

    dev = d["q"].device
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    pin_in = {k: v.pin_memory() for k, v in host.items() if v is not None}
    dev_in = [{k: (torch.empty_like(pin_in[k], device=dev) if k in pin_in else None) for k in host}
              for _ in range(2)]
    dev_out = [outputs] + [{k: torch.empty_like(t) for k, t in outputs.items()}]
    pin_out = {k: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for k, t in outputs.items()}
    h2d = sum(v.numel() * v.element_size() for v in pin_in.values())
    d2h = sum(v.numel() * v.element_size() for v in pin_out.values())
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def full_step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(done[b])  # the compute that read this input set has finished
            for k, v in pin_in.items():
                dev_in[b][k].copy_(v, non_blocking=True)
            in_ready[b].record(s_in)
        comp.wait_event(in_ready[b])
        if used[b]:
            comp.wait_event(out_read[b])  # this output set has been read back
        step(dev_in[b], dev_out[b])
        done[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[b])
            for k, v in pin_out.items():
                v.copy_(dev_out[b][k], non_blocking=True)
            out_read[b].record(s_out)
        used[b] = True

    for i in range(2):
        full_step(i)
    torch.cuda.synchronize()
    n = max(3, min(50, args.steps // 2))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(s_in)
    for i in range(n):
        full_step(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1) / n, world)
    # the same copies with no compute: the host link's share of the step
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e2.record(s_in)
    s_out.wait_event(e2)
    for i in range(n):
        b = i % 2
        with torch.cuda.stream(s_in):
            for k, v in pin_in.items():
                dev_in[b][k].copy_(v, non_blocking=True)
        with torch.cuda.stream(s_out):
            for k, v in pin_out.items():
                v.copy_(dev_out[b][k], non_blocking=True)
    s_in.wait_stream(s_out)
    e3.record(s_in)
    torch.cuda.synchronize()
    copy_ms = e2.elapsed_time(e3) / n
    tokens = host["q"].shape[0] * host["q"].shape[1]
    return {"value": round(world * tokens / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "copies_only_ms_per_step": round(copy_ms, 4),
            "link_gbs_per_direction": round(max(h2d, d2h) / (copy_ms / 1e3) / 1e9, 1),
            "overlap": "inputs and results copied on their own streams, double-buffered against compute"}


def decode_leg(dev):
    """Recurrent kernel: decode steps (T = 1) with the state read and written once.
    B2 H48: L2 flushed before every step (a buffer twice the L2 size is read), the
    kernel timed alone by the library's per-launch events, queued behind a spin
    kernel so that no host launch gap falls inside the measurement. B32 H48 (state
    201 MB > L2): 30 steps back to back between two CUDA events, all queued behind a
    spin kernel first. Then replay decode on the B32 batch and the 2048-token prefill
    of the same geometry, token-recurrent and through the chunked forward."""
    import torch

    import gated_deltanet_gdn_gb300 as gdn
    from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs

    res = {}
    # read (not written) between steps, so no dirty lines are written back inside a timed step
    flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    for B, label in ((2, "B2 H48 Dk=Dv=128 fp32 (L2 flushed before each step, kernel events)"),
                     (32, "B32 H48 Dk=Dv=128 fp32 (state 201 MB > L2, 30 steps back to back)")):
        w = WORKLOADS["recurrent"].with_(B=B, T=1, h0_std=0.01)
        d = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(w).items()}
        state = d["h0"].clone()
        out = torch.empty_like(d["v"])

        def one():
            gdn.gdn_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], state, out=out, h_final=state)

        for _ in range(5):
            one()
        torch.cuda.synchronize()
        if B == 2:
            times = []
            for _ in range(30):
                flush.sum()
                # a spin kernel keeps the GPU busy while the host submits the step, so the
                # library's begin event and the kernel run back to back (no launch gap)
                torch.cuda._sleep(200_000)
                gdn.gdn_profile_enable(True)
                one()
                prof = gdn.gdn_profile_read()
                gdn.gdn_profile_enable(False)
                times.append(sum(v[0] for v in prof.values()))
            ms = statistics.median(times)
        else:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(4_000_000)  # every step is queued before the timed region starts
            e0.record()
            for _ in range(30):
                one()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / 30
        sb = w.B * w.H * w.Dk * w.Dv * 4
        io_b = w.B * w.H * (2 * w.Dk + 2 * w.Dv + 2) * 4
        b = 2 * sb + io_b
        res["B%d" % B] = {"workload": label, "ms_per_step": round(ms, 5), "bytes_per_step": b,
                          "hbm_gbs": round(b / (ms / 1e3) / 1e9, 1)}
    res["replay_B32"] = replay_leg(dev, res["B32"]["ms_per_step"])
    w = WORKLOADS["recurrent"]
    d = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(w).items()}
    gdn.gdn_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], None)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        gdn.gdn_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], None)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / 3
    res["prefill_B2_T2048_H48"] = {"ms": round(ms, 4), "tokens_per_s": round(w.B * w.T / (ms / 1e3), 1)}
    # the same prefill through the chunked forward (out and h_final; scalar decay with the
    # wipes), fp32 operands and bf16 operands, residuals preallocated
    for dt in ("f32", "bf16"):
        wv = w.with_(dtype=dt)
        dv = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(wv).items()}
        dims = gdn.make_dims(dv["q"], dv["v"], dv["g"], 0)
        rbuf = torch.empty(gdn.gdn_chunk_residual_bytes(dims), dtype=torch.uint8, device=dev)
        for _ in range(3):
            gdn.gdn_chunk_fwd(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], None, residuals=rbuf)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(10):
            gdn.gdn_chunk_fwd(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], None, residuals=rbuf)
        e1.record()
        torch.cuda.synchronize()
        cms = e0.elapsed_time(e1) / 10
        res["prefill_chunked_B2_T2048_H48_" + dt] = {
            "ms": round(cms, 4), "tokens_per_s": round(w.B * w.T / (cms / 1e3), 1),
            "speedup_vs_recurrent": round(ms / cms, 2),
            "workload": "B2 T2048 H48 Dk=Dv=128 %s operands, scalar decay with wipes, chunked forward" % dt}
        del dv, rbuf
    peaks = load_peaks()
    res["hbm_peak_gbs"] = peaks["hbm_gbs"]
    return res


def replay_leg(dev, recurrent_ms, L=8):
    """Replay decode (checkpoint + L-token buffer) on the B32 H48 Dk=Dv=128 fp32 decode
    batch: 2 L warm-up steps reach the steady fill cycle, then 4 L steps (4 folds) back to
    back between two CUDA events, queued behind a spin kernel. Bytes per step are averaged over the cycle: the
    checkpoint read, (L + 1) / 2 buffer slots read, one slot written, the checkpoint
    written once per L steps, the token row in and the output out."""
    import torch

    import gated_deltanet_gdn_gb300 as gdn
    from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs

    w = WORKLOADS["recurrent"].with_(B=32, T=1, h0_std=0.01)
    d = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(w).items()}
    ckpt, buffer, fill = gdn.replay_init(d["h0"], L)
    out = torch.empty_like(d["v"])

    def one():
        gdn.gdn_replay_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], ckpt, buffer, fill, L, out=out)

    for _ in range(2 * L):
        one()
    torch.cuda.synchronize()
    steps = 4 * L
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(4_000_000)  # every step is queued before the timed region starts
    e0.record()
    for _ in range(steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    heads = w.B * w.H
    sb = w.Dk * w.Dv * 4
    slot = (2 * w.Dk + w.Dv) * 4
    io = (2 * w.Dk + 2 * w.Dv + 2) * 4
    b = heads * (sb + (L + 1) / 2 * slot + slot + sb / L + io)
    return {"workload": "B32 H48 Dk=Dv=128 fp32, buffer L=%d, %d steps back to back" % (L, steps),
            "ms_per_step": round(ms, 5), "bytes_per_step": int(b), "hbm_gbs": round(b / (ms / 1e3) / 1e9, 1),
            "speedup_vs_recurrent_decode": round(recurrent_ms / ms, 3)}


def oracle_sample(w, host, pairs):
    """float64 oracle forward + reverse pass over the listed (b, h) pairs, full T."""
    import numpy as np

    import oracle
    from gated_deltanet_gdn_gb300.synthetic import to_f64

    def sl(name, state=False):
        t = host[name]
        if t is None:
            return None
        if state:
            return np.ascontiguousarray(np.stack([to_f64(t[b, h]) for b, h in pairs], 0)[None])
        return np.ascontiguousarray(np.stack([to_f64(t[b, :, h]) for b, h in pairs], 1)[None])

    a = {n: sl(n, n in ("h0", "dh_final")) for n in ("q", "k", "v", "g", "beta", "h0", "dout", "dh_final")}
    t0 = time.perf_counter()
    o, h = oracle.fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], nthreads=len(pairs))
    g = oracle.bwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], a["dout"], a["dh_final"],
                   nthreads=len(pairs))
    sec = time.perf_counter() - t0
    return sec, dict(g, out=o, h_final=h, pairs=pairs)


def cpu_pairs(w):
    """Up to 16 (batch, head) pairs (one per host core), spread evenly over all B * H."""
    cores = os.cpu_count() or 1
    n = w.B * w.H
    p = max(1, min(cores, 16, n))
    return [(j // w.H, j % w.H) for j in (i * n // p for i in range(p))]


def cpu_baseline(w, host):
    """The float64 oracle's forward + reverse pass on a bounded sample of (b, h) pairs,
    timed on the host cores. Returns the baseline line and the oracle's results for
    those pairs (the benchmark's correctness gate compares the GPU step with them)."""
    import oracle

    oracle.build()
    pairs = cpu_pairs(w)
    sec, ref = oracle_sample(w, host, pairs)
    tokens = len(pairs) * w.T / w.H  # head-sequences expressed in tokens of all H heads
    return ({"value": round(tokens / sec, 1), "unit": "tokens/s", "cores": len(pairs), "kind": "oracle",
             "sample": f"float64 token-serial forward + reverse pass of {len(pairs)} (batch, head) pairs "
                       f"x {w.T} tokens = {tokens:.0f} tokens of the {w.H}-head workload, {sec:.2f} s"}, ref)


def oracle_gate(ref, got, tol=2e-2):
    """rel-L2 of the GPU results at the oracle sample's (b, h) pairs, per tensor."""
    import numpy as np

    pairs = ref["pairs"]
    res = {}
    for n in ("out", "h_final", "dq", "dk", "dv", "dg", "dbeta", "dh0"):
        t = got[n].detach().double().cpu()
        if n in ("h_final", "dh0"):
            x = np.stack([t[b, h].numpy() for b, h in pairs], 0)[None]
        else:
            x = np.stack([t[b, :, h].numpy() for b, h in pairs], 1)[None]
        y = ref[n]
        res[n] = float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300))
    return {"vs_oracle_rel_l2": {k: round(v, 6) for k, v in res.items()}, "tolerance": tol,
            "pairs": len(pairs), "passed": all(v <= tol for v in res.values())}


def run_reference(args, world, rank):
    """The float64 CPU oracle timed on the host cores, same workload, metric and unit."""
    if rank != 0:
        return
    import oracle
    from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs

    oracle.build()
    w = WORKLOADS[WORKLOAD]
    host = make_inputs(w)
    pairs = cpu_pairs(w)
    tokens = len(pairs) * w.T / w.H
    steps = max(1, min(args.steps, 10))
    warm = max(3, min(args.warmup, 5))  # at least three, and bounded: each step is seconds of CPU
    for _ in range(warm):
        oracle_sample(w, host, pairs)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_sample(w, host, pairs)[0]
    sec = (time.perf_counter() - t0) / steps
    value = tokens / sec
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": steps, "warmup": warm, "ms_per_step": round(sec * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "chunked fwd+bwd, B8 T4096 H6 Dk=Dv=128 (bounded sample, see cpu_baseline)"},
            "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": len(pairs), "kind": "oracle",
                             "sample": f"{len(pairs)} (batch, head) pairs x {w.T} tokens per step"},
            "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return
    world, rank, local = dist_setup()
    run_gdn(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
