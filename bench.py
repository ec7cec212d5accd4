#!/usr/bin/env python
"""Benchmark of the KDA hot path on one GB300 (replicas on N GPUs).

Default line: the fused decode step over the state pool, 256 sequences x 32
heads, dk = dv = 128, bf16 q/k/v/b, fp32 g, 4096-slot fp32 pool (8 GiB).
One step = one kda_decode launch over one batch of synthetic inputs; the
batch and its slot set rotate over 16 disjoint slot sets so that each step
touches 512 MiB of state that the previous step did not (more than the
129 MB L2).  Extra paths measured in the same run (``paths`` key):
speculative verify + commit (128 x 7 draft tokens x 32 heads), the fused
ShortConv + decode + RMS-norm-gate step at the decode workload's size, chunked
prefill (T = 8192 x 32 heads) and the long-context mix (T = 102400 prefill,
256 decode steps on its final state, 1024 x 64-head decode over a
16384-slot pool).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
        [--paths decode,spec,fused,prefill,longmix] [--no-cpu-baseline]
With N > 1 it must run under torchrun (one process per GPU); every rank runs
an independent replica (the recurrence has no cross-GPU exchange) and rank 0
prints one JSON line with the whole-job throughput.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_delta_rule_decode_gb300 import inputs  # noqa: E402

METRIC = "KDA decode token-heads/s + HBM GB/s vs peak; chunked-prefill tokens/s"
UNIT = "token-heads/s"
L2_BYTES = 129 * 1024 * 1024

# Algorithmic bytes per unit (token-head for decode):
#   decode: state read + write 2 * dv * dk * 4, q/k/v 3 * d * 2 (bf16),
#           g dk * 4, b 2, out dv * 2
DECODE_BYTES_PER_TH = 2 * 128 * 128 * 4 + 3 * 128 * 2 + 128 * 4 + 2 + 128 * 2  # 132610


def verify_bytes_per_sh(D):
    # state read once + per draft token: q,k,v (768) + g (512) + b (2) + out (256)
    # + record k_hat (512) + v (256) + g (512) + beta (4)
    return 128 * 128 * 4 + D * (768 + 512 + 2 + 256 + 512 + 256 + 512 + 4)


def commit_bytes_per_sh(a):
    # a >= 1: state read + write + a records (k_hat 512, v 256, g 512, beta 4)
    return 0 if a == 0 else 2 * 128 * 128 * 4 + a * (512 + 256 + 512 + 4)


PREFILL_BYTES_PER_TH = 3 * 128 * 2 + 128 * 4 + 2 + 128 * 2  # q,k,v,g,b in + out = 1538
PREFILL_FLOP_PER_TH = 180224  # listed MMAs of the chunk form, per token-head


# --------------------------------------------------------------------------- utils

def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                source="fallback")


def kernel_source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "gated_delta_rule_decode_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key, digest):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source has not changed since it was captured (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel_key:
                if parts[1] == digest:
                    return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clock/throttle sampling in the background."""

    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.rows = []
        self.proc = None
        self.gpu = gpu_index
        self.period = period_ms
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def mark_on(self):
        self.t_on = time.time()

    def mark_off(self):
        self.t_off = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = [r for t, r in self.rows if self.t_on and self.t_off and self.t_on <= t <= self.t_off]
        window = "timed steps and the 0.5 s continuation of the same launches"
        if len(inside) < 3:
            inside = [r for t, r in self.rows]
            window = "whole run (timed region shorter than the sampling period)"
        sm = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in inside if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4)
                          if len(r) > 6 + i and r[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside), "window": window}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------- decode (main line)

def build_decode_sets(n_sets=16, n_inputs=8, device="cuda"):
    w = inputs.WORKLOADS["decode_b256_h32_d128_pool4096_bf16"]
    B, H, dk, dv, NS = w["B"], w["H"], w["dk"], w["dv"], w["num_slots"]
    base = inputs.decode_inputs(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=0,
                                g_mean=3.0, pool_std=0.02, device=device)
    gen = torch.Generator(device=device)
    gen.manual_seed(1234)
    perm = torch.randperm(NS, generator=gen, device=device).to(torch.int32)
    slot_sets = [base.slot_ids] + [perm[i * B:(i + 1) * B].contiguous() for i in range(1, n_sets)]
    batches = [base] + [inputs.decode_inputs(B, H, dk, dv, dtype="bf16", num_slots=1,
                                             seed=100 + i, g_mean=3.0, device=device)
                        for i in range(1, n_inputs)]
    for bt in batches[1:]:
        bt.pool = None  # only the per-token tensors of the extra batches are used
    return w, base.pool, slot_sets, batches


def run_decode(args, world, rank, kda, peaks, sampler):
    w, pool, slot_sets, batches = build_decode_sets()
    B, H = w["B"], w["H"]
    stream = torch.cuda.current_stream()
    outs = torch.empty((B, H, w["dv"]), dtype=torch.bfloat16, device="cuda")
    # one prepared C-ABI call per (input batch, slot set): the timed loop only
    # launches (no Python marshalling between kernels)
    calls = {}
    for bi, bt in enumerate(batches):
        for si, ss in enumerate(slot_sets):
            calls[(bi, si)] = kda.decode(bt.q, bt.k, bt.v, bt.g, bt.b, ss, pool, outs,
                                         stream=stream, _prepare=True)

    def step(i):
        calls[(i % len(batches), i % len(slot_sets))]()

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    sampler.mark_on()
    t0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    t1.record(stream)
    # the same launches continue for about half a second so that the clock
    # samples cover the timed region's conditions; event pairs every 100
    # launches give a sustained per-launch time beside the timed one
    sus = []
    j = args.warmup + args.steps
    deadline = time.time() + 0.5
    while time.time() < deadline or len(sus) < 3:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(100):
            step(j)
            j += 1
        b.record(stream)
        sus.append((a, b))
        if len(sus) % 4 == 0:
            b.synchronize()
    torch.cuda.synchronize()
    sampler.mark_off()
    barrier(world)
    total_ms = t0.elapsed_time(t1)
    sus_us = statistics.median([a.elapsed_time(b) * 10.0 for a, b in sus])
    ms_per_step = max_over_ranks(total_ms / args.steps, world)
    units = B * H
    value = sum_over_ranks(units * args.steps, world) / (ms_per_step * args.steps / 1e3)
    # one kernel per step: its average duration is the step time
    avg_kernel_s = total_ms / args.steps / 1e3
    achieved = DECODE_BYTES_PER_TH * units / avg_kernel_s / 1e9
    digest = kernel_source_digest(["kda_decode.cu", "kda_rowmath.cuh"])
    traffic = ncu_traffic("decode_kernel", digest)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": traffic, "kernel": "kda::decode_kernel<128,bf16,4>",
                "algorithmic_bytes_per_launch": DECODE_BYTES_PER_TH * units,
                "peak_source": f"{peaks['source']} hbm_gbs (copy)",
                "avg_kernel_us": round(avg_kernel_s * 1e6, 2),
                "frac_of_nominal_8000_gbs": round(achieved / 8000.0, 4),
                "sustained_us_per_launch_median": round(sus_us, 2),
                "sustained_launches": 100 * len(sus)}

    # e2e: host buffers through the same C ABI entry point.  As in a serving
    # loop, step i+1's inputs are uploaded and step i-1's outputs read back on
    # copy streams while step i computes (two device buffer sets).
    pinned = {}
    for name in ("q", "k", "v", "g", "b"):
        pinned[name] = [getattr(bt, name).cpu().pin_memory() for bt in batches]
    pinned["slots"] = [s.cpu().pin_memory() for s in slot_sets]
    NB = 2
    dev_in = [{n: torch.empty_like(getattr(batches[0], n)) for n in ("q", "k", "v", "g", "b")} for _ in range(NB)]
    dev_slots = [torch.empty_like(slot_sets[0]) for _ in range(NB)]
    dev_out = [torch.empty((B, H, w["dv"]), dtype=torch.bfloat16, device="cuda") for _ in range(NB)]
    host_out = [torch.empty((B, H, w["dv"]), dtype=torch.bfloat16).pin_memory() for _ in range(NB)]
    h2d = sum(pinned[n][0].numel() * pinned[n][0].element_size() for n in ("q", "k", "v", "g", "b"))
    h2d += pinned["slots"][0].numel() * 4
    d2h = host_out[0].numel() * host_out[0].element_size()
    up_s, down_s = torch.cuda.Stream(), torch.cuda.Stream()
    up_done = [torch.cuda.Event() for _ in range(NB)]
    comp_done = [torch.cuda.Event() for _ in range(NB)]
    down_done = [torch.cuda.Event() for _ in range(NB)]

    def e2e_step(i):
        j, bi = i % NB, i % len(batches)
        up_s.wait_event(comp_done[j])  # buffer set j: step i - NB has consumed it
        with torch.cuda.stream(up_s):
            for n in ("q", "k", "v", "g", "b"):
                dev_in[j][n].copy_(pinned[n][bi], non_blocking=True)
            dev_slots[j].copy_(pinned["slots"][i % len(slot_sets)], non_blocking=True)
        up_done[j].record(up_s)
        stream.wait_event(up_done[j])
        stream.wait_event(down_done[j])  # output buffer j has been read back
        kda.decode(dev_in[j]["q"], dev_in[j]["k"], dev_in[j]["v"], dev_in[j]["g"], dev_in[j]["b"],
                   dev_slots[j], pool, dev_out[j], stream=stream)
        comp_done[j].record(stream)
        down_s.wait_event(comp_done[j])
        with torch.cuda.stream(down_s):
            host_out[j].copy_(dev_out[j], non_blocking=True)
        down_done[j].record(down_s)

    n_e2e = max(3, min(args.steps, 200))
    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up_s.wait_event(e0)
    for i in range(n_e2e):
        e2e_step(i)
    for j in range(NB):
        stream.wait_event(down_done[j])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world)
    e2e_value = sum_over_ranks(units * n_e2e, world) / (e2e_ms * n_e2e / 1e3)

    # the same steps with copy, kernel and read-back in order on one stream
    def serial_step(i):
        bi = i % len(batches)
        for n in ("q", "k", "v", "g", "b"):
            dev_in[0][n].copy_(pinned[n][bi], non_blocking=True)
        dev_slots[0].copy_(pinned["slots"][i % len(slot_sets)], non_blocking=True)
        kda.decode(dev_in[0]["q"], dev_in[0]["k"], dev_in[0]["v"], dev_in[0]["g"], dev_in[0]["b"],
                   dev_slots[0], pool, dev_out[0], stream=stream)
        host_out[0].copy_(dev_out[0], non_blocking=True)

    for i in range(3):
        serial_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0.record(stream)
    for i in range(n_e2e):
        serial_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    serial_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world)
    serial_value = sum_over_ranks(units * n_e2e, world) / (serial_ms * n_e2e / 1e3)
    e2e = {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
           "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 4), "steps": n_e2e,
           "copies": "pinned host buffers; uploads and read-backs on two copy streams, "
                     "overlapping the neighbouring steps' kernels (two device buffer sets)",
           "serial": {"value": round(serial_value, 1), "ms_per_step": round(serial_ms, 4),
                      "copies": "upload, kernel and read-back in order on one stream"}}
    del pool
    return dict(value=value, ms_per_step=ms_per_step, roofline=roofline, e2e=e2e,
                launches=args.steps, kernel_us=avg_kernel_s * 1e6,
                sustained_launches=100 * len(sus))


# --------------------------------------------------------------------------- extra paths

def time_launches(fn, n, warmup=3):
    """Average microseconds per call of fn(i) over n back-to-back calls,
    bracketed by one pair of CUDA events on the launching stream."""
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s)
    for i in range(n):
        fn(warmup + i)
    b.record(s)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / n


def run_spec(kda, peaks):
    w = inputs.WORKLOADS["verify_commit_b128_d7_h32_d128_bf16"]
    B, D, H, dk, dv, NS = w["B"], w["D"], w["H"], w["dk"], w["dv"], w["num_slots"]
    x = inputs.verify_inputs(B, D, H, dk, dv, dtype="bf16", num_slots=NS, seed=0, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(99)
    perm = torch.randperm(NS, generator=gen, device="cuda").to(torch.int32)
    sets = [perm[i * B:(i + 1) * B].contiguous() for i in range(NS // B)]
    out = torch.empty((B, D, H, dv), dtype=torch.bfloat16, device="cuda")
    rec = kda.alloc_records(B, D, H, dk, dv, torch.bfloat16, "cuda")
    acc = x.num_accepted
    n = 30
    vws_bytes = kda.verify_workspace_bytes(H, dk, dv, kda.KDA_DT_BF16, B, D)
    vws = torch.empty(max(vws_bytes, 1), dtype=torch.uint8, device="cuda")
    vcalls = [kda.verify_record(x.q, x.k, x.v, x.g, x.b, ss, x.pool, out, rec, workspace=vws,
                                _prepare=True)
              for ss in sets]
    tv = time_launches(lambda i: vcalls[i % len(sets)](), n)
    kda.verify_record(x.q, x.k, x.v, x.g, x.b, x.slot_ids, x.pool, out, rec)
    ccalls = [kda.replay_commit(rec, acc, ss, x.pool, _prepare=True) for ss in sets]
    tc = time_launches(lambda i: ccalls[i % len(sets)](), n)
    a_list = acc.tolist()
    vbytes = B * H * verify_bytes_per_sh(D)
    cbytes = H * sum(commit_bytes_per_sh(a) for a in a_list)
    vt = tv / 1e6
    ct = tc / 1e6
    # the u-record variant: verify into u records, commit without dot
    # products, and the previous window's commit fused with the next verify
    recu = kda.alloc_records_u(B, D, H, dk, dv, "cuda")
    rec2 = kda.alloc_records_u(B, D, H, dk, dv, "cuda")
    kda.verify_record_u(x.q, x.k, x.v, x.g, x.b, x.slot_ids, x.pool, out, recu, workspace=vws)
    ucalls = [kda.verify_record_u(x.q, x.k, x.v, x.g, x.b, ss, x.pool, out, rec2, workspace=vws, _prepare=True)
              for ss in sets]
    tvu = time_launches(lambda i: ucalls[i % len(sets)](), n) / 1e6
    cucalls = [kda.replay_commit_u(recu, acc, ss, x.pool, _prepare=True) for ss in sets]
    tcu = time_launches(lambda i: cucalls[i % len(sets)](), n) / 1e6
    fcalls = [kda.commit_verify_u(recu, acc, x.q, x.k, x.v, x.g, x.b, ss, x.pool, out, rec2, workspace=vws,
                                  _prepare=True) for ss in sets]
    tf = time_launches(lambda i: fcalls[i % len(sets)](), n) / 1e6
    ubytes_rec = 512 + 512 + 512  # k_hat, g, u per token-head
    cubytes = H * sum(0 if a == 0 else 2 * 128 * 128 * 4 + a * ubytes_rec for a in a_list)
    vubytes = B * H * (128 * 128 * 4 + D * (768 + 512 + 2 + 256 + ubytes_rec))
    fbytes = H * sum((2 if a else 1) * 128 * 128 * 4 + a * ubytes_rec for a in a_list) + \
        B * H * D * (768 + 512 + 2 + 256 + ubytes_rec)
    urec = {
        "verify_u": {"us": round(tvu * 1e6, 2), "GB/s": round(vubytes / tvu / 1e9, 1),
                     "frac_hbm": round(vubytes / tvu / 1e9 / peaks["hbm_gbs"], 4)},
        "commit_u": {"us": round(tcu * 1e6, 2), "GB/s": round(cubytes / tcu / 1e9, 1),
                     "frac_hbm": round(cubytes / tcu / 1e9 / peaks["hbm_gbs"], 4),
                     "algorithmic_bytes": cubytes,
                     "bytes_per_seq_head_a": "131072 + 1536 a (a >= 1); value records 131072 + 1284 a"},
        # kda_commit_verify_u: on this shape the commit and the verify are two
        # launches in one call; the bytes are the call's minimum (one state
        # read and one write where something was accepted)
        "commit_then_verify": {"us": round(tf * 1e6, 2), "GB/s": round(fbytes / tf / 1e9, 1),
                               "frac_hbm": round(fbytes / tf / 1e9 / peaks["hbm_gbs"], 4),
                               "algorithmic_bytes": fbytes,
                               "separate_calls_us": round((tcu + tvu) * 1e6, 2)},
    }
    return {
        "workload": "verify_commit_b128_d7_h32_d128_bf16",
        "verify": {"us": round(vt * 1e6, 2), "GB/s": round(vbytes / vt / 1e9, 1),
                   "frac_hbm": round(vbytes / vt / 1e9 / peaks["hbm_gbs"], 4),
                   "algorithmic_bytes": vbytes,
                   "draft_token_heads_per_s": round(B * D * H / vt, 1)},
        "commit": {"us": round(ct * 1e6, 2), "GB/s": round(cbytes / ct / 1e9, 1),
                   "frac_hbm": round(cbytes / ct / 1e9 / peaks["hbm_gbs"], 4),
                   "algorithmic_bytes": cbytes, "mean_accepted": round(sum(a_list) / B, 3)},
        "verify_workspace_bytes": vws_bytes,
        "u_records": urec,
        "launches": 3 * n,  # verify: window + state kernels; commit: replay kernel
    }


# fused decode (ShortConv + decode step + RMS norm and gate), per token-head:
# the decode bytes + z (dv * 2) + the conv state read and write
# (2 * 3 * (2 dk + dv) * 2); per launch once: conv taps H * (2 dk + dv) * 16
# and the norm weight dv * 4
FUSED_BYTES_PER_TH = DECODE_BYTES_PER_TH + 128 * 2 + 2 * 3 * 384 * 2  # 137474


def run_fused(kda, peaks, B=256, H=32, NS=4096, n=200):
    """The fused decode at the decode workload's size, rotating over 16
    disjoint slot sets like the main line, beside the plain decode launch."""
    dk = dv = 128
    x = inputs.decode_inputs(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=0, device="cuda")
    ex = inputs.fused_extras(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=0, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    perm = torch.randperm(NS, generator=gen, device="cuda").to(torch.int32)
    sets = [perm[i * B:(i + 1) * B].contiguous() for i in range(NS // B)]
    out = torch.empty((B, H, dv), dtype=torch.bfloat16, device="cuda")
    fcalls = [kda.decode_fused(x.q, x.k, x.v, x.g, x.b, ex.z, ss, x.pool, ex.conv_state, ex.conv_w,
                               ex.norm_w, out, _prepare=True) for ss in sets]
    dcalls = [kda.decode(x.q, x.k, x.v, x.g, x.b, ss, x.pool, out, _prepare=True) for ss in sets]
    tf = time_launches(lambda i: fcalls[i % len(sets)](), n) / 1e6
    td = time_launches(lambda i: dcalls[i % len(sets)](), n) / 1e6
    fbytes = B * H * FUSED_BYTES_PER_TH + H * (2 * dk + dv) * 16 + dv * 4
    gbs = fbytes / tf / 1e9
    return {
        "workload": "fused_decode_b256_h32_d128_pool4096_bf16",
        "us": round(tf * 1e6, 2), "GB/s": round(gbs, 1),
        "frac_hbm": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": fbytes,
        "token_heads_per_s": round(B * H / tf, 1),
        "plain_decode_us": round(td * 1e6, 2),
        "bytes_per_token_head": FUSED_BYTES_PER_TH,
        "launches": 2 * n,
    }


def run_prefill(kda, peaks, T=8192, H=32, steps=10, key="prefill_t8192_h32_d128_bf16", x=None):
    if x is None:
        x = inputs.prefill_inputs([T], H, 128, 128, dtype="bf16", seed=0, device="cuda")
    out = torch.empty((T, H, 128), dtype=torch.bfloat16, device="cuda")
    ws_bytes = kda.prefill_workspace_bytes(H, 128, 128, kda.KDA_DT_BF16, 1, T)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    try:
        call = kda.prefill_chunked(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, x.pool, out,
                                   workspace=ws, _prepare=True)
        t = time_launches(lambda i: call(), steps, warmup=2) / 1e6
    except kda.KdaError as e:
        return {"workload": key, "unavailable": str(e)}
    bytes_ = T * H * PREFILL_BYTES_PER_TH + H * 128 * 128 * 4
    flops = T * H * PREFILL_FLOP_PER_TH
    t_roof = max(bytes_ / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
    snap = None
    if T % 1024 == 0 and T <= 16384:
        # the same prefill writing the state every 1024 tokens into pool slots
        # (the prefix-cache snapshots): its extra cost
        n_snap = T // 1024
        pool2 = torch.zeros((n_snap + 1, H, 128, 128), device="cuda")
        snaps = (torch.zeros(n_snap, dtype=torch.int32, device="cuda"),
                 torch.arange(1, n_snap + 1, dtype=torch.int32, device="cuda") * 1024,
                 torch.arange(1, n_snap + 1, dtype=torch.int32, device="cuda"))
        slot0 = torch.zeros(1, dtype=torch.int32, device="cuda")
        call_s = kda.prefill_chunked(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, slot0, pool2, out,
                                     workspace=ws, snapshots=snaps, _prepare=True)
        ts = time_launches(lambda i: call_s(), steps, warmup=2) / 1e6
        snap = {"snapshots": n_snap, "every_tokens": 1024, "us": round(ts * 1e6, 1),
                "extra_us": round((ts - t) * 1e6, 1),
                "extra_bytes": n_snap * H * 128 * 128 * 4}
        del pool2
    return {"workload": key, "us": round(t * 1e6, 1), "tokens_per_s": round(T / t, 1),
            "token_heads_per_s": round(T * H / t, 1), "GB/s": round(bytes_ / t / 1e9, 1),
            "frac_hbm": round(bytes_ / t / 1e9 / peaks["hbm_gbs"], 4),
            "TFLOP/s": round(flops / t / 1e12, 2),
            "frac_tc_dense_bf16": round(flops / t / 1e12 / peaks["bf16_tflops"], 4),
            "frac_roofline": round(t_roof / t, 4), "algorithmic_bytes": bytes_,
            "algorithmic_flop": flops, "with_snapshots": snap}


def run_prefill_fused(kda, peaks, T=8192, H=32, steps=10):
    """The fused ShortConv + prefill + gated RMS norm at the prefill
    workload's size, beside the plain prefill's figure."""
    x = inputs.prefill_inputs([T], H, 128, 128, dtype="bf16", seed=0, device="cuda")
    ex = inputs.fused_prefill_extras(T, 1, H, 128, 128, dtype="bf16", seed=0, device="cuda")
    out = torch.empty((T, H, 128), dtype=torch.bfloat16, device="cuda")
    ws_bytes = kda.prefill_workspace_bytes(H, 128, 128, kda.KDA_DT_BF16, 1, T)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    try:
        call = kda.prefill_fused(x.q, x.k, x.v, x.g, x.b, ex.z, x.cu_seqlens, x.slot_ids, x.pool,
                                 ex.conv_state, ex.conv_w, ex.norm_w, out, workspace=ws, _prepare=True)
        t = time_launches(lambda i: call(), steps, warmup=2) / 1e6
    except kda.KdaError as e:
        return {"workload": "prefill_fused_t8192_h32_d128_bf16", "unavailable": str(e)}
    # the plain prefill's bytes plus z (dv x 2 per token-head) and the conv
    # state read and written (2 x 3 x 384 x 2 per head)
    bytes_ = T * H * (PREFILL_BYTES_PER_TH + 128 * 2) + H * 128 * 128 * 4 + H * 2 * 3 * 384 * 2
    return {"workload": "prefill_fused_t8192_h32_d128_bf16", "us": round(t * 1e6, 1),
            "tokens_per_s": round(T / t, 1), "GB/s": round(bytes_ / t / 1e9, 1),
            "frac_hbm": round(bytes_ / t / 1e9 / peaks["hbm_gbs"], 4), "algorithmic_bytes": bytes_}


def run_longmix(kda, peaks):
    res = {"workload": "longmix_prefill_t102400_h32_decode256_b1024_h64_pool16384"}
    T, H = 102400, 32
    xp = inputs.prefill_inputs([T], H, 128, 128, dtype="bf16", seed=0, device="cuda")
    res["prefill_t102400"] = run_prefill(kda, peaks, T=T, H=H, steps=3,
                                         key="prefill_t102400_h32_d128_bf16", x=xp)
    # 256 decode steps, batch 1 x 32 heads, on the prefill's final state (its
    # slot; L2-resident: latency-bound), captured in one CUDA graph.  Every
    # timed replay starts again from the prefill's final state.
    pool, slots = xp.pool, xp.slot_ids
    del xp
    torch.cuda.empty_cache()
    s_final = pool.clone()
    x = inputs.decode_inputs(1, H, 128, 128, dtype="bf16", num_slots=1, seed=7, device="cuda",
                             tokens=256)
    out = torch.empty((256, 1, H, 128), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for t in range(256):
            kda.decode(x.q[t], x.k[t], x.v[t], x.g[t], x.b[t], slots, pool, out[t], stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for t in range(256):
            kda.decode(x.q[t], x.k[t], x.v[t], x.g[t], x.b[t], slots, pool, out[t], stream=s)
    times = []
    cur = torch.cuda.current_stream()
    for i in range(7):
        pool.copy_(s_final)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(cur)
        graph.replay()
        b.record(cur)
        torch.cuda.synchronize()
        if i >= 2:
            times.append(a.elapsed_time(b) * 1e3)
    ts = statistics.median(times)
    res["decode_256_steps_b1_h32"] = {"us_per_step": round(ts / 256, 3), "graph": True,
                                      "state": "the T = 102400 prefill's final state",
                                      "replays": len(times), "us_per_replay_median": round(ts, 1)}
    del pool, s_final, x, out, graph
    # 1024 x 64 heads over a 16384-slot pool (64 GiB)
    B2, H2, NS2 = 1024, 64, 16384
    try:
        big = inputs.decode_inputs(B2, H2, 128, 128, dtype="bf16", num_slots=NS2, seed=11,
                                   g_mean=3.0, pool_std=0.02, device="cuda")
    except torch.cuda.OutOfMemoryError as e:  # pragma: no cover
        res["decode_b1024_h64"] = {"unavailable": f"out of memory: {e}"}
        return res
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    perm = torch.randperm(NS2, generator=gen, device="cuda").to(torch.int32)
    sets = [perm[i * B2:(i + 1) * B2].contiguous() for i in range(NS2 // B2)]
    out2 = torch.empty((B2, H2, 128), dtype=torch.bfloat16, device="cuda")
    dcalls = [kda.decode(big.q, big.k, big.v, big.g, big.b, ss, big.pool, out2, _prepare=True)
              for ss in sets]
    t = time_launches(lambda i: dcalls[i % len(sets)](), 10) / 1e6
    bytes_ = B2 * H2 * DECODE_BYTES_PER_TH
    res["decode_b1024_h64"] = {"us": round(t * 1e6, 1), "token_heads_per_s": round(B2 * H2 / t, 1),
                               "GB/s": round(bytes_ / t / 1e9, 1),
                               "frac_hbm": round(bytes_ / t / 1e9 / peaks["hbm_gbs"], 4)}
    del big
    torch.cuda.empty_cache()
    return res


# --------------------------------------------------------------------------- CPU oracle

def _timed_reps(fn, seconds):
    """Repeat fn() for about `seconds` (at least once); (reps, elapsed s)."""
    fn()  # warm
    reps, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds or reps == 0:
        fn()
        reps += 1
    return reps, time.perf_counter() - t0


def cpu_baseline(seconds_budget=6.0, threads=None, per_path=True):
    """The fp64 oracle as it stands, on bounded samples of the workloads, on
    the host cores.  The headline figure is decode (a 32-sequence subset of
    the 256 x 32-head batch) on every core; `paths` adds decode on one core,
    verify + commit (16 sequences x 7 draft tokens x 32 heads, the accepted
    lengths of the workload's draw) and the 8192-token prefill (1 head on one
    core, 16 heads on every core), each on one core and on all of them."""
    import oracle
    threads = threads or os.cpu_count() or 1
    used = oracle.set_threads(threads)
    w = inputs.WORKLOADS["decode_b256_h32_d128_pool4096_bf16"]
    H, Bs = w["H"], 32
    x = inputs.decode_inputs(Bs, H, 128, 128, dtype="bf16", num_slots=Bs, seed=0,
                             g_mean=3.0, pool_std=0.02)
    pool = x.pool.double()

    def dec():
        oracle.decode(x.q, x.k, x.v, x.g, x.b, x.slot_ids, pool)

    reps, dt = _timed_reps(dec, seconds_budget)
    done = reps * Bs * H
    res = {"value": round(done / dt, 2), "unit": UNIT, "cores": used, "kind": "oracle",
           "sample": f"{reps} oracle decode calls of {Bs} sequences x {H} heads "
                     f"(dk = dv = 128, fp64) = {done} token-heads in {dt:.1f} s"}
    if not per_path:
        return res
    paths = {}
    budget = max(1.0, seconds_budget / 3)
    for nthr in (1, used):
        oracle.set_threads(nthr)
        tag = f"{nthr}_core" if nthr == 1 else f"{nthr}_cores"
        if nthr == 1:
            r1, d1 = _timed_reps(dec, budget)
            paths["decode_b256_h32_d128_1_core"] = {
                "value": round(r1 * Bs * H / d1, 2), "unit": "token-heads/s", "cores": 1,
                "sample": f"{r1} calls of {Bs} x {H} token-heads in {d1:.1f} s"}
        y = inputs.verify_inputs(16, 7, H, 128, 128, dtype="bf16", num_slots=16, seed=0)
        ypool = y.pool.double()

        def spec():
            _, rec, _ = oracle.verify(y.q, y.k, y.v, y.g, y.b, y.slot_ids, ypool)
            oracle.replay(rec, y.num_accepted, y.slot_ids, ypool.clone())

        r2, d2 = _timed_reps(spec, budget)
        paths[f"verify_commit_b128_d7_h32_d128_{tag}"] = {
            "value": round(r2 * 16 * 7 * H / d2, 2), "unit": "draft token-heads/s (verify + commit)",
            "cores": nthr,
            "sample": f"{r2} verify + commit rounds of 16 sequences x 7 draft tokens x {H} heads "
                      f"in {d2:.1f} s"}
        Hp = 1 if nthr == 1 else min(16, H)
        z = inputs.prefill_inputs([8192], Hp, 128, 128, dtype="bf16", seed=0)
        zpool = z.pool.double()

        def pre():
            oracle.prefill(z.q, z.k, z.v, z.g, z.b, z.cu_seqlens, z.slot_ids, zpool)

        t0 = time.perf_counter()
        pre()
        d3 = time.perf_counter() - t0
        paths[f"prefill_t8192_d128_{tag}"] = {
            "value": round(8192 * Hp / d3, 2), "unit": "token-heads/s", "cores": nthr,
            "sample": f"one oracle prefill of 8192 tokens x {Hp} head(s) in {d3:.1f} s"}
    oracle.set_threads(used)
    res["paths"] = paths
    return res


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    cb = cpu_baseline(seconds_budget=max(2.0, min(30.0, 1.5 * (args.steps + args.warmup))),
                      per_path=False)
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(256 * 32 / cb["value"] * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "decode_b256_h32_d128_pool4096_bf16",
                       "note": "fp64 CPU oracle on host cores; each step a bounded sample"},
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- ncu cases

def run_ncu_case(name, steps, kda):
    """Small cases of each kernel for ncu --set full captures: inputs larger
    than L2 but at most ~1-2 GB on the device.  Prints nothing useful; the
    profile is the product."""
    if name == "decode_small":
        # 256 x 32 heads, dk = dv = 128, over a 512-slot pool (1 GiB): each
        # launch touches 512 MiB of state, two disjoint slot sets alternate
        x = inputs.decode_inputs(256, 32, 128, 128, dtype="bf16", num_slots=512, seed=0,
                                 device="cuda")
        sets = [x.slot_ids, torch.arange(512, dtype=torch.int32, device="cuda")[
            ~torch.isin(torch.arange(512, device="cuda"), x.slot_ids.long())].contiguous()]
        for i in range(steps):
            kda.decode(x.q, x.k, x.v, x.g, x.b, sets[i % 2], x.pool)
    elif name == "spec_small":
        x = inputs.verify_inputs(128, 7, 32, 128, 128, dtype="bf16", num_slots=256, seed=0,
                                 device="cuda")
        out, rec = None, None
        for i in range(steps):
            out, rec = kda.verify_record(x.q, x.k, x.v, x.g, x.b, x.slot_ids, x.pool, out, rec)
            kda.replay_commit(rec, x.num_accepted, x.slot_ids, x.pool)
    elif name == "fused_small":
        # the fused decode at 256 x 32 heads over a 512-slot pool, two
        # disjoint slot sets alternating (512 MiB of state per launch)
        x = inputs.decode_inputs(256, 32, 128, 128, dtype="bf16", num_slots=512, seed=0,
                                 device="cuda")
        ex = inputs.fused_extras(256, 32, 128, 128, dtype="bf16", num_slots=512, seed=0, device="cuda")
        sets = [x.slot_ids, torch.arange(512, dtype=torch.int32, device="cuda")[
            ~torch.isin(torch.arange(512, device="cuda"), x.slot_ids.long())].contiguous()]
        for i in range(steps):
            kda.decode_fused(x.q, x.k, x.v, x.g, x.b, ex.z, sets[i % 2], x.pool, ex.conv_state,
                             ex.conv_w, ex.norm_w)
    elif name == "prefill_fused_small":
        x = inputs.prefill_inputs([8192], 32, 128, 128, dtype="bf16", seed=0, device="cuda")
        ex = inputs.fused_prefill_extras(8192, 1, 32, 128, 128, dtype="bf16", seed=0, device="cuda")
        for i in range(steps):
            kda.prefill_fused(x.q, x.k, x.v, x.g, x.b, ex.z, x.cu_seqlens, x.slot_ids, x.pool, ex.conv_state,
                              ex.conv_w, ex.norm_w)
    elif name == "prefill_small":
        x = inputs.prefill_inputs([8192], 32, 128, 128, dtype="bf16", seed=0, device="cuda")
        for i in range(steps):
            kda.prefill_chunked(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, x.pool)
    else:
        raise SystemExit(f"unknown ncu case {name}")
    torch.cuda.synchronize()
    print(json.dumps({"ncu_case": name, "steps": steps, "status": "ok"}))
    return 0


# --------------------------------------------------------------------------- main

def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--paths", default="decode,spec,fused,prefill,longmix")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ncu-case", default=None,
                    help="run one small profiling case (decode_small, spec_small, fused_small, prefill_small, "
                         "prefill_fused_small)")
    args = ap.parse_args(argv)
    if args.ncu_case:
        from gated_delta_rule_decode_gb300 import kda
        return run_ncu_case(args.ncu_case, args.steps, kda)
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    from gated_delta_rule_decode_gb300 import kda
    peaks = read_peaks()
    sampler = ClockSampler(local)
    sampler.start()
    try:
        main_res = run_decode(args, world, rank, kda, peaks, sampler)
    finally:
        sampler.stop()
    paths = {}
    wanted = set(args.paths.split(","))
    launches = main_res["launches"]
    if rank == 0:
        if "spec" in wanted:
            paths["verify_commit"] = run_spec(kda, peaks)
        if "fused" in wanted:
            paths["fused_decode"] = run_fused(kda, peaks)
        if "prefill" in wanted:
            paths["prefill"] = run_prefill(kda, peaks)
            paths["prefill_fused"] = run_prefill_fused(kda, peaks)
        if "longmix" in wanted:
            paths["longmix"] = run_longmix(kda, peaks)
    barrier(world)
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": round(main_res["value"], 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(main_res["ms_per_step"], 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "decode_b256_h32_d128_pool4096_bf16",
                   "sequences": 256, "heads": 32, "dk": 128, "dv": 128, "pool_slots": 4096,
                   "state": "fp32", "inputs": "bf16 q/k/v/b, fp32 g",
                   "l2": "inputs larger than L2: each step touches 512 MiB of state, "
                         "slot sets rotate over 16 disjoint sets",
                   "parallelism": f"replicas x{world}"},
        "roofline": main_res["roofline"],
        "e2e": main_res["e2e"],
        "gpu_launches": launches,
        "clocks": sampler.summary(),
        "paths": paths,
        "gpu": torch.cuda.get_device_name(),
    }
    if not args.no_cpu_baseline and world >= 1:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
