#!/usr/bin/env python3
"""Benchmark of the seg_la hot path on GB300: tokens/s and the fraction of the HBM/tensor roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload NAME] [--headline-only]
    python bench.py --profile-calls C [--workload NAME | --profile-case CASE]   (untimed)

A step is one call of the path over one batch of the chosen workload (inputs resident in HBM):
  decode         256 requests x 1 token, H=16, layer 3 of L=8, 1024-slot pool   (default)
  varlen_extend  8 requests, lengths uniform in [512, 4096], H=16, layer 0 of L=4
  long_prefill   1 request of 32768 tokens, H=32, layer 5 of L=12
  verify         128 requests x 5 draft tokens, H=64, layer 10 of L=20, 512-slot pool
  verify_tree    the same requests with an 8-token binary draft tree each
  varlen_extend_tracked  varlen_extend plus a state-tracking snapshot per request
  verify_commit  verify followed by the accepted-state commit (two library calls)
  varlen_extend_b1024  1024 requests, lengths uniform in [32, 512], H=16 (the persistent grid,
                 longest first; also timed without a workspace: one CTA per (request, head))
  varlen_extend_skewed  8 requests: two of 4096-8192 tokens, six of 256-1024, H=16 (the balanced
                 schedule; also timed with it switched off: one CTA per (request, head) and the
                 column split)
Every workload's inputs exceed the 129 MB L2, so no flush is needed between steps.  With N > 1
(torchrun), every rank runs its own replica of the workload (weak scaling, no collective on the
data path); timing is bracketed by a barrier and the slowest rank's time is reported.

The default run prints ONE JSON line for the decode workload and, unless --headline-only, adds
the other workloads under "other_workloads" (each timed the same way, three times over, with its
own clock record, end-to-end rate and oracle baseline).  `--impl reference` times the fp64 CPU
oracle instead, on a bounded sample of the same workload.

Timing: after the warm-up, a barrier and a synchronize, one untimed lead step is enqueued and then
the CUDA start event, the K timed steps and the end event, so that the GPU is already busy when
the timed region opens (the host's enqueue of the first timed call would otherwise count as
device time).  The host time spent enqueueing the K calls is reported per call.
"""
from __future__ import annotations

import argparse
import hashlib
import re
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

from lightning_attention_gb300 import workloads  # noqa: E402

METRIC = "seg-LA tokens/s (extend, decode, verify) and % of GB300 HBM/tensor roofline"
HEADLINE = "decode"
D = 128
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# Which source files hold the kernels a workload's step launches (used to invalidate stored ncu
# traffic).
KERNEL_SOURCE = {
    "decode": "la_recurrent.cu",
    "verify": "la_recurrent.cu",
    "varlen_extend": "la_extend_w.cu",
    "long_prefill": ("la_extend_w.cu", "la_extend_seg.cu"),
    "verify_tree": "la_recurrent.cu",
    "varlen_extend_tracked": "la_extend_w.cu",
    "verify_commit": "la_recurrent.cu",
    "varlen_extend_b1024": "la_extend_many.cu",
    "varlen_extend_skewed": "la_extend_bal.cu",
}
KERNEL_NAME = {
    "decode": "recurrent_kernel<0>",
    "verify": "recurrent_kernel<1>",
    "varlen_extend": "extend_wide_kernel",
    "long_prefill": "extend_wide_kernel",
    "verify_tree": "recurrent_kernel<3>",
    "varlen_extend_tracked": "extend_wide_kernel",
    "verify_commit": "recurrent_kernel<1>",
    "varlen_extend_b1024": "extend_many_kernel",
    "varlen_extend_skewed": "extend_bal_kernel",
}
# Small cases of the same kernels for multi-pass ncu captures (--profile-calls); a few GB at most.
PROFILE_CASES = {
    "verify_b32": lambda: workloads.verify_chain(0, B=32, num_slots=64),
    "verify_tree_b32": lambda: workloads.verify_tree(0, B=32, num_slots=64),
    # a quarter of the 1024-request batch: still 4,096 (request, head) pairs, the persistent grid
    "extend_many_b256": lambda: workloads.varlen_extend_many(0, B=256, num_slots=512),
}


# ----------------------------------------------------------------------------------------------
# distributed plumbing (host logic, also exercised on CPU with gloo by tests/test_multirank.py)

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(backend: str):
    world, rank, _ = dist_env()
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)
    return world, rank


def barrier(world: int, device=None):
    if world > 1:
        if device is not None and device.type == "cuda":
            torch.distributed.barrier(device_ids=[device.index])
        else:
            torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base: int, rank: int) -> int:
    """Each rank draws its own replica of the workload (weak scaling): seed base + rank."""
    return base + rank


def aggregate_throughput(units_per_rank_step: float, steps: int, world: int,
                         max_seconds: float) -> float:
    return units_per_rank_step * steps * world / max_seconds


# ----------------------------------------------------------------------------------------------
# workload geometry: tokens and algorithmic HBM bytes / tensor flops per call

CHUNK = 128  # the extend kernel's chunk length

def algorithmic(w) -> dict:
    H = w.H
    if w.kind == "decode":
        tokens = w.B
        byts = 2 * w.B * H * D * D * 4 + 4 * w.B * H * D * 2
        flops = w.B * H * 4 * D * D
        issued = flops
    elif w.kind in ("verify", "tree"):
        # tree: the same minimum (root state read once, every draft state written once); states a
        # fork re-reads from the intermediate buffer are not counted
        tokens = w.B * w.N
        byts = w.B * H * D * D * 4 * (1 + w.N) + 4 * w.B * w.N * H * D * 2
        if w.accept_idx is not None:
            # the commit: each accepted state read from the intermediate buffer, written to its slot
            byts += 2 * int((w.accept_idx >= 0).sum()) * H * D * D * 4
        flops = tokens * H * 4 * D * D
        issued = flops
    else:
        tokens = w.T
        n_prefix = int(w.prefix_mask.sum())
        byts = 4 * w.T * H * D * 2 + (n_prefix + w.B) * H * D * D * 4
        if w.track_lens is not None:
            byts += int((w.track_lens >= 0).sum()) * H * D * D * 4   # the snapshots
        flops = w.T * H * 4 * D * D           # the recurrence's own 4 d^2 per token-head
        # what the tensor cores are given per token-head, C = 128: Q K^T 2Cd, then Q S, the state
        # update and P V each as a bf16 hi + lo pair, 2 x 2d^2 + 2 x 2d^2 + 2 x 2Cd
        issued = w.T * H * (6 * CHUNK * D + 8 * D * D)
    return {"tokens": tokens, "bytes": byts, "flops": flops, "issued_flops": issued}


def make_workload(name: str, seed: int):
    return workloads.WORKLOADS[name](seed)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "of measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "of fallback"}


def source_digest(fname) -> str:
    """Digest of a kernel source file (or a tuple of them) and the local headers they include
    (recursively)."""
    csrc = os.path.join(ROOT, "lightning_attention_gb300", "csrc")
    h = hashlib.sha256()
    seen, todo = set(), [fname] if isinstance(fname, str) else list(fname)
    while todo:
        name = todo.pop(0)
        if name in seen:
            continue
        seen.add(name)
        with open(os.path.join(csrc, name), "rb") as f:
            text = f.read()
        h.update(text)
        for inc in re.findall(rb'^#include "([^"]+)"', text, flags=re.M):
            if os.path.exists(os.path.join(csrc, inc.decode())):
                todo.append(inc.decode())
    return h.hexdigest()[:16]


def stored_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current kernel
    source; else None."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            key, val = line.split(":", 1)
            vals[key.strip()] = val.strip()
    try:
        if vals.get("source_sha256_16") != source_digest(KERNEL_SOURCE[workload]):
            return None
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------------------------
# clocks sampled during the timed region

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------------------------
# GPU arm

class GpuCase:
    """Device-resident inputs and a step() that makes exactly one library call."""

    def __init__(self, w, dev, name):
        import lightning_attention_gb300 as la
        self.la = la
        self.w = w
        self.dev = dev
        self.q, self.k, self.v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
        self.slopes = la.slopes(w.H, w.layer_id, w.L).to(dev)
        self.pool = w.materialize_pool(dev)
        self.idx = w.state_idx.to(dev)
        self.out = torch.empty_like(self.q)
        self.launches_per_step = 1
        self.kernel = KERNEL_NAME[name]
        if w.kind == "extend":
            self.cu = w.cu_seqlens.to(dev)
            self.pm = w.prefix_mask.to(dev)
            lens = w.cu_seqlens[1:] - w.cu_seqlens[:-1]
            self.max_seqlen = int(lens.max()) if w.B else 0
            self.workspace = None  # the binding supplies what la_extend_workspace_size asks for
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            nbytes = la.extend_workspace_size(w.B, w.T, w.H, D, self.max_seqlen)
            if nbytes > 0:
                if w.B * w.H > sms:
                    # more (request, head) pairs than SMs: the request-record pre-pass, then the
                    # persistent grid
                    self.launches_per_step = 2
                    self.kernel = "item_records_kernel + extend_many_kernel (one la_extend call)"
                elif w.B > 256:
                    # a large batch: the ranking pre-pass, then the extend kernel
                    self.launches_per_step = 2
                    self.kernel = "rank_requests_kernel + extend_wide_kernel (one la_extend call)"
                elif nbytes < 65536:
                    # a skewed one-wave batch: the plan on the device, then the balanced grid
                    self.launches_per_step = 2
                    self.kernel = "seg_plan_kernel + extend_bal_kernel (one la_extend call)"
                else:
                    # long requests split into segments: block-state kernel, state scan, then
                    # the extend kernel
                    self.launches_per_step = 3
                    self.kernel = ("block_state_kernel + state_scan_kernel + extend_wide_kernel "
                                   "(one la_extend call)")
            self.track = None
            if w.track_lens is not None:
                self.track = (w.track_lens.to(dev), w.track_idx.to(dev))
                self.kernel = self.kernel.replace("extend_wide_kernel",
                                                  "extend_wide_kernel<true>").replace(
                                                      "extend_many_kernel", "extend_many_kernel<true>").replace(
                                                      "extend_bal_kernel", "extend_bal_kernel<true>")
        if w.kind in ("verify", "tree"):
            self.inter = torch.empty((w.B, w.N, w.H, D, D), dtype=torch.float32, device=dev)
        if w.kind == "tree":
            self.parents = w.parents.to(dev)
        self.accept = None
        if w.accept_idx is not None:
            self.accept = w.accept_idx.to(dev)
            self.launches_per_step += 1
            self.kernel += " + commit_kernel"

    def step(self, q=None, k=None, v=None, idx=None, out=None):
        la, w = self.la, self.w
        out = self.out if out is None else out
        q = self.q if q is None else q
        k = self.k if k is None else k
        v = self.v if v is None else v
        idx = self.idx if idx is None else idx
        if w.kind == "decode":
            la.decode(q, k, v, self.slopes, self.pool, idx, out=out)
        elif w.kind == "verify":
            la.verify_chain(q, k, v, self.slopes, self.pool, idx, w.N,
                            inter_states=self.inter, out=out)
            if self.accept is not None:
                la.commit_accepted(self.inter, self.accept, self.pool, idx)
        elif w.kind == "tree":
            la.verify_tree(q, k, v, self.slopes, self.pool, idx, self.parents, w.N,
                           inter_states=self.inter, out=out)
        elif self.track is not None:
            la.extend(q, k, v, self.slopes, self.pool, idx, self.cu, self.pm, out=out,
                      max_seqlen=self.max_seqlen, track_lens=self.track[0],
                      track_state_idx=self.track[1])
        else:
            la.extend(q, k, v, self.slopes, self.pool, idx, self.cu, self.pm, out=out,
                      max_seqlen=self.max_seqlen, workspace=self.workspace)
        return out


def timed_region(case, steps, world, dev, stream):
    """Device time of exactly `steps` steps between CUDA events on the launching stream, with a
    barrier and a synchronize on both sides.  One untimed lead step is enqueued after the
    synchronize and before the first event, so that the GPU is busy when the timed region opens
    and the host's enqueue of the first timed call is not counted as device time.  Returns
    (device seconds, host seconds spent enqueueing the timed calls)."""
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    case.step()  # the lead step (untimed)
    ev0.record(stream)
    h0 = time.perf_counter()
    for _ in range(steps):
        case.step()
    h1 = time.perf_counter()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    return ev0.elapsed_time(ev1) / 1e3, h1 - h0


def time_gpu(name, steps, warmup, world, rank, dev, peaks, with_e2e=True, sampler=None,
             repeats=1):
    import lightning_attention_gb300 as la
    w = make_workload(name, rank_seed(0, rank))
    geo = algorithmic(w)
    case = GpuCase(w, dev, name)
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        case.step()
    la.poll_error()

    if sampler:
        sampler.start()
    wall0 = time.perf_counter()
    runs = [timed_region(case, steps, world, dev, stream) for _ in range(repeats)]
    wall1 = time.perf_counter()
    clocks = sampler.stop() if sampler else None
    la.poll_error()
    # the reported run is the median one (the first when there is one); the others give the spread
    order = sorted(range(repeats), key=lambda i: runs[i][0])
    dev_s, host_s = runs[order[(repeats - 1) // 2]]
    max_s = max_over_ranks(dev_s, world, dev)
    per_launch = dev_s / steps  # one la_extend / la_decode / la_verify_chain call per step
    value = aggregate_throughput(geo["tokens"], steps, world, max_s)
    spread = None
    if repeats > 1:
        ms = sorted(r[0] / steps * 1e3 for r in runs)
        spread = {"repeats": repeats, "steps_each": steps, "ms_per_step_min": round(ms[0], 4),
                  "ms_per_step_median": round(ms[(repeats - 1) // 2], 4),
                  "ms_per_step_max": round(ms[-1], 4)}

    achieved_gbs = geo["bytes"] / per_launch / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved_gbs / peaks["hbm_gbs"], 4),
            "traffic": stored_traffic(name), "peak_source": peaks["source"],
            "algorithmic_bytes_per_launch": geo["bytes"], "kernel": case.kernel,
            "launch_ms": round(per_launch * 1e3, 4)}
    # for a step of two launches (long prefill, verify + commit) the stored traffic covers both
    tensor = None
    if w.kind == "extend":
        tflops = geo["flops"] / per_launch / 1e12
        itflops = geo["issued_flops"] / per_launch / 1e12
        tensor = {"recurrence_tflops": round(tflops, 2),
                  "frac_of_bf16_peak": round(tflops / peaks["bf16_tflops"], 4),
                  "note": "4 d^2 flops per token-head (the recurrence's own count)",
                  "issued_tflops": round(itflops, 2),
                  "issued_frac_of_bf16_peak": round(itflops / peaks["bf16_tflops"], 4),
                  "issued_note": "6 C d + 8 d^2 flops per token-head at C = 128: Q K^T, and Q S, "
                                 "the state update and P V each as a bf16 hi + lo pair; the "
                                 "time includes every launch of the call"}

    index_order = None
    if w.kind == "extend" and w.B > 256 and w.track_lens is None:
        # the same batch in index order (no workspace: no ranking pre-pass), for comparison
        case.workspace = False
        case.launches_per_step -= 1
        case.step()
        io_s, _ = timed_region(case, steps, world, dev, stream)
        case.workspace = None
        case.launches_per_step += 1
        index_order = {"ms_per_step": round(max_over_ranks(io_s, world, dev) / steps * 1e3, 4),
                       "note": "without a workspace: one CTA per (request, head), requests in "
                               "index order"}
    if "extend_bal_kernel" in case.kernel:
        # the same batch with the balanced schedule switched off, for comparison
        la.set_balanced(False)
        saved = (case.kernel, case.launches_per_step)
        case.launches_per_step = 1
        case.step()
        ub_s, _ = timed_region(case, steps, world, dev, stream)
        la.set_balanced(True)
        case.kernel, case.launches_per_step = saved
        index_order = {"ms_per_step": round(max_over_ranks(ub_s, world, dev) / steps * 1e3, 4),
                       "note": "balanced schedule off: one CTA per (request, head), the longest "
                               "requests' value columns split over idle SMs"}

    e2e = None
    if with_e2e:
        e2e = time_e2e(case, w, geo, steps, world, dev)
    res = {"value": value, "ms_per_step": max_s / steps * 1e3, "tokens_per_step": geo["tokens"],
           "gpu_launches": steps * case.launches_per_step,
           "host_enqueue_us_per_call": round(host_s / steps * 1e6, 2),
           "roofline": roof, "wall_s": wall1 - wall0, "clocks": clocks, "e2e": e2e,
           "workload": w, "geo": geo, "spread": spread, "index_order": index_order}
    if tensor:
        res["tensor"] = tensor
    return res


def time_e2e(case, w, geo, steps, world, dev):
    """Same metric through the public API with host buffers: per step, pinned-host -> device
    copies of the step's inputs (q, k, v, slot indices) and a device -> host read of the output,
    all inside the timed region, and the host waits for every step's result.  Steps are
    pipelined as a serving loop would: inputs and outputs are double-buffered, the copies run on
    their own streams, so step k+1's inputs travel while step k computes and step k's output
    travels while step k+1 computes; the library calls stay in order on one stream (decode and
    extend update the pool in place).  The state pool stays resident on the device."""
    hq, hk, hv = (t.pin_memory() for t in (w.q, w.k, w.v))
    hidx = w.state_idx.pin_memory()
    houts = [torch.empty(case.out.shape, dtype=case.out.dtype).pin_memory() for _ in range(2)]
    dins = [(torch.empty_like(case.q), torch.empty_like(case.k), torch.empty_like(case.v),
             torch.empty_like(case.idx)) for _ in range(2)]
    douts = [torch.empty_like(case.out) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hidx))
    d2h = houts[0].numel() * houts[0].element_size()
    e2e_steps = max(1, min(steps, 50))
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    e_in, e_done, e_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def issue(n):
        j = n & 1
        dq, dk, dv, didx = dins[j]
        with torch.cuda.stream(s_in):
            if n >= 2:
                s_in.wait_event(e_done[j])      # step n-2 is done with input buffers j
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            didx.copy_(hidx, non_blocking=True)
            e_in[j].record(s_in)
        comp.wait_event(e_in[j])
        if n >= 2:
            comp.wait_event(e_out[j])           # step n-2's output has left buffer j
        case.step(dq, dk, dv, didx, out=douts[j])
        e_done[j].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(e_done[j])
            houts[j].copy_(douts[j], non_blocking=True)
            e_out[j].record(s_out)

    issue(0)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    t0 = time.perf_counter()
    for n in range(e2e_steps):
        issue(n)
        if n >= 1:
            e_out[(n - 1) & 1].synchronize()    # the host reads step n-1's result
    e_out[(e2e_steps - 1) & 1].synchronize()
    t1 = time.perf_counter()
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    max_s = max_over_ranks(t1 - t0, world, dev)
    return {"value": aggregate_throughput(geo["tokens"], e2e_steps, world, max_s),
            "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": e2e_steps, "pipelined": "copies on their own streams, double-buffered"}


# ----------------------------------------------------------------------------------------------
# oracle (CPU) timing: the cpu_baseline leg and the --impl reference arm

def oracle_sample(w, budget_pairs: int):
    """A bounded sample of the workload for the fp64 oracle: whole requests (all heads) for
    decode/verify/varlen extend; for the single long request, a token prefix of it."""
    import numpy as np
    H = w.H
    if w.kind == "decode":
        B = min(w.B, max(1, budget_pairs // H))
        return {"kind": "decode", "B": B, "tokens": B,
                "desc": f"{B} of {w.B} requests x {H} heads (1 token each)"}
    if w.kind in ("verify", "tree"):
        B = min(w.B, max(1, budget_pairs // (H * w.N)))
        return {"kind": w.kind, "B": B, "tokens": B * w.N,
                "desc": f"{B} of {w.B} requests x {w.N} draft tokens x {H} heads"}
    lens = (w.cu_seqlens[1:] - w.cu_seqlens[:-1]).numpy()
    # token-heads budget: budget_pairs counts token-heads here
    if w.B == 1:
        n = int(min(lens[0], max(1, budget_pairs // H)))
        return {"kind": "extend_prefix", "n": n, "tokens": n,
                "desc": f"first {n} of {int(lens[0])} tokens x {H} heads"}
    keep, tok = [], 0
    for b in np.argsort(lens):
        if (tok + lens[b]) * H > budget_pairs and keep:
            break
        keep.append(int(b))
        tok += int(lens[b])
    return {"kind": "extend_requests", "reqs": sorted(keep), "tokens": tok,
            "desc": f"{len(keep)} of {w.B} requests ({tok} tokens) x {H} heads"}


def run_oracle_sample(w, sample, threads):
    import numpy as np
    import oracle
    s = oracle.slopes(w.H, w.layer_id, w.L).astype(np.float32).astype(np.float64)
    if sample["kind"] == "decode":
        B = sample["B"]
        q, k, v = (t[:B].float().numpy().astype(np.float64) for t in (w.q, w.k, w.v))
        idx = w.state_idx[:B].long()
        pool = w.pool_fill[idx].double().numpy()
        t0 = time.perf_counter()
        oracle.decode(q, k, v, s, pool, np.arange(B, dtype=np.int32), w.H, D, nthreads=threads)
        return time.perf_counter() - t0
    if sample["kind"] == "verify":
        B = sample["B"]
        rows = B * w.N
        q, k, v = (t[:rows].float().numpy().astype(np.float64) for t in (w.q, w.k, w.v))
        pool = w.prefix_states[:B].double().numpy()
        t0 = time.perf_counter()
        _, inter = oracle.verify_chain(q, k, v, s, pool, np.arange(B, dtype=np.int32), w.N, w.H,
                                       D, nthreads=threads)
        if w.accept_idx is not None:
            oracle.commit_accepted(inter, w.accept_idx[:B].numpy(), pool,
                                   np.arange(B, dtype=np.int32))
        return time.perf_counter() - t0
    if sample["kind"] == "tree":
        B = sample["B"]
        rows = B * w.N
        q, k, v = (t[:rows].float().numpy().astype(np.float64) for t in (w.q, w.k, w.v))
        pool = w.prefix_states[:B].double().numpy()
        t0 = time.perf_counter()
        oracle.verify_tree(q, k, v, s, pool, np.arange(B, dtype=np.int32), w.parents[:B].numpy(),
                           w.N, w.H, D)
        return time.perf_counter() - t0
    if sample["kind"] == "extend_prefix":
        n = sample["n"]
        q, k, v = (t[:n].float().numpy().astype(np.float64) for t in (w.q, w.k, w.v))
        pool = np.zeros((1, w.H, D, D))
        t0 = time.perf_counter()
        oracle.extend(q, k, v, s, pool, [0], [0, n], [0], w.H, D, nthreads=threads)
        return time.perf_counter() - t0
    reqs = sample["reqs"]
    cu = w.cu_seqlens.numpy()
    rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in reqs])
    q, k, v = (t.float().numpy()[rows].astype(np.float64) for t in (w.q, w.k, w.v))
    lens = [int(cu[b + 1] - cu[b]) for b in reqs]
    sub_cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    pool = w.prefix_states[reqs].double().numpy()
    pm = w.prefix_mask.numpy()[reqs]
    nr = len(reqs)
    if w.track_lens is not None:
        # snapshots go to slots nr .. 2 nr - 1 of the sample's pool
        pool = np.concatenate([pool, np.zeros_like(pool)])
        t0 = time.perf_counter()
        oracle.extend_tracked(q, k, v, s, pool, np.arange(nr, dtype=np.int32), sub_cu, pm,
                              w.track_lens.numpy()[reqs], np.arange(nr, 2 * nr, dtype=np.int32),
                              w.H, D, nthreads=threads)
        return time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.extend(q, k, v, s, pool, np.arange(nr, dtype=np.int32), sub_cu, pm, w.H, D,
                  nthreads=threads)
    return time.perf_counter() - t0


ORACLE_BUDGET = {  # (request, head) pairs or token-heads per sample: ~1-10 s of fp64 CPU work
    "decode": 4096, "verify": 64 * 5 * 16, "varlen_extend": 16 * 2400, "long_prefill": 32 * 1200,
    "verify_tree": 64 * 8 * 8, "varlen_extend_tracked": 16 * 2400, "verify_commit": 64 * 5 * 16,
    "varlen_extend_b1024": 16 * 2400, "varlen_extend_skewed": 16 * 2400}


def cpu_baseline(name, w, threads):
    """The oracle as it stands on all host cores, and on one thread (on a quarter of the sample,
    so that the single-thread leg stays within seconds)."""
    sample = oracle_sample(w, ORACLE_BUDGET[name])
    secs = run_oracle_sample(w, sample, threads)
    single = oracle_sample(w, max(1, ORACLE_BUDGET[name] // 4))
    secs1 = run_oracle_sample(w, single, 1)
    return {"value": sample["tokens"] / secs, "unit": "tokens/s", "cores": threads,
            "kind": "oracle", "sample": sample["desc"], "seconds": round(secs, 3),
            "single_thread": {"value": single["tokens"] / secs1, "cores": 1,
                              "sample": single["desc"], "seconds": round(secs1, 3)}}


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


# ----------------------------------------------------------------------------------------------

def workload_config(name, w, world):
    cfg = {"workload": w.name, "H": w.H, "head_dim": D, "layer_id": w.layer_id, "L": w.L,
           "requests_per_gpu": w.B, "tokens_per_gpu_step": algorithmic(w)["tokens"],
           "parallelism": f"replicas{world}" if world > 1 else "single_gpu",
           "l2": "inputs larger than L2 (129 MB); no flush"}
    if w.kind in ("verify", "tree"):
        cfg["draft_tokens"] = w.N
    if w.kind == "tree":
        cfg["tree_parents"] = [int(x) for x in w.parents[0]]
    if w.kind == "decode":
        cfg["pool_slots"] = w.num_slots
    return cfg


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", choices=list(KERNEL_SOURCE), default=HEADLINE)
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--profile-calls", type=int, default=0,
                    help="untimed: make this many library calls on --workload (or "
                         "--profile-case) on cuda:0 and exit; the command an ncu capture runs")
    ap.add_argument("--profile-case", choices=list(PROFILE_CASES), default=None)
    args = ap.parse_args()

    if args.impl == "reference":
        return main_reference(args)
    if args.profile_calls > 0:
        return main_profile(args)

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    init_dist("nccl")
    import lightning_attention_gb300 as la
    la.load()
    peaks = read_peaks()

    sampler = ClockSampler(local) if rank == 0 else None
    head = time_gpu(args.workload, args.steps, args.warmup, world, rank, dev, peaks,
                    with_e2e=True, sampler=sampler)
    w = head["workload"]
    line = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if w.kind != "extend" else "bf16",
            "data": "synthetic (seeded; see lightning_attention_gb300/workloads.py)",
            "config": workload_config(args.workload, w, world),
            "roofline": head["roofline"], "e2e": head["e2e"], "gpu_launches": head["gpu_launches"],
            "host_enqueue_us_per_call": head["host_enqueue_us_per_call"],
            "clocks": head["clocks"]}
    if "tensor" in head:
        line["tensor"] = head["tensor"]
    if head.get("index_order"):
        line["index_order"] = head["index_order"]
    threads = os.cpu_count() or 1
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(args.workload, w, threads)
        line["cpu_baseline"]["cpu"] = cpu_model()
    del head, w
    torch.cuda.empty_cache()

    if not args.headline_only:
        others = []
        for name in OTHER_ORDER:
            if name == args.workload:
                continue
            steps = max(3, min(args.steps, 20))
            smp = ClockSampler(local) if rank == 0 else None
            r = time_gpu(name, steps, max(3, args.warmup), world, rank, dev, peaks,
                         with_e2e=True, sampler=smp, repeats=3)
            others.append(compact_entry(r, steps, cpu_baseline(name, r["workload"], threads)
                                        if rank == 0 else None))
            del r
            torch.cuda.empty_cache()
        line["other_workloads"] = others
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# The other workloads, each timed like the headline (3 repeats of up to 20 steps, clocks sampled
# over them).  The chain verify of 128 x 5 draft tokens comes last so that it is in the tail of
# the printed line.
OTHER_ORDER = ("varlen_extend_b1024", "varlen_extend_skewed", "verify_tree",
               "varlen_extend_tracked", "verify_commit", "varlen_extend", "long_prefill", "verify")


def compact_entry(r, steps, cpu):
    roof = r["roofline"]
    e = {"workload": r["workload"].name, "value": r["value"], "unit": "tokens/s",
         "steps": steps, "ms_per_step": round(r["ms_per_step"], 4), "spread": r["spread"],
         "roofline": {"bound": roof["bound"], "achieved": roof["achieved"], "peak": roof["peak"],
                      "unit": roof["unit"], "frac": roof["frac"], "traffic": roof["traffic"],
                      "algorithmic_bytes_per_launch": roof["algorithmic_bytes_per_launch"],
                      "kernel": roof["kernel"]},
         "gpu_launches": r["gpu_launches"],
         "host_enqueue_us_per_call": r["host_enqueue_us_per_call"]}
    if r.get("index_order"):
        e["index_order"] = r["index_order"]
    if r.get("clocks"):
        c = r["clocks"]
        e["clocks"] = {"sm_mhz": c.get("sm_mhz"), "sm_max_mhz": c.get("sm_max_mhz"),
                       "reasons": c.get("reasons")}
    if r.get("e2e"):
        x = r["e2e"]
        e["e2e"] = {"value": x["value"], "unit": x["unit"],
                    "h2d_bytes_per_step": x["h2d_bytes_per_step"],
                    "d2h_bytes_per_step": x["d2h_bytes_per_step"]}
    if "tensor" in r:
        t = r["tensor"]
        e["tensor"] = {"recurrence_frac_of_bf16_peak": t["frac_of_bf16_peak"],
                       "issued_frac_of_bf16_peak": t["issued_frac_of_bf16_peak"]}
    if cpu is not None:
        e["cpu_baseline"] = {"value": cpu["value"], "cores": cpu["cores"], "kind": "oracle",
                             "single_thread_value": cpu["single_thread"]["value"]}
    return e


def main_profile(args):
    """The workload's step, args.profile_calls times, with nothing timed or printed but a final
    status line: what an ncu capture of one kernel runs (-k / -s / -c select the launch)."""
    import lightning_attention_gb300 as la
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.profile_case:
        w, name = PROFILE_CASES[args.profile_case](), args.profile_case
        kname = {"verify_b32": "verify", "verify_tree_b32": "verify_tree",
                 "extend_many_b256": "varlen_extend_b1024"}[name]
    else:
        w, name = make_workload(args.workload, 0), args.workload
        kname = name
    case = GpuCase(w, dev, kname)
    for _ in range(args.profile_calls):
        case.step()
    la.poll_error()
    torch.cuda.synchronize(dev)
    print(f"profile run ok: {w.name}, {args.profile_calls} calls", flush=True)


def calibrated_sample(name, w, threads, seconds_per_step):
    """Shrink the oracle sample so that one step takes about seconds_per_step (never larger
    than the workload's default sample)."""
    budget = ORACLE_BUDGET[name]
    probe = oracle_sample(w, max(1, budget // 16))
    t = run_oracle_sample(w, probe, threads)
    per_token = t / max(1, probe["tokens"])
    full = oracle_sample(w, budget)
    if per_token * full["tokens"] <= seconds_per_step:
        return full
    scale = seconds_per_step / (per_token * full["tokens"])
    return oracle_sample(w, max(1, int(budget * scale)))


def main_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return  # rank 0 alone times the CPU oracle
    import oracle
    oracle.build()
    name = args.workload
    w = make_workload(name, 0)
    threads = os.cpu_count() or 1
    # size each step so that warmup + steps take about two minutes in all
    per_step = min(10.0, 120.0 / max(1, args.steps + args.warmup))
    sample = calibrated_sample(name, w, threads, per_step)
    for _ in range(args.warmup):
        run_oracle_sample(w, sample, threads)
    total = 0.0
    for _ in range(args.steps):
        total += run_oracle_sample(w, sample, threads)
    value = sample["tokens"] * args.steps / total
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; see lightning_attention_gb300/workloads.py)",
            "config": workload_config(name, w, 1), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                             "kind": "oracle", "sample": sample["desc"], "cpu": cpu_model()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "note": "the reference arm is the fp64 CPU oracle (there is no reference code for "
                    "this path); each step is a bounded sample of the workload"}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
