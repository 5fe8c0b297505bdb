#!/usr/bin/env python
"""Throughput benchmark for index-gathered attention with sinks on GB300.

Default workload: the windowed vision-encoder attention (bf16): 256 varlen
sequences with lengths ~ U{64..1024}, 16 query heads, head dim 128, window 128,
non-causal. One step runs the whole workload: both KV-head counts (16 and 8)
and both sink semantics (key-0 bias and null logit), four launches of
sattn_window_fwd over device-resident inputs. The metric is queries/s (query
tokens per second, all four passes counted).

Other workloads (--workload decode | prefill | decode_fp8 | prefill_fp8 |
block | select | index | compress) measure the gathered decode / prefill path
(bf16 or FP8 cache), the chunked block-sparse path, the block selection that
produces its mask, the cache bookkeeping (index lists + ring write) and the
compressor's gated pooling the same way.

Output: one JSON line on rank 0. Timing: W warm-up steps, then K steps between
a barrier + device synchronisation on both sides, CUDA events on the launch
stream around every launch; inputs are larger than L2 (config "l2" says
which).

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# the ncu record behind each workload's roofline.traffic: (kernel, source file);
# bytes per unit of the workload (query, or compressed row)
TRAFFIC_RECORD = {
    "decode": ("sparse_decode_kernel", "sparse_decode.cu"),
    "prefill": ("sparse_tc_kernel<prefill>", "sparse_tc.cu"),
    "decode_fp8": ("sparse_decode_kernel<fp8>", "sparse_decode.cu"),
    "prefill_fp8": ("sparse_tc_kernel<prefill_fp8>", "sparse_tc.cu"),
    "block": ("attn_tc_kernel<block>", "attn_tc.cu"),
    "select": ("xattn_tc_kernel<1>", "xattn.cu"),
    "compress": ("compress_kernel", "compress.cu"),
}


def code_sha256(path):
    """sha256 of a C/C++/CUDA source with its comments and whitespace removed:
    it changes when the code changes, not when a comment does."""
    import hashlib
    import re

    with open(path) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return hashlib.sha256("".join(src.split()).encode()).hexdigest()


def profiled_traffic(kernel, source_name, units):
    """DRAM bytes per launch from the committed ncu record, scaled to `units`
    query tokens; None when the kernel's code changed since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel]
        sha = code_sha256(os.path.join(ROOT, "windowed_attention_sinks_gb300", "csrc", source_name))
    except (OSError, KeyError, ValueError):
        return None
    if sha != rec.get("code_sha256"):
        return None
    return rec["bytes_per_query_token"] * units


# ---------------------------------------------------------------- workloads

def window_work(seed, num_seqs=256):
    """Both KV-head variants and both sink modes of the vision workload."""
    from windowed_attention_sinks_gb300 import workloads as W

    passes = []
    for hkv in (16, 8):
        case = W.window_vision_bf16(seed, hkv, num_seqs=num_seqs)
        for mode in (W.SINK_KEY0_BIAS, W.SINK_NULL_LOGIT):
            passes.append((case, mode))
    return passes


def window_counts(case):
    """Algorithmic bytes and FLOPs of one window pass over the workload."""
    lens = np.diff(case.cu_seqlens).astype(np.int64)
    T, H, Hkv, d, w = case.T, case.H, case.Hkv, case.d, case.window_left
    pairs = 0
    for L in lens:
        i = np.arange(L)
        pairs += int((np.minimum(L - 1, i + w) - np.maximum(0, i - w) + 1).sum())
    bytes_ = 2 * T * H * d * 2 + 2 * T * Hkv * d * 2 + T * H * 4
    flops = 4 * d * pairs * H
    return bytes_, flops


def run_sattn(args, rank, world, device):
    import torch

    import windowed_attention_sinks_gb300 as sa

    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream()
    peaks, peaks_src = load_peaks()
    seed = rank_seed(rank)  # each rank owns an independent batch (weak scaling)
    if args.workload != "window":
        return run_other(args, rank, world, device, peaks, peaks_src)

    passes = window_work(seed, args.seqs)
    dev_inputs = {}
    launches = []
    total_q, total_bytes, total_flops = 0, 0, 0
    for case, mode in passes:
        key = id(case)
        if key not in dev_inputs:
            bf = torch.bfloat16
            dev_inputs[key] = dict(
                q=torch.from_numpy(case.q).to(bf).to(device),
                k=torch.from_numpy(case.k).to(bf).to(device),
                v=torch.from_numpy(case.v).to(bf).to(device),
                cu=torch.from_numpy(case.cu_seqlens).to(device),
                sinks=torch.from_numpy(case.sinks).to(device))
            dev_inputs[key]["o"] = torch.empty_like(dev_inputs[key]["q"])
            dev_inputs[key]["lse"] = torch.empty((case.T, case.H), dtype=torch.float32,
                                                 device=device)
        t = dev_inputs[key]
        b, f = window_counts(case)
        launches.append((case, mode, t, b, f))
        total_q += case.T
        total_bytes += b
        total_flops += f

    def one_step(events=None):
        for i, (case, mode, t, _, _) in enumerate(launches):
            if events is not None:
                events[i][0].record(stream)
            sa.window_fwd(t["q"], t["k"], t["v"], t["cu"], case.max_seqlen, case.window_left,
                          case.window_right, False, t["sinks"], mode, case.scale,
                          o=t["o"], lse=t["lse"], stream=stream)
            if events is not None:
                events[i][1].record(stream)

    for _ in range(args.warmup):
        one_step()
    sa.check_device(stream)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in launches] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(gpu_index(device)) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for s in range(args.steps):
            one_step(ev[s])
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = t0.elapsed_time(t1)
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    launch_ms = [[a.elapsed_time(b) for a, b in row] for row in ev]
    avg_launch_ms = float(np.mean(launch_ms))
    sa.check_device(stream)

    ms_per_step = elapsed_ms / args.steps
    value = whole_job_rate(total_q, world, ms_per_step)
    # Roofline of the dominant launch (Hkv = 16: the most bytes per launch),
    # the median over its key-0 and null-logit launches; beside it every
    # launch's own figure and the whole step's (all four launches' bytes over
    # the sum of their median times).
    lm = np.array(launch_ms)  # [steps, launches]
    med = np.median(lm, axis=0)
    dom = [i for i, (c, _, _, _, _) in enumerate(launches) if c.Hkv == max(x[0].Hkv for x in launches)]
    dom_ms = float(np.median(lm[:, dom]))
    dom_bytes, dom_flops = launches[dom[0]][3], launches[dom[0]][4]
    achieved_gbs = dom_bytes / (dom_ms / 1e3) / 1e9
    achieved_tf = dom_flops / (dom_ms / 1e3) / 1e12
    peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    traffic = profiled_traffic("attn_tc_kernel<window>", "attn_tc.cu", launches[dom[0]][0].T)
    variants = [{"hkv": c.Hkv, "sink_mode": "key0_bias" if m == 1 else "null_logit",
                 "ms": float(med[i]), "gbs": b / (float(med[i]) / 1e3) / 1e9,
                 "frac": b / (float(med[i]) / 1e3) / 1e9 / peak}
                for i, (c, m, _, b, _) in enumerate(launches)]
    step_gbs = total_bytes / (float(med.sum()) / 1e3) / 1e9
    out = {
        "metric": "queries/s (window attention, bf16, 256 varlen seqs, H=16, Hkv 16+8, "
                  "d=128, w=128, key0_bias+null_logit)",
        "value": value, "unit": "queries/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded numpy PCG64, bf16)",
        "config": {"workload": "window-vision-bf16: %d seqs U{64..1024}, H=16, Hkv in {16,8}, "
                               "d=128, w=128, non-causal, sinks key0_bias and null_logit "
                               "(4 launches per step)" % args.seqs,
                   "tokens_per_pass": int(launches[0][0].T), "launches_per_step": len(launches),
                   "l2": "inputs larger than L2 (1.7-2.3 GB per launch), no flush",
                   "parallelism": "replicas (dp%d, independent batches)" % world},
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                     "frac": achieved_gbs / peak, "traffic": traffic,
                     "peak_source": peaks_src,
                     "kernel": "attn_tc_kernel<window> (Hkv=16 launches)",
                     "launch_ms": dom_ms, "algorithmic_bytes": dom_bytes,
                     "avg_launch_ms_all": avg_launch_ms, "tflops": achieved_tf,
                     "tensor_frac": achieved_tf / peaks.get("bf16_tflops_sustained", 1700.0),
                     "variants": variants,
                     "whole_step": {"achieved": step_gbs, "frac": step_gbs / peak,
                                    "bytes": int(total_bytes), "ms": float(med.sum())},
                     "timing": "median of %d steps per launch" % args.steps},
        "gpu_launches": len(launches) * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_e2e:
        out["e2e"] = e2e_window(args, launches, device, stream)
    if not args.no_paths:
        # the other paths of the hot path, each timed in this run (median of 50)
        for t in dev_inputs.values():
            t.clear()
        torch.cuda.empty_cache()
        out["paths"] = measure_paths(["decode", "prefill", "block"], rank, world, device, peaks,
                                     peaks_src)
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_window(launches)
    return out


def e2e_window(args, launches, device, stream):
    """Same metric through the public API with host buffers. Every step copies
    each distinct input (q/k/v/cu/sinks of a KV-head variant; its two sink
    modes share them) host->device from pinned memory and reads every pass's
    o/lse back. Input copies run on one stream, the kernels on the compute
    stream, the result reads on a third, ordered by events, so that copies in
    both directions overlap the kernels of neighbouring passes."""
    import torch

    import windowed_attention_sinks_gb300 as sa

    inputs = {}  # one host/device set per distinct case
    passes = []
    h2d = d2h = 0
    for case, mode, t, _, _ in launches:
        key = id(case)
        if key not in inputs:
            hx = {n: t[n].cpu().pin_memory() for n in ("q", "k", "v", "cu", "sinks")}
            inputs[key] = dict(host=hx, dev={n: t[n] for n in hx},
                               ready=torch.cuda.Event(), used=[])
            h2d += sum(x.numel() * x.element_size() for x in hx.values())
        o = torch.empty_like(t["o"])  # each pass its own output
        lse = torch.empty_like(t["lse"])
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hl = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        d2h += ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
        ps = dict(case=case, mode=mode, inp=inputs[key], o=o, lse=lse, ho=ho, hl=hl,
                  done=torch.cuda.Event(), read=torch.cuda.Event())
        inputs[key]["used"].append(ps)
        passes.append(ps)
    s_in = torch.cuda.Stream(device=device)
    s_out = torch.cuda.Stream(device=device)
    first_step = [True]

    def step():
        copied = set()
        for ps in passes:
            inp = ps["inp"]
            if id(inp) not in copied:
                copied.add(id(inp))
                if not first_step[0]:  # the previous step's kernels read these buffers
                    for u in inp["used"]:
                        s_in.wait_event(u["done"])
                with torch.cuda.stream(s_in):
                    for n, hx in inp["host"].items():
                        inp["dev"][n].copy_(hx, non_blocking=True)
                inp["ready"].record(s_in)
            stream.wait_event(inp["ready"])
            if not first_step[0]:
                stream.wait_event(ps["read"])  # o / lse of the previous step were read back
            d, case = inp["dev"], ps["case"]
            sa.window_fwd(d["q"], d["k"], d["v"], d["cu"], case.max_seqlen, case.window_left,
                          case.window_right, False, d["sinks"], ps["mode"], case.scale,
                          o=ps["o"], lse=ps["lse"], stream=stream)
            ps["done"].record(stream)
            s_out.wait_event(ps["done"])
            with torch.cuda.stream(s_out):
                ps["ho"].copy_(ps["o"], non_blocking=True)
                ps["hl"].copy_(ps["lse"], non_blocking=True)
            ps["read"].record(s_out)
        first_step[0] = False

    steps = max(3, min(args.steps, 10))
    step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    q = sum(ps["case"].T for ps in passes)
    return {"value": q / dt, "unit": "queries/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps,
            "schedule": "inputs copied once per step on a copy stream, kernels on the compute "
                        "stream, results read back on a third stream (event-ordered)"}


def cpu_baseline_window(launches, budget_s=15.0):
    """The fp64 oracle, as it stands, on a bounded sample of the same workload:
    whole sequences (all heads) until ~budget_s of CPU work is spent."""
    import oracle

    oracle.build()
    cores = oracle.get_threads()
    done_q, spent, seqs = 0, 0.0, 0
    case, mode = launches[0][0], launches[0][1]
    lens = np.diff(case.cu_seqlens)
    t_start = time.perf_counter()
    for s in range(len(lens)):
        a, b = int(case.cu_seqlens[s]), int(case.cu_seqlens[s + 1])
        rows = np.arange(a * case.H, b * case.H, dtype=np.int64)
        oracle.window(case.q, case.k, case.v, case.cu_seqlens, case.H, case.Hkv, case.d,
                      case.window_left, case.window_right, 0, case.sinks, mode, case.scale,
                      rows=rows)
        done_q += b - a
        seqs += 1
        spent = time.perf_counter() - t_start
        if spent > budget_s:
            break
    return {"value": done_q / spent, "unit": "queries/s", "cores": cores, "kind": "oracle",
            "sample": "%d of 256 sequences (%d query tokens x 16 heads) of the Hkv=16 key0_bias "
                      "pass, fp64, %.1f s" % (seqs, done_q, spent)}


class Path:
    """One measured path: a launch function over device-resident inputs and
    its algorithmic work per step."""

    def __init__(self, **kw):
        self.__dict__.update(kw)


def build_path(workload, seed, device, stream):
    """Inputs and launch function of a non-window workload (decode | prefill |
    decode_fp8 | prefill_fp8 | block | select | index | compress)."""
    import torch

    import windowed_attention_sinks_gb300 as sa
    from windowed_attention_sinks_gb300 import workloads as W

    bf = torch.bfloat16
    if workload in ("decode", "prefill", "decode_fp8", "prefill_fp8"):
        fp8 = workload.endswith("_fp8")
        decode = workload.startswith("decode")
        case = W.sparse_decode_bf16(seed) if decode else W.sparse_prefill_bf16(seed)
        # a step's inputs (q, index lists) and outputs (o, lse) each live in one
        # device buffer, so that the end-to-end step moves each way in one copy
        qb, ib = case.q.size * 2, case.idx.size * 4
        inbuf = torch.empty(qb + ib, dtype=torch.uint8, device=device)
        q = inbuf[:qb].view(bf).view(case.q.shape)
        q.copy_(torch.from_numpy(case.q).to(bf))
        idx = inbuf[qb:].view(torch.int32).view(case.idx.shape)
        idx.copy_(torch.from_numpy(case.idx))
        kv = torch.from_numpy(case.kv).to(bf).to(device)
        sinks = torch.from_numpy(case.sinks).to(device)
        outbuf = torch.empty(qb + case.B * case.M * case.H * 4, dtype=torch.uint8, device=device)
        o = outbuf[:qb].view(bf).view(case.q.shape)
        lse = outbuf[qb:].view(torch.float32).view(case.B, case.M, case.H)
        nb = sa.sparse_workspace_bytes(case.B, case.M, case.H, case.d, case.K)
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=device)
        valid = int((case.idx >= 0).sum())
        # a gathered row: 2 d bytes, or (FP8 cache, RoPE half in bf16) d/2 codes +
        # d bytes of RoPE part + a 4-byte scale
        row_bytes = (case.d // 2 + case.d + 4) if fp8 else case.d * 2
        nbytes = valid * row_bytes + case.idx.size * 4 + 2 * q.numel() * 2 + lse.numel() * 4
        if fp8:
            kv_nope, kv_rope, kv_scale = sa.quantize_kv_fp8(kv, case.d // 2)
            del kv

        def launch(st=None):
            if fp8:
                sa.sparse_fp8_fwd(q, kv_nope, kv_rope, kv_scale, idx, sinks, case.sink_mode,
                                  case.scale, o=o, lse=lse, workspace=ws, stream=st or stream)
            else:
                sa.sparse_fwd(q, kv, idx, sinks, case.sink_mode, case.scale, o=o, lse=lse,
                              workspace=ws, stream=st or stream)
        # launches per step: the cluster kernel alone for decode (its splits
        # merge on chip), the persistent kernel for prefill
        if decode:
            kernel, launches = "sparse_decode_kernel" + ("<fp8>" if fp8 else ""), 1
        else:
            kernel, launches = "sparse_tc_kernel<%s>" % workload, 1
        return Path(
            launch=launch, units=case.B * case.M, nbytes=nbytes,
            # end to end: a step's queries and index lists come from the host,
            # its o and lse go back (one staging buffer each way); the cache
            # stays resident
            e2e_in=[inbuf], e2e_out=[outbuf],
            flops=4 * case.d * valid * case.H,
            # decode is tiny: a scratch buffer larger than L2 is rewritten before each step
            flush=decode, graph=decode, launches=launches, kernel=kernel,
            bound="tensor" if not decode else "hbm",
            traffic_key=workload,
            name="sparse %s %s: B=%d M=%d H=%d d=%d N=%d K=%d null_logit" % (
                workload.replace("_fp8", ""),
                "bf16 q, FP8 cache (e4m3 + row scale, bf16 RoPE half)" if fp8 else "bf16",
                case.B, case.M, case.H, case.d, case.N, case.K))
    if workload == "index":
        # cache bookkeeping of the prefill layout: index lists of 8192 queries
        # (K = 2048, window 128, ratio 4) and the ring write of the prompt's KV
        M, K, win, ratio, d = 8192, 2048, 128, 4, 128
        starts = torch.zeros(1, dtype=torch.int32, device=device)
        idx_out = torch.empty((1, M, K), dtype=torch.int32, device=device)
        cache = torch.zeros((1, win + 8192, d), dtype=bf, device=device)
        new_kv = torch.randn((1, M, d), device=device).to(bf)

        side = torch.cuda.Stream(device=device)

        def launch(st=None):
            # the two are independent (the lists do not read the ring): the ring
            # write runs on a second stream, joined before the step ends
            s0 = st or stream
            side.wait_stream(s0)
            sa.build_topk_idxs(starts, M, K, win, ratio, out=idx_out, stream=s0)
            with torch.cuda.stream(side):
                sa.kv_ring_write(cache, new_kv, starts, win, stream=side)
            s0.wait_stream(side)
        # the 67 MB of lists fit in L2: a larger scratch is rewritten before each step
        return Path(launch=launch, units=M, nbytes=idx_out.numel() * 4 + 2 * win * d * 2,
                    flops=0, flush=True, graph=True, launches=2, kernel="topk_idxs_kernel",
                    bound="hbm", traffic_key=None,
                    name="cache bookkeeping: topk index lists (8192 queries, K=2048, win 128, "
                         "ratio 4) + ring write")
    if workload == "select":
        # block selection over the chunked block-sparse workload's shape: the
        # last 4096 positions of a 32768-token context, H=32 over 8 KV heads,
        # eight 4096-key chunks (stats, merge, block sums, threshold 0.9)
        case = W.block_sparse_bf16(seed)
        q = torch.from_numpy(case.q).to(bf).to(device)
        k = torch.from_numpy(case.k).to(bf).to(device)
        M, H, d = case.q.shape
        Nctx = case.k.shape[0]
        chunk = case.chunks[0][1] - case.chunks[0][0]
        ws = torch.empty(sa.xattn_select_workspace_bytes(M, H, Nctx, chunk), dtype=torch.uint8,
                         device=device)
        bs = torch.empty((H, -(-M // 128), -(-Nctx // 128)), dtype=torch.float32, device=device)
        sel = torch.empty(bs.shape, dtype=torch.uint8, device=device)
        # visible (row, key) pairs of all heads; each costs one exponential per pass
        pairs = H * sum(min(Nctx, case.q_pos0 + i + 1) for i in range(M))

        def launch(st=None):
            # stats of all chunks, merge, block sums, threshold 0.9: four launches
            sa.xattn_select_blocks(q, k, case.q_pos0, True, 0.9, case.scale, chunk=chunk,
                                   workspace=ws, block_sum=bs, mask=sel, stream=st or stream)
        return Path(launch=launch, units=M, nbytes=0, flops=2 * 2 * d * pairs, pairs=pairs,
                    flush=False, graph=False, launches=4, kernel="xattn_tc_kernel",
                    bound="tensor", traffic_key="select",
                    name="block selection: ctx 32768, 4096 queries, H=32, Hkv=8, d=128, "
                         "8 x 4096-key chunks, threshold 0.9, one call")
    if workload == "compress":
        # compressor gated pooling: eight 32K-token prefills at ratio 4 with
        # overlapping windows, fp32 projections in, bf16 rows into the
        # compressed region of each request's cache
        case = W.compress_case(seed)
        B, S, Wd = case.kv.shape
        d, ratio, win = case.d, case.ratio, 128
        nwin = S // ratio
        kvp = torch.from_numpy(case.kv).to(device)
        scp = torch.from_numpy(case.score).to(device)
        ape = torch.from_numpy(case.ape).to(device)
        cache = torch.zeros((B, win + nwin, d), dtype=bf, device=device)
        rows = cache[:, win:]

        def launch(st=None):
            sa.compress_kv(kvp, scp, ape, ratio, case.overlap, out=rows, stream=st or stream)
        # every projection element read once (the last window's first half is
        # never needed), each row written once
        nbytes = (B * (nwin * ratio * d * (2 if case.overlap else 1)
                       - (ratio * d if case.overlap else 0)) * 2 * 4 + B * nwin * d * 2)
        return Path(launch=launch, units=B * nwin, nbytes=nbytes, flops=0, flush=False,
                    graph=False, launches=1, kernel="compress_kernel", bound="hbm",
                    traffic_key="compress",
                    name="compressor gated pooling: B=%d S=%d d=%d ratio=%d overlap, fp32 in, "
                         "bf16 rows" % (B, S, d, ratio))
    # block: the chunked block-sparse workload
    case = W.block_sparse_bf16(seed)
    q = torch.from_numpy(case.q).to(bf).to(device)
    k = torch.from_numpy(case.k).to(bf).to(device)
    v = torch.from_numpy(case.v).to(bf).to(device)
    mask = torch.from_numpy(case.mask).to(device)
    C = len(case.chunks)
    op = torch.empty((C, case.M * case.H, case.d), dtype=torch.float32, device=device)
    lp = torch.empty((C, case.M * case.H), dtype=torch.float32, device=device)
    o = torch.empty((case.M * case.H, case.d), dtype=bf, device=device)
    lse = torch.empty((case.M * case.H,), dtype=torch.float32, device=device)
    nblk = int(case.mask.sum())
    nbytes = (q.numel() * 2 + k.numel() * 2 + v.numel() * 2 + 2 * op.numel() * 4
              + 2 * lp.numel() * 4 + o.numel() * 2 + lse.numel() * 4)
    chunk = case.chunks[0][1] - case.chunks[0][0]

    def launch(st=None):
        # every chunk in one launch over (chunk, query block, head), then
        # the LSE merge of the eight partials
        st = st or stream
        sa.block_sparse_chunks_fwd(q, k, v, mask, case.q_pos0, 0, case.k.shape[0], chunk, True,
                                   case.scale, o_parts=op.view(C, case.M, case.H, case.d),
                                   lse_parts=lp.view(C, case.M, case.H), stream=st)
        sa.merge_lse(op, lp, case.H, o=o, lse=lse, stream=st)
    # causal pairs inside kept blocks (diagonal blocks are half visible)
    flops = 4 * case.d * (nblk * 128 * 128 - case.H * (case.M // 128) * (128 * 127 // 2))
    return Path(launch=launch, units=case.M, nbytes=nbytes, flops=flops, flush=False,
                graph=False, launches=2, kernel="attn_tc_kernel<block>", bound="hbm",
                traffic_key="block",
                name="block-sparse bf16: ctx 32768, 4096 queries, H=32, Hkv=8, d=128, 8 chunks "
                     "in one launch + merge")


def time_path(p, steps, warmup, stream, world=1, clk=None):
    """Per-step device times (ms) of a path, each step bracketed by CUDA events
    on the launch stream: `cold` with L2 flushed (p.flush) or inputs larger
    than L2, and `warm`, the same steps back to back without a flush."""
    import torch

    import windowed_attention_sinks_gb300 as sa

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=stream.device) if p.flush else None
    for _ in range(warmup):
        p.launch()
    sa.check_device(stream)
    graph = None
    if p.graph:
        # a step of ~10-30 us of device work is replayed from a CUDA graph so
        # that host-side enqueue time stays out of the timed region
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            p.launch(torch.cuda.current_stream())
        graph.replay()
        torch.cuda.synchronize()
        sa.check_device(stream)

    def run(n, flushed, use_graph=True):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        barrier(world)
        torch.cuda.synchronize()
        for s in range(n):
            if flushed and flush is not None:
                flush.fill_(s & 0xff)
            evs[s][0].record(stream)
            if graph is not None and use_graph:
                graph.replay()
            else:
                p.launch()
            evs[s][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return [a.elapsed_time(b) for a, b in evs]

    if clk is not None:
        with clk:
            cold = run(steps, True)
    else:
        cold = run(steps, True)
    warm = run(max(steps, 20), False)
    if graph is not None:
        # 100 replays back to back between two events: launches pipeline
        # behind each other, which exposes what one launch costs in a stream
        # of them
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(100):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        p.back_to_back_ms = e0.elapsed_time(e1) / 100
        if flush is not None:
            # the same steps launched directly: behind the flush kernel the
            # host's enqueue stays out of the timed region as well, and a
            # directly launched cluster kernel starts sooner than one replayed
            # from a graph
            p.direct_ms = max_over_ranks(float(np.median(run(steps, True, use_graph=False))),
                                         world)
    sa.check_device(stream)
    return cold, warm, graph is not None


def time_path_e2e(p, steps, stream):
    """Queries/s through the public API with host buffers: every step copies
    its inputs host->device from pinned memory, launches, and reads its
    outputs back (one stream, synchronised at the end of each step)."""
    import torch

    hin = [t.cpu().pin_memory() for t in p.e2e_in]
    hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in p.e2e_out]
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout)

    def step():
        with torch.cuda.stream(stream):
            for d, h in zip(p.e2e_in, hin):
                d.copy_(h, non_blocking=True)
            p.launch(stream)
            for h, d in zip(hout, p.e2e_out):
                h.copy_(d, non_blocking=True)
        stream.synchronize()

    def timed(fn):
        for _ in range(3):
            fn()
        t0 = time.perf_counter()
        for _ in range(steps):
            fn()
        return (time.perf_counter() - t0) / steps

    dt = timed(step)
    rec = {"value": p.units / dt, "unit": "queries/s", "ms": dt * 1e3,
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
           "schedule": "queries and index lists copied in from one pinned host buffer, the call, "
                       "o and lse copied back into one, one stream, synchronised every step"}
    if p.graph:
        # the way a decode server runs a step: the copy in, the call and the copy
        # back captured once as a CUDA graph over the same pinned staging
        # buffers (new inputs are written there before each replay)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):  # captured on a side stream of torch's
            cs = torch.cuda.current_stream()
            for d, h in zip(p.e2e_in, hin):
                d.copy_(h, non_blocking=True)
            p.launch(cs)
            for h, d in zip(hout, p.e2e_out):
                h.copy_(d, non_blocking=True)

        def replay():
            g.replay()
            torch.cuda.synchronize()

        dt_g = timed(replay)
        rec["direct"] = {"value": rec["value"], "ms": rec["ms"], "schedule": rec["schedule"]}
        rec.update({"value": p.units / dt_g, "ms": dt_g * 1e3,
                    "schedule": "copy in from one pinned host buffer, the call, copy back into "
                                "one: captured once as a CUDA graph and replayed, synchronised "
                                "every step (`direct`: the same issued call by call)"})
    return rec


def path_record(p, cold, warm, peaks, peaks_src, world, clk_mhz=None, sm_count=152):
    """Median step time, its roofline and the labelled warm-L2 figure."""
    ms = max_over_ranks(float(np.median(cold)), world)
    ms_warm = max_over_ranks(float(np.median(warm)), world)
    gbs = p.nbytes / (ms / 1e3) / 1e9
    tf = p.flops / (ms / 1e3) / 1e12
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    tpeak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    if p.bound == "tensor":
        roof = {"bound": "tensor", "achieved": tf, "peak": tpeak, "unit": "TFLOP/s",
                "frac": tf / tpeak}
        if p.nbytes:
            # the gathered-bytes convention beside it (the cache may live in L2)
            roof["gathered_bytes"] = {"achieved": gbs, "peak": hbm, "unit": "GB/s",
                                      "frac": gbs / hbm}
        if getattr(p, "pairs", None):
            # one MUFU ex2 per visible pair and pass, 32 per clock per SM
            ex2_peak = 32 * sm_count * (clk_mhz or 2070.0) * 1e6 / 1e12
            ex2 = 2 * p.pairs / (ms / 1e3) / 1e12
            roof["ex2"] = {"achieved": ex2, "peak": ex2_peak, "unit": "Tex2/s",
                           "frac": ex2 / ex2_peak}
    else:
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                "frac": gbs / hbm}
    roof["traffic"] = (profiled_traffic(*TRAFFIC_RECORD[p.traffic_key], p.units)
                       if p.traffic_key in TRAFFIC_RECORD else None)
    roof["peak_source"] = peaks_src
    roof["tflops"] = tf
    roof["tensor_frac"] = tf / peaks.get("bf16_tflops_sustained", 1700.0)
    rec = {"ms": ms, "ms_mean": float(np.mean(cold)), "runs": len(cold),
           "value": whole_job_rate(p.units, world, ms), "unit": "queries/s",
           "warm_l2_ms": ms_warm, "launches_per_step": p.launches, "kernel": p.kernel,
           "roofline": roof}
    if getattr(p, "back_to_back_ms", None) is not None:
        rec["back_to_back_ms"] = p.back_to_back_ms
    if getattr(p, "direct_ms", None) is not None:
        rec["direct_launch_ms"] = p.direct_ms  # the same steps launched directly (labelled)
    return rec


def run_other(args, rank, world, device, peaks, peaks_src):
    """Decode / prefill / block-sparse / ... measurement lines (same JSON shape)."""
    import torch

    stream = torch.cuda.current_stream()
    p = build_path(args.workload, rank_seed(rank), device, stream)
    clk = ClockSampler(gpu_index(device))
    cold, warm, graphed = time_path(p, args.steps, args.warmup, stream, world, clk)
    summ = clk.summary()
    rec = path_record(p, cold, warm, peaks, peaks_src, world, summ.get("sm_mhz"),
                      torch.cuda.get_device_properties(device).multi_processor_count)
    unit_name = "compressed rows" if args.workload == "compress" else "queries"
    e2e = None
    if getattr(p, "e2e_in", None) and not args.no_e2e:
        e2e = time_path_e2e(p, max(args.steps, 10), stream)
    out = {
        "metric": "%s/s (%s)" % (unit_name, args.workload),
        "value": rec["value"],
        "unit": "%s/s" % unit_name, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": rec["ms"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if args.workload == "compress" else "bf16",
        "data": "synthetic (seeded numpy PCG64%s)" % (
            ", fp32 projections" if args.workload == "compress" else ", bf16"),
        "config": {"workload": p.name,
                   "l2": "scratch > L2 rewritten before each step" if p.flush
                   else "inputs larger than L2",
                   "launch": "CUDA graph replay" if graphed else "direct",
                   "timing": "median of %d steps (ms_mean beside it); warm_l2_ms: the same "
                             "steps back to back, no flush" % args.steps},
        "roofline": rec["roofline"],
        "ms_mean": rec["ms_mean"], "warm_l2_ms": rec["warm_l2_ms"],
        "back_to_back_ms": rec.get("back_to_back_ms"),
        "direct_launch_ms": rec.get("direct_launch_ms"),
        "gpu_launches": args.steps * p.launches,
        "clocks": summ,
    }
    if e2e is not None:
        out["e2e"] = e2e
    return out


def measure_paths(names, rank, world, device, peaks, peaks_src, steps=50, warmup=5):
    """The `paths` record of the default line: each named path measured in the
    same run (median of `steps` timed steps after `warmup`)."""
    import torch

    stream = torch.cuda.current_stream()
    out = {}
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    for name in names:
        p = build_path(name, rank_seed(rank), device, stream)
        cold, warm, graphed = time_path(p, steps, warmup, stream, world)
        rec = path_record(p, cold, warm, peaks, peaks_src, world, None, sms)
        rec["workload"] = p.name
        rec["launch"] = "CUDA graph replay, L2 flushed" if graphed else "direct"
        if getattr(p, "e2e_in", None):
            rec["e2e"] = time_path_e2e(p, steps, stream)
        out[name] = rec
        del p
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    """The fp64 oracle timed on the host cores: each step is a bounded sample
    (two whole sequences, all heads, one pass) of the default workload."""
    import oracle
    from windowed_attention_sinks_gb300 import workloads as W

    if rank != 0:
        return None
    oracle.build()
    case = W.window_vision_bf16(1000, 16)
    lens = np.diff(case.cu_seqlens)

    def step(s):
        a = int(case.cu_seqlens[(2 * s) % 256])
        b = int(case.cu_seqlens[(2 * s) % 256 + 2])
        rows = np.arange(a * case.H, b * case.H, dtype=np.int64)
        oracle.window(case.q, case.k, case.v, case.cu_seqlens, case.H, case.Hkv, case.d,
                      case.window_left, case.window_right, 0, case.sinks, 1, case.scale,
                      rows=rows)
        return b - a

    for s in range(args.warmup):
        step(s)
    t0 = time.perf_counter()
    q = sum(step(args.warmup + s) for s in range(args.steps))
    dt = time.perf_counter() - t0
    value = q / dt
    cores = oracle.get_threads()
    sample = "two whole sequences (all 16 heads) of the Hkv=16 key0_bias pass per step, fp64"
    return {"impl": "reference", "metric": "queries/s (window attention, bf16, 256 varlen seqs, "
            "H=16, Hkv 16+8, d=128, w=128, key0_bias+null_logit)",
            "value": value, "unit": "queries/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy PCG64, bf16 inputs)",
            "config": {"workload": "window-vision-bf16: 256 seqs U{64..1024}, H=16, Hkv in "
                                   "{16,8}, d=128, w=128 (oracle sample: two sequences of the "
                                   "Hkv=16 key0_bias pass per step)"},
            "cpu_baseline": {"value": value, "unit": "queries/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


# ---------------------------------------------------------------- distributed plumbing

def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(rank):
    """Seed of the batch rank `rank` owns: every rank runs an independent batch of
    the same shape (weak scaling, no data-path collective)."""
    return 1000 + rank


def whole_job_rate(units_per_rank, world, ms_max):
    """Units all ranks processed per second, over the slowest rank's time."""
    return units_per_rank * world / (ms_max / 1e3)


def gpu_index(device):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v for v in vis.split(",") if v.strip()]
        if device < len(ids) and ids[device].strip().isdigit():
            return int(ids[device])
    return device


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="sattn", choices=["sattn", "reference"])
    ap.add_argument("--workload", default="window", choices=["window", "decode", "prefill",
                                                              "block", "index", "compress",
                                                              "decode_fp8", "prefill_fp8",
                                                              "select"])
    ap.add_argument("--seqs", type=int, default=256,
                    help="window workload: number of sequences (256 = the full workload)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-paths", action="store_true",
                    help="window workload: skip the decode / prefill / block-sparse sub-record")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    import torch

    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    from windowed_attention_sinks_gb300 import build

    build.build()
    out = run_sattn(args, rank, world, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
