"""Throughput of the tile-sparse masked attention hot path on one GB300.

A step is one pass of the whole path over one batch of synthetic input:
fa_create_block_mask + fa_forward_prepare_backward + fa_backward_prepared (the
forward and backward of fa_forward / fa_backward, with the clearing of the
backward's fp32 dq accumulator moved into the forward).  The default workload is the
largest single-GPU one, the window-growth sweep (B=1, H=16, S=65536, D=128,
causal & same document & window W, ALiBi, log-normal document lengths): one
step runs the path once for every W of the sweep, 64..1792 in steps of 64,
each W read by the kernels from a device int32 (no rebuild).  The metric is
attention TFLOP/s counted over visible tiles only: forward 4*128*128*D per
visible tile per (b, h), backward 2.5x that (five tile GEMMs against two).
The other workloads are timed in the same run for the per-config keys.

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import WORKLOADS, make_doc_ids, make_qkv  # noqa: E402

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
METRIC = "attention TFLOP/s over visible tiles (fwd+bwd)"


# The translation unit each profiled kernel is compiled from; every kernel also
# includes the shared headers and the C header.
KERNEL_SOURCES = {"fwd_kernel": "fwd.cu", "bwd_kernel": "bwd.cu", "classify_kernel": "builder.cu",
                  "row_segs_kernel": "builder.cu", "decode_partial_kernel": "decode.cu"}
SHARED_HEADERS = ("common.cuh", "internal.h", "ptx.cuh")


def source_digest(kernel: str, read=None) -> str:
    """sha256 over the files `kernel` is compiled from: its .cu, the shared
    headers and include/fa.h.  `read(relpath) -> bytes` defaults to the
    working tree (a recording script passes the sources of the capture)."""
    import hashlib

    def _read(rel):
        with open(os.path.join(ROOT, rel), "rb") as f:
            return f.read()

    read = read or _read
    h = hashlib.sha256()
    csrc = "block_sparse_masked_fa_gb300/csrc/"
    for name in sorted((KERNEL_SOURCES[kernel],) + SHARED_HEADERS):
        h.update(name.encode() + b"\0" + read(csrc + name))
    h.update(read("include/fa.h"))
    return h.hexdigest()


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu record, or None when
    the record is missing, was taken on another workload, or the kernel's sources
    have changed since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    for entry in rec.get("records", []):
        if (entry.get("kernel") == kernel and entry.get("workload") == workload
                and entry.get("source_sha256") == source_digest(kernel)):
            return entry.get("dram_bytes_per_launch")
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return PEAKS_FALLBACK, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return self.summarise(self.lines)

    @staticmethod
    def summarise(lines):
        """Median and maximum SM clock and the throttle reasons seen active, from
        nvidia-smi lines of FIELDS (unparsable lines are skipped)."""
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def workload_tensors(w, seed=None):
    seed = w.seed if seed is None else seed
    q, k, v, do = make_qkv(w.B, w.H, w.S, w.D, seed)
    docs = make_doc_ids(w.docs, w.S, w.doc_seed or seed) if w.docs is not None else None
    return q, k, v, do, docs


def mask_nodes(w, docs, W):
    """The binding's node list of the workload's mask program (docs / W on the device)."""
    nodes = []
    for node in w.mask.nodes:
        if node[0] == "same_doc":
            nodes.append(("same_doc", docs))
        elif node[0] == "window":
            nodes.append(("window", W if w.windows else int(node[1])))
        elif node[0] == "sink":
            nodes.append(("sink", int(node[1])))
        else:
            nodes.append((node[0],))
    return nodes


def builder_scaled(fa, w, W, dev, S=262144, reps=10):
    """fa_create_block_mask alone at a scaled length (the workload's mask program,
    documents drawn for S tokens): its time and achieved bandwidth over the
    algorithmic bytes -- doc ids read, four count vectors and four padded tile
    lists written."""
    import torch

    docs = None
    if w.docs is not None:
        docs = torch.as_tensor(make_doc_ids(w.docs, S, w.doc_seed or w.seed), dtype=torch.int32, device=dev)
    spec = fa.make_mask_spec(mask_nodes(w, docs, W), device=dev)
    buf = torch.empty(fa.fa_block_mask_bytes(1, 1, S, S, 128), dtype=torch.uint8, device=dev)
    for _ in range(3):
        fa.fa_create_block_mask(spec, 1, 1, S, S, 128, buffer=buf)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fa.fa_create_block_mask(spec, 1, 1, S, S, 128, buffer=buf)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    nt = S // 128
    nbytes = (S * 4 if docs is not None else 0) + 4 * nt * 4 + 4 * nt * nt * 4
    return {"S": S, "ms": round(ms, 4), "algorithmic_bytes": int(nbytes), "GB_s": round(nbytes / (ms * 1e-3) / 1e9, 1)}


def decode_point(fa, dev, hbm_gbs, B=1, H=16, kv_len=65536, D=128, reps=20):
    """The short-query forward alone (q_len 1, every key visible, a single long
    context per head): its time and achieved bandwidth over the algorithmic
    bytes -- K and V of every key, read once -- between L2 flushes."""
    import torch

    g = torch.Generator(device=dev).manual_seed(7)
    q = torch.randn(B, H, 1, D, device=dev, generator=g).to(torch.bfloat16)
    k = torch.randn(B, H, kv_len, D, device=dev, generator=g).to(torch.bfloat16)
    v = torch.randn(B, H, kv_len, D, device=dev, generator=g).to(torch.bfloat16)
    bm = fa.fa_create_block_mask([("true",)], 1, 1, 1, kv_len, 128)
    ws = torch.empty(fa.fa_forward_decode_workspace_bytes(B, H, 1, kv_len, D), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty(B, H, 1, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        fa.fa_forward_decode(q, k, v, bm, out=out, lse=lse, workspace=ws)
    times = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fa.fa_forward_decode(q, k, v, bm, out=out, lse=lse, workspace=ws)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = sorted(times)[reps // 2]
    nbytes = 2 * k.numel() * k.element_size()
    gbs = nbytes / (ms * 1e-3) / 1e9
    assert fa.fa_get_status(bm) == 0
    return {"shape": f"B{B} H{H} q_len 1 kv_len {kv_len} D{D}", "ms": round(ms, 4), "algorithmic_bytes": int(nbytes),
            "GB_s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_gbs, 3)}


def small_block_point(fa, dev, peak, S=32768, H=16, D=128, reps=10):
    """A fine-grained mask -- causal & same document, documents of geometric
    mean length 40 -- with block masks of 128 and of 64 (tutorial, sharp edge
    4): forward and backward times (median of `reps`, L2 flushed) and the tiles
    each walks.  At block 64 the forward walks 128 x 64 tiles (FLOPs
    4 * 128 * 64 * D each), the backward the same 128 x 128 tiles as at 128."""
    import torch

    q, k, v, do = (t.to(dev) for t in make_qkv(1, H, S, D, 4040))
    docs = torch.as_tensor(make_doc_ids(("geometric", 40.0), S, 4040), dtype=torch.int32, device=dev)
    spec = fa.make_mask_spec([("causal",), ("same_doc", docs), ("and",)], device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {"shape": f"B1 H{H} S{S} D{D}, causal & same document, geometric(40) documents"}
    for block in (128, 64):
        bm = fa.fa_create_block_mask(spec, 1, 1, S, S, block)
        o, lse = fa.fa_forward(q, k, v, bm)
        fa.fa_backward(q, k, v, o, lse, do, bm)
        torch.cuda.synchronize()
        assert fa.fa_get_status(bm) == 0
        times = {"fwd": [], "bwd": []}
        for _ in range(reps):
            for what in ("fwd", "bwd"):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                if what == "fwd":
                    fa.fa_forward(q, k, v, bm, out=o, lse=lse)
                else:
                    fa.fa_backward(q, k, v, o, lse, do, bm)
                e1.record()
                torch.cuda.synchronize()
                times[what].append(e0.elapsed_time(e1))
        fms, bms = (sorted(times[x])[reps // 2] for x in ("fwd", "bwd"))
        if block == 128:
            L = bm.lists()
            ft = int((L["kv_num_blocks"].long() + L["full_kv_num_blocks"].long()).sum()) * H
            bt, fkv = ft, 128
        else:
            L = bm.kernel_lists()
            ft = int((L["fwd_kv_num_blocks"].long() + L["fwd_full_kv_num_blocks"].long()).sum()) * H
            bt = int((L["bwd_q_num_blocks"].long() + L["bwd_full_q_num_blocks"].long()).sum()) * H
            fkv = 64
        fflops, bflops = ft * 4.0 * 128 * fkv * D, 2.5 * bt * 4.0 * 128 * 128 * D
        out[f"block{block}"] = {"fwd_ms": round(fms, 4), "bwd_ms": round(bms, 4),
                                "fwd_tiles": f"{ft} of 128 x {fkv}", "bwd_tiles": f"{bt} of 128 x 128",
                                "fwd_tflops": round(fflops / (fms * 1e-3) / 1e12, 2),
                                "bwd_tflops": round(bflops / (bms * 1e-3) / 1e12, 2),
                                "fwd_frac": round(fflops / (fms * 1e-3) / 1e12 / peak, 4)}
    out["fwd_time_ratio_64_over_128"] = round(out["block64"]["fwd_ms"] / out["block128"]["fwd_ms"], 3)
    return out


def visible_tiles(fa, bm, B, H):
    """Sum over (b, h) of non-empty tiles, from the block mask's counts."""
    L = bm.lists()
    per_row = (L["kv_num_blocks"].long() + L["full_kv_num_blocks"].long()).sum().item()
    rep = (B // bm.struct.Bm) * (H // bm.struct.Hm)
    return per_row * rep


def rank_env():
    """(world size, rank, local rank) from the launcher's environment; (1, 0, 0) alone."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica_seed(w, rank):
    """Each rank runs an independent replica of the workload with its own seed
    (its own documents and inputs), as data-parallel ranks each hold a sequence."""
    return w.seed + 97 * rank


def reduce_over_ranks(dist, device, times_ms, work):
    """Max over ranks of each timed region (the job is as slow as its slowest
    rank) and the sum over ranks of the work (the replicas' visible tiles differ
    with their documents)."""
    import torch

    t = torch.tensor([float(x) for x in times_ms], dtype=torch.float64, device=device)
    f = torch.tensor([float(work)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(f, op=dist.ReduceOp.SUM)
    return [float(x) for x in t.tolist()], float(f.item())


class Problem:
    """One workload resident on the device: inputs, outputs, the backward's
    workspace, the block-mask buffer and one mask spec per window of the sweep
    (one spec for a fixed mask).  Every spec of a sweep reads its W from its own
    element of one device int32 tensor, so the sweep changes W with no rebuild of
    anything but the block mask (speedrun notes, Record #13)."""

    def __init__(self, fa, w, dev, host, windows):
        import torch

        self.fa, self.w, self.dev = fa, w, dev
        q_h, k_h, v_h, do_h, docs_np = host
        self.q, self.k, self.v, self.do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
        self.docs = torch.as_tensor(docs_np, dtype=torch.int32, device=dev) if docs_np is not None else None
        self.windows = list(windows)
        self.W = torch.tensor([x or 0 for x in self.windows], dtype=torch.int32, device=dev)
        self.specs = [fa.make_mask_spec(mask_nodes(w, self.docs, self.W[i:i + 1]), device=dev)
                      for i in range(len(self.windows))]
        self.score = None
        if w.score[0] == "softcap":
            self.score = fa.make_score_spec("softcap", [float(w.score[1])], device=dev)
        elif w.score[0] == "alibi":
            from synth import make_alibi_slopes
            self.score = fa.make_score_spec("alibi", torch.as_tensor(make_alibi_slopes(w.H)), device=dev)
        self.bm_buf = torch.empty(fa.fa_block_mask_bytes(1, 1, w.S, w.S, 128), dtype=torch.uint8, device=dev)
        self.ws = torch.empty(fa.fa_backward_workspace_bytes(w.B, w.H, w.S, w.D), dtype=torch.uint8, device=dev)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty(w.B, w.H, w.S, dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = (torch.empty_like(t) for t in (self.q, self.k, self.v))

    def sub_step(self, i, stream, ev=None):
        """Block mask of window i, forward, backward; events 0..3 around them when given."""
        fa, w = self.fa, self.w
        if ev:
            ev[0].record(stream)
        bm = fa.fa_create_block_mask(self.specs[i], 1, 1, w.S, w.S, 128, buffer=self.bm_buf)
        if ev:
            ev[1].record(stream)
        # the forward clears the workspace's dq accumulator beside its own work
        # (hidden under its tensor-core time); the backward then skips that pass
        fa.fa_forward_prepare_backward(self.q, self.k, self.v, bm, self.ws, score=self.score, out=self.out,
                                       lse=self.lse)
        if ev:
            ev[2].record(stream)
        fa.fa_backward_prepared(self.q, self.k, self.v, self.out, self.lse, self.do, bm, self.ws, score=self.score,
                                dq=self.dq, dk=self.dk, dv=self.dv)
        if ev:
            ev[3].record(stream)
        return bm

    def visible_tiles(self, stream):
        """Visible tiles (all b, h) of every window's block mask."""
        import torch

        out = []
        for i in range(len(self.windows)):
            bm = self.fa.fa_create_block_mask(self.specs[i], 1, 1, self.w.S, self.w.S, 128, buffer=self.bm_buf)
            torch.cuda.synchronize()
            out.append(visible_tiles(self.fa, bm, self.w.B, self.w.H))
        return out


def launches_per_sub_step(w):
    # builder: tile_summary + doc_runs (documents only) + row_segs + classify + compact + order;
    # forward 1; backward pre + main + dq convert
    return (6 if w.docs is not None else 4) + 1 + 3


def timed_steps(prob, stream, steps):
    """Runs `steps` steps (each a pass over every window) between CUDA events on
    `stream`; returns total ms and per-window summed ms of build, forward, backward."""
    import torch

    ev = lambda: torch.cuda.Event(enable_timing=True)
    n = len(prob.windows)
    marks = []
    t0, t1 = ev(), ev()
    t0.record(stream)
    for _ in range(steps):
        for i in range(n):
            e = [ev() for _ in range(4)]
            prob.sub_step(i, stream, e)
            marks.append((i, e))
    t1.record(stream)
    torch.cuda.synchronize()
    per = [[0.0, 0.0, 0.0] for _ in range(n)]
    for i, e in marks:
        for j in range(3):
            per[i][j] += e[j].elapsed_time(e[j + 1])
    return t0.elapsed_time(t1), per


def tile_flops(n_vis, D):
    """Forward FLOPs of n_vis visible 128 x 128 tiles at head dim D (two tile GEMMs)."""
    return n_vis * 4.0 * 128 * 128 * D


def per_config(fa, w, dev, steps, warmup, peak):
    """Device-timed fwd / bwd throughput of one more workload (no e2e): the same
    step as the headline, for the per-config keys of the line."""
    import torch

    prob = Problem(fa, w, dev, workload_tensors(w), [None])
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        prob.sub_step(0, stream)
    n_vis = prob.visible_tiles(stream)[0]
    ms, per = timed_steps(prob, stream, steps)
    assert fa.fa_get_status(prob.sub_step(0, stream)) == 0
    ff = tile_flops(n_vis, w.D)
    b, f, d = (x / steps for x in per[0])
    res = {"workload": w.name, "visible_tiles": int(n_vis), "ms_per_step": round(ms / steps, 4),
           "tflops": round(3.5 * ff / (ms / steps * 1e-3) / 1e12, 2),
           "build_ms": round(b, 4), "fwd_ms": round(f, 4), "bwd_ms": round(d, 4),
           "fwd_tflops": round(ff / (f * 1e-3) / 1e12, 2), "bwd_tflops": round(2.5 * ff / (d * 1e-3) / 1e12, 2)}
    res["fwd_frac"] = round(res["fwd_tflops"] / peak, 4)
    res["bwd_frac"] = round(res["bwd_tflops"] / peak, 4)
    del prob
    torch.cuda.empty_cache()
    return res


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import block_sparse_masked_fa_gb300 as fa

    world, rank, local = rank_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")

    w = WORKLOADS[args.workload]
    if args.heads:
        if not args.profile:
            raise SystemExit("--heads is for --profile runs only (the headline keeps the workload's heads)")
        w = dataclasses.replace(w, H=args.heads)
    dev = torch.device("cuda", local)
    windows = [args.window] if (w.windows and args.window) else (list(w.windows) or [None])
    host = workload_tensors(w, seed=replica_seed(w, rank))
    prob = Problem(fa, w, dev, host, windows)
    stream = torch.cuda.current_stream()
    n_sub = len(windows)

    for _ in range(args.warmup):
        for i in range(n_sub):
            prob.sub_step(i, stream)
    torch.cuda.synchronize()
    n_vis = prob.visible_tiles(stream)
    fwd_w = [tile_flops(n, w.D) for n in n_vis]
    fwd_flops = sum(fwd_w)
    bwd_flops = 2.5 * fwd_flops
    step_flops = fwd_flops + bwd_flops

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ms_total, per = timed_steps(prob, stream, args.steps)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    build_ms = sum(p[0] for p in per) / args.steps
    fwd_ms = sum(p[1] for p in per) / args.steps
    bwd_ms = sum(p[2] for p in per) / args.steps
    assert fa.fa_get_status(prob.sub_step(n_sub - 1, stream)) == 0, "device status reported an error"

    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    e2e = None
    if not args.profile:
        ref_out = prob.out.cpu()  # the last window's output, for the e2e run's check
        e2e = run_e2e(fa, w, dev, host, windows, prob, stream, max(4, args.steps // 2), ref_out)
    job_flops = step_flops  # the work of all ranks
    e2e_ms = e2e["ms"] if e2e else 0.0
    if world > 1:
        (ms_total, e2e_ms), job_flops = reduce_over_ranks(dist, dev, (ms_total, e2e_ms), step_flops)
    ms_step = ms_total / args.steps

    dominant = "bwd" if bwd_ms > fwd_ms else "fwd"
    dom_ms = bwd_ms if dominant == "bwd" else fwd_ms
    dom_flops = bwd_flops if dominant == "bwd" else fwd_flops
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    value = job_flops / (ms_step * 1e-3) / 1e12
    sweep = len(windows) > 1
    name = w.name + (f" (W {windows[0]}..{windows[-1]} step {windows[1] - windows[0]}, one sweep of "
                     f"{len(windows)} windows per step)" if sweep else (f" (W {windows[0]})" if windows[0] else ""))
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v/dO in bf16, log-normal document lengths)",
        "config": {"workload": name, "B": w.B, "H": w.H, "S": w.S, "D": w.D,
                   "mask": " ".join(n[0] if len(n) == 1 else f"{n[0]}:{n[1]}" for n in w.mask.nodes)
                   + (" (W from a device int32, swept)" if sweep else ""),
                   "score_mod": w.score[0], "block": 128, "visible_tiles": int(sum(n_vis)),
                   "l2": "inputs larger than L2 (q, k, v, dO: 4 x %d MiB)" % (prob.q.numel() * 2 >> 20),
                   "parallelism": f"replicas x{world}"},
        "breakdown_ms": {"create_block_mask": round(build_ms, 4), "forward": round(fwd_ms, 4),
                         "backward": round(bwd_ms, 4)},
        "fwd_tflops": round(fwd_flops / (fwd_ms * 1e-3) / 1e12, 2),
        "bwd_tflops": round(bwd_flops / (bwd_ms * 1e-3) / 1e12, 2),
        "roofline": {"kernel": dominant, "bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "peak_source": f"bf16_tflops ({peak_src}, burst)", "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic("bwd_kernel" if dominant == "bwd" else "fwd_kernel", w.name),
                     "traffic_note": "DRAM bytes of one launch at W 1024 (ncu on 4 heads, scaled to 16); "
                                     "null when the kernel's sources changed since the capture"},
        "gpu_launches": launches_per_sub_step(w) * n_sub * args.steps,
        "clocks": clk,
    }
    if sweep:
        pick = [i for i, x in enumerate(windows) if x in (64, 1024, 1792)]
        res["per_window"] = {str(windows[i]): {
            "visible_tiles": int(n_vis[i]),
            "fwd_tflops": round(fwd_w[i] / (per[i][1] / args.steps * 1e-3) / 1e12, 2),
            "bwd_tflops": round(2.5 * fwd_w[i] / (per[i][2] / args.steps * 1e-3) / 1e12, 2),
            "build_ms": round(per[i][0] / args.steps, 4)} for i in pick}
    if e2e:
        res["e2e"] = {"value": round(job_flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                      "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": e2e["h2d"],
                      "d2h_bytes_per_step": e2e["d2h"],
                      "overlap": "two device buffer sets; copies of a window's step overlap its neighbours' compute"}
    del prob
    torch.cuda.empty_cache()
    if rank == 0 and not args.profile:
        res["builder_scaled"] = builder_scaled(fa, w, prob_window(w, windows), dev)
        res["decode"] = decode_point(fa, dev, float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"])))
        res["small_block"] = small_block_point(fa, dev, peak)
        res["per_config"] = {str(n): per_config(fa, WORKLOADS[n], dev, max(3, args.steps // 2), 3, peak)
                             for n in sorted(WORKLOADS) if n != args.workload}
    if rank == 0 and not args.no_cpu_baseline and not args.profile:
        res["cpu_baseline"] = cpu_baseline(w, args.cpu_sample_tokens)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


def prob_window(w, windows):
    """A device W for builder_scaled: the largest window of the run (or the fixed one)."""
    import torch

    return torch.tensor([max(x or 0 for x in windows) or 1024], dtype=torch.int32, device="cuda")


def run_e2e(fa, w, dev, host, windows, prob, stream, steps, ref_out):
    """End to end through the public API: every window's step copies its inputs in
    from pinned host memory and its results back.  Two device buffer sets and
    three streams let the copies of one window's step overlap the compute of its
    neighbours (the inputs of the next load while one computes, the results of
    one return while the next computes), as a training loop that prefetches its
    batches does; each window's step still moves all of its own bytes."""
    import torch

    q_h, k_h, v_h, do_h, docs_np = host
    pin = lambda t: t.pin_memory()
    hq, hk, hv, hdo = (pin(t) for t in (q_h, k_h, v_h, do_h))
    hdocs = pin(torch.as_tensor(docs_np, dtype=torch.int32)) if docs_np is not None else None
    h_out, h_lse = pin(torch.empty_like(q_h)), pin(torch.empty(w.B, w.H, w.S, dtype=torch.float32))
    h_dq, h_dk, h_dv = (pin(torch.empty_like(t)) for t in (q_h, k_h, v_h))
    n = len(windows)
    h2d = n * (sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo)) +
               (hdocs.numel() * 4 if hdocs is not None else 0))
    d2h = n * (h_out.numel() * 2 + h_lse.numel() * 4 + 3 * h_dq.numel() * 2)
    sets = [prob, Problem(fa, w, dev, host, windows)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def e2e_sub(j):
        b = j % 2
        st = sets[b]
        with torch.cuda.stream(s_in):  # this set's inputs, once step j - 2 has finished with them
            s_in.wait_event(ev_comp[b])
            for dst, src in ((st.q, hq), (st.k, hk), (st.v, hv), (st.do, hdo)):
                dst.copy_(src, non_blocking=True)
            if hdocs is not None:
                st.docs.copy_(hdocs, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])  # step j - 2's results have left this set
        st.sub_step(j % n, stream)
        ev_comp[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            for dst, src in ((h_out, st.out), (h_lse, st.lse), (h_dq, st.dq), (h_dk, st.dk), (h_dv, st.dv)):
                dst.copy_(src, non_blocking=True)
            ev_out[b].record(s_out)

    for j in range(2):
        e2e_sub(j)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for j in range(steps * n):
        e2e_sub(j)
    e1.record(s_out)
    torch.cuda.synchronize()
    # the device-timed run ended on the same window with the same inputs
    assert torch.equal(h_out, ref_out), "e2e results differ from the device-timed run"
    del sets[1]
    return {"ms": e0.elapsed_time(e1) / steps, "h2d": int(h2d), "d2h": int(d2h)}


def _sample_visible_tiles(mask, docs_row, S):
    import oracle

    cls = oracle.classify_tiles(oracle.Program(mask, doc_row=docs_row), S, S, 128)
    return int((cls > 0).sum())


def cpu_baseline(w, tokens, heads=1):
    """The oracle, as it stands, on the first `tokens` positions of `heads` heads.

    The workload's masks are causal, so a prefix of the sequence is a
    self-contained problem of the same kind; its visible tiles give the FLOP
    count in the metric's convention."""
    import torch

    import oracle

    S = min(tokens, w.S)
    q, k, v, do = make_qkv(1, heads, S, w.D, w.seed)
    docs = make_doc_ids(w.docs, w.S, w.doc_seed or w.seed)[0][:S] if w.docs is not None else None
    mask = w.mask.with_window(1024) if w.windows else w.mask
    prog = oracle.Program(mask, doc_row=docs)
    score = ("none",)
    if w.score[0] == "softcap":
        score = ("softcap", float(w.score[1]))
    elif w.score[0] == "alibi":
        from synth import make_alibi_slopes
        score = ("alibi", make_alibi_slopes(w.H))
    scale = 1.0 / np.sqrt(w.D)
    t = time.perf_counter()
    for h in range(heads):
        f = lambda x: x[0, h].to(torch.float64).numpy()
        oracle.forward_head(f(q), f(k), f(v), prog, score, h, scale)
        oracle.backward_head(f(q), f(k), f(v), f(do), prog, score, h, scale)
    dt = time.perf_counter() - t
    n_vis = _sample_visible_tiles(mask, docs, S) * heads
    flops = 3.5 * n_vis * 4.0 * 128 * 128 * w.D
    cores = int(os.environ.get("OMP_NUM_THREADS", len(os.sched_getaffinity(0))))
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "seconds": round(dt, 2),
            "sample": f"fwd+bwd of {heads} head(s) on the first {S} tokens of {w.name} "
                      f"({n_vis} visible tiles, same mask and score mod"
                      + (", W 1024 of the sweep)" if w.windows else ")")}


def run_reference(args):
    """--impl reference: the CPU oracle as it stands, on a bounded sample per step."""
    _, rank, _ = rank_env()
    if rank != 0:  # under torchrun only rank 0 runs and prints
        return
    w = WORKLOADS[args.workload]
    vals = []
    for _ in range(args.warmup):
        cpu_baseline(w, args.ref_sample_tokens)
    t = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(w, args.ref_sample_tokens))
    total = time.perf_counter() - t
    v = statistics.median(x["value"] for x in vals)
    res = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1000 * total / max(1, args.steps), 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D},
           "cpu_baseline": {"value": v, "unit": "TFLOP/s", "kind": "oracle", "cores": vals[0]["cores"],
                            "sample": vals[0]["sample"]},
           "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", type=int, default=5, choices=sorted(WORKLOADS))
    ap.add_argument("--window", type=int, default=None,
                    help="one fixed window for the sweep workload (5) instead of the whole sweep")
    ap.add_argument("--heads", type=int, default=0,
                    help="with --profile: fewer heads than the workload's, for a smaller profiler capture")
    ap.add_argument("--profile", action="store_true",
                    help="the timed steps only (no e2e buffer set, scaled builder, decode point, other "
                         "configs or CPU baseline): a small device footprint for profiler captures")
    ap.add_argument("--cpu-sample-tokens", type=int, default=32768,
                    help="tokens of the oracle sample timed as cpu_baseline")
    ap.add_argument("--ref-sample-tokens", type=int, default=16384,
                    help="tokens of the oracle sample per step of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
