"""Throughput of the tile-sparse masked attention hot path on one GB300.

A step is one pass of the whole path over one batch of synthetic input:
fa_create_block_mask + fa_forward + fa_backward, on the packed 64K-token
workload (B=1, H=6, S=65536, D=128, causal & same document & 1024 window,
log-normal document lengths).  The metric is attention TFLOP/s counted over
visible tiles only: forward 4*128*128*D per visible tile per (b, h), backward
2.5x that (five tile GEMMs against two).

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload instead.
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
    entry = rec.get("kernels", {}).get(kernel)
    if not entry or entry.get("workload") != workload or entry.get("source_sha256") != source_digest(kernel):
        return None
    return entry.get("dram_bytes_per_launch")


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


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import block_sparse_masked_fa_gb300 as fa

    world, rank, local = rank_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")

    w = WORKLOADS[args.workload]
    q_h, k_h, v_h, do_h, docs_np = workload_tensors(w, seed=replica_seed(w, rank))
    dev = torch.device("cuda", local)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    docs = torch.as_tensor(docs_np, dtype=torch.int32, device=dev) if docs_np is not None else None
    W = torch.tensor([args.window if w.windows else 1024], dtype=torch.int32, device=dev)
    nodes = mask_nodes(w, docs, W)
    spec, keep = fa.make_mask_spec(nodes, device=dev)
    score = None
    if w.score[0] == "softcap":
        score = fa.make_score_spec("softcap", [float(w.score[1])], device=dev)
    elif w.score[0] == "alibi":
        from synth import make_alibi_slopes
        score = fa.make_score_spec("alibi", torch.as_tensor(make_alibi_slopes(w.H)), device=dev)
    stream = torch.cuda.current_stream()
    bm_buf = torch.empty(fa.fa_block_mask_bytes(1, 1, w.S, w.S, 128), dtype=torch.uint8, device=dev)
    ws = torch.empty(fa.fa_backward_workspace_bytes(w.B, w.H, w.S, w.D), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.S, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    have_bwd = True
    bm0 = fa.fa_create_block_mask((spec, keep), 1, 1, w.S, w.S, 128, buffer=bm_buf)
    fa.fa_forward(q, k, v, bm0, score=score, out=out, lse=lse)
    try:
        fa.fa_backward(q, k, v, out, lse, do, bm0, score=score, dq=dq, dk=dk, dv=dv, workspace=ws)
    except fa.FaError:
        have_bwd = False
    torch.cuda.synchronize()

    ev = lambda: torch.cuda.Event(enable_timing=True)
    marks = []

    def step(record):
        e = [ev() for _ in range(4)] if record else None
        if record:
            e[0].record(stream)
        bm = fa.fa_create_block_mask((spec, keep), 1, 1, w.S, w.S, 128, buffer=bm_buf)
        if record:
            e[1].record(stream)
        fa.fa_forward(q, k, v, bm, score=score, out=out, lse=lse)
        if record:
            e[2].record(stream)
        if have_bwd:
            fa.fa_backward(q, k, v, out, lse, do, bm, score=score, dq=dq, dk=dk, dv=dv, workspace=ws)
        if record:
            e[3].record(stream)
            marks.append(e)
        return bm

    for _ in range(args.warmup):
        bm = step(False)
    torch.cuda.synchronize()
    n_vis = visible_tiles(fa, bm, w.B, w.H)
    fwd_flops = n_vis * 4.0 * 128 * 128 * w.D
    bwd_flops = 2.5 * fwd_flops
    step_flops = fwd_flops + (bwd_flops if have_bwd else 0.0)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = ev(), ev()
    t0.record(stream)
    for _ in range(args.steps):
        step(True)
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms_total = t0.elapsed_time(t1)
    build_ms = sum(m[0].elapsed_time(m[1]) for m in marks) / args.steps
    fwd_ms = sum(m[1].elapsed_time(m[2]) for m in marks) / args.steps
    bwd_ms = sum(m[2].elapsed_time(m[3]) for m in marks) / args.steps
    assert fa.fa_get_status(bm) == 0, "device status reported an error"

    # end to end through the public API: every step copies its inputs in from
    # pinned host memory and its results back.  Two device buffer sets and three
    # streams let the copies of one step overlap the compute of its neighbours
    # (the inputs of step i + 1 load while step i computes, the results of step
    # i return while step i + 1 computes), as a training loop that prefetches
    # its batches does; each step still moves all of its own bytes.
    pin = lambda t: t.pin_memory()
    hq, hk, hv, hdo = (pin(t) for t in (q_h, k_h, v_h, do_h))
    hdocs = pin(torch.as_tensor(docs_np, dtype=torch.int32)) if docs_np is not None else None
    h_out, h_lse = pin(torch.empty_like(q_h)), pin(torch.empty(w.B, w.H, w.S, dtype=torch.float32))
    h_dq, h_dk, h_dv = (pin(torch.empty_like(t)) for t in (q_h, k_h, v_h))
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo)) + \
        (hdocs.numel() * 4 if hdocs is not None else 0)
    d2h = h_out.numel() * 2 + h_lse.numel() * 4 + (3 * h_dq.numel() * 2 if have_bwd else 0)

    sets = [dict(q=q, k=k, v=v, do=do, docs=docs, spec=(spec, keep), out=out, lse=lse, dq=dq, dk=dk, dv=dv)]
    q2, k2, v2, do2 = (torch.empty_like(t) for t in (q, k, v, do))
    docs2 = torch.empty_like(docs) if docs is not None else None
    nodes2 = [("same_doc", docs2) if nd[0] == "same_doc" else nd for nd in nodes]
    sets.append(dict(q=q2, k=k2, v=v2, do=do2, docs=docs2, spec=fa.make_mask_spec(nodes2, device=dev),
                     out=torch.empty_like(out), lse=torch.empty_like(lse), dq=torch.empty_like(dq),
                     dk=torch.empty_like(dk), dv=torch.empty_like(dv)))
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def e2e_step(i):
        b = i % 2
        st = sets[b]
        with torch.cuda.stream(s_in):  # this set's inputs, once step i - 2 has finished with them
            s_in.wait_event(ev_comp[b])
            st["q"].copy_(hq, non_blocking=True)
            st["k"].copy_(hk, non_blocking=True)
            st["v"].copy_(hv, non_blocking=True)
            st["do"].copy_(hdo, non_blocking=True)
            if hdocs is not None:
                st["docs"].copy_(hdocs, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])  # step i - 2's results have left this set
        bm = fa.fa_create_block_mask(st["spec"], 1, 1, w.S, w.S, 128, buffer=bm_buf)
        fa.fa_forward(st["q"], st["k"], st["v"], bm, score=score, out=st["out"], lse=st["lse"])
        if have_bwd:
            fa.fa_backward(st["q"], st["k"], st["v"], st["out"], st["lse"], st["do"], bm, score=score,
                           dq=st["dq"], dk=st["dk"], dv=st["dv"], workspace=ws)
        ev_comp[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            h_out.copy_(st["out"], non_blocking=True)
            h_lse.copy_(st["lse"], non_blocking=True)
            if have_bwd:
                h_dq.copy_(st["dq"], non_blocking=True)
                h_dk.copy_(st["dk"], non_blocking=True)
                h_dv.copy_(st["dv"], non_blocking=True)
            ev_out[b].record(s_out)
        return bm

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    e2e_steps = max(4, args.steps // 2)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    job_flops = step_flops  # the work of all ranks
    if world > 1:
        (ms_total, e2e_ms), job_flops = reduce_over_ranks(dist, dev, (ms_total, e2e_ms), step_flops)
    ms_step = ms_total / args.steps
    assert torch.equal(h_out, out.cpu()), "e2e results differ from the device-timed run"

    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    dominant = "bwd" if (have_bwd and bwd_ms > fwd_ms) else "fwd"
    dom_ms = bwd_ms if dominant == "bwd" else fwd_ms
    dom_flops = bwd_flops if dominant == "bwd" else fwd_flops
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    value = job_flops / (ms_step * 1e-3) / 1e12
    # builder: (tile_summary + doc_runs) + row_segs + classify + compact + order; forward 1;
    # backward pre + main + dq convert
    launches_per_step = (6 if docs is not None else 4) + 1 + (3 if have_bwd else 0)
    res = {
        "metric": METRIC if have_bwd else "attention TFLOP/s over visible tiles (fwd only; bwd not built)",
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
        "config": {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D,
                   "mask": " ".join(n[0] if len(n) == 1 else f"{n[0]}:{n[1]}" for n in w.mask.nodes),
                   "score_mod": w.score[0], "block": 128, "visible_tiles": int(n_vis),
                   "l2": "inputs larger than L2 (q, k, v, dO: 4 x %d MiB)" % (q.numel() * 2 >> 20),
                   "parallelism": f"replicas x{world}"},
        "breakdown_ms": {"create_block_mask": round(build_ms, 4), "forward": round(fwd_ms, 4),
                         "backward": round(bwd_ms, 4) if have_bwd else None},
        "fwd_tflops": round(fwd_flops / (fwd_ms * 1e-3) / 1e12, 2),
        "bwd_tflops": round(bwd_flops / (bwd_ms * 1e-3) / 1e12, 2) if have_bwd else None,
        "roofline": {"kernel": dominant, "bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "peak_source": f"bf16_tflops ({peak_src}, burst)", "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic("bwd_kernel" if dominant == "bwd" else "fwd_kernel", w.name)},
        "e2e": {"value": round(job_flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "overlap": "two device buffer sets; copies of a step overlap neighbouring steps' compute"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if rank == 0:
        res["builder_scaled"] = builder_scaled(fa, w, W, dev)
        res["decode"] = decode_point(fa, dev, float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"])))
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, args.cpu_sample_tokens)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


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
                      f"({n_vis} visible tiles, same mask and score mod)"}


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
    ap.add_argument("--workload", type=int, default=2, choices=sorted(WORKLOADS))
    ap.add_argument("--window", type=int, default=1024, help="window of the sweep workload (5)")
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
