#!/usr/bin/env python
"""Decode-step benchmark of the MXFP4 lightning-indexer path on one GB300.

One step is the whole decode hot path over one batch of 64 sequences with
contexts uniform in [8K, 32K] (H = 32 index heads, head_dim 128, page 64,
next_n = 1, top-k 2048; 1% outlier channels x8 in K and q):
  1. quantise and insert the step's new key of every sequence (idx_quant_insert),
  2. quantise the step's query heads (idx_quant_q),
  3. paged MQA logits + top-k 2048 of every row, fused (idx_paged_logits_topk).
The cache holds the rest of every context before timing starts.

The metric is key-tokens scored per second (sum over query rows of the keys
in the row's window, per second of step time) with the algorithmic HBM GB/s
beside it.  L2 is flushed (a 256 MiB buffer written, then read) before every timed step and each
step is timed alone with CUDA events on the launching stream.

--impl reference times the CPU oracle (the plain fp64 statement of the same
path) on a bounded sample of the same workload, on the host cores.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode K-tokens scored/s + HBM GB/s (paged MXFP4 MQA logits + top-k)"
UNIT = "key-tokens/s"
TOPK = 2048
L2_FLUSH_BYTES = 256 << 20   # 2x the 129 MB L2
SMS_GB300 = 152
# sources of the fused decode entry (scoring + select launches); the committed
# traffic figure is only used while their digest matches
FUSED_SOURCES = ["paged_topk.cu", "paged_logits.cu", "paged_core.cuh", "select_row.cuh",
                 "topk_select.cuh", "common.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-sample-seqs", type=int, default=1 << 30,
                    help="sequences of the batch the CPU oracle baseline covers (default: all)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="the CPU oracle baseline repeats decode steps for at least this long")
    ap.add_argument("--no-also", action="store_true",
                    help="skip the secondary insert / prefill measurements")
    ap.add_argument("--ref-budget-s", type=float, default=90.0,
                    help="reference arm: seconds of oracle work for warmup + steps")
    ap.add_argument("--workload", default="batched_decode",
                    choices=sorted(WORKLOADS),
                    help="decode workload; the default is the headline configuration")
    ap.add_argument("--case", nargs="+", metavar=("NAME", "T"),
                    help="run one step of the path alone a few times for a profiler and "
                         "print its median time: 'prefill T' (mqa_logits then topk_rows on "
                         "a T-token causal prefill, H=32, then the logits + top-k entry), "
                         "'decode' (the fused paged logits + top-k of the headline batch), "
                         "'quant T' (q-quant and insert of a T-token prefill), 'next' "
                         "(q-RoPE + q-quant and K-pool insert of the 32768-token prefill), "
                         "'step' (the two- and four-launch decode steps)")
    ap.add_argument("--reps", type=int, default=5, help="repetitions of a --case step")
    return ap.parse_args()


# decode workloads (the pages' shapes): name -> (builder name, description)
WORKLOADS = {
    "batched_decode": ("batched_decode", "64 sequences, contexts uniform [8192, 32768], H=32, next_n=1"),
    "pr_ref": ("pr_ref", "1 sequence of 8192 tokens, H=32, next_n=1"),
    "long_decode": ("long_decode", "16 sequences x 131072 tokens, H=64, next_n=2"),
    "mixed_decode": ("mixed_decode_part", "128 sequences, contexts uniform [1024, 131072], H=32, next_n=1"),
}


def make_workload(name, rank=0, **sizes):
    """Rank r's shard of a decode workload: the workload's recipe with its
    seed moved by 1000 * r, so every rank owns different sequences and no
    data crosses ranks (the decode path has no exchange step).  `sizes`
    overrides the recipe's sizes (tests use small shards)."""
    from sparse_attention_indexer_quant_gb300 import workloads as wl
    builder = getattr(wl, WORKLOADS[name][0])
    import inspect
    seed = inspect.signature(builder).parameters["seed"].default
    return builder(seed=seed + 1000 * rank, **sizes)


def dist_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def workload_config(p, name="batched_decode"):
    return {"workload": name, "description": WORKLOADS[name][1], "sequences": p.B,
            "H": p.H, "head_dim": 128,
            "page_size": 64, "next_n": p.next_n, "topk": p.topk,
            "scored_key_tokens_per_step": int(scored_tokens(p)),
            "l2": "flushed before every timed step: a 256 MiB buffer (2x L2) written, then "
                  "read back, so no input is resident and no dirty line is left"}


def scored_tokens(p) -> int:
    st, en = p.row_windows()
    return int((en.astype(np.int64) - st).sum())


def fused_algorithmic_bytes(p) -> int:
    """Bytes the fused kernel must move: every cached key of every sequence
    (64 value + 4 scale bytes), the block-table entries for those pages, the
    context lengths, the query pairs and weights, and the top-k output."""
    L = p.context_lens.astype(np.int64)
    return int((68 * L + 4 * ((L + 63) // 64) + 4).sum() + p.rows * p.H * (68 + 4)
               + p.rows * p.topk * 4)


def step_algorithmic_bytes(p) -> int:
    n_new = len(p.new_token_rows())
    insert = n_new * (256 + 8 + 68)
    qquant = p.rows * p.H * (256 + 68)
    return fused_algorithmic_bytes(p) + insert + qquant


def source_digest():
    h = hashlib.sha256()
    for f in FUSED_SOURCES:
        with open(os.path.join(ROOT, "sparse_attention_indexer_quant_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic():
    """DRAM bytes per launch of the fused kernel from the committed ncu summary,
    if it was taken on the current source."""
    path = os.path.join(ROOT, "profiles", "fused_decode_traffic.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
    except (OSError, ValueError):
        return None
    if d.get("source_sha256") != source_digest():
        return None
    return d.get("dram_bytes_per_launch")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def bf16_tensor(a, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def run_ours(args, rank, world, local_rank):
    import torch
    from sparse_attention_indexer_quant_gb300 import binding as idx
    from sparse_attention_indexer_quant_gb300 import workloads as wl

    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    idx.check_device(local_rank)
    p = make_workload(args.workload, rank)
    new_rows = p.new_token_rows()
    old_mask = np.ones(p.total_tokens, bool)
    old_mask[new_rows] = False

    # resident state: the cache with every context except the newest token
    cache = torch.from_numpy(wl.poisoned_cache(p.num_blocks)).to(dev)
    k_old = bf16_tensor(p.k[old_mask], dev)
    idx.quant_insert(k_old, torch.from_numpy(p.slots[old_mask]).to(dev), cache)
    del k_old
    new_k = bf16_tensor(p.k[new_rows], dev)
    new_slots = torch.from_numpy(p.slots[new_rows]).to(dev)
    q = bf16_tensor(p.q, dev)
    w = torch.from_numpy(p.weights).to(dev)
    bt = torch.from_numpy(p.block_table).to(dev)
    cl = torch.from_numpy(p.context_lens).to(dev)
    max_blocks = p.block_table.shape[1]
    ws = idx.new_paged_topk_workspace(p.B, p.next_n, max_blocks, TOPK, dev)
    qv = torch.empty((p.rows * p.H, 64), dtype=torch.uint8, device=dev)
    qs = torch.empty((p.rows * p.H, 4), dtype=torch.uint8, device=dev)
    out = torch.empty((p.rows, TOPK), dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2():
        # write a buffer twice the size of L2, then read it back: afterwards no
        # input of the step is resident and no dirty line is left for the
        # timed kernels to write back
        flush.fill_(1)
        torch.sum(flush, 0, dtype=torch.int64, out=flush_sink)

    stream = torch.cuda.current_stream()

    def step():
        idx.quant_insert(new_k, new_slots, cache)
        idx.quant_q(q, out_vals=qv, out_scales=qs)

    def fused():
        idx.paged_logits_topk(qv, qs, w, cache, bt, cl, p.next_n, p.H, TOPK, workspace=ws,
                              out=out)

    for _ in range(args.warmup):
        flush_l2()
        step()
        fused()
    torch.cuda.synchronize()

    # A decode loop replays its step as a CUDA graph: the step (insert, q-quant,
    # fused logits + top-k, captured through the C ABI calls above) is timed as
    # one graph replay, with no event between its kernels (an event between two
    # dependent launches keeps the second from starting during the first one's
    # tail, and host launch gaps would land inside the step); the fused call is
    # timed alone the same way for its roofline, and the step once more as
    # eager calls for reference.
    g_step = graph_of(lambda: (step(), fused()))
    g_fused = graph_of(fused)
    K = args.steps
    K_eager = min(K, 200)

    def timed(n, body):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for i in range(n):
            flush_l2()
            evs[i][0].record(stream)
            body()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return [e[0].elapsed_time(e[1]) for e in evs]

    for _ in range(args.warmup):
        flush_l2()
        g_step.replay()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        step_ms = timed(K, g_step.replay)
        fused_ms = timed(K, g_fused.replay)
        eager_ms = timed(K_eager, lambda: (step(), fused()))
    barrier(world)
    total_ms = sum(step_ms)
    total_ms_max = reduce_max(total_ms, world, dev)

    # ---- end to end through the public API with host buffers: the step's
    # inputs live in one pinned staging buffer (16-byte aligned sections), so
    # one host->device copy carries them all; the indices come back in one copy
    host_parts = [bf16_tensor(p.k[new_rows], "cpu"), torch.from_numpy(p.slots[new_rows]),
                  bf16_tensor(p.q, "cpu"), torch.from_numpy(p.weights),
                  torch.from_numpy(p.block_table), torch.from_numpy(p.context_lens)]
    offs, total = [], 0
    for t in host_parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 15) // 16 * 16
    h_stage = torch.empty(total, dtype=torch.uint8).pin_memory()
    d_stage = torch.empty(total, dtype=torch.uint8, device=dev)

    def section(buf, i):
        t = host_parts[i]
        n = t.numel() * t.element_size()
        return buf[offs[i]:offs[i] + n].view(t.dtype).view(t.shape)

    for i, t in enumerate(host_parts):
        section(h_stage, i).copy_(t)
    d_new_k, d_new_slots, d_q, d_w, d_bt, d_cl = (section(d_stage, i) for i in range(6))
    h_out = torch.empty((p.rows, TOPK), dtype=torch.int32).pin_memory()
    h2d = total
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step(engine=False):
        # the copies run on the SMs through the library's idx_copy_async
        # (engine=True: the same copies by the copy engine, for comparison)
        if engine:
            d_stage.copy_(h_stage, non_blocking=True)
        else:
            idx.copy_async(d_stage, h_stage)
        idx.quant_insert(d_new_k, d_new_slots, cache)
        idx.quant_q(d_q, out_vals=qv, out_scales=qs)
        idx.paged_logits_topk(qv, qs, d_w, cache, d_bt, d_cl, p.next_n, p.H, TOPK,
                              workspace=ws, out=out)
        if engine:
            h_out.copy_(out, non_blocking=True)
        else:
            idx.copy_async(h_out, out)

    def e2e_time(engine):
        for _ in range(3):
            e2e_step(engine)
        torch.cuda.synchronize()
        ts = []
        for _ in range(args.e2e_steps):
            flush_l2()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            e2e_step(engine)
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        # correctness spot check of the last e2e result against the device result
        assert torch.equal(h_out, out.cpu())
        return reduce_max(sum(ts) / len(ts), world, dev)

    e2e_engine_mean = e2e_time(True)
    e2e_mean = e2e_time(False)

    also = None
    if rank == 0 and not args.no_also:
        also = secondary_measurements(idx, dev, flush_l2, stream,
                                      decode=(p, cache, qv, qs, w, bt, cl),
                                      decode_desc=WORKLOADS[args.workload][1])
        also.update(insert_entries(idx, dev, flush_l2, stream))
        also.update(next_entries(idx, dev, flush_l2, stream))
        also.update(step_entries(idx, dev, flush_l2, stream))
        also.update(mixed_prefill_entry(idx, dev, flush_l2, stream))
        for other in ("long_decode", "mixed_decode", "pr_ref"):
            if other != args.workload:
                also[other] = decode_workload_entry(other, idx, dev, flush_l2, stream)

    cpu = None
    if rank == 0:
        cpu = cpu_baseline(p, args.cpu_sample_seqs, args.cpu_seconds)

    if rank != 0:
        return
    tokens = scored_tokens(p) * world
    ms_per_step = total_ms_max / K
    value = tokens / (ms_per_step * 1e-3)
    hbm_gbs = step_algorithmic_bytes(p) * world / (ms_per_step * 1e-3) / 1e9
    fused_mean = sum(fused_ms) / K
    achieved = fused_algorithmic_bytes(p) / (fused_mean * 1e-3) / 1e9
    peak, peak_src = peaks()
    traffic = measured_traffic()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "mxfp4 (e2m1 x e2m1, fp32 accumulate)",
        "data": "synthetic (seeded bf16 N(0,1) keys/queries, shuffled block tables)",
        "config": workload_config(p, args.workload),
        "hbm_gbs": hbm_gbs,
        "fused_kernel_ms": fused_mean,
        "step_ms_eager_calls": sum(eager_ms) / len(eager_ms),
        "step_timing": ("each step one replay of a CUDA graph captured from the C-ABI calls "
                        "(insert, q-quant, fused logits + top-k); L2 flushed before each"),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": (f"idx_paged_logits_topk (paged_logits_kernel<{p.H},{p.next_n}> "
                                "scoring + paged_select_kernel, timed together)"),
                     "peak_source": f"{peak_src} (hbm_gbs, burst)",
                     "algorithmic_bytes_per_launch": fused_algorithmic_bytes(p)},
        "cpu_baseline": cpu,
        "e2e": {"value": scored_tokens(p) * world / (e2e_mean * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_mean,
                "copies": ("one pinned staging buffer in and the indices out per step, each "
                           "by idx_copy_async (the SMs over NVLink-C2C)"),
                "ms_per_step_copy_engine": e2e_engine_mean},
        # per timed step: quant_insert, quant_q, the scoring and the select kernels
        "gpu_launches": 4 * K,
        "clocks": clocks.summary(),
        "also": also,
    }
    print(json.dumps(line), flush=True)


def mxf4_peak_tflops():
    """Dense MXF4 tensor peak: the measured bf16 GEMM burst rate times the
    nominal fp4 : bf16 ratio (13.5 / 2.25 PFLOP/s)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return float(json.load(fh)["bf16_tflops"]) * 6.0, "measured bf16 x 6"
    except (OSError, ValueError, KeyError):
        return 1900.0 * 6.0, "fallback bf16 x 6"


def time_op(fn, flush_l2, stream, reps):
    import torch
    ts = []
    for _ in range(reps):
        flush_l2()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    ts.sort()
    return ts[len(ts) // 2]


def fill_cache(idx, p, dev, rows=None, chunk=1 << 21):
    """A poisoned cache with the given rows of a problem's keys inserted
    (all of them by default), uploaded in bounded chunks."""
    import torch
    from sparse_attention_indexer_quant_gb300 import workloads as wl
    cache = torch.from_numpy(wl.poisoned_cache(p.num_blocks)).to(dev)
    rows = np.arange(p.total_tokens) if rows is None else np.asarray(rows)
    for lo in range(0, len(rows), chunk):
        r = rows[lo:lo + chunk]
        idx.quant_insert(bf16_tensor(p.k[r], dev), torch.from_numpy(p.slots[r]).to(dev), cache)
    return cache


def graph_of(fn):
    """A CUDA graph of fn's launches (captured after one warm call on a side
    stream)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def decode_workload_entry(name, idx, dev, flush_l2, stream, reps=50, cpu_seconds=5.0):
    """The fused decode call (paged logits + top-k) on another decode workload:
    its CUDA-graph replay time with L2 flushed before each (median of reps),
    its roofline fraction on the same algorithmic bytes as the headline, and
    the oracle on a bounded sample of the same workload."""
    import torch
    import oracle
    p = make_workload(name)
    cache = fill_cache(idx, p, dev)
    qv, qs = idx.quant_q(bf16_tensor(p.q, dev))
    w = torch.from_numpy(p.weights).to(dev)
    bt = torch.from_numpy(p.block_table).to(dev)
    cl = torch.from_numpy(p.context_lens).to(dev)
    ws = idx.new_paged_topk_workspace(p.B, p.next_n, p.block_table.shape[1], TOPK, dev)
    out = torch.empty((p.rows, TOPK), dtype=torch.int32, device=dev)
    g = graph_of(lambda: idx.paged_logits_topk(qv, qs, w, cache, bt, cl, p.next_n, p.H, TOPK,
                                               workspace=ws, out=out))
    ms = time_op(g.replay, flush_l2, stream, reps)
    hbm, src = peaks()
    gbs = fused_algorithmic_bytes(p) / (ms * 1e-3) / 1e9
    n_seq = max(1, min(p.B, oracle.num_threads() // p.next_n))
    cpu = cpu_baseline(p, n_seq, cpu_seconds, max_steps=20)
    del cache
    return {"workload": name, "description": WORKLOADS[name][1],
            "fused_ms": ms, "timing": f"median of {reps} CUDA-graph replays, L2 flushed before each",
            "value": scored_tokens(p) / (ms * 1e-3), "unit": UNIT,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm, "peak_source": f"{src} (hbm_gbs, burst)",
                         "algorithmic_bytes_per_launch": fused_algorithmic_bytes(p)},
            "cpu_baseline": cpu}


def insert_entries(idx, dev, flush_l2, stream, reps=10):
    """The insert where it streams: the headline batch's whole cache (every
    context, 1.3 M keys) in one call, and the mixed step's insert batch (8 x
    8192 chunked-prefill keys + 128 decode keys, with 5% padding rows)."""
    import torch
    from sparse_attention_indexer_quant_gb300 import workloads as wl
    hbm, _ = peaks()
    res = {}
    p = wl.batched_decode()
    cache = torch.from_numpy(wl.poisoned_cache(p.num_blocks)).to(dev)
    k = bf16_tensor(p.k, dev)
    slots = torch.from_numpy(p.slots).to(dev)
    ms = time_op(lambda: idx.quant_insert(k, slots, cache), flush_l2, stream, reps)
    n = p.total_tokens
    b = n * (256 + 8 + 68)
    res["insert_batched_cache"] = {
        "workload": f"the batched decode's whole cache: {n} bf16 keys in one call", "ms": ms,
        "tokens_per_s": n / (ms * 1e-3), "gbs": b / (ms * 1e-3) / 1e9,
        "frac_of_hbm": b / (ms * 1e-3) / 1e9 / hbm}
    del cache, k, slots
    ib = wl.mixed_insert_batch()
    cache = torch.from_numpy(wl.poisoned_cache(ib.num_blocks)).to(dev)
    idx.quant_insert(bf16_tensor(ib.pre_k, dev), torch.from_numpy(ib.pre_slots).to(dev), cache)
    k = bf16_tensor(ib.k, dev)
    slots = torch.from_numpy(ib.slots).to(dev)
    ms = time_op(lambda: idx.quant_insert(k, slots, cache), flush_l2, stream, reps)
    real, pads = ib.real_rows, len(ib.slots) - ib.real_rows
    b = real * (256 + 8 + 68) + pads * 8
    res["insert_mixed_batch"] = {
        "workload": f"the mixed step's insert batch: {real} keys + {pads} padding rows", "ms": ms,
        "tokens_per_s": real / (ms * 1e-3), "gbs": b / (ms * 1e-3) / 1e9,
        "frac_of_hbm": b / (ms * 1e-3) / 1e9 / hbm}
    return res


def prefill_oracle_sample(p, qv, qs, kv, ks, logits_dev, n_rows=512, seed=4242):
    """The oracle's prefill (logits and top-k) on a seeded sample of query rows
    of the causal prefill, timed on the host cores, with the full-size time
    extrapolated by valid (query, key) pairs; and a parity check of the GPU's
    logits on those rows against the oracle (tolerance 1e-5 of the summed
    magnitudes)."""
    import oracle
    g = np.random.default_rng(seed)
    st, en = p.windows()
    rows = np.sort(np.concatenate([g.choice(p.T, size=n_rows - 8, replace=False),
                                   np.arange(8) * 37]))  # a few rows shorter than k
    rows = np.unique(rows)
    qv_h = qv.cpu().numpy().reshape(p.T, p.H, 64)[rows].reshape(-1, 64)
    qs_h = qs.cpu().numpy().reshape(p.T, p.H, 4)[rows].reshape(-1, 4)
    kv_h, ks_h = kv.cpu().numpy(), ks.cpu().numpy()
    S = kv_h.shape[0]
    t0 = time.perf_counter()
    lg, mag = oracle.mqa_logits(qv_h, qs_h, p.H, kv_h, ks_h, p.weights[rows], st[rows], en[rows],
                                ld=S)
    oracle.topk_rows(np.nan_to_num(lg, nan=-np.inf), st[rows], en[rows], p.topk)
    dt = time.perf_counter() - t0
    pairs_s = int((en[rows].astype(np.int64) - st[rows]).sum())
    pairs = int((en.astype(np.int64) - st).sum())
    ok = True
    for i, r in enumerate(rows):
        a, b_ = int(st[r]), int(en[r])
        got = logits_dev[int(r), a:b_].cpu().numpy().astype(np.float64)
        ok &= bool((np.abs(got - lg[i, a:b_]) <= 1e-5 * mag[i, a:b_]).all())
    return {"kind": "oracle", "sample": f"{len(rows)} seeded query rows of the {p.T}-row causal "
                                        f"prefill ({pairs_s} of {pairs} valid pairs)",
            "cores": oracle.num_threads(), "sample_seconds": dt,
            "extrapolated_full_seconds": dt * pairs / pairs_s, "extrapolated": True,
            "tflops": 2.0 * p.H * 128 * pairs_s / dt / 1e12,
            "gpu_logits_match_oracle_on_sample": ok}


def step_entries(idx, dev, flush_l2, stream, reps=50):
    """The two-launch decode step (insert and q-quant inside the scoring
    launch) against the four separate calls, each step captured as a CUDA
    graph and replayed with L2 flushed before each: on the 8K
    single-sequence decode and on the 64-sequence batched decode."""
    import torch
    res = {}
    for name in ("pr_ref", "batched_decode"):
        p = make_workload(name)
        new = p.new_token_rows()
        old = np.setdiff1d(np.arange(p.total_tokens), new)
        cache = fill_cache(idx, p, dev, rows=old)
        new_k = bf16_tensor(p.k[new], dev)
        new_slots = torch.from_numpy(p.slots[new]).to(dev)
        q = bf16_tensor(p.q, dev)
        w = torch.from_numpy(p.weights).to(dev)
        bt = torch.from_numpy(p.block_table).to(dev)
        cl = torch.from_numpy(p.context_lens).to(dev)
        mb = p.block_table.shape[1]
        ws = idx.new_paged_topk_workspace(p.B, p.next_n, mb, TOPK, dev)
        ws_step = torch.empty(idx.paged_decode_step_workspace_bytes(p.B, p.next_n, p.H, mb, TOPK),
                              dtype=torch.uint8, device=dev)
        qv = torch.empty((p.rows * p.H, 64), dtype=torch.uint8, device=dev)
        qs = torch.empty((p.rows * p.H, 4), dtype=torch.uint8, device=dev)
        out = torch.empty((p.rows, TOPK), dtype=torch.int32, device=dev)

        def four():
            idx.quant_insert(new_k, new_slots, cache)
            idx.quant_q(q, out_vals=qv, out_scales=qs)
            idx.paged_logits_topk(qv, qs, w, cache, bt, cl, p.next_n, p.H, TOPK, workspace=ws,
                                  out=out)

        def two():
            idx.paged_decode_step(new_k, q, w, cache, bt, cl, p.next_n, p.H, TOPK,
                                  workspace=ws_step, out=out)

        ms4 = time_op(graph_of(four).replay, flush_l2, stream, reps)
        ms2 = time_op(graph_of(two).replay, flush_l2, stream, reps)
        res[f"decode_step_{name}"] = {
            "workload": WORKLOADS[name][1],
            "two_launch_step_us": ms2 * 1e3, "four_launch_step_us": ms4 * 1e3,
            "timing": f"median of {reps} CUDA-graph replays, L2 flushed before each",
            "note": "the two-launch step's scoring launch first quantises the query heads and "
                    "inserts the new keys in chunks its CTAs claim; a CTA waits for a "
                    "sequence's chunks before reading its keys"}
        del cache
    return res


def next_entries(idx, dev, flush_l2, stream, reps=10):
    """The fused q-RoPE + q-quant on the causal prefill's query heads and the
    K-pool insert of its keys (pool 4, seeded gates)."""
    import torch
    from sparse_attention_indexer_quant_gb300 import workloads as wl
    hbm, _ = peaks()
    p = wl.prefill()
    q = bf16_tensor(p.q, dev)
    g = wl.rng(4711)
    half = 32
    ang = np.arange(p.T, dtype=np.float64)[:, None] * 10000.0 ** (-np.arange(half) / half)[None, :]
    cs = torch.from_numpy(np.cos(ang).astype(np.float32)).to(dev)
    sn = torch.from_numpy(np.sin(ang).astype(np.float32)).to(dev)
    pos = torch.arange(p.T, dtype=torch.int32, device=dev)
    qv, qs = idx.rope_quant_q(q, pos, cs, sn, 64)
    ms = time_op(lambda: idx.rope_quant_q(q, pos, cs, sn, 64, out_vals=qv, out_scales=qs),
                 flush_l2, stream, reps)
    rows = p.T * p.H
    b = rows * (256 + 68) + p.T * (4 + 2 * half * 4)
    res = {"rope_quant_q": {"workload": f"{rows} query-head rows of the causal prefill, rot_dim 64",
                            "ms": ms, "gbs": b / (ms * 1e-3) / 1e9,
                            "frac_of_hbm": b / (ms * 1e-3) / 1e9 / hbm}}
    P = 4
    n = p.T
    k = bf16_tensor(p.k, dev)
    gate = torch.from_numpy(g.standard_normal((n, 128)).astype(np.float32)).to(dev)
    ape = torch.from_numpy(g.standard_normal((P, 128)).astype(np.float32)).to(dev)
    slots = np.full(n, -1, np.int64)
    slots[P - 1::P] = np.arange(n // P)
    num_blocks = (n // P + 63) // 64
    cache = torch.from_numpy(wl.poisoned_cache(num_blocks)).to(dev)
    sl = torch.from_numpy(slots).to(dev)
    ms = time_op(lambda: idx.kpool_insert(k, gate, ape, sl, cache), flush_l2, stream, reps)
    b = n * (256 + 512 + 8) + P * 512 + (n // P) * 68
    res["kpool_insert"] = {"workload": f"{n} keys of the causal prefill in pools of {P}",
                           "ms": ms, "gbs": b / (ms * 1e-3) / 1e9,
                           "frac_of_hbm": b / (ms * 1e-3) / 1e9 / hbm}
    return res


def secondary_measurements(idx, dev, flush_l2, stream, reps=10, decode=None, decode_desc=""):
    """The other steps of the path, each timed alone with a flushed L2: insert,
    q-quant, gather, prefill logits and top-k on the 32K-token causal prefill
    (one sequence, H = 32); with `decode` (the timed decode workload's state,
    described by `decode_desc`), the unfused paged logits and the top-k of its
    rows."""
    import torch
    from sparse_attention_indexer_quant_gb300 import workloads as wl
    hbm, _ = peaks()
    res = {}
    if decode is not None:
        dp, dcache, dqv, dqs, dw, dbt, dcl = decode
        ld = dp.block_table.shape[1] * 64
        lg = torch.empty((dp.rows, ld), dtype=torch.float32, device=dev)
        pl_ms = time_op(lambda: idx.paged_mqa_logits(dqv, dqs, dw, dcache, dbt, dcl, dp.next_n,
                                                     dp.H, ld=ld, out=lg), flush_l2, stream, reps)
        st_r, en_r = dp.row_windows()
        n_logits = int((en_r.astype(np.int64) - st_r).sum())
        pl_bytes = fused_algorithmic_bytes(dp) - dp.rows * dp.topk * 4 + 4 * n_logits
        en_d = torch.from_numpy(en_r).to(dev)
        dout = torch.empty((dp.rows, TOPK), dtype=torch.int32, device=dev)
        dk_ms = time_op(lambda: idx.topk_rows(lg, en_d, TOPK, out=dout), flush_l2, stream, reps)
        res["paged_logits_unfused"] = {
            "workload": f"{decode_desc}: logits rows written to HBM (unclean)", "ms": pl_ms,
            "gbs": pl_bytes / (pl_ms * 1e-3) / 1e9,
            "frac_of_hbm": pl_bytes / (pl_ms * 1e-3) / 1e9 / hbm}
        res["decode_topk_rows"] = {
            "workload": f"the decode's {dp.rows} logits rows, k=2048", "ms": dk_ms,
            "read_gbs": (4 * n_logits + dp.rows * TOPK * 4) / (dk_ms * 1e-3) / 1e9}
        del lg
    p = wl.prefill()
    S = int(p.tok_offsets[-1])
    cache = torch.from_numpy(wl.poisoned_cache(p.num_blocks)).to(dev)
    k = bf16_tensor(p.k, dev)
    slots = torch.from_numpy(p.slots).to(dev)
    ins_ms = time_op(lambda: idx.quant_insert(k, slots, cache), flush_l2, stream, reps)
    ins_bytes = S * (256 + 8 + 68)
    kv, ks = idx.gather_k(cache, torch.from_numpy(p.block_table).to(dev),
                          torch.from_numpy(p.new_lens.astype(np.int32)).to(dev),
                          torch.zeros(1, dtype=torch.int64, device=dev), S)
    g_bt = torch.from_numpy(p.block_table).to(dev)
    g_lens = torch.from_numpy(p.new_lens.astype(np.int32)).to(dev)
    g_off = torch.zeros(1, dtype=torch.int64, device=dev)
    g_ms = time_op(lambda: idx.gather_k(cache, g_bt, g_lens, g_off, S), flush_l2, stream, reps)
    q_bf = bf16_tensor(p.q, dev)
    qv, qs = idx.quant_q(q_bf)
    qq_ms = time_op(lambda: idx.quant_q(q_bf, out_vals=qv, out_scales=qs), flush_l2, stream, reps)
    q_rows = p.T * p.H
    w = torch.from_numpy(p.weights).to(dev)
    st, en = p.windows()
    st_d, en_d = torch.from_numpy(st).to(dev), torch.from_numpy(en).to(dev)
    logits = torch.empty((p.T, S), dtype=torch.float32, device=dev)
    pre_ms = time_op(lambda: idx.mqa_logits(qv, qs, w, kv, ks, st_d, en_d, p.H, out=logits),
                     flush_l2, stream, reps)
    pairs = int((en.astype(np.int64) - st).sum())
    flops = 2.0 * p.H * 128 * pairs
    peak_tf, peak_src = mxf4_peak_tflops()
    out = torch.empty((p.T, TOPK), dtype=torch.int32, device=dev)
    topk_ms = time_op(lambda: idx.topk_rows(logits, en_d, TOPK, row_start=st_d, out=out),
                      flush_l2, stream, reps)
    pre_cpu = prefill_oracle_sample(p, qv, qs, kv, ks, logits)
    del logits
    # the same rows' top-k without a logits tensor (candidate lists)
    ws_tk = torch.empty(idx.mqa_logits_topk_workspace_bytes(p.T, S, TOPK), dtype=torch.uint8,
                        device=dev)
    fused_ms = time_op(lambda: idx.mqa_logits_topk(qv, qs, w, kv, ks, st_d, en_d, p.H, TOPK,
                                                   workspace=ws_tk, out=out),
                       flush_l2, stream, reps)
    del ws_tk
    tf = flops / (pre_ms * 1e-3) / 1e12
    res.update({
        "q_quant": {"workload": f"{q_rows} query-head rows of the causal prefill", "ms": qq_ms,
                    "gbs": q_rows * (256 + 68) / (qq_ms * 1e-3) / 1e9,
                    "frac_of_hbm": q_rows * (256 + 68) / (qq_ms * 1e-3) / 1e9 / hbm},
        "gather": {"workload": "32768 cached keys of the causal prefill", "ms": g_ms,
                   "gbs": S * 2 * 68 / (g_ms * 1e-3) / 1e9,
                   "frac_of_hbm": S * 2 * 68 / (g_ms * 1e-3) / 1e9 / hbm},
        "insert": {"workload": "32768 bf16 keys of the causal prefill", "ms": ins_ms,
                   "tokens_per_s": S / (ins_ms * 1e-3),
                   "gbs": ins_bytes / (ins_ms * 1e-3) / 1e9,
                   "frac_of_hbm": ins_bytes / (ins_ms * 1e-3) / 1e9 / hbm},
        "prefill_logits": {"workload": "causal 32768 x 32768, H=32 (unclean rows)",
                           "ms": pre_ms, "tflops": tf, "peak_tflops": peak_tf,
                           "peak_source": peak_src, "frac": tf / peak_tf,
                           "store_gbs": pairs * 4 / (pre_ms * 1e-3) / 1e9,
                           "store_frac_of_hbm": pairs * 4 / (pre_ms * 1e-3) / 1e9 / hbm,
                           "valid_pairs": pairs,
                           # the CUDA-core epilogue: one max and one multiply-add per
                           # accumulator value (pairs x H); at the ALU pipe's rate for the
                           # max, 64 values per cycle per SM at the 2070 MHz SM clock
                           "epilogue_values": pairs * p.H,
                           "epilogue_floor_ms": pairs * p.H / (64.0 * SMS_GB300 * 2.07e9) * 1e3},
        "prefill_topk": {"workload": "32768 causal rows, k=2048", "ms": topk_ms,
                         "read_gbs": pairs * 4 / (topk_ms * 1e-3) / 1e9,
                         # the logits read once and k indices written per row
                         "frac_of_hbm": (pairs * 4 + p.T * TOPK * 4) / (topk_ms * 1e-3) / 1e9
                                        / hbm},
        "prefill_cpu_baseline": pre_cpu,
        "prefill_logits_topk_fused": {
            "workload": "causal 32768 x 32768, H=32, k=2048, no logits tensor",
            "ms": fused_ms, "unfused_ms": pre_ms + topk_ms,
            "tflops": tf * pre_ms / fused_ms},
    })
    return res


def mixed_prefill_entry(idx, dev, flush_l2, stream, reps=5):
    """The chunked-prefill half of the mixed batch (8 sequences, prefixes
    U[0, 65536], 8192 new tokens each): the gather of every sequence's cached
    keys, then per sequence the causal logits over its gathered keys and the
    top-k of its rows, as a serving step issues them; L2 flushed once before
    each repetition."""
    import torch
    from sparse_attention_indexer_quant_gb300 import workloads as wl
    p = wl.mixed_prefill_part()
    cache = torch.from_numpy(wl.poisoned_cache(p.num_blocks)).to(dev)
    idx.quant_insert(bf16_tensor(p.k, dev), torch.from_numpy(p.slots).to(dev), cache)
    lens = (p.prefix_lens.astype(np.int64) + p.new_lens).astype(np.int32)
    offs = p.tok_offsets[:-1].astype(np.int64)
    S = int(p.tok_offsets[-1])
    bt, ln, of = (torch.from_numpy(x).to(dev) for x in (p.block_table, lens, offs))
    kv, ks = idx.gather_k(cache, bt, ln, of, S)
    qv, qs = idx.quant_q(bf16_tensor(p.q, dev))
    w = torch.from_numpy(p.weights).to(dev)
    q_off = np.concatenate([[0], np.cumsum(p.new_lens)]).astype(np.int64)
    H = p.H
    Tmax, Lmax = int(p.new_lens.max()), int(lens.max())
    # two streams, each with its own logits buffer, take the sequences in
    # turn, so that one sequence's top-k overlaps the next one's logits
    n_streams = 2
    logits = [torch.empty((Tmax, Lmax), dtype=torch.float32, device=dev) for _ in range(n_streams)]
    out = [torch.empty((Tmax, TOPK), dtype=torch.int32, device=dev) for _ in range(n_streams)]
    side = [torch.cuda.Stream(device=dev) for _ in range(n_streams)]
    calls, pairs = [], 0
    for b in range(p.B):
        L, P, T = int(lens[b]), int(p.prefix_lens[b]), int(p.new_lens[b])
        st = torch.zeros(T, dtype=torch.int32, device=dev)
        en = torch.from_numpy((P + np.arange(T) + 1).astype(np.int32)).to(dev)
        qa, qb = int(q_off[b]), int(q_off[b + 1])
        pairs += int(T * P + T * (T + 1) // 2)
        calls.append((qv[qa * H:qb * H], qs[qa * H:qb * H], w[qa:qb], kv[offs[b]:offs[b] + L],
                      ks[offs[b]:offs[b] + L], st, en, T, L))

    def step():
        main = torch.cuda.current_stream()
        idx.gather_k(cache, bt, ln, of, S)
        for sd in side:
            sd.wait_stream(main)
        for i, (qvb, qsb, wb, kvb, ksb, st, en, T, L) in enumerate(calls):
            j = i % n_streams
            lg = logits[j][:T].view(-1)[:T * L].view(T, L)
            idx.mqa_logits(qvb, qsb, wb, kvb, ksb, st, en, H, out=lg, stream=side[j])
            idx.topk_rows(lg, en, TOPK, out=out[j][:T], stream=side[j])
        for sd in side:
            main.wait_stream(sd)

    ms = time_op(step, flush_l2, stream, reps)
    flops = 2.0 * H * 128 * pairs
    peak_tf, peak_src = mxf4_peak_tflops()
    return {"mixed_prefill": {
        "workload": "the mixed batch's 8 chunked prefills (prefix U[0, 65536] + 8192 new, "
                    "H=32): gather, then per sequence logits and top-k, the sequences in turn "
                    "on two streams",
        "ms": ms, "valid_pairs": pairs, "tflops": flops / (ms * 1e-3) / 1e12,
        "frac_of_mxf4_peak": flops / (ms * 1e-3) / 1e12 / peak_tf, "peak_source": peak_src,
        "note": "the step's time includes the top-k of every row and the gather"}}


def host_cpu_info():
    """The host the CPU baseline runs on: logical CPUs, the ones this process
    may use, the CPU model, and the OpenMP thread count the oracle runs with."""
    import oracle
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() in ("Model name", "Model"):
                model = ln.split(":", 1)[1].strip()
                if ln.startswith("Model name"):
                    break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as fh:
                for ln in fh:
                    if ln.lower().startswith(("model name", "cpu part")):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    try:
        usable = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        usable = os.cpu_count()
    threads = oracle.num_threads()
    env = os.environ.get("OMP_NUM_THREADS")
    why = (f"OMP_NUM_THREADS={env}" if env else
           f"OpenMP's default: the {usable} CPUs in this process's affinity mask")
    return {"nproc": os.cpu_count(), "usable_cpus": usable, "cpu_model": model,
            "threads": threads, "threads_capped_by": why}


def cpu_baseline(p, n_seq, min_seconds=10.0, max_steps=200):
    """The oracle, as it stands, on the first n_seq sequences of the batch:
    insert of their new keys, query quantisation, paged logits and top-k,
    repeated as whole decode steps until at least min_seconds of work."""
    import oracle
    from sparse_attention_indexer_quant_gb300 import workloads as wl
    n_seq = max(1, min(n_seq, p.B))
    hi_tok = int(p.tok_offsets[n_seq])
    cache = wl.poisoned_cache(p.num_blocks)
    new_rows = [r for r in p.new_token_rows() if r < hi_tok]
    old = np.setdiff1d(np.arange(hi_tok), new_rows)
    oracle.quant_insert(p.k[old], p.slots[old], cache)
    rows = n_seq * p.next_n
    ld = p.block_table.shape[1] * 64
    st, en = p.row_windows()
    toks = int((en[:rows].astype(np.int64) - st[:rows]).sum())
    steps, dt = 0, 0.0
    while steps < max_steps and (steps == 0 or dt < min_seconds):
        t0 = time.perf_counter()
        oracle.quant_insert(p.k[new_rows], p.slots[new_rows], cache)
        qv, qs = oracle.quant_q(p.q[:rows])
        lg, _ = oracle.paged_mqa_logits(qv, qs, n_seq, p.next_n, p.H, cache, p.block_table[:n_seq],
                                        p.context_lens[:n_seq], p.weights[:rows], ld)
        oracle.topk_rows(np.nan_to_num(lg, nan=-np.inf), st[:rows], en[:rows], p.topk)
        dt += time.perf_counter() - t0
        steps += 1
    return {"value": steps * toks / dt, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{steps} decode steps over the first {n_seq} of {p.B} sequences "
                      f"({toks} key-tokens per step)",
            "seconds": dt, "host": host_cpu_info()}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is the oracle's decode step
    over a bounded sample of the workload's sequences."""
    if rank != 0:
        return
    import oracle
    from sparse_attention_indexer_quant_gb300 import workloads as wl
    p = make_workload(args.workload)
    # calibrate the per-step sample so that warmup + steps take about 90 s: as
    # many sequences as the oracle has threads (it parallelises over query
    # rows), each window cut short to fit (the rate is per key-token)
    budget_s = args.ref_budget_s
    n_steps = args.steps + args.warmup
    n_seq = max(1, min(p.B, oracle.num_threads()))
    probe = cpu_baseline(p, n_seq, min_seconds=0.0)
    rate = probe["value"]
    per_step_tokens = max(2048 * n_seq, int(rate * budget_s / max(n_steps, 1)))
    per_seq = max(1, per_step_tokens // n_seq)
    cache = wl.poisoned_cache(p.num_blocks)
    hi_tok = int(p.tok_offsets[n_seq])
    oracle.quant_insert(p.k[:hi_tok], p.slots[:hi_tok], cache)
    ctx = np.minimum(p.context_lens[:n_seq], per_seq).astype(np.int32)
    rows = n_seq * p.next_n
    new_rows = [r for r in p.new_token_rows() if r < hi_tok]
    ld = p.block_table.shape[1] * 64

    def one():
        oracle.quant_insert(p.k[new_rows], p.slots[new_rows], cache)
        qv, qs = oracle.quant_q(p.q[:rows])
        lg, _ = oracle.paged_mqa_logits(qv, qs, n_seq, p.next_n, p.H, cache,
                                        p.block_table[:n_seq], ctx, p.weights[:rows], ld)
        en = ctx.astype(np.int32)
        oracle.topk_rows(np.nan_to_num(lg, nan=-np.inf), np.zeros_like(en), en, p.topk)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = time.perf_counter() - t0
    toks = int(ctx.astype(np.int64).sum())
    value = toks * args.steps / dt
    sample = (f"first {n_seq} of {p.B} sequences, contexts cut to at most {per_seq} keys, "
              f"{toks} key-tokens per step (oracle decode step: insert, q-quant, logits, top-k)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": workload_config(p, args.workload),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample, "host": host_cpu_info()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


_PG = None


def init_dist(world, backend=None):
    """One process per GPU (torchrun); the process group carries only the
    barrier and the max-over-ranks of the timing, never the data path."""
    global _PG
    if world <= 1:
        return
    import torch.distributed as dist
    if not dist.is_initialized():
        if backend is None:
            backend = "nccl" if __import__("torch").cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    _PG = dist


def barrier(world):
    if world > 1 and _PG is not None:
        _PG.barrier()


def reduce_max(x: float, world: int, device) -> float:
    """Largest value of x over the ranks (the whole job ends with its slowest rank)."""
    if world <= 1 or _PG is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    _PG.all_reduce(t, op=_PG.ReduceOp.MAX)
    return float(t.item())


def run_case(args):
    """One step of the path alone, args.reps times with L2 flushed before each,
    for a profiler to capture (ncu -k on the step's kernel); prints the median
    CUDA-event time of each timed call."""
    import torch
    from sparse_attention_indexer_quant_gb300 import binding as idx
    from sparse_attention_indexer_quant_gb300 import workloads as wl
    dev = torch.device("cuda")
    idx.check_device(torch.cuda.current_device())
    buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    sink = torch.empty((), dtype=torch.int64, device=dev)

    def flush():
        buf.fill_(1)
        torch.sum(buf, 0, dtype=torch.int64, out=sink)

    stream = torch.cuda.current_stream()
    name, rest = args.case[0], args.case[1:]
    if name == "prefill":
        T = int(rest[0]) if rest else 8192
        p = wl.prefill(T=T)
        S = int(p.tok_offsets[-1])
        cache = torch.from_numpy(wl.poisoned_cache(p.num_blocks)).to(dev)
        idx.quant_insert(bf16_tensor(p.k, dev), torch.from_numpy(p.slots).to(dev), cache)
        kv, ks = idx.gather_k(cache, torch.from_numpy(p.block_table).to(dev),
                              torch.from_numpy(p.new_lens.astype(np.int32)).to(dev),
                              torch.zeros(1, dtype=torch.int64, device=dev), S)
        qv, qs = idx.quant_q(bf16_tensor(p.q, dev))
        w = torch.from_numpy(p.weights).to(dev)
        st, en = p.windows()
        st_d, en_d = torch.from_numpy(st).to(dev), torch.from_numpy(en).to(dev)
        logits = torch.empty((p.T, S), dtype=torch.float32, device=dev)
        out = torch.empty((p.T, TOPK), dtype=torch.int32, device=dev)
        ms = time_op(lambda: idx.mqa_logits(qv, qs, w, kv, ks, st_d, en_d, p.H, out=logits),
                     flush, stream, args.reps)
        pairs = int((en.astype(np.int64) - st).sum())
        print(f"prefill T={T}: mqa_logits {ms:.3f} ms "
              f"({2.0 * p.H * 128 * pairs / (ms * 1e-3) / 1e12:.0f} TFLOP/s)")
        ms = time_op(lambda: idx.topk_rows(logits, en_d, TOPK, row_start=st_d, out=out), flush,
                     stream, args.reps)
        print(f"prefill T={T}: topk_rows {ms:.3f} ms")
        del logits
        ws = torch.empty(idx.mqa_logits_topk_workspace_bytes(p.T, S, TOPK), dtype=torch.uint8,
                         device=dev)
        ms = time_op(lambda: idx.mqa_logits_topk(qv, qs, w, kv, ks, st_d, en_d, p.H, TOPK,
                                                 workspace=ws, out=out), flush, stream, args.reps)
        print(f"prefill T={T}: mqa_logits_topk {ms:.3f} ms")
    elif name == "decode":
        p = wl.batched_decode()
        cache = torch.from_numpy(wl.poisoned_cache(p.num_blocks)).to(dev)
        idx.quant_insert(bf16_tensor(p.k, dev), torch.from_numpy(p.slots).to(dev), cache)
        qv, qs = idx.quant_q(bf16_tensor(p.q, dev))
        w = torch.from_numpy(p.weights).to(dev)
        bt = torch.from_numpy(p.block_table).to(dev)
        cl = torch.from_numpy(p.context_lens).to(dev)
        ws = idx.new_paged_topk_workspace(p.B, p.next_n, p.block_table.shape[1], TOPK, dev)
        out = torch.empty((p.rows, TOPK), dtype=torch.int32, device=dev)
        ms = time_op(lambda: idx.paged_logits_topk(qv, qs, w, cache, bt, cl, p.next_n, p.H, TOPK,
                                                   workspace=ws, out=out), flush, stream,
                     args.reps)
        print(f"batched decode: paged_logits_topk {ms * 1e3:.1f} us")
    elif name == "quant":
        T = int(rest[0]) if rest else 32768
        p = wl.prefill(T=T)
        q = bf16_tensor(p.q, dev)
        qv, qs = idx.quant_q(q)
        ms = time_op(lambda: idx.quant_q(q, out_vals=qv, out_scales=qs), flush, stream,
                     args.reps)
        print(f"prefill T={T}: quant_q of {T * p.H} rows {ms * 1e3:.1f} us")
        cache = torch.from_numpy(wl.poisoned_cache(p.num_blocks)).to(dev)
        k = bf16_tensor(p.k, dev)
        slots = torch.from_numpy(p.slots).to(dev)
        ms = time_op(lambda: idx.quant_insert(k, slots, cache), flush, stream, args.reps)
        print(f"prefill T={T}: quant_insert of {k.shape[0]} keys {ms * 1e3:.1f} us")
    elif name == "next":
        for key, v in next_entries(idx, dev, flush, stream, args.reps).items():
            print(f"{key}: {v['workload']}: {v['ms'] * 1e3:.1f} us, {v['frac_of_hbm']:.2f} of HBM")
    elif name == "step":
        for key, v in step_entries(idx, dev, flush, stream, args.reps).items():
            print(f"{key}: two-launch step {v['two_launch_step_us']:.1f} us, four-launch "
                  f"{v['four_launch_step_us']:.1f} us")
    else:
        raise SystemExit(f"unknown --case {name!r}")


def main():
    args = parse_args()
    if args.case:
        run_case(args)
        return
    rank, world, local_rank = dist_info()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    init_dist(world)
    run_ours(args, rank, world, local_rank)
    if world > 1 and _PG is not None:
        _PG.destroy_process_group()


if __name__ == "__main__":
    main()
