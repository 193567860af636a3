#!/usr/bin/env python
"""Benchmark of the sink-attention hot path on GB300.

Headline (one JSON line on rank 0): paged decode of the gpt-oss-20b-shaped
batch -- 64 query / 8 KV heads, head_dim 64, 64 requests with kv_len uniform
in [1, 4096], bf16 paged KV (16-token pages, shuffled), sinks ~ N(0, 2) with
-inf and +8 heads -- in algorithmic KV GB/s, with its roofline fraction
against the measured HBM copy bandwidth.  Extra sections time the other
workloads of the same path (long-context split-KV decode, ragged causal
prefill in TFLOP/s, the mixed serving batch) and the float64 CPU oracle.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Inputs are synthetic, seeded and resident in HBM before timing (``value``);
``e2e`` repeats the decode through the public API with pinned host buffers
and the per-step copies inside the timed region (uploads and downloads on
their own streams, double-buffered, as a serving loop overlaps them).  Copies of each KV pool
are cycled one per step, like the pools of consecutive layers, so that a page comes back only
after 4 GB of other pages: no step finds an earlier step's KV in L2.
Under torchrun each rank runs its own seeded batch (weak scaling, no
collective on the data path); rank 0 prints the max-over-ranks time.
"""

import argparse
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

METRIC = "sink-attn decode KV GB/s (% of HBM peak); prefill TFLOP/s (% BF16 peak)"
HEAD_DIM = 64
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DECODE_WORKLOAD = ("gpt-oss-20b decode: 64 q / 8 KV heads, head_dim 64, batch 64, "
                   "kv_len U[1,4096], bf16 paged KV (page 16, shuffled), sinks N(0,2) with -inf/+8 heads")


# ----------------------------------------------------------------- helpers

# DRAM bytes (read + write) per launch of a kernel from one ncu capture of
# the same workload, each valid only for the kernel sources it was taken on:
# once a source changes, the traffic is reported as unknown (null).
TRAFFIC = {
    "decode": {"sources": ("gqa_attention_learned_gb300/csrc/decode.cu",
                           "gqa_attention_learned_gb300/csrc/kernels.cuh",
                           "gqa_attention_learned_gb300/csrc/ptx.cuh"),
               "sha256_16": "32c82e9d91842e7b", "bytes": 261_699_328 + 2_998_272},
    "prefill": {"sources": ("gqa_attention_learned_gb300/csrc/prefill.cu",
                            "gqa_attention_learned_gb300/csrc/kernels.cuh",
                            "gqa_attention_learned_gb300/csrc/ptx.cuh"),
                "sha256_16": "5c75eae3ef74e629", "bytes": 222_833_920 + 139_865_856},
}


def sources_hash(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def kernel_traffic(kernel):
    t = TRAFFIC[kernel]
    try:
        ok = t["sha256_16"] is not None and sources_hash(t["sources"]) == t["sha256_16"]
    except OSError:
        return None
    return t["bytes"] if ok else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def decode_bytes(kv_lens, num_qo_heads, num_kv_heads, head_dim=HEAD_DIM, page_size=16):
    """Algorithmic bytes of one decode pass: every K and V row once, plus q,
    out, lse, sinks, kv_lens and the page-table entries in use."""
    kv = sum(int(n) for n in kv_lens)
    pages = sum((int(n) + page_size - 1) // page_size for n in kv_lens)
    b = len(kv_lens)
    return (kv * num_kv_heads * head_dim * 2 * 2          # K and V, bf16
            + 2 * b * num_qo_heads * head_dim * 2          # q in, out
            + b * num_qo_heads * 4 + num_qo_heads * 4      # lse, sinks
            + b * 4 + pages * 4)                           # kv_lens, table


def verify_bytes(kv_lens, q_len, num_qo_heads, num_kv_heads, tree, head_dim=HEAD_DIM,
                 page_size=16):
    """Algorithmic bytes of one verification pass: every K and V row once,
    q_len query/output rows and lse per request, sinks, kv_lens, the table
    entries in use and the tree masks."""
    kv = sum(int(n) for n in kv_lens)
    pages = sum((int(n) + page_size - 1) // page_size for n in kv_lens)
    b = len(kv_lens)
    return (kv * num_kv_heads * head_dim * 2 * 2
            + 2 * b * q_len * num_qo_heads * head_dim * 2
            + b * q_len * num_qo_heads * 4 + num_qo_heads * 4
            + b * 4 + pages * 4 + (b * q_len * 8 if tree else 0))


def prologue_bytes(tokens, num_qo_heads, num_kv_heads, head_dim=HEAD_DIM):
    """Algorithmic bytes of the prologue: the qkv rows and the token's position
    and slot read once, q written once, k and v written to their cache slot,
    plus the bias row."""
    heads = num_qo_heads + 2 * num_kv_heads
    return tokens * (2 * heads * head_dim * 2 + 8) + heads * head_dim * 2


def prefill_flops(seqlens, num_qo_heads, head_dim=HEAD_DIM):
    """QK^T and PV over the causal (lower-triangular incl. diagonal) pairs."""
    return sum(4 * head_dim * num_qo_heads * n * (n + 1) // 2 for n in seqlens)


def extend_flops(q_lens, kv_lens, num_qo_heads, head_dim=HEAD_DIM):
    tot = 0
    for lq, lk in zip(q_lens, kv_lens):
        prefix = lk - lq
        tot += 4 * head_dim * num_qo_heads * (lq * prefix + lq * (lq + 1) // 2)
    return tot


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0, period_ms=100):
        self.index, self.period = index, period_ms
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        time.sleep(0.15)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.close()

    def summary(self):
        rows = []
        try:
            with open(self.file.name) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) == 9 and parts[1].replace(".", "").isdigit():
                        rows.append(parts)
        finally:
            os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


# ------------------------------------------------------------ distributed

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(backend):
    import torch.distributed as dist
    world, rank, _ = dist_info()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return world, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_scalar(x, op, device="cpu"):
    """All-reduce one float (MAX or SUM) across ranks; identity when alone."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(units_this_rank, seconds_this_rank, device="cpu"):
    """Whole-job throughput: units of all ranks / slowest rank's time."""
    t = reduce_scalar(seconds_this_rank, "max", device)
    u = reduce_scalar(units_this_rank, "sum", device)
    return u, t, (u / t if t > 0 else 0.0)


# ------------------------------------------------------------------ GPU arm

def _time_steps(torch, fn, steps, warmup, stream):
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        fn(i)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3


# Bytes of other pages read before a page comes back (about 30x L2).
REUSE_BYTES = 4e9


def kv_pools(torch, k, v, dev):
    """Copies of a KV pool on `dev`, cycled one per step like the pools of
    consecutive layers: a page is read again only after REUSE_BYTES of other
    pages, so no step finds pages of an earlier one in L2, whatever eviction
    priority the kernels give their loads."""
    import math
    pool_bytes = 2 * k.numel() * k.element_size()
    n = min(32, max(2, math.ceil(REUSE_BYTES / pool_bytes) + 1))
    first = (k.to(dev), v.to(dev))
    return [first] + [(first[0].clone(), first[1].clone()) for _ in range(n - 1)]


def pools_label(pools):
    mb = 2 * pools[0][0].numel() * pools[0][0].element_size() / 1e6
    return f"{len(pools)} KV pool copies ({len(pools)} x {mb:.0f} MB) cycled, one per step"


def run_decode_arm(args, rank, dev):
    import torch

    import gqa_attention_learned_gb300 as sa
    from gqa_attention_learned_gb300 import workloads

    w = workloads.decode_batch(seed=1 + 1000 * rank)
    hq, hkv = w["num_qo_heads"], w["num_kv_heads"]
    lens = [int(x) for x in w["kv_lens"]]
    nbytes = decode_bytes(lens, hq, hkv)
    q = w["q"].to(dev)
    pools = kv_pools(torch, w["k_cache"], w["v_cache"], dev)
    table, kv_lens, sinks = w["page_table"].to(dev), w["kv_lens"].to(dev), w["sinks"].to(dev)
    max_kv = w["max_kv_len"]
    splits, ws_bytes = sa.decode_plan(64, hq, hkv, max_kv, args.splits)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[0], hq, dtype=torch.float32, device=dev)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(i, mode=None):
        kc, vc = pools[i % len(pools)]
        sa.decode(q, kc, vc, table, kv_lens, sinks, w["scale"], max_kv, out=out, lse=lse,
                  num_splits=args.splits, workspace=ws, stream=stream, programmatic=mode)

    with ClockSampler(index=torch.cuda.current_device()) as clocks:
        secs = _time_steps(torch, step, args.steps, args.warmup, stream)
    units, t_max, gbps = aggregate(nbytes * args.steps, secs, dev)
    launches_per_step = 1
    # the same steps with every launch plain: each kernel starts only after
    # the previous one has finished (no overlap of neighbouring launches)
    plain_steps = max(args.steps, 100)
    plain_secs = _time_steps(torch, lambda i: step(i, False), plain_steps, args.warmup, stream)
    _, _, plain_gbps = aggregate(nbytes * plain_steps, plain_secs, dev)

    # the same plain launches replayed from one CUDA graph (a step on every
    # pool copy): still no overlap of neighbouring kernels, but the device has
    # the next launch queued when a kernel ends
    def plain_on(i, s):
        kc, vc = pools[i % len(pools)]
        sa.decode(q, kc, vc, table, kv_lens, sinks, w["scale"], max_kv, out=out, lse=lse,
                  num_splits=args.splits, workspace=ws, stream=s, programmatic=False)

    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        plain_on(0, side)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    plain_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(plain_graph):
        cs = torch.cuda.current_stream()
        for i in range(len(pools)):
            plain_on(i, cs)
    graph_reps = max(10, plain_steps // len(pools))
    g_secs = _time_steps(torch, lambda i: plain_graph.replay(), graph_reps, 3, stream)
    _, _, plain_graph_gbps = aggregate(nbytes * graph_reps * len(pools), g_secs, dev)
    del plain_graph

    # end to end through the public call: each step's inputs (q, page table,
    # kv_lens) go host -> device in one copy of a packed pinned buffer, the
    # results (out, lse) come back in one copy; the sinks are weights and stay
    # resident like the KV cache
    def packed(parts):
        offs, total = [], 0
        for t in parts:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, total

    def views(buf, parts, offs):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                for t, o in zip(parts, offs)]

    ins = [w["q"], w["page_table"], w["kv_lens"]]
    in_offs, in_bytes = packed(ins)
    in_h = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    for t, v in zip(ins, views(in_h, ins, in_offs)):
        v.copy_(t)
    in_d = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    q_e, table_e, lens_e = views(in_d, ins, in_offs)
    outs = [out, lse]
    out_offs, out_bytes = packed(outs)
    out_d = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
    out_h = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    out_e, lse_e = views(out_d, outs, out_offs)
    h2d, d2h = in_bytes, out_bytes

    def e2e_step(i):
        in_d.copy_(in_h, non_blocking=True)
        kc, vc = pools[i % len(pools)]
        sa.decode(q_e, kc, vc, table_e, lens_e, sinks, w["scale"], max_kv, out=out_e, lse=lse_e,
                  num_splits=args.splits, workspace=ws, stream=stream)
        out_h.copy_(out_d, non_blocking=True)

    # Pipelined as a serving loop runs it: two sets of device buffers; step
    # i's upload (copy stream 1) and step i-2's download (copy stream 2)
    # overlap the decode of step i-1 on the compute stream, with events
    # guarding each buffer's reuse.  Every step still uploads its own inputs
    # and downloads its own results inside the timed region.
    sets = []
    for _ in range(2):
        ib = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        ob = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
        sets.append(dict(in_d=ib, ins=views(ib, ins, in_offs), out_d=ob,
                         outs=views(ob, outs, out_offs),
                         out_h=torch.empty(out_bytes, dtype=torch.uint8).pin_memory(),
                         up=torch.cuda.Event(), done=torch.cuda.Event(),
                         down=torch.cuda.Event()))
    up_s, down_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_pipelined(steps, cs):
        up_s.wait_stream(cs)
        down_s.wait_stream(cs)
        for i in range(steps):
            b = sets[i & 1]
            if i >= 2:
                up_s.wait_event(b["done"])          # decode i-2 has read this input set
            with torch.cuda.stream(up_s):
                b["in_d"].copy_(in_h, non_blocking=True)
            b["up"].record(up_s)
            cs.wait_event(b["up"])
            if i >= 2:
                cs.wait_event(b["down"])            # download i-2 has read this output set
            kc, vc = pools[i % len(pools)]
            q_b, table_b, lens_b = b["ins"]
            out_b, lse_b = b["outs"]
            sa.decode(q_b, kc, vc, table_b, lens_b, sinks, w["scale"], max_kv, out=out_b,
                      lse=lse_b, num_splits=args.splits, workspace=ws, stream=cs)
            b["done"].record(cs)
            down_s.wait_event(b["done"])
            with torch.cuda.stream(down_s):
                b["out_h"].copy_(b["out_d"], non_blocking=True)
            b["down"].record(down_s)
        cs.wait_stream(up_s)
        cs.wait_stream(down_s)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        fn()
        t1.record(stream)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / 1e3

    e2e_steps = max(10, args.steps // 10)
    eager_secs = timed(lambda: e2e_pipelined(e2e_steps, stream))
    _, _, eager_gbps = aggregate(nbytes * e2e_steps, eager_secs, dev)
    # the same pipelined steps captured once in a CUDA graph (no host work per
    # step: the Python issue rate no longer bounds the loop)
    graph_err = None
    try:
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            e2e_pipelined(2, cap)                   # warm-up outside capture
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph):
            e2e_pipelined(e2e_steps, torch.cuda.current_stream())
        graph_secs = timed(e2e_graph.replay)
        _, _, graph_gbps = aggregate(nbytes * e2e_steps, graph_secs, dev)
        del e2e_graph
    except RuntimeError as exc:                     # capture refused: report, keep the rest
        graph_err, graph_gbps = str(exc).splitlines()[0], None
    e2e_gbps = graph_gbps if graph_gbps is not None else eager_gbps
    # the same calls one after another on one stream, no overlap
    ser_secs = _time_steps(torch, e2e_step, e2e_steps, args.warmup, stream)
    _, _, ser_gbps = aggregate(nbytes * e2e_steps, ser_secs, dev)

    # same, with the whole paged KV pool copied host -> device every step
    k_h, v_h = w["k_cache"].pin_memory(), w["v_cache"].pin_memory()
    kv_pool_bytes = 2 * k_h.numel() * k_h.element_size()

    def e2e_kv_step(i):
        kc, vc = pools[i % len(pools)]
        kc.copy_(k_h, non_blocking=True)
        vc.copy_(v_h, non_blocking=True)
        e2e_step(i)

    kv_steps = max(5, args.steps // 200)
    kv_secs = _time_steps(torch, e2e_kv_step, kv_steps, 2, stream)
    _, _, kv_gbps = aggregate(nbytes * kv_steps, kv_secs, dev)

    pool_label = pools_label(pools)
    return dict(w=w, nbytes=nbytes, secs=t_max, gbps=gbps / 1e9, splits=splits,
                plain_gbps=plain_gbps / 1e9, plain_steps=plain_steps, pool_label=pool_label,
                plain_graph_gbps=plain_graph_gbps / 1e9,
                launches_per_step=launches_per_step, clocks=clocks.summary(),
                e2e=dict(value=e2e_gbps / 1e9, unit="GB/s", h2d_bytes_per_step=h2d,
                         d2h_bytes_per_step=d2h, steps=e2e_steps,
                         mode="pipelined, CUDA graph" if graph_gbps is not None else
                              "pipelined, eager",
                         eager_pipelined_value=round(eager_gbps / 1e9, 2),
                         serialized_value=round(ser_gbps / 1e9, 2),
                         graph_error=graph_err,
                         note="paged KV cache and sinks resident on the device (serving state); "
                              "per step one H2D copy of packed q / page table / kv_lens and one "
                              "D2H copy of packed out / lse, from/to pinned memory, pipelined "
                              "over two buffer sets (uploads and downloads on their own streams "
                              "overlap the neighbouring steps' decodes), all steps captured in "
                              "one CUDA graph; eager_pipelined_value: the same issued from "
                              "Python step by step; serialized_value: the same calls back to "
                              "back on one stream"),
                e2e_kv_h2d=dict(value=kv_gbps / 1e9, unit="GB/s",
                                h2d_bytes_per_step=h2d + kv_pool_bytes, d2h_bytes_per_step=d2h,
                                steps=kv_steps))


def run_graph_decode(args, rank, dev, peaks):
    """The headline decode step replayed from CUDA graphs (one per KV pool
    copy) instead of launched from Python: same kernel, no host work."""
    import torch

    import gqa_attention_learned_gb300 as sa
    from gqa_attention_learned_gb300 import workloads

    w = workloads.decode_batch(seed=1 + 1000 * rank)
    hq, hkv = w["num_qo_heads"], w["num_kv_heads"]
    lens = [int(x) for x in w["kv_lens"]]
    nbytes = decode_bytes(lens, hq, hkv)
    q = w["q"].to(dev)
    pools = kv_pools(torch, w["k_cache"], w["v_cache"], dev)
    table, kv_lens, sinks = w["page_table"].to(dev), w["kv_lens"].to(dev), w["sinks"].to(dev)
    max_kv = w["max_kv_len"]
    _, ws_bytes = sa.decode_plan(64, hq, hkv, max_kv)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[0], hq, dtype=torch.float32, device=dev)

    def call(i):
        kc, vc = pools[i % len(pools)]
        sa.decode(q, kc, vc, table, kv_lens, sinks, w["scale"], max_kv, out=out, lse=lse,
                  workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(0)
        call(1)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    # one graph per step (per pool copy), and one graph holding a step on
    # every pool copy, whose launches keep their programmatic edges
    per_graph = len(pools)
    graphs = []
    for i in range(len(pools)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call(i)
        graphs.append(g)
    g10 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g10):
        for i in range(per_graph):
            call(i)
    stream = torch.cuda.current_stream()

    def step(i):
        graphs[i % len(graphs)].replay()

    steps = max(100, args.steps // 2)
    secs = _time_steps(torch, step, steps, args.warmup, stream)
    _, t, bps = aggregate(nbytes * steps, secs, dev)
    reps = max(10, steps // per_graph)
    secs10 = _time_steps(torch, lambda i: g10.replay(), reps, args.warmup, stream)
    _, t10, bps10 = aggregate(nbytes * reps * per_graph, secs10, dev)
    del graphs, g10, pools
    torch.cuda.empty_cache()
    return dict(workload=DECODE_WORKLOAD + " (CUDA graph replay)", steps=steps,
                ms_per_step=1e3 * t / steps, value=round(bps / 1e9, 2), unit="GB/s",
                frac_of_hbm=round(bps / 1e9 / peaks["hbm_gbs"], 4),
                multi_step_graph=dict(steps=reps * per_graph, steps_per_graph=per_graph,
                                    ms_per_step=1e3 * t10 / (reps * per_graph),
                                    value=round(bps10 / 1e9, 2), unit="GB/s",
                                    frac_of_hbm=round(bps10 / 1e9 / peaks["hbm_gbs"], 4)),
                note="plan from host-side sizes; chunks per request derived on the device from "
                     "kv_lens, so the captured launch serves new lengths and page tables; value: "
                     "one graph per step (no programmatic edge between graph launches); "
                     "multi_step_graph: one graph holding a step on every pool copy")


def run_long_decode(args, rank, dev):
    import torch

    import gqa_attention_learned_gb300 as sa
    from gqa_attention_learned_gb300 import workloads

    w = workloads.long_decode(seed=2 + 1000 * rank)
    hq, hkv = w["num_qo_heads"], w["num_kv_heads"]
    lens = [int(x) for x in w["kv_lens"]]
    nbytes = decode_bytes(lens, hq, hkv)
    q, table, kv_lens, sinks = (w[n].to(dev) for n in ("q", "page_table", "kv_lens", "sinks"))
    pools = kv_pools(torch, w["k_cache"], w["v_cache"], dev)
    res = {}
    for label, splits in (("auto", 0), ("8 splits", 8)):
        s, ws_bytes = sa.decode_plan(len(lens), hq, hkv, w["max_kv_len"], splits)
        ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        out = torch.empty_like(q)
        lse = torch.empty(len(lens), hq, dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream()

        def step(i, splits=splits, ws=ws, out=out, lse=lse):
            kc, vc = pools[i % len(pools)]
            sa.decode(q, kc, vc, table, kv_lens, sinks, w["scale"], w["max_kv_len"], out=out,
                      lse=lse, num_splits=splits, workspace=ws, stream=stream)

        steps = max(20, args.steps // 50)
        secs = _time_steps(torch, step, steps, args.warmup, stream)
        _, t, gbps = aggregate(nbytes * steps, secs, dev)
        res[label] = dict(splits=s, ms_per_step=1e3 * t / steps, value=gbps / 1e9, unit="GB/s")
    label = pools_label(pools)
    del pools
    torch.cuda.empty_cache()
    return dict(workload="long-context split-KV decode: 64 q / 8 KV heads, batch 8, "
                         "kv_len U[32768,131072], bf16 paged KV (page 16); " + label,
                kv_bytes=nbytes, runs=res)


def run_verify(args, rank, dev, peaks):
    import torch

    import gqa_attention_learned_gb300 as sa
    from gqa_attention_learned_gb300 import workloads

    res = {}
    for label, q_len, tree in (("mtp 2 tokens", 2, False), ("4 tokens causal", 4, False),
                               ("8-node tree", 8, True)):
        w = workloads.verify_batch(seed=5 + 1000 * rank, q_len=q_len, tree=tree)
        hq, hkv = w["num_qo_heads"], w["num_kv_heads"]
        lens = [int(x) for x in w["kv_lens"]]
        nbytes = verify_bytes(lens, q_len, hq, hkv, tree)
        q = w["q"].to(dev)
        pools = kv_pools(torch, w["k_cache"], w["v_cache"], dev)
        table, kv_lens, sinks = w["page_table"].to(dev), w["kv_lens"].to(dev), w["sinks"].to(dev)
        mask = None if w["tree_mask"] is None else w["tree_mask"].to(dev)
        splits, ws_bytes = sa.verify_plan(len(lens), q_len, hq, hkv, w["max_kv_len"])
        ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream()

        def step(i, q=q, pools=pools, table=table, kv_lens=kv_lens, sinks=sinks, mask=mask,
                 w=w, out=out, lse=lse, ws=ws):
            kc, vc = pools[i % len(pools)]
            sa.verify(q, kc, vc, table, kv_lens, sinks, w["scale"], w["max_kv_len"],
                      tree_mask=mask, out=out, lse=lse, workspace=ws, stream=stream)

        steps = max(50, args.steps // 20)
        secs = _time_steps(torch, step, steps, args.warmup, stream)
        _, t, bps = aggregate(nbytes * steps, secs, dev)
        res[label] = dict(q_len=q_len, tree=tree, splits=splits, bytes_per_step=nbytes,
                          kernel=verify_kernel(len(lens), q_len, hq, hkv, w["max_kv_len"]),
                          ms_per_step=1e3 * t / steps, value=round(bps / 1e9, 2), unit="GB/s",
                          frac_of_hbm=round(bps / 1e9 / peaks["hbm_gbs"], 4))
        del pools, q
        torch.cuda.empty_cache()
    return dict(workload="draft-token verification on the gpt-oss-20b decode batch: 64 requests, "
                         "kv_len U[q_len,4096], 64 q / 8 KV heads, bf16 paged KV; copies of the KV "
                         "pool cycled one per step (a page re-read after 4 GB of others)",
                runs=res)


def verify_kernel(batch, q_len, hq, hkv, max_kv_len, num_sms=152):
    """Which kernel sinkattn_verify runs for these sizes with num_splits = 0
    (the library's rule, stated in include/sinkattn.h): the tensor-core
    kernel for >= 24 query rows per KV head, a group dividing 128, at most
    8192 keys and a wave of (request, KV head) tiles; else the mma.sync
    decode kernel with 8 or 16 rows per CTA."""
    g = hq // hkv
    tiles = -(-q_len // max(1, 128 // g)) if 128 % g == 0 else 0
    if (q_len >= 2 and 128 % g == 0 and q_len * g >= 24 and -(-max_kv_len // 16) <= 512
            and tiles * batch * hkv >= 2 * num_sms):
        if q_len * g <= 64:               # every key tile split between two softmax warps
            return ("prefill_kernel<true, true, true> (tcgen05, key halves; rows = tokens x heads "
                    "of a KV head)")
        return "prefill_kernel<true, true> (tcgen05; rows = tokens x heads of a KV head)"
    nb = 2 if q_len * g > 8 else 1
    return f"decode_kernel<{nb}, true> (mma.sync; rows = tokens x heads of a KV head)"


def run_prologue(args, rank, dev, peaks):
    import numpy as np
    import torch

    import gqa_attention_learned_gb300 as sa
    from gqa_attention_learned_gb300 import workloads

    inv, ms = sa.yarn_table()                     # base 150000, factor 32, L 4096, beta 32 / 1
    pre = workloads.ragged_prefill(seed=3 + 1000 * rank)
    cu = [int(x) for x in pre["cu_seqlens"]]
    lens = [b - a for a, b in zip(cu, cu[1:])]
    res = {}
    for label, seq_lens, starts in (("prefill 4 sequences", lens, [0] * len(lens)),
                                    ("decode 64 tokens", [1] * 64,
                                     [int(x) for x in np.random.default_rng(1).integers(0, 4096, 64)])):
        w = workloads.prologue_batch(seq_lens, starts, seed=6 + 1000 * rank)
        tokens = sum(seq_lens)
        nbytes = prologue_bytes(tokens, 64, 8)
        qkv, bias = w["qkv"].to(dev), w["bias"].to(dev)
        pos, slots = w["positions"].to(dev), w["slot_mapping"].to(dev)
        kc, vc = w["k_cache"].to(dev), w["v_cache"].to(dev)
        q_out = torch.empty(tokens, 64, 64, dtype=torch.bfloat16, device=dev)
        stream = torch.cuda.current_stream()

        def call(qkv=qkv, bias=bias, pos=pos, slots=slots, kc=kc, vc=vc, q_out=q_out):
            sa.qkv_prologue(qkv, bias, pos, slots, inv, ms, kc, vc, 64, 8, q_out=q_out)

        # launches replayed from a CUDA graph (10 per replay), so the small
        # case measures the device, not the Python call
        per_graph = 10
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            call()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(per_graph):
                call()

        def step(i, g=g):
            g.replay()

        steps = max(10, args.steps // 200)
        secs = _time_steps(torch, step, steps, args.warmup, stream)
        _, t, bps = aggregate(nbytes * steps * per_graph, secs, dev)
        t /= per_graph
        res[label] = dict(tokens=tokens, bytes_per_step=nbytes, ms_per_step=1e3 * t / steps,
                          value=round(bps / 1e9, 2), unit="GB/s",
                          frac_of_hbm=round(bps / 1e9 / peaks["hbm_gbs"], 4))
        del qkv, kc, vc, q_out, g
        torch.cuda.empty_cache()
    return dict(workload="attention prologue (QKV bias + YaRN rotary on q/k + paged k/v write), "
                         "64 q / 8 KV heads, head_dim 64, bf16; YaRN base 150000, factor 32, "
                         "original context 4096, beta 32 / 1 (the pages give no values)",
                kernel="prologue_kernel",
                note="timed as CUDA-graph replays of 10 launches; the decode-sized batch "
                     "(1.3 MB) is L2-resident",
                runs=res)


def run_prefill(args, rank, dev, peaks):
    import torch

    import gqa_attention_learned_gb300 as sa
    from gqa_attention_learned_gb300 import workloads

    w = workloads.ragged_prefill(seed=3 + 1000 * rank)
    cu = [int(x) for x in w["cu_seqlens"]]
    lens = [b - a for a, b in zip(cu, cu[1:])]
    flops = prefill_flops(lens, w["num_qo_heads"])
    args_d = [w[n].to(dev) for n in ("q", "k", "v", "cu_seqlens", "sinks")]
    out = torch.empty_like(args_d[0])
    lse = torch.empty(args_d[0].shape[0], w["num_qo_heads"], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        sa.prefill(*args_d, w["scale"], w["max_seqlen"], out=out, lse=lse, stream=stream)

    steps = max(10, args.steps // 200)
    secs = _time_steps(torch, step, steps, args.warmup, stream)
    _, t, fps = aggregate(flops * steps, secs, dev)
    tf = fps / 1e12
    return dict(workload="causal ragged prefill: 64 q / 8 KV heads, head_dim 64, 4 sequences "
                         f"{lens} ({sum(lens)} tokens), bf16, fp32 LSE",
                flops_per_step=flops, steps=steps, ms_per_step=1e3 * t / steps,
                value=round(tf, 2), unit="TFLOP/s",
                roofline={"bound": "tensor", "achieved": round(tf, 2),
                          "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                          "frac": round(tf / peaks["bf16_tflops"], 4),
                          "frac_of_sustained": round(tf / peaks["bf16_tflops_sustained"], 4),
                          "traffic": kernel_traffic("prefill"),
                          "kernel": "prefill_kernel<false, false>"})


def run_mixed(args, rank, dev, peaks):
    import torch

    import gqa_attention_learned_gb300 as sa
    from gqa_attention_learned_gb300 import workloads

    m = workloads.mixed_batch(seed=4 + 1000 * rank)
    d, e = m["decode"], m["extend"]
    hq, hkv = m["num_qo_heads"], m["num_kv_heads"]
    pools = kv_pools(torch, m["k_cache"], m["v_cache"], dev)
    sinks = m["sinks"].to(dev)
    dq, dt, dl = d["q"].to(dev), d["page_table"].to(dev), d["kv_lens"].to(dev)
    eq, ecu, et, el = (e["q"].to(dev), e["cu_seqlens_q"].to(dev), e["page_table"].to(dev),
                       e["kv_lens"].to(dev))
    dec_lens = [int(x) for x in d["kv_lens"]]
    ext_kv = [int(x) for x in e["kv_lens"]]
    ext_q = [e["max_q_len"]] * len(ext_kv)
    nbytes = decode_bytes(dec_lens, hq, hkv)
    flops = extend_flops(ext_q, ext_kv, hq)
    _, ws_bytes = sa.decode_plan(len(dec_lens), hq, hkv, d["max_kv_len"], 0)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    dout = torch.empty_like(dq)
    dlse = torch.empty(dq.shape[0], hq, dtype=torch.float32, device=dev)
    eout = torch.empty_like(eq)
    else_ = torch.empty(eq.shape[0], hq, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    steps = max(10, args.steps // 200)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]

    def step(i, record=False):
        kc, vc = pools[i % len(pools)]
        if record:
            ev[i][0].record(stream)
        sa.decode(dq, kc, vc, dt, dl, sinks, m["scale"], d["max_kv_len"], out=dout, lse=dlse,
                  workspace=ws, stream=stream)
        if record:
            ev[i][1].record(stream)
        sa.prefill_paged(eq, ecu, kc, vc, et, el, sinks, m["scale"], e["max_q_len"],
                         e["max_kv_len"], out=eout, lse=else_, stream=stream)
        if record:
            ev[i][2].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    barrier()
    for i in range(steps):
        step(i, record=True)
    torch.cuda.synchronize()
    t_dec = sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)) / 1e3
    t_ext = sum(ev[i][1].elapsed_time(ev[i][2]) for i in range(steps)) / 1e3
    t_all = sum(ev[i][0].elapsed_time(ev[i][2]) for i in range(steps)) / 1e3
    _, t_all, _ = aggregate(0, t_all, dev)
    dec_gbs = nbytes * steps / t_dec / 1e9
    ext_tf = flops * steps / t_ext / 1e12
    ideal = nbytes / (peaks["hbm_gbs"] * 1e9) + flops / (peaks["bf16_tflops"] * 1e12)
    return dict(workload="mixed serving batch: 32 decode requests (kv_len U[512,16384]) + 4 "
                         "chunked-prefill requests of 2048 tokens on prefixes U[0,14336], one "
                         "shuffled page pool, two launches on one stream; " + pools_label(pools),
                steps=steps, ms_per_step=1e3 * t_all / steps,
                decode={"value": round(dec_gbs, 2), "unit": "GB/s", "bytes": nbytes,
                        "ms": 1e3 * t_dec / steps},
                extend={"value": round(ext_tf, 2), "unit": "TFLOP/s", "flops": flops,
                        "ms": 1e3 * t_ext / steps},
                combined_roofline_frac=round(ideal / (t_all / steps), 4))


def run_gqa(args, rank, dev, peaks):
    """Decode over GQA group sizes (query / KV heads 64/8, 48/4, 64/4, 128/8,
    64/2) at 64 and 128 requests, kv_len U[1,4096]: groups above 8 run 16
    heads per CTA when those CTAs fill a wave."""
    import torch

    import gqa_attention_learned_gb300 as sa
    from gqa_attention_learned_gb300 import workloads

    res = {}
    for hq, hkv, b in ((64, 8, 64), (48, 4, 64), (64, 4, 64), (64, 4, 128), (128, 8, 64),
                       (64, 2, 64)):
        w = workloads.decode_batch(seed=1 + 1000 * rank, batch=b, num_qo_heads=hq,
                                   num_kv_heads=hkv)
        nbytes = decode_bytes([int(x) for x in w["kv_lens"]], hq, hkv)
        q = w["q"].to(dev)
        pools = kv_pools(torch, w["k_cache"], w["v_cache"], dev)
        table, lens, sinks = w["page_table"].to(dev), w["kv_lens"].to(dev), w["sinks"].to(dev)
        splits, ws_bytes = sa.decode_plan(b, hq, hkv, w["max_kv_len"])
        ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream()
        run = {"splits": splits}
        for mode in (True, False):
            def step(i, mode=mode, q=q, pools=pools, table=table, lens=lens, sinks=sinks, w=w,
                     ws=ws):
                kc, vc = pools[i % len(pools)]
                sa.decode(q, kc, vc, table, lens, sinks, w["scale"], w["max_kv_len"],
                          workspace=ws, stream=stream, programmatic=mode)
            steps = max(50, args.steps // 20)
            secs = _time_steps(torch, step, steps, args.warmup, stream)
            _, _, bps = aggregate(nbytes * steps, secs, dev)
            key = "programmatic" if mode else "plain"
            run[key] = round(bps / 1e9, 1)
            run[key + "_frac"] = round(bps / 1e9 / peaks["hbm_gbs"], 4)
        res[f"{hq} q / {hkv} kv heads, {b} requests"] = run
        del pools, q
        torch.cuda.empty_cache()
    return dict(workload="decode, kv_len U[1,4096], bf16 paged KV (page 16, shuffled), copies of "
                         "the KV pool cycled one per step", runs=res)


def run_layer(args, rank, dev, peaks):
    """The attention of a decode layer as a model runs it: per step the
    prologue of the step's 64 new tokens (QKV bias, YaRN rotation of q and k,
    k and v written into each request's newest cache slot), then the decode
    over the cache that now holds them, each step on its own pool copy.  With
    programmatic launch the decode ranks its requests and reads its page ids
    while the prologue runs; the same steps with plain launches beside."""
    import torch

    import gqa_attention_learned_gb300 as sa
    from gqa_attention_learned_gb300 import workloads

    w = workloads.decode_batch(seed=1 + 1000 * rank)
    hq, hkv = w["num_qo_heads"], w["num_kv_heads"]
    lens = [int(x) for x in w["kv_lens"]]
    b = len(lens)
    table_h = w["page_table"]
    pools = kv_pools(torch, w["k_cache"], w["v_cache"], dev)
    table, kv_lens, sinks = table_h.to(dev), w["kv_lens"].to(dev), w["sinks"].to(dev)
    # request r's newest token: position kv_len - 1 and its cache slot
    pos = torch.tensor([max(n - 1, 0) for n in lens], dtype=torch.int32, device=dev)
    slots = torch.tensor([int(table_h[r, (n - 1) // 16]) * 16 + (n - 1) % 16 if n > 0 else -1
                          for r, n in enumerate(lens)], dtype=torch.int32, device=dev)
    gen = torch.Generator().manual_seed(11 + 1000 * rank)
    width = (hq + 2 * hkv) * HEAD_DIM
    qkv = torch.randn(b, width, generator=gen).to(torch.bfloat16).to(dev)
    bias = (0.5 * torch.randn(width, generator=gen)).to(torch.bfloat16).to(dev)
    inv, msc = sa.yarn_table()
    q_new = torch.empty(b, hq, HEAD_DIM, dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q_new)
    lse = torch.empty(b, hq, dtype=torch.float32, device=dev)
    _, ws_bytes = sa.decode_plan(b, hq, hkv, w["max_kv_len"])
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    nbytes = prologue_bytes(b, hq, hkv) + decode_bytes(lens, hq, hkv)
    res = {}
    for mode in (True, False):
        def step(i, mode=mode):
            kc, vc = pools[i % len(pools)]
            sa.qkv_prologue(qkv, bias, pos, slots, inv, msc, kc, vc, hq, hkv, q_out=q_new,
                            stream=stream)
            sa.decode(q_new, kc, vc, table, kv_lens, sinks, w["scale"], w["max_kv_len"], out=out,
                      lse=lse, workspace=ws, stream=stream, programmatic=mode)

        steps = max(200, args.steps // 10)
        secs = _time_steps(torch, step, steps, args.warmup, stream)
        _, t, bps = aggregate(nbytes * steps, secs, dev)
        res["programmatic" if mode else "plain"] = dict(
            us_per_step=round(1e6 * t / steps, 2), value=round(bps / 1e9, 2), unit="GB/s",
            frac_of_hbm=round(bps / 1e9 / peaks["hbm_gbs"], 4))
    label = pools_label(pools)
    del pools
    torch.cuda.empty_cache()
    return dict(workload="decode layer: prologue of 64 new tokens (bias, YaRN q/k, paged k/v write) "
                         "then decode of the gpt-oss-20b batch, two launches per step; " + label,
                bytes_per_step=nbytes, launches_per_step=2, runs=res)


SECTIONS = {"long": "long_decode", "graph": "graph_decode", "verify": "verify",
            "prologue": "prologue", "prefill": "prefill", "mixed": "mixed", "gqa": "gqa",
            "layer": "layer"}


def only_section(args):
    """One extra section alone (no headline decode, no CPU baseline): its
    figures as one JSON line, for profiling a single kernel's workload."""
    import torch

    world, rank, local = dist_info()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_init("nccl" if world > 1 else "gloo")
    import gqa_attention_learned_gb300 as sa
    sa.load()
    sa.set_programmatic_launch(not args.plain_launch)
    peaks, _ = load_peaks()
    fn = {"long": lambda: run_long_decode(args, rank, dev),
          "graph": lambda: run_graph_decode(args, rank, dev, peaks),
          "verify": lambda: run_verify(args, rank, dev, peaks),
          "prologue": lambda: run_prologue(args, rank, dev, peaks),
          "prefill": lambda: run_prefill(args, rank, dev, peaks),
          "mixed": lambda: run_mixed(args, rank, dev, peaks),
          "gqa": lambda: run_gqa(args, rank, dev, peaks),
          "layer": lambda: run_layer(args, rank, dev, peaks)}[args.only]
    out = fn()
    if rank == 0:
        print(json.dumps({"section": SECTIONS[args.only], **out}), flush=True)


def section_summary(extra, peaks):
    """Flat numeric figures of the extra sections (GB/s, TFLOP/s and
    fractions of the measured peaks) for the printed line; the full sections
    go to --details."""
    hbm, tf = peaks["hbm_gbs"], peaks["bf16_tflops"]
    out = {}
    if "long_decode" in extra:
        r = extra["long_decode"]["runs"]["auto"]
        out.update(long_decode_gbps=round(r["value"], 1), long_decode_frac=round(r["value"] / hbm, 4),
                   long_decode_splits=r["splits"])
        r8 = extra["long_decode"]["runs"]["8 splits"]
        out.update(long_decode_8split_frac=round(r8["value"] / hbm, 4))
    if "graph_decode" in extra:
        g = extra["graph_decode"]
        out.update(graph_decode_frac=g["frac_of_hbm"],
                   graph_multi_step_decode_frac=g["multi_step_graph"]["frac_of_hbm"])
    if "verify" in extra:
        for key, label in (("verify_mtp2", "mtp 2 tokens"), ("verify_4tok", "4 tokens causal"),
                           ("verify_tree8", "8-node tree")):
            r = extra["verify"]["runs"].get(label)
            if r:
                out[key + "_gbps"] = r["value"]
                out[key + "_frac"] = r["frac_of_hbm"]
    if "prefill" in extra:
        p = extra["prefill"]["roofline"]
        out.update(prefill_tflops=p["achieved"], prefill_frac=p["frac"],
                   prefill_frac_sustained=p["frac_of_sustained"], prefill_traffic=p["traffic"])
    if "mixed" in extra:
        m = extra["mixed"]
        out.update(mixed_decode_gbps=m["decode"]["value"],
                   mixed_decode_frac=round(m["decode"]["value"] / hbm, 4),
                   mixed_extend_tflops=m["extend"]["value"],
                   mixed_extend_frac=round(m["extend"]["value"] / tf, 4),
                   mixed_combined_frac=m["combined_roofline_frac"])
    if "prologue" in extra:
        r = extra["prologue"]["runs"].get("prefill 4 sequences")
        if r:
            out.update(prologue_prefill_frac=r["frac_of_hbm"])
    if "layer" in extra:
        r = extra["layer"]["runs"]
        out.update(layer_frac=r["programmatic"]["frac_of_hbm"],
                   layer_us_per_step=r["programmatic"]["us_per_step"],
                   layer_plain_frac=r["plain"]["frac_of_hbm"])
    return out


def gpu_arm(args):
    import torch

    world, rank, local = dist_info()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_init("nccl" if world > 1 else "gloo")
    import gqa_attention_learned_gb300 as sa
    sa.load()
    sa.set_programmatic_launch(not args.plain_launch)
    peaks, peak_src = load_peaks()

    sections = set(args.sections.split(","))
    d = run_decode_arm(args, rank, dev)
    ms = 1e3 * d["secs"] / args.steps
    kernel_gbps = d["nbytes"] / (d["secs"] / args.steps) / 1e9     # per launch, this rank
    extra = {}
    if not args.quick:
        if "long" in sections:
            extra["long_decode"] = run_long_decode(args, rank, dev)
        if "graph" in sections:
            extra["graph_decode"] = run_graph_decode(args, rank, dev, peaks)
        if "verify" in sections:
            extra["verify"] = run_verify(args, rank, dev, peaks)
        if "prologue" in sections:
            extra["prologue"] = run_prologue(args, rank, dev, peaks)
        if "prefill" in sections:
            extra["prefill"] = run_prefill(args, rank, dev, peaks)
        if "mixed" in sections:
            extra["mixed"] = run_mixed(args, rank, dev, peaks)
        if "gqa" in sections:
            extra["gqa"] = run_gqa(args, rank, dev, peaks)
        if "layer" in sections:
            extra["layer"] = run_layer(args, rank, dev, peaks)
    roofline = {"bound": "hbm", "achieved": round(kernel_gbps, 2), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(kernel_gbps / peaks["hbm_gbs"], 4),
                "traffic": kernel_traffic("decode"), "peak_source": peak_src,
                "kernel": "decode_kernel<1, false>",
                "bytes_per_launch": d["nbytes"],
                "plain_launch_gbps": round(d["plain_gbps"], 1),
                "plain_launch_frac": round(d["plain_gbps"] / peaks["hbm_gbs"], 4),
                "plain_launch_graph_frac": round(d["plain_graph_gbps"] / peaks["hbm_gbs"], 4)}
    roofline.update(section_summary(extra, peaks))
    line = {
        "metric": METRIC, "value": round(d["gbps"], 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q/k/v, shuffled page pool)",
        "config": {"workload": DECODE_WORKLOAD, "batch": 64, "num_qo_heads": 64,
                   "num_kv_heads": 8, "head_dim": 64, "page_size": 16,
                   "kv_tokens": sum(int(x) for x in d["w"]["kv_lens"]),
                   "num_splits": d["splits"],
                   "launch": "plain" if args.plain_launch else "programmatic dependent launch",
                   "l2": "inputs larger than L2: " + d["pool_label"]},
        "roofline": roofline,
        "e2e": {k: v for k, v in d["e2e"].items() if k != "note"},
        "gpu_launches": args.steps * d["launches_per_step"],
        "clocks": d["clocks"],
    }
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds)
    if rank == 0 and args.details:
        with open(args.details, "w") as f:
            json.dump(dict(line=line, e2e=d["e2e"], e2e_kv_h2d=d["e2e_kv_h2d"],
                           plain_launch=dict(steps=d["plain_steps"],
                                             value=round(d["plain_gbps"], 2)),
                           extra=extra), f, indent=1)
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------- CPU oracle

def oracle_worker(spec):
    """Runs in a fresh single-threaded process: the float64 oracle, as it
    stands, decoding (request, KV head) groups of the gpt-oss-20b batch in
    turn.  spec: warmup/steps/units_per_step, or budget_s (run until spent)."""
    import numpy as np

    import oracle
    from gqa_attention_learned_gb300 import workloads

    class Pool:  # float64 view of a bf16 pool, converted row by row on gather
        def __init__(self, t):
            self.t, self.shape = t, tuple(t.shape)

        def __getitem__(self, idx):
            import torch
            idx = tuple(torch.as_tensor(i) if isinstance(i, np.ndarray) else i for i in idx)
            return self.t[idx].float().numpy().astype(np.float64)

    w = workloads.decode_batch(seed=1)
    hq, hkv = w["num_qo_heads"], w["num_kv_heads"]
    g = hq // hkv
    q = w["q"].float().numpy().astype(np.float64)
    table, lens = w["page_table"].numpy(), w["kv_lens"].numpy()
    sinks = w["sinks"].numpy().astype(np.float64)
    pools = [(Pool(w["k_cache"][:, h:h + 1]), Pool(w["v_cache"][:, h:h + 1])) for h in range(hkv)]
    units = [(b, h) for b in range(len(lens)) for h in range(hkv)]
    cursor = [0]

    def step(n):
        nbytes = 0
        for _ in range(n):
            b, h = units[cursor[0] % len(units)]
            cursor[0] += 1
            kc, vc = pools[h]
            oracle.decode(q[b:b + 1, g * h:g * (h + 1)], kc, vc, table[b:b + 1], lens[b:b + 1],
                          sinks[g * h:g * (h + 1)], w["scale"])
            nbytes += decode_bytes(lens[b:b + 1], g, 1)
        return nbytes

    per = int(spec.get("units_per_step", 1))
    for _ in range(int(spec.get("warmup", 0))):
        step(per)
    t0 = time.perf_counter()
    done, steps = 0, 0
    while True:
        done += step(per)
        steps += 1
        el = time.perf_counter() - t0
        if spec.get("steps") and steps >= spec["steps"]:
            break
        if not spec.get("steps") and el >= spec.get("budget_s", 10.0):
            break
    return dict(bytes=done, seconds=el, steps=steps, units=steps * per)


def _run_oracle(spec):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-worker",
                        json.dumps(spec)], env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(budget_s=15.0):
    """The float64 oracle on one host core (BLAS pinned to one thread in a
    fresh process) over (request, KV head) groups of the same batch."""
    res = _run_oracle({"budget_s": budget_s, "units_per_step": 8})
    return {"value": round(res["bytes"] / res["seconds"] / 1e9, 5), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{res['units']} (request, KV head) groups of the gpt-oss-20b decode batch, "
                      f"cycled in order, {res['seconds']:.1f} s, float64 NumPy, 1 BLAS thread",
            "host_cores": os.cpu_count()}


def reference_arm(args):
    """The oracle as the reference arm: W untimed steps, then exactly K timed
    steps, each step a bounded sample of the decode batch ((request, KV head)
    groups), sized from a probe so the whole run ends within a few minutes."""
    world, rank, _ = dist_info()
    if rank != 0:
        return
    probe = _run_oracle({"steps": 8, "units_per_step": 1})
    t_unit = probe["seconds"] / probe["steps"]
    budget = 100.0
    per = max(1, int(budget / (args.steps + args.warmup) / t_unit))
    res = _run_oracle({"warmup": args.warmup, "steps": args.steps, "units_per_step": per})
    value = res["bytes"] / res["seconds"] / 1e9
    sample = f"{per} (request, KV head) group(s) of the gpt-oss-20b decode batch per step, cycled"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s",
            "n_gpus": world, "steps": res["steps"], "warmup": args.warmup,
            "ms_per_step": round(1e3 * res["seconds"] / res["steps"], 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16 q/k/v, shuffled page pool)",
            "config": {"workload": DECODE_WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--splits", type=int, default=0, help="decode split count (0 = planned)")
    ap.add_argument("--quick", action="store_true", help="headline decode only")
    ap.add_argument("--sections", default="graph,long,verify,prologue,prefill,mixed,layer",
                    help="extra sections after the headline decode")
    ap.add_argument("--plain-launch", action="store_true",
                    help="launch decode kernels without programmatic dependent launch")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--only", choices=sorted(SECTIONS), default=None,
                    help="run one extra section alone and print its figures (profiling)")
    ap.add_argument("--details", default=None,
                    help="write the full sections (e2e variants, per-run figures) to this JSON file")
    ap.add_argument("--oracle-worker", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_worker is not None:
        print(json.dumps(oracle_worker(json.loads(args.oracle_worker))))
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        reference_arm(args)
    elif args.only:
        only_section(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
