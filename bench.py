#!/usr/bin/env python3
"""Benchmark of the GB300 sparse paged attention hot path.

Headline: one prefill call of 8192 queries from position 0 (64 heads, head_dim 512, window 128,
top-k 512 of the causally valid compressed entries, ratio 4, page size 64; the "sparse prefill r4
S8192" shape of the FreeToken PR 633 "Kernel time" table), in microseconds per call, L2 flushed
before every call.  The same JSON line carries the other four configurations (the tiny case, decode
B=1, decode B=8 at ratios 128/4/0, the e4m3 prefill chunk) with their achieved GB/s or TFLOP/s
against the measured GB300 peaks.  The remaining shapes of the pages' tables (the other decode and
prefill shapes, the paged KV write, the compressor's gated pool, the indexer logits and top-k) are
printed on one more JSON line, to stderr, before it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload NAME] [--headline-only] [--sub NAME,...] [--no-cpu-baseline]

For N > 1 (torchrun, one rank per GPU) the job is a batch of N independent copies of the workload's
sequences (N prefill sequences, or 8N decode sequences for the B=8 shapes), partitioned by
sequence: rank r holds and computes shard r only, with no data-path collective (a barrier and a
max over ranks time the job).  Scaling is weak.  ``--impl reference`` times the float64 CPU oracle
on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse attn µs/call; decode HBM GB/s and prefill TFLOP/s as % of GB300 peak"
HEADLINE = "prefill_s8192_r4"
# the five configurations: c1 tiny, c2 decode B=1, c3 decode B=8 (three ratios), c4 prefill
# S=8192, c5 the e4m3 prefill chunk
CONFIGS = {"c1": ["tiny_r4"], "c2": ["decode_b1_r4"],
           "c3": ["decode_b8_r128", "decode_b8_r4", "decode_b8_r0"],
           "c4": ["prefill_s8192_r4"], "c5": ["prefill_fp8_s4096_r4"]}
OTHER_SHAPES = ["decode_b1_r128", "decode_b1_r0", "prefill_s2048_r4", "prefill_s4096at28672_r4",
                "prefill_s8192_r128", "prefill_s8192_r0"]
KV_WRITES = {"kv_write_fp8_t65536": True, "kv_write_t65536": False}   # name -> e4m3 pool
GATED_POOLS = {"gated_pool_b%d_r%d_d%d" % s: s for s in
               [(b, r, d) for b in (1, 8) for r in (8, 128) for d in (128, 512)]}
# the indexer shapes of FreeToken PR 634 ("All shapes"): name -> (mode, n queries, first position,
# ratio, sequences, candidates); decode shapes put each sequence's one query at ctx - 1
INDEXERS = {
    "indexer_full_prefill_n2048_start0_r2": ("full", 2048, 0, 2, 1, None),
    "indexer_full_prefill_n8192_start0_r2": ("full", 8192, 0, 2, 1, None),
    "indexer_full_prefill_n2048_start129024_r2": ("full", 2048, 129024, 2, 1, None),
    "indexer_full_prefill_n128_start8064_r1": ("full", 128, 8064, 1, 1, None),
    "indexer_full_prefill_n128_start130944_r1": ("full", 128, 130944, 1, 1, None),
    "indexer_cand_prefill_n128_start8064_nc16384": ("cand", 128, 8064, 1, 1, 16384),
    "indexer_cand_prefill_n128_start130944_nc16384": ("cand", 128, 130944, 1, 1, 16384),
    "indexer_full_decode_b1_ctx32768_r2": ("full", 1, 32767, 2, 1, None),
    "indexer_full_decode_b4_ctx32768_r2": ("full", 1, 32767, 2, 4, None),
    "indexer_full_decode_b1_ctx131072_r2": ("full", 1, 131071, 2, 1, None),
    "indexer_full_decode_b1_ctx131072_r1": ("full", 1, 131071, 1, 1, None),
    "indexer_cand_decode_b1_ctx131072_nc16384": ("cand", 1, 131071, 1, 1, 16384),
    "indexer_cand_decode_b4_ctx131072_nc16384": ("cand", 1, 131071, 1, 4, 16384),
}
TOPK_SHAPES = {"topk_t1_n65536_k512": (1, 65536, 512), "topk_t128_n8192_k512": (128, 8192, 512),
               "topk_t2048_n32768_k512": (2048, 32768, 512)}
FLUSH_BYTES = 512 << 20   # > 129 MB of L2
E2E_CHUNK = 1024          # tokens a chunk of the host-buffer prefill (e2e)
# a device-side wait enqueued before each timed call, so that the GPU is still busy with it while
# the host enqueues the start event, the call and the end event: the events then bracket device
# time only (about 100 us at GB300 clocks)
SPIN_CYCLES = 200_000
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------------------------
# distributed plumbing (timing only: barriers and a max over ranks, never on the data path)
# ----------------------------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """Largest value over all ranks (the slowest rank sets the time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------------------------
# accounting
# ----------------------------------------------------------------------------------------------
def algorithmic_work(w):
    """Bytes the method must move and flops it must do for one call (the dense attention it
    avoids is not counted): every resolved K and V row once, q in, out, the index lists."""
    from workloads import pool_rows_referenced
    cols = pool_rows_referenced(w)
    elt = 1 if w.fp8 else 2
    row_bytes = 2 * w.head_dim * elt + (8 if w.fp8 else 0)   # K row + V row (+ two fp32 scales)
    T, H, D = w.q.shape
    nbytes = cols * row_bytes + 2 * T * H * D * 2 + T * (w.topk + 1) * 4
    flops = 4.0 * H * D * cols
    return {"columns": cols, "bytes": nbytes, "flops": flops}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, \
            "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def roofline_of(w, us, peaks):
    """Achieved rate of one call against its bound: decode HBM bytes against the copy peak,
    prefill flops against the dense tensor peak of the kernel's operand type (bf16 measured
    burst; e4m3 twice that, the nominal fp8/bf16 ratio), both for a kernel timed alone."""
    work = algorithmic_work(w)
    if w.decode or w.name == "tiny_r4":
        gbs = work["bytes"] / (us * 1e-6) / 1e9
        return {"bound": "hbm", "achieved": round(gbs, 1), "unit": "GB/s",
                "peak": peaks["hbm_gbs"], "frac": round(gbs / peaks["hbm_gbs"], 4)}, work
    tf = work["flops"] / (us * 1e-6) / 1e12
    peak = peaks["bf16_tflops"] * (2.0 if w.fp8 else 1.0)
    return {"bound": "tensor", "achieved": round(tf, 1), "unit": "TFLOP/s", "peak": peak,
            "frac": round(tf / peak, 4)}, work


def _code_only(text: str) -> str:
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    """Hash of what compiles into the attention kernel, with comments and blank space removed: its
    translation unit (spa_attention.cu), the library headers it includes (spa_launch.h,
    spa_device.cuh) and, of the public header, the status codes the kernel raises.  A counter
    capture stays valid across comment edits and changes to other kernels or to host code, and no
    longer once any of this code changes."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_paged_attention_gb300", "csrc")
    for name in ("spa_attention.cu", "spa_device.cuh", "spa_launch.h"):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    with open(os.path.join(ROOT, "include", "sparse_attn_paged.h"), encoding="utf-8") as f:
        pub = _code_only(f.read())
    m = re.search(r"typedef enum spa_status \{.*?\} spa_status_t;", pub)
    h.update(b"spa_status" + (m.group(0).encode() if m else b""))
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------------------------
# clocks sampled while the GPU is busy
# ----------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except OSError:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        busy = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------------
class Runner:
    """One workload resident on the GPU plus the C-ABI call that computes it, its argument structs
    built once (so a timed call is the library call and nothing else)."""

    def __init__(self, name, device, seed=0):
        import torch
        import sparse_paged_attention_gb300 as spa
        from workloads import make
        self.spa = spa
        self.w = w = make(name, seed=seed)
        g = lambda t: None if t is None else t.to(device)
        self.q, self.pos = g(w.q), g(w.positions)
        self.tk = g(w.topk_idx) if w.topk > 0 else None
        self.sot = g(w.seq_of_token)
        self.win = spa.PagedPool(g(w.win.kv), g(w.win.block_table), g(w.win.k_scale),
                                 g(w.win.v_scale))
        self.cmp = None if w.cmp is None else spa.PagedPool(
            g(w.cmp.kv), g(w.cmp.block_table), g(w.cmp.k_scale), g(w.cmp.v_scale))
        self.out = torch.empty_like(self.q)
        self.call = self.bind(self.q, self.tk, self.pos, self.out)
        # a decode plan with a workspace adds the merge kernel; every other plan is one launch
        self.launches_per_call = 2 if getattr(self.call, "workspace", None) is not None and \
            self.call.workspace.numel() > 16 else 1

    def bind(self, q, tk, pos, out):
        w = self.w
        kw = dict(window=w.window, ratio=w.ratio, scale=w.scale, seq_of_token=self.sot, out=out,
                  fp8=w.fp8)
        if w.decode:
            return self.spa.bind_decode(q, self.win, self.cmp, tk, pos, **kw)
        return self.spa.bind_prefill(q, self.win, self.cmp, tk, pos, **kw)


def time_calls(fn, steps, warmup, flush, dist=None):
    """Per-call device time (ms) of `steps` calls: L2 flushed before each, then a device-side
    wait that keeps the GPU busy while the host enqueues the start event, the call and the end
    event (outside the events), so each event pair brackets the call's device time."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    barrier(dist)
    torch.cuda.synchronize()
    for a, b in ev:
        flush.zero_()
        torch.cuda._sleep(SPIN_CYCLES)
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    return [a.elapsed_time(b) for a, b in ev]


def stats_us(times_ms):
    us = [1e3 * t for t in times_ms]
    return {"us": round(statistics.mean(us), 3), "us_median": round(statistics.median(us), 3),
            "us_min": round(min(us), 3), "us_max": round(max(us), 3), "calls": len(us)}


def time_graph(fn, reps=20, rounds=10):
    """Per-call device time (ms) of `reps` calls captured in one CUDA graph and replayed with L2
    warm: the median over `rounds` replays.  This is how the pages' tables were measured."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    out = []
    for _ in range(rounds):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b) / reps)
    del g
    return statistics.median(out)


def time_e2e(r, steps, warmup, flush, dist=None):
    """The same call from host buffers, every copy inside the timed region (the pools are the
    resident KV cache).  Prefill goes through the library's host-buffer entry point
    (sparse_attn_paged_prefill_host): q, the top-k lists and the positions from pinned host
    memory and out back to it, a chunk of E2E_CHUNK tokens at a time, the copies in, kernels and
    copies out of consecutive chunks overlapping.  Decode, a few hundred KB, copies with torch
    around the device call."""
    import torch
    q_h = r.w.q.pin_memory()
    pos_h = r.w.positions.pin_memory()
    tk_h = r.w.topk_idx.pin_memory() if r.tk is not None else None
    sot_h = r.w.seq_of_token.pin_memory() if r.w.seq_of_token is not None else None
    h2d = q_h.numel() * 2 + pos_h.numel() * 4 + (tk_h.numel() * 4 if tk_h is not None else 0) + \
        (sot_h.numel() * 4 if sot_h is not None else 0)
    d2h = q_h.numel() * 2
    if not r.w.decode:
        w = r.w
        step = r.spa.bind_prefill_host(q_h, r.win, r.cmp, tk_h, pos_h, window=w.window,
                                       ratio=w.ratio, scale=w.scale, seq_of_token=sot_h,
                                       chunk_tokens=E2E_CHUNK, fp8=w.fp8)
        return time_calls(step, steps, warmup, flush, dist), h2d, d2h
    out_h = torch.empty(r.out.shape, dtype=r.out.dtype, pin_memory=True)
    q_d, pos_d = torch.empty_like(r.q), torch.empty_like(r.pos)
    tk_d = torch.empty_like(r.tk) if r.tk is not None else None
    out_d = torch.empty_like(r.out)
    call = r.bind(q_d, tk_d, pos_d, out_d)

    def step():
        q_d.copy_(q_h, non_blocking=True)
        pos_d.copy_(pos_h, non_blocking=True)
        if tk_d is not None:
            tk_d.copy_(tk_h, non_blocking=True)
        call()
        out_h.copy_(out_d, non_blocking=True)

    return time_calls(step, steps, warmup, flush, dist), h2d, d2h


def measure_workload(name, device, steps, warmup, flush, peaks, graph=True):
    import torch
    r = Runner(name, device)
    r.call()
    torch.cuda.synchronize()
    st = r.spa.sparse_attn_paged_check_errors()
    if st:
        raise RuntimeError(f"{name}: device error word {st}")
    s = stats_us(time_calls(r.call, steps, warmup, flush))
    roof, _ = roofline_of(r.w, s["us"], peaks)
    d = dict(s, **roof)
    if graph:
        try:
            d["us_warm_graph"] = round(1e3 * time_graph(r.call, reps=20 if r.w.decode else 3), 3)
        except Exception as e:  # noqa: BLE001 - reported, never fatal to the cold-L2 number
            d["us_warm_graph"] = None
            d["graph_error"] = str(e)[:120]
    del r
    torch.cuda.empty_cache()
    return d


def measure_kv_write(name, device, steps, flush, peaks):
    """The paged KV write of 65536 new tokens (head_dim 512, pages of 64) into a pool twice that
    size: HBM-bound, bytes = 4·D read per token plus 2·D (e4m3 codes, and two fp32 scales) or
    4·D (bf16) written."""
    import numpy as np
    import torch
    import sparse_paged_attention_gb300 as spa
    from workloads import kv_write_inputs
    fp8 = KV_WRITES[name]
    T, D, ps = 65536, 512, 64
    inp = kv_write_inputs([np.arange(T)], D, ps, seed=3, specials=False)
    nb = inp.num_blocks
    kv = torch.zeros((nb, ps, 2, D), dtype=torch.uint8 if fp8 else torch.bfloat16, device=device)
    ks = torch.zeros(nb * ps, dtype=torch.float32, device=device)
    vs = torch.zeros_like(ks)
    pool = spa.PagedPool(kv, inp.block_table.to(device), ks, vs)
    k, v = inp.k.to(device), inp.v.to(device)
    pos, sot = inp.positions.to(device), inp.seq_of_token.to(device)
    fn = spa.sparse_attn_paged_kv_write_fp8 if fp8 else spa.sparse_attn_paged_kv_write
    call = lambda: fn(k, v, pos, pool, seq_of_token=sot)
    call()
    if spa.sparse_attn_paged_check_errors():
        raise RuntimeError(f"{name}: device error word")
    s = stats_us(time_calls(call, steps, 3, flush))
    nbytes = T * (4 * D + (2 * D + 8 if fp8 else 4 * D))
    gbs = nbytes / (s["us"] * 1e-6) / 1e9
    return dict(s, bound="hbm", achieved=round(gbs, 1), unit="GB/s", peak=peaks["hbm_gbs"],
                frac=round(gbs / peaks["hbm_gbs"], 4))


def measure_gated_pool(name, device, steps, flush, peaks):
    """The compressor's gated pool at one of the pages' shapes (B entries of R rows, D channels,
    fp32 output): HBM- and latency-bound, bytes = 8·B·R·D read (kv and gates) + 4·B·D written."""
    import torch
    import sparse_paged_attention_gb300 as spa
    from workloads import gated_pool_inputs
    B, R, D = GATED_POOLS[name]
    _, kv, _, gate = gated_pool_inputs(B, R, D, seed=4)
    kv, gate = kv.to(device), gate.to(device)
    out = torch.empty((B, D), dtype=torch.float32, device=device)
    call = lambda: spa.sparse_attn_gated_pool(kv, gate, out)
    call()
    s = stats_us(time_calls(call, steps, 3, flush))
    warm = 1e3 * time_graph(call)
    nbytes = 8 * B * R * D + 4 * B * D
    gbs = nbytes / (s["us"] * 1e-6) / 1e9
    return dict(s, us_warm_graph=round(warm, 3), bound="hbm", achieved=round(gbs, 1), unit="GB/s",
                peak=peaks["hbm_gbs"], frac=round(gbs / peaks["hbm_gbs"], 4))


def measure_indexer(name, device, flush, peaks):
    """Indexer logits at one of the pages' shapes.  Work: 2·32·128 flop per (query, scored entry)
    on the tensor cores; bytes: the packed key rows scored (68 B each, once per query group that
    shares them), q, the weights and the logits written."""
    import numpy as np
    import torch
    import sparse_paged_attention_gb300 as spa
    from workloads import indexer_inputs
    mode, n, start, ratio, B, nc = INDEXERS[name]
    seqs = [np.arange(start, start + n)] * B
    x = indexer_inputs(seqs, ratio, page_size=64, seed=5, cand_count=nc)
    g = lambda t: None if t is None else t.to(device)
    q, w, kp, bt, pos = g(x.q), g(x.weights), g(x.key_pool), g(x.block_table), g(x.positions)
    cand, sot = g(x.cand), (g(x.seq_of_token) if B > 1 else None)
    out = torch.empty((x.q.shape[0], x.num_cols), dtype=torch.float32, device=device)
    call = lambda: spa.sparse_attn_indexer_logits(q, w, kp, bt, pos, ratio=ratio,
                                                  num_cols=x.num_cols, cand=cand,
                                                  seq_of_token=sot, num_seqs=B, out=out)
    call()
    if spa.sparse_attn_paged_check_errors():
        raise RuntimeError(f"{name}: device error word")
    big = n * x.num_cols >= (1 << 24)
    s = stats_us(time_calls(call, 5 if big else 30, 3, flush))
    warm = 1e3 * time_graph(call, reps=3 if big else 20, rounds=5)
    p = x.positions.numpy().astype(np.int64)
    if x.cand is None:
        scored = np.minimum((p + 1) // ratio, x.num_cols)
        rows = B * int(scored.max()) if n > 1 else int(scored.sum())
    else:
        c = x.cand.numpy().astype(np.int64)
        scored = ((c >= 0) & (ratio * c + ratio - 1 <= p[:, None])).sum(axis=1)
        rows = int(scored.sum())
    flops = 2.0 * 32 * 128 * float(scored.sum())
    nbytes = 68 * rows + x.q.numel() * 2 + x.weights.numel() * 4 + out.numel() * 4
    tf = flops / (s["us"] * 1e-6) / 1e12
    gbs = nbytes / (s["us"] * 1e-6) / 1e9
    return dict(s, us_warm_graph=round(warm, 3), tflops=round(tf, 2),
                frac_bf16_tensor=round(tf / peaks["bf16_tflops"], 4), gbs=round(gbs, 1),
                frac_hbm=round(gbs / peaks["hbm_gbs"], 4))


def measure_topk(name, device, flush, peaks):
    """Top-k selection over indexer logits (T rows of N fp32 logits, k entries kept): bytes = the
    logits read once (the kernel's passes re-read them from L2) plus the int32 lists written."""
    import numpy as np
    import torch
    import sparse_paged_attention_gb300 as spa
    T, N, k = TOPK_SHAPES[name]
    rng = np.random.default_rng(6)
    lg = torch.from_numpy(rng.standard_normal((T, N)).astype(np.float32)).to(device)
    out = torch.empty((T, k), dtype=torch.int32, device=device)
    call = lambda: spa.sparse_attn_indexer_topk(lg, k, out=out)
    call()
    s = stats_us(time_calls(call, 30, 3, flush))
    nbytes = T * N * 4 + T * k * 4
    gbs = nbytes / (s["us"] * 1e-6) / 1e9
    return dict(s, gbs=round(gbs, 1), frac_hbm=round(gbs / peaks["hbm_gbs"], 4))


def cpu_baseline(name, seconds):
    """The float64 oracle as it stands, on the host cores, in a fresh process."""
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.oracle_timing(%r, %f)))" % (ROOT, name, seconds))
    try:
        p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                           timeout=600)
        return json.loads(p.stdout.strip().splitlines()[-1])
    except Exception as e:  # noqa: BLE001 - reported, never fatal to the GPU numbers
        return {"error": str(e)[:200]}


def sample_args(a, toks):
    """The oracle's arguments restricted to the queries `toks` (their q, positions, sequence ids
    and top-k lists; the pools and block tables whole), so that its cost is that of those
    queries alone."""
    b = dict(a)
    for k in ("q_bits", "positions", "seq_ids", "topk_idx"):
        b[k] = a[k][toks]
    return b


def oracle_timing(name, seconds, max_queries=None):
    """Time the oracle on about `seconds` of work for workload `name`: queries are drawn at random
    in groups of up to 8 and the time per query is scaled to a full call of all the workload's
    queries (a decode call of a few queries runs whole)."""
    import numpy as np
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from oracle_io import oracle_args
    import oracle
    from workloads import make
    w = make(name)
    a = oracle_args(w)
    T = w.num_tokens
    rng = np.random.default_rng(0)
    t0 = time.perf_counter()
    queries = 0
    while time.perf_counter() - t0 < seconds and (max_queries is None or queries < max_queries):
        toks = np.sort(rng.choice(T, size=min(T, 8), replace=False))
        oracle.sparse_paged_attention(**sample_args(a, toks))
        queries += len(toks)
    el = time.perf_counter() - t0
    per_query = el / queries
    return {"us_per_call": per_query * T * 1e6, "queries": int(queries), "seconds": round(el, 2),
            "cores": os.cpu_count(), "per_call_queries": T}


DESCRIBE = {
    "prefill_s8192_r4": "prefill S=8192 from position 0, 64 heads, head_dim 512, window 128, "
                        "top-k 512 of the causally valid compressed entries (ratio 4), page size "
                        "64, bf16 pools",
    "decode_b1_r4": "decode B=1 at position 32767, 64 heads, head_dim 512, window 128, top-k 512 "
                    "of 8192 (ratio 4), page size 64, bf16 pools",
    "prefill_fp8_s4096_r4": "e4m3 prefill chunk of 4096 queries at 28672..32767, 64 heads, "
                            "head_dim 512, window 128, top-k 512 of 8192 (ratio 4), page size 64, "
                            "e4m3 pools with per-row fp32 scales",
}


def describe(name):
    return DESCRIBE.get(name, name)


def run_gpu(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    peaks, peak_src = load_peaks()
    import sparse_paged_attention_gb300 as spa
    spa.load_library()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    headline = args.workload
    only = None if args.sub is None else set(args.sub.split(","))
    keep = lambda name: only is None or name in only
    with ClockSampler(local) as clk:
        # shard `rank` of a batch of `world` independent copies of the workload's sequences
        r = Runner(headline, device, seed=rank)
        r.call()
        if spa.sparse_attn_paged_check_errors():
            raise RuntimeError("device error word set by the first call")
        times = time_calls(r.call, args.steps, args.warmup, flush, dist)
        st = spa.sparse_attn_paged_check_errors()
        if st:
            raise RuntimeError(f"device error word {st}")
        head = stats_us(times)
        us_job = max_over_ranks(dist, head["us"], device)
        med_job = max_over_ranks(dist, head["us_median"], device)
        max_job = max_over_ranks(dist, head["us_max"], device)
        roof, work = roofline_of(r.w, us_job, peaks)
        work_job = {k: sum_over_ranks(dist, float(v), device) for k, v in work.items()}
        warm_us = 1e3 * time_graph(r.call, reps=20 if r.w.decode else 3)
        e2e_times, h2d, d2h = time_e2e(r, args.steps, args.warmup, flush, dist)
        e2e_us = max_over_ranks(dist, 1e3 * statistics.mean(e2e_times), device)
        launches = r.launches_per_call * args.steps
        w_desc = r.w
        del r
        torch.cuda.empty_cache()
        configs, detail = {}, {}
        if not args.headline_only:
            for cid, names in CONFIGS.items():
                for name in names:
                    if name == headline or not keep(name):
                        continue
                    try:
                        n = 50 if name.startswith("decode") or name == "tiny_r4" else 10
                        configs[name] = dict(config=cid, **measure_workload(
                            name, device, n, 3, flush, peaks))
                    except Exception as e:  # noqa: BLE001 - reported, not fatal
                        configs[name] = {"config": cid, "error": str(e)[:200]}
            for name in filter(keep, OTHER_SHAPES):
                try:
                    n = 50 if name.startswith("decode") else 10
                    detail[name] = measure_workload(name, device, n, 3, flush, peaks)
                except Exception as e:  # noqa: BLE001 - reported, not fatal
                    detail[name] = {"error": str(e)[:200]}
            for name in filter(keep, KV_WRITES):
                try:
                    detail[name] = measure_kv_write(name, device, 50, flush, peaks)
                except Exception as e:  # noqa: BLE001 - reported, not fatal
                    detail[name] = {"error": str(e)[:200]}
            for name in filter(keep, GATED_POOLS):
                try:
                    detail[name] = measure_gated_pool(name, device, 50, flush, peaks)
                except Exception as e:  # noqa: BLE001 - reported, not fatal
                    detail[name] = {"error": str(e)[:200]}
            for name in filter(keep, INDEXERS):
                try:
                    detail[name] = measure_indexer(name, device, flush, peaks)
                except Exception as e:  # noqa: BLE001 - reported, not fatal
                    detail[name] = {"error": str(e)[:200]}
            for name in filter(keep, TOPK_SHAPES):
                try:
                    detail[name] = measure_topk(name, device, flush, peaks)
                except Exception as e:  # noqa: BLE001 - reported, not fatal
                    detail[name] = {"error": str(e)[:200]}
        # keep the GPU busy long enough for the clock sampler to see it under load
        r = Runner(headline, device, seed=rank)
        t_end = time.time() + 1.0
        while time.time() < t_end:
            for _ in range(20):
                r.call()
            torch.cuda.synchronize()
        del r
    clocks = clk.summary()

    if rank != 0:
        return
    roof.update(kernel="attn_kernel", traffic=ncu_traffic("attn_kernel", headline),
                peak_source=f"{peak_src} ({'hbm_gbs' if roof['bound'] == 'hbm' else 'bf16_tflops burst'})",
                note="algorithmic work of one call / its device time (one launch of the "
                     "attention kernel per call)")
    if world > 1:
        roof["note"] += "; all ranks' work over the slowest rank's time"
        if roof["bound"] == "tensor":
            roof["achieved"] = round(work_job["flops"] / (us_job * 1e-6) / 1e12, 1)
        else:
            roof["achieved"] = round(work_job["bytes"] / (us_job * 1e-6) / 1e9, 1)
        roof["frac"] = round(roof["achieved"] / (roof["peak"] * world), 4)
    seqs = w_desc.num_seqs
    line = {
        "metric": METRIC,
        "value": round(us_job, 3),
        "unit": "us/call",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(us_job / 1e3, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) rows, random block tables and top-k; no dataset)",
        "config": {"workload": describe(headline),
                   "l2": f"flushed before every call ({FLUSH_BYTES >> 20} MiB write)",
                   "parallelism": (f"batch of {world} independent copies of the workload "
                                   f"({world * seqs} sequences), one shard per rank by sequence, "
                                   f"no collective" if world > 1 else "one GPU")},
        "timing": {"us_median": round(med_job, 3), "us_max": round(max_job, 3),
                   "us_min": head["us_min"], "calls": args.steps,
                   "how": "CUDA events on the launching stream around each call; L2 flush and a "
                          "device-side wait enqueued before the start event"},
        "roofline": roof,
        "e2e": {"value": round(e2e_us, 3), "unit": "us/call", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "warm_l2_graph_us": round(warm_us, 3),
        "clocks": clocks,
        "configs": {k: {kk: v[kk] for kk in ("config", "us", "us_median", "us_max",
                                             "us_warm_graph", "achieved", "unit", "frac", "error")
                        if kk in v} for k, v in configs.items()},
    }
    if not args.no_cpu_baseline:
        cb = cpu_baseline(headline, args.cpu_seconds)
        if "us_per_call" in cb:
            line["cpu_baseline"] = {
                "value": round(cb["us_per_call"], 1), "unit": "us/call", "cores": cb["cores"],
                "kind": "oracle",
                "sample": f"{cb['queries']} of the {cb['per_call_queries']} queries, drawn at "
                          f"random, in {cb['seconds']} s (float64 numpy, BLAS threads at the "
                          f"library default), scaled to a full call"}
        else:
            line["cpu_baseline"] = {"value": None, "kind": "oracle", "error": cb.get("error")}
    if detail:
        compact = {k: {kk: v[kk] for kk in ("us", "us_median", "us_warm_graph", "achieved", "unit",
                                            "frac", "tflops", "gbs", "frac_hbm",
                                            "frac_bf16_tensor", "error") if kk in v}
                   for k, v in detail.items()}
        print(json.dumps({"bench_detail": compact}), file=sys.stderr, flush=True)
    print(json.dumps(line), flush=True)


def run_reference(args):
    """The reference arm: the float64 oracle on the host cores, rank 0 only.  A full call of the
    prefill workloads takes the oracle minutes, so each step is a bounded sample of the call's
    queries (at most --ref-queries, drawn at random), timed and scaled to the full call."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from oracle_io import oracle_args
    import oracle
    from workloads import make
    w = make(args.workload)
    a = oracle_args(w)
    T = w.num_tokens
    rng = np.random.default_rng(0)
    nq = min(T, args.ref_queries)

    def step():
        toks = np.sort(rng.choice(T, size=nq, replace=False)) if nq < T else np.arange(T)
        t0 = time.perf_counter()
        oracle.sparse_paged_attention(**sample_args(a, toks))
        return (time.perf_counter() - t0) * T / nq

    for _ in range(args.warmup):
        step()
    per_call = [step() for _ in range(args.steps)]
    us = statistics.mean(per_call) * 1e6
    sample = (f"{nq} of the {T} queries per step, drawn at random, scaled to the full call"
              if nq < T else "every query of the call")
    line = {
        "metric": METRIC, "value": round(us, 1), "unit": "us/call", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) rows, random block tables and top-k; no dataset)",
        "config": {"workload": describe(args.workload),
                   "parallelism": "rank 0 only, host cores"},
        "impl": "reference",
        "cpu_baseline": {"value": round(us, 1), "unit": "us/call", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": f"float64 numpy oracle; {sample}"},
        "e2e": {"value": round(us, 1), "unit": "us/call", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=HEADLINE,
                    help="headline workload (default: prefill S=8192, ratio 4); see workloads.make")
    ap.add_argument("--headline-only", action="store_true",
                    help="the headline workload only (no other configurations or shapes)")
    ap.add_argument("--sub", default=None,
                    help="comma-separated names: measure only these of the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-queries", type=int, default=32,
                    help="reference arm: queries of the call timed per step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.sub is not None:
        known = (set(sum(CONFIGS.values(), [])) | set(OTHER_SHAPES) | set(KV_WRITES)
                 | set(GATED_POOLS) | set(INDEXERS) | set(TOPK_SHAPES))
        unknown = set(args.sub.split(",")) - known
        if unknown:
            ap.error(f"unknown --sub workload(s): {sorted(unknown)}")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
