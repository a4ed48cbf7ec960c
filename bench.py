#!/usr/bin/env python3
"""Benchmark: paged decode attention on GB300 (one JSON line on rank 0).

A step is one pass of the whole hot path over one batch: the cache write of
the step's new tokens (fp16 -> E5M2 cast for an E5M2 cache) followed by paged
decode attention over every sequence's blocks (one decode launch; split units are
combined inside it).

    python bench.py [--config 8b] [--steps K] [--warmup W] [--gpus N]
    python bench.py --impl reference ...   # the CPU oracle on the same workload

Workloads (seeded, synthetic; see paged_kv_cache_252_gb300/workloads.py):
  tiny, 8b (default: Llama-3-8B-shaped decode layer, batch 64, fp16 KV),
  8b_fp8, 8b_int8, long, 70b_spec, mixed (decode + 4-token verify rows packed together).

value  = algorithmic bytes of the step / device time per step (GB/s), inputs
         resident in HBM. Algorithmic bytes: every visible token's K and V once,
         q in, out out, plus the cache write's reads and writes. The K timed
         steps are captured as one CUDA graph and replayed (as a serving loop
         replays its decode steps); the same steps issued one by one from Python
         are reported beside (ms_per_step_host_issued).
roofline = the decode launch alone: algorithmic bytes / mean time per launch,
         from CUDA events around graphs of back-to-back launches (the binding's
         Python time per call is about the kernel's, so launches issued one by
         one with an event pair each, also reported, partly time the host).
e2e    = the same metric through the public Python API with host buffers: the
         step's q, new K/V tokens, slot mapping, block table and lengths copied
         from pinned host memory (one packed copy), and the output copied back,
         inside the timing; copies run on copy streams, double-buffered, and
         overlap the neighbouring steps' kernels as in a serving loop, and the
         --steps steps are captured once in a CUDA graph and replayed
         (--no-graph: direct calls).
per_config = the decode op of each other workload (8b_fp8, 8b_int8, long,
         70b_spec, mixed), timed in the same run with CUDA events.
Several KV pools are rotated so that one cycle touches more than 4x the L2.

Multi-GPU: replicas only. Each rank runs the same workload on its own GPU;
value = total bytes of all ranks / max elapsed over ranks (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode-attention HBM GB/s (% of GB300 peak) and seq-steps/s"


# ---------------------------------------------------------------------------------
# distributed helpers (replicas only)
# ---------------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int, device=None):
    if world > 1:
        if device is not None and device.type == "cuda":
            torch.distributed.barrier(device_ids=[device.index])
        else:
            torch.distributed.barrier()


def aggregate(elapsed_s: float, units: float, world: int, device=None):
    """Whole-job view of a replicated run: max elapsed over ranks, total units."""
    if world <= 1:
        return elapsed_s, units
    dev = device if (device is not None and device.type == "cuda") else torch.device("cpu")
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.gpu_index = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="pkv_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.interval_ms}"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)   # let the first sample land before the timed region
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            lines = f.read().splitlines()
        os.unlink(self.path)
        return summarize_clocks(lines)


def summarize_clocks(lines):
    """nvidia-smi CSV rows (noheader, nounits) -> median SM clock, max, reasons seen."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                         "hw": parts[5], "hw_thermal": parts[6], "sw_thermal": parts[7],
                         "sw_power": parts[8]})
        except ValueError:
            continue
    if not rows:
        return None
    reasons = set()
    for r in rows:
        for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
            if r[key].lower().startswith("active"):
                reasons.add(name)
    return {"sm_mhz": float(np.median([r["sm"] for r in rows])),
            "sm_max_mhz": float(max(r["max"] for r in rows)),
            "power_w_max": float(max(r["power"] for r in rows)),
            "samples": len(rows), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------------
# roofline helpers
# ---------------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# Sources that decide the decode launch of a workload: the host side and the
# shared device code, plus the kernel family that runs it (the tcgen05 kernel
# for E5M2 head-128 units of more than 16 rows, the mma.sync kernel otherwise).
_DECODE_COMMON = ["capi.cu", "pkv_internal.h", "pkv_ptx.cuh", "decode_common.cuh"]
_DECODE_FAMILY = {
    "tc": ["decode_tc.cu", "decode_tc_kernel.cuh", "pkv_tc.cuh"],
    "mma": ["decode_kernel.cuh", "decode_f16.cu", "decode_bf16.cu", "decode_e5m2.cu", "decode_int8.cu"],
}


def decode_family(w) -> str:
    rows = w.q_per_seq * (w.num_q_heads // w.num_kv_heads)
    return "tc" if (w.kv_dtype == "e5m2" and w.head_size == 128 and rows > 16) else "mma"


def product_source(text: str) -> str:
    """A source file as the product library compiles it, as far as the profiling
    build's hooks go: the branches of `#ifdef PKV_TIMELINE` blocks and the lines that
    call the PKV_TL* macros (which expand to nothing without PKV_TIMELINE) are left
    out; `#else` branches are kept."""
    out, stack = [], []      # stack: per open #if*, whether its current branch is dropped
    for line in text.splitlines(keepends=True):
        t = line.strip()
        if t.startswith("#if"):
            stack.append(t == "#ifdef PKV_TIMELINE")
            if stack[-1]:
                continue
        elif t.startswith("#else") and stack:
            if stack[-1] is not False:
                stack[-1] = "else"
                continue
        elif t.startswith("#endif") and stack:
            if stack.pop() is not False:
                continue
        if any(x is True for x in stack) or "PKV_TL" in line:
            continue
        out.append(line)
    return "".join(out)


def csrc_digest(family: str) -> str:
    src = hashlib.sha256()
    d = os.path.join(ROOT, "paged_kv_cache_252_gb300", "csrc")
    for fn in sorted(_DECODE_COMMON + _DECODE_FAMILY[family]):
        with open(os.path.join(d, fn), encoding="utf-8") as f:
            src.update(fn.encode())
            src.update(product_source(f.read()).encode())
    return src.hexdigest()


def profiled_traffic(config: str):
    """DRAM bytes per decode launch from a committed ncu summary, if it was taken on
    the current source of the kernel that runs this workload (else None)."""
    from paged_kv_cache_252_gb300 import workloads as wl
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    entry = d.get(config)
    if not entry or entry.get("csrc_sha256") != csrc_digest(decode_family(wl.by_name(config))):
        return None
    return float(entry["dram_bytes_per_launch"])


# ---------------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------------

def l2_bytes(dev=None) -> int:
    """L2 size of the device (the GB300's when no device is visible)."""
    if dev is not None or torch.cuda.is_available():
        props = torch.cuda.get_device_properties(dev if dev is not None else 0)
        return int(getattr(props, "L2_cache_size", 126 << 20))
    return 126 << 20


def pool_count(w, l2: int, pools_arg: int = 0) -> int:
    """KV pools rotated so that one cycle touches more than 4x the L2."""
    return pools_arg or max(2, math.ceil(4 * l2 / w.kv_bytes_read()))


def bench_config(w, pools: int, l2: int, world: int) -> dict:
    """The `config` object of the JSON line (identical in both arms)."""
    return {**w.describe(), "l2_policy": f"{pools} KV pools rotated, "
            f"{pools * w.kv_bytes_read() / 1e9:.2f} GB per cycle > 4x L2 ({l2 / 1e6:.0f} MB)",
            "parallelism": f"replicas x{world}"}


class Prepared:
    """One workload resident on the device: `pools` prefilled KV caches, the step's
    new tokens, block table, lengths, and per-pool query/output buffers."""

    def __init__(self, w, dev, pools: int):
        import paged_kv_cache_252_gb300 as pkv
        from paged_kv_cache_252_gb300 import workloads as wl
        self.pkv, self.w, self.dev, self.pools = pkv, w, dev, pools
        self.int8 = w.kv_dtype == "int8"
        vals = wl.token_values(w, device=dev)
        self.caches = []   # (k_cache, v_cache[, scales])
        for _ in range(pools):
            kc, vc = pkv.alloc_kv_cache(w.num_blocks, w.num_kv_heads, w.head_size, w.kv_dtype, dev)
            c = (kc, vc) + ((pkv.alloc_kv_scales(w.num_blocks, w.num_kv_heads, dev),) if self.int8 else ())
            self.write(vals["k_all"], vals["v_all"], vals["slot_all"], c)   # prefill
            self.caches.append(c)
        new_idx = vals["new_idx"]
        self.k_new = vals["k_all"][new_idx].contiguous()
        self.v_new = vals["v_all"][new_idx].contiguous()
        self.s_new = vals["slot_all"][new_idx].contiguous()
        self.bt = torch.from_numpy(w.block_tables).to(dev)
        self.cl = torch.from_numpy(w.context_lens).to(dev)
        self.cu = torch.from_numpy(w.cu_q_lens()).to(dev) if w.q_lens is not None else None
        self.qs = [vals["q"].clone() for _ in range(pools)]
        self.outs = [torch.empty_like(vals["q"]) for _ in range(pools)]
        del vals
        torch.cuda.synchronize(dev)
        self.kv_bytes = w.kv_bytes_read()
        self.attn_bytes = self.kv_bytes + w.q_out_bytes()
        self.step_bytes = self.attn_bytes + w.write_bytes()

    def write(self, kn, vn, sn, c):
        if self.int8:
            self.pkv.kv_cache_write_int8(kn, vn, sn, *c)
        else:
            self.pkv.kv_cache_write(kn, vn, sn, c[0], c[1])

    def decode(self, o, q, c, bt, cl, cu):
        w, pkv = self.w, self.pkv
        if self.int8:
            pkv.paged_attention_decode_int8(o, q, *c, bt, cl, w.q_per_seq, w.scale)
        elif cu is not None:
            pkv.paged_attention_decode_varlen(o, q, cu, c[0], c[1], bt, cl, w.q_per_seq, w.scale)
        else:
            pkv.paged_attention_decode(o, q, c[0], c[1], bt, cl, w.q_per_seq, w.scale)

    def step(self, i):
        """One step: the new tokens' cache write, then decode attention (2 launches)."""
        p = i % self.pools
        self.write(self.k_new, self.v_new, self.s_new, self.caches[p])
        self.decode_pool(p)

    def decode_pool(self, p):
        self.decode(self.outs[p], self.qs[p], self.caches[p], self.bt, self.cl, self.cu)

    def time_decode_host_issued(self, n: int) -> float:
        """Mean seconds per decode launch over n launches issued one by one from
        Python (rotating pools), an event pair on the launching stream around each.
        When the binding's per-call host time exceeds the kernel's, the GPU idles
        between the first event and the launch and this overstates the kernel."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize(self.dev)
        for i in range(n):
            evs[i][0].record()
            self.decode_pool(i % self.pools)
            evs[i][1].record()
        torch.cuda.synchronize(self.dev)
        return float(np.mean([a.elapsed_time(b) for a, b in evs])) / 1e3

    def graph_of(self, n: int, body):
        """A CUDA graph of body(0), ..., body(n-1) (library calls only), captured on
        a side stream. One call runs on that stream before the capture, so the
        binding's workspace for it exists outside the capture."""
        cur = torch.cuda.current_stream(self.dev)
        s = torch.cuda.Stream(self.dev)
        s.wait_stream(cur)
        with torch.cuda.stream(s):
            body(0)
        cur.wait_stream(s)
        torch.cuda.synchronize(self.dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(n):
                body(i)
        torch.cuda.synchronize(self.dev)
        return g

    def time_graph(self, g, replays: int = 1) -> float:
        """Seconds for `replays` back-to-back replays of g, an event pair on the
        current stream around them (after one untimed replay that uploads it)."""
        cur = torch.cuda.current_stream(self.dev)
        g.replay()
        torch.cuda.synchronize(self.dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for _ in range(replays):
            g.replay()
        b.record(cur)
        torch.cuda.synchronize(self.dev)
        return a.elapsed_time(b) / 1e3

    def time_decode(self, n: int, per_graph: int = 200):
        """Mean seconds per decode launch over about n launches run back to back from
        CUDA graphs of up to per_graph launches (rotating pools), as a serving loop
        replays them; returns (seconds per launch, launches timed)."""
        k = min(per_graph, n)
        k = max(self.pools, (k + self.pools - 1) // self.pools * self.pools)
        replays = max(1, -(-n // k))
        g = self.graph_of(k, lambda i: self.decode_pool(i % self.pools))
        t = self.time_graph(g, replays)
        del g
        return t / (k * replays), k * replays


# The other workloads, measured as decode-op timings in the same run.
PER_CONFIG = ["8b_fp8", "8b_int8", "long", "70b_spec", "mixed"]


def measure_per_config(keys, dev, peak, min_launches=50, min_seconds=1.0):
    """Decode-op time per launch of each workload (CUDA events, at least min_launches
    launches and about min_seconds of launches each), with the clocks sampled during
    each timing loop."""
    from paged_kv_cache_252_gb300 import workloads as wl
    res = {}
    l2 = l2_bytes(dev)
    for key in keys:
        w = wl.by_name(key)
        P = Prepared(w, dev, pool_count(w, l2))
        for i in range(5):
            P.decode_pool(i % P.pools)
        est, _ = P.time_decode(20)
        n = max(min_launches, int(math.ceil(min_seconds / max(est, 1e-6))))
        sampler = ClockSampler(dev.index)
        sampler.start()
        t, n = P.time_decode(n)
        clocks = sampler.stop()
        t_host = P.time_decode_host_issued(min_launches)
        achieved = P.attn_bytes / t / 1e9
        res[key] = {"workload": w.name, "kv_dtype": w.kv_dtype, "launches": n,
                    "us_per_launch": round(t * 1e6, 3),
                    "us_per_launch_host_issued": round(t_host * 1e6, 3),
                    "achieved_gbs": round(achieved, 2), "frac": round(achieved / peak, 4),
                    "algorithmic_bytes_per_launch": int(P.attn_bytes),
                    "seq_steps_per_s": round(w.num_seqs / t, 1),
                    "tokens_per_s": round(w.num_new_tokens / t, 1),
                    "clocks": clocks}
        del P
        torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, local):
    import paged_kv_cache_252_gb300 as pkv
    from paged_kv_cache_252_gb300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pkv.load_library()
    w = wl.by_name(args.config)
    l2 = l2_bytes(dev)
    pools = pool_count(w, l2, args.pools)
    P = Prepared(w, dev, pools)
    step_bytes, attn_bytes = P.step_bytes, P.attn_bytes

    for i in range(args.warmup):
        P.step(i)
    torch.cuda.synchronize(dev)

    # The K timed steps run as one CUDA graph replay (as a serving loop replays its
    # decode steps), so the binding's host time does not enter the measurement; the
    # graph is captured and replayed once untimed first.
    g_steps = P.graph_of(args.steps, P.step) if not args.no_graph else None
    if g_steps is not None:
        g_steps.replay()
    torch.cuda.synchronize(dev)
    barrier(world, dev)

    sampler = ClockSampler(local) if not args.no_clocks else None
    if sampler:
        sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record()
    if g_steps is not None:
        g_steps.replay()
    else:
        for i in range(args.steps):
            P.step(i)
    e1.record()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    barrier(world, dev)
    elapsed = e0.elapsed_time(e1) / 1e3
    job_elapsed, job_bytes = aggregate(elapsed, step_bytes * args.steps, world, dev)
    del g_steps

    # The same K steps issued one by one from Python (reported beside: the binding's
    # per-call host time is close to the kernel's, so this is partly host-bound).
    torch.cuda.synchronize(dev)
    h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h0.record()
    for i in range(args.steps):
        P.step(i)
    h1.record()
    torch.cuda.synchronize(dev)
    host_issued_step_s = h0.elapsed_time(h1) / 1e3 / args.steps

    # Decode op alone (one decode launch, split-KV combine fused): CUDA events on its
    # stream around graphs of back-to-back launches; and, beside it, launches issued
    # one by one from Python with an event pair around each.
    dec_s, n_r = P.time_decode(max(args.steps, 50))
    dec_host_s = P.time_decode_host_issued(max(args.steps, 50))

    # End to end through the public API with pinned host buffers, run the way a
    # serving loop runs it: each step's inputs travel in one packed host->device
    # copy and its output in one device->host copy, on an upload and a download
    # stream, double-buffered, so the copies of neighbouring steps overlap this
    # step's kernels. Every step still copies its own inputs and reads back its output
    # inside the timed region.
    e2e = None
    if not args.no_e2e:
        caches, outs, qs = P.caches, P.outs, P.qs
        named = [("q", qs[0]), ("k_new", P.k_new), ("v_new", P.v_new), ("s_new", P.s_new), ("bt", P.bt),
                 ("cl", P.cl)]
        if P.cu is not None:
            named.append(("cu", P.cu))
        layout, off = [], 0
        for n, t in named:
            nbytes = t.numel() * t.element_size()
            layout.append((n, off, nbytes, t.dtype, tuple(t.shape)))
            off += (nbytes + 255) // 256 * 256
        host_in = torch.empty(off, dtype=torch.uint8).pin_memory()
        for (n, o, nbytes, dt, shp), (_, t) in zip(layout, named):
            host_in[o:o + nbytes].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
        dev_in = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]
        views = [{n: buf[o:o + nbytes].view(dt).view(shp) for n, o, nbytes, dt, shp in layout} for buf in dev_in]
        out_h = [torch.empty(outs[0].shape, dtype=outs[0].dtype).pin_memory() for _ in range(2)]
        h2d = off
        d2h = out_h[0].numel() * out_h[0].element_size()
        cs_in, cs_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)   # uploads, downloads
        comp = torch.cuda.current_stream(dev)
        ev = lambda: torch.cuda.Event()
        ready = [ev(), ev()]        # inputs of buffer b landed
        free = [ev(), ev()]         # kernels that read buffer b are done
        out_done = [ev() for _ in range(pools)]   # outs[p] copied back
        for e_ in free + out_done:
            e_.record(comp)

        def e2e_step(i, captured=False):
            """One step. Inside a graph capture it waits only on events recorded by
            earlier steps of the same capture: earlier replays already precede it in
            stream order."""
            p, b = i % pools, i % 2
            v = views[b]
            with torch.cuda.stream(cs_in):
                if not captured or i >= 2:
                    cs_in.wait_event(free[b])
                dev_in[b].copy_(host_in, non_blocking=True)
                ready[b].record(cs_in)
            comp.wait_event(ready[b])
            if not captured or i >= pools:
                comp.wait_event(out_done[p])
            P.write(v["k_new"], v["v_new"], v["s_new"], caches[p])
            P.decode(outs[p], v["q"], caches[p], v["bt"], v["cl"], v.get("cu"))
            free[b].record(comp)
            with torch.cuda.stream(cs_out):
                cs_out.wait_event(free[b])
                out_h[b].copy_(outs[p], non_blocking=True)
                out_done[p].record(cs_out)

        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        graph = None
        e2e_steps = args.steps
        if not args.no_graph:
            # A serving loop replays captured steps: the timed steps are captured
            # once as one graph, with the copy streams forked from and joined back
            # into the capture, replayed once untimed and once timed.
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(comp)
            with torch.cuda.stream(cap):          # the binding's workspace for this stream, outside the capture
                P.decode(outs[0], qs[0], caches[0], P.bt, P.cl, P.cu)
            comp.wait_stream(cap)
            torch.cuda.synchronize(dev)
            graph = torch.cuda.CUDAGraph()
            comp_outer = comp
            with torch.cuda.graph(graph, stream=cap):
                comp = torch.cuda.current_stream(dev)
                cs_in.wait_stream(comp)
                cs_out.wait_stream(comp)
                for i in range(e2e_steps):
                    e2e_step(i, captured=True)
                comp.wait_stream(cs_in)
                comp.wait_stream(cs_out)
            comp = comp_outer
            graph.replay()
            torch.cuda.synchronize(dev)
        barrier(world, dev)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(comp)
        if graph is not None:
            graph.replay()
        else:
            cs_in.wait_stream(comp)   # the first upload starts inside the timed region
            for i in range(e2e_steps):
                e2e_step(i)
            comp.wait_stream(cs_in)
            comp.wait_stream(cs_out)  # the last outputs are back on the host
        a1.record(comp)
        torch.cuda.synchronize(dev)
        e2e_el = a0.elapsed_time(a1) / 1e3
        e2e_job_el, e2e_job_bytes = aggregate(e2e_el, step_bytes * e2e_steps, world, dev)
        e2e = {"value": round(e2e_job_bytes / e2e_job_el / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e2e_el / e2e_steps * 1e3, 5), "steps": e2e_steps,
               "copies": "one packed H2D and one D2H per step on copy streams, double-buffered",
               "launch": (f"CUDA graph of the {e2e_steps} steps, replayed once" if graph is not None
                          else "direct calls")}

    peak, peak_kind = measured_peaks()
    per_config = None
    if not args.no_per_config and world == 1:
        keys = [k for k in PER_CONFIG if k != args.config]
        del P
        torch.cuda.empty_cache()
        per_config = measure_per_config(keys, dev, peak)
    if rank != 0:
        return
    achieved = attn_bytes / dec_s / 1e9
    cpu = None if (args.no_cpu_baseline or world > 1) else cpu_baseline(w, args.cpu_budget_s)
    value = job_bytes / job_elapsed / 1e9
    dtype = ("fp16 q / " + w.kv_dtype + " KV, fp32 accumulate") if w.q_dtype == "fp16" \
        else "bf16 q / bf16 KV, fp32 accumulate"
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed / args.steps * 1e3, 5),
        "ms_per_step_host_issued": round(host_issued_step_s * 1e3, 5),
        "launch": ("the K steps as one CUDA graph replay" if not args.no_graph
                   else "the K steps issued one by one from Python"),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype,
        "data": "synthetic (seeded N(0,1) K/V/q, shuffled block pool)",
        "config": bench_config(w, pools, l2, world),
        "seq_steps_per_s": round(w.num_seqs * world * args.steps / job_elapsed, 1),
        "tokens_per_s": round(w.num_new_tokens * world * args.steps / job_elapsed, 1),
        "pct_of_hbm_peak": round(100 * value / peak, 2),
        "roofline": {"bound": "hbm", "kernel": "paged_attention_decode (one launch, split-KV combine fused)",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "traffic": profiled_traffic(args.config),
                     "algorithmic_bytes_per_launch": int(attn_bytes),
                     "us_per_launch": round(dec_s * 1e6, 3), "launches_timed": n_r,
                     "timing": "CUDA events around graphs of back-to-back decode launches",
                     "us_per_launch_host_issued": round(dec_host_s * 1e6, 3)},
        "e2e": e2e,
        # per step: the cache write and the decode, one launch each
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "per_config": per_config,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------------

def _oracle_inputs(w, seqs):
    """Host inputs for the oracle: cache images holding the sample's tokens."""
    import oracle
    from paged_kv_cache_252_gb300 import workloads as wl
    vals = wl.token_values(w, device="cpu")
    starts = w.seq_starts()
    mask = np.zeros(w.num_tokens_total, dtype=bool)
    for s in seqs:
        mask[starts[s]:starts[s + 1]] = True
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    k_all, v_all = bits(vals["k_all"]), bits(vals["v_all"])
    slots = vals["slot_all"].numpy()
    new = np.zeros(w.num_tokens_total, dtype=bool)
    new[w.new_token_index()] = True
    pre, stp = mask & ~new, mask & new
    dt = {"e5m2": np.uint8, "int8": np.int8}.get(w.kv_dtype, np.uint16)
    shape = (w.num_blocks, w.num_kv_heads, 16, w.head_size)
    kc, vc = np.zeros(shape, dt), np.zeros(shape, dt)
    code = {"fp16": 0, "bf16": 1, "e5m2": 2, "int8": 3}[w.kv_dtype]
    src = 1 if w.kv_dtype == "bf16" else 0
    ks = vs = None
    if code == 3:
        ks, vs = np.zeros(shape[:3], np.float32), np.zeros(shape[:3], np.float32)
    inp = {"kc": kc, "vc": vc, "ks": ks, "vs": vs, "q": bits(vals["q"]), "k_new": k_all[stp],
           "v_new": v_all[stp], "s_new": slots[stp], "src": src, "code": code}
    _oracle_write(inp, k_all[pre], v_all[pre], slots[pre])
    return inp


def _oracle_write(inp, k, v, slots):
    import oracle
    if inp["code"] == 3:
        oracle.kv_cache_write_int8(k, v, slots, inp["kc"], inp["vc"], inp["ks"], inp["vs"])
    else:
        oracle.kv_cache_write(k, v, inp["src"], slots, inp["kc"], inp["vc"], inp["code"])


def _oracle_step(w, inp, seqs, threads):
    import oracle
    _oracle_write(inp, inp["k_new"], inp["v_new"], inp["s_new"])
    qcode = 1 if w.q_dtype == "bf16" else 0
    _, _, rc = oracle.paged_attention(inp["q"], qcode, w.q_per_seq, inp["kc"], inp["vc"], inp["code"],
                                      w.block_tables, w.context_lens, w.scale, seqs=seqs,
                                      num_threads=threads,
                                      cu_q_lens=w.cu_q_lens() if w.q_lens is not None else None,
                                      k_scale=inp["ks"], v_scale=inp["vs"])
    assert rc == 0


def _sample_bytes(w, seqs):
    lens = w.context_lens[seqs].astype(np.int64)
    row = w.head_size * w.kv_elem_bytes + w.kv_row_extra_bytes
    kv = int(lens.sum()) * w.num_kv_heads * row * 2
    t = int(w.query_lens()[seqs].sum())
    qo = 2 * t * w.num_q_heads * w.head_size * 2
    wr = t * w.num_kv_heads * (w.head_size * 4 + 2 * row) + 4 * t
    return kv + qo + wr


def _pick_sample(w, budget_s, threads):
    """Leading sequences whose oracle step takes about budget_s on `threads` threads,
    estimated from a one-sequence probe."""
    probe = [0]
    inp = _oracle_inputs(w, probe)
    t0 = time.perf_counter()
    _oracle_step(w, inp, probe, 1)
    per_token = (time.perf_counter() - t0) / max(1, int(w.context_lens[0]))
    total_tokens = budget_s * threads / max(per_token, 1e-9)
    seqs, acc = [], 0
    for s in range(w.num_seqs):
        if seqs and acc + int(w.context_lens[s]) > total_tokens:
            break
        seqs.append(s)
        acc += int(w.context_lens[s])
    return seqs


def cpu_baseline(w, budget_s):
    import oracle
    threads = oracle.hardware_threads()
    seqs = _pick_sample(w, budget_s, threads)
    inp = _oracle_inputs(w, seqs)
    t0 = time.perf_counter()
    _oracle_step(w, inp, seqs, threads)
    el = time.perf_counter() - t0
    return {"value": round(_sample_bytes(w, seqs) / el / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{len(seqs)} of {w.num_seqs} sequences (their new-token cache write + fp64 "
                      f"decode attention), {el:.1f} s on {threads} threads"}


def run_reference(args, rank, world, local):
    """The CPU oracle as the reference arm: bounded sample per step, same metric."""
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_252_gb300 import workloads as wl
    oracle.build()
    w = wl.by_name(args.config)
    threads = oracle.hardware_threads()
    per_step = max(1.0, args.cpu_budget_s / max(1, args.steps + args.warmup))
    seqs = _pick_sample(w, per_step, threads)
    inp = _oracle_inputs(w, seqs)
    for _ in range(args.warmup):
        _oracle_step(w, inp, seqs, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(w, inp, seqs, threads)
    el = time.perf_counter() - t0
    v = _sample_bytes(w, seqs) * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) K/V/q, shuffled block pool)",
        "config": bench_config(w, pool_count(w, l2_bytes()), l2_bytes(), world),
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{len(seqs)} of {w.num_seqs} sequences per step"},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="8b", choices=["tiny", "8b", "8b_fp8", "8b_int8", "long", "70b_spec", "mixed"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--pools", type=int, default=0, help="KV pools to rotate (default: >4x L2)")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="steps and e2e by direct calls instead of graph replays")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the decode-op timings of the other workloads")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world, local)
        return
    init_dist(world, "nccl")
    try:
        run_ours(args, rank, world, local)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
