"""Per-CTA timeline of one decode launch (profiling aid).

    python -m paged_kv_cache_252_gb300.timeline --config 8b [--num-seqs N] [--iters 5]

Builds the profiling variant of the library (libpagedkv_timeline.so, compiled
with -DPKV_TIMELINE; the product library has no timeline code), runs the
workload's decode --iters times back to back from a CUDA graph (CUDA events
around the replay give the mean time per launch) and keeps from the last
launch every CTA's
global-timer readings: kernel entry, share planned, first / last tile copy
issued, first block landed, last block consumed, exit (epilogue and split
merges done), plus its SM, pieces and blocks. Prints a summary (times in us
from the earliest CTA entry): quantiles of each event over the CTAs, the launch
span, and how the span divides into ramp (entry to first data), streaming and
tail (after the median CTA exit). --raw PATH saves the per-CTA rows as CSV.
"""
from __future__ import annotations

import argparse
import ctypes

import numpy as np
import torch

from . import api
from . import build
from . import workloads as wl

EVENTS = ["start", "planned", "first_issue", "last_issue", "first_data", "last_data", "exit"]
LATE = ["piece_out", "counted", "merged"]   # events 8..10: the last piece's epilogue
NEV = 28                                     # 64-bit words per CTA (pkv_timeline.cuh)
# tcgen05 kernel: cycles per chunk of the softmax loop's steps (thread 0), the MMA
# thread's waits and the producer's wait for a free ring buffer (words 12..26)
STEP_NAMES = ["top: next chunk / queries", "wait S + read scores", "wait ring (next chunk)",
              "widen K (next chunk)", "scores, max vote", "rare rescale", "wait O (previous chunk)",
              "exp2 + write P", "widen V (next chunk)", "end of piece"]
# mma.sync kernel: SM cycles of consumer thread 0 summed over the CTA's pieces, per
# phase (words 12..19), and the producer's wait for a free ring stage (words 25, 26)
MMA_STEPS = ["query rows load + barrier", "Q fragments, masks", "wait for a block", "block compute",
             "stream merge (barrier)", "merge + output", "split finish", "next piece / exit"]
MAX_CTAS = 4096


def run(config: str, num_seqs: int = 0, iters: int = 5):
    lib = api.load_library(build.build(variant="timeline"))
    if not hasattr(lib, "pkv_timeline_attach"):
        raise RuntimeError("the loaded library is not the timeline build")
    lib.pkv_timeline_attach.argtypes = [ctypes.c_void_p, ctypes.c_int32]
    lib.pkv_timeline_attach.restype = ctypes.c_int
    dev = torch.device("cuda:0")
    w = wl.by_name(config)
    if num_seqs:
        w = wl.reduced(w, num_seqs=num_seqs)
    vals = wl.token_values(w, device=dev)
    kc, vc = api.alloc_kv_cache(w.num_blocks, w.num_kv_heads, w.head_size, w.kv_dtype, dev)
    int8 = w.kv_dtype == "int8"
    sc = None
    if int8:
        sc = api.alloc_kv_scales(w.num_blocks, w.num_kv_heads, dev)
        api.kv_cache_write_int8(vals["k_all"], vals["v_all"], vals["slot_all"], kc, vc, sc)
    else:
        api.kv_cache_write(vals["k_all"], vals["v_all"], vals["slot_all"], kc, vc)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    cu = torch.from_numpy(w.cu_q_lens()).to(dev) if w.q_lens is not None else None
    out = torch.empty_like(vals["q"])
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    tl = torch.zeros(MAX_CTAS * NEV, dtype=torch.int64, device=dev)

    def decode():
        if int8:
            api.paged_attention_decode_int8(out, vals["q"], kc, vc, sc, bt, cl, w.q_per_seq, w.scale,
                                            device_status=status)
        elif cu is not None:
            api.paged_attention_decode_varlen(out, vals["q"], cu, kc, vc, bt, cl, w.q_per_seq, w.scale,
                                              device_status=status)
        else:
            api.paged_attention_decode(out, vals["q"], kc, vc, bt, cl, w.q_per_seq, w.scale,
                                       device_status=status)

    # Every launch records (each overwrites the buffer), so all of them run the same
    # instrumented code: the last one's rows are kept. The launches run back to back
    # from a CUDA graph (no host time between them), and the mean time per launch
    # from an event pair around the replay is the same build's op time to compare
    # the span with.
    lib.pkv_timeline_attach(ctypes.c_void_p(tl.data_ptr()), MAX_CTAS)
    n = max(iters, 2)
    cur = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(cur)
    with torch.cuda.stream(side):
        decode()                 # the binding's workspace for this stream, outside the capture
    cur.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for _ in range(n):
            decode()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    lib.pkv_timeline_attach(None, 0)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    rows = tl.view(MAX_CTAS, NEV).cpu().numpy().view(np.uint64)
    ncta = int((rows[:, 0] != 0).sum())
    ev_us = e0.elapsed_time(e1) * 1e3 / n
    return w, rows[:ncta], ev_us


def summarize(w, rows, event_us: float | None = None) -> str:
    t = rows[:, :7].astype(np.float64)
    info = rows[:, 7]
    t0 = t[:, 0].min()
    rel = np.where(t > 0, (t - t0) / 1e3, np.nan)
    busy = rows[:, 4] != 0
    lines = [f"workload {w.name}: {w.num_seqs} seqs, {w.kv_bytes_read() / 1e6:.1f} MB KV, "
             f"{len(rows)} CTAs ({int(busy.sum())} with work)",
             "",
             "| event (us from first entry) | min | p10 | median | p90 | max |",
             "|---|---|---|---|---|---|"]
    for k, name in enumerate(EVENTS):
        v = rel[:, k][~np.isnan(rel[:, k])]
        if v.size:
            q = np.percentile(v, [0, 10, 50, 90, 100])
            lines.append(f"| {name} | " + " | ".join(f"{x:.2f}" for x in q) + " |")
    late = rows[:, 8:11].astype(np.float64)
    late_rel = np.where(late > 0, (late - t0) / 1e3, np.nan)
    # Only the last piece's epilogue events are comparable: a merge or count that
    # happened mid-share is older than that piece's last data.
    ld = rel[:, 5]
    for k, name in enumerate(LATE):
        v = late_rel[:, k]
        ok = ~np.isnan(v) & (v >= ld - 1e-9)
        if ok.any():
            d = v[ok] - ld[ok]
            q = np.percentile(d, [0, 10, 50, 90, 100])
            lines.append(f"| {name} - last_data ({int(ok.sum())} CTAs) | " + " | ".join(f"{x:.2f}" for x in q) + " |")
    steps = rows[:, 12:12 + len(STEP_NAMES)].astype(np.float64)
    chunks = ((info >> 32) // 8).astype(np.float64)          # tcgen05 kernel: blocks / 8 per chunk
    is_tc = rows[busy, 24].astype(np.float64).sum() > 0      # only the tcgen05 kernel's MMA thread writes 24
    if steps[busy].sum() > 0 and not is_tc:
        per = steps[busy][:, :len(MMA_STEPS)]
        tot = per.sum(axis=1)
        lines += ["", "mma.sync consumer thread 0, SM cycles per CTA summed over its pieces:",
                  "| phase | median cycles | share of the CTA's total |", "|---|---|---|"]
        for k, name in enumerate(MMA_STEPS):
            lines.append(f"| {name} | {np.median(per[:, k]):.0f} | {np.median(per[:, k] / tot):.3f} |")
        lines.append(f"| total | {np.median(tot):.0f} | 1 |")
        prod = rows[busy, 25:27].astype(np.float64)
        lines.append(f"producer: waiting for a free stage {np.median(prod[:, 0]):.0f} of "
                     f"{np.median(prod[:, 1]):.0f} cycles (median per CTA)")
    if steps[busy].sum() > 0 and is_tc:
        per = steps[busy] / np.maximum(chunks[busy], 1)[:, None]
        lines += ["", "tcgen05 chunk loop, SM cycles per chunk (median over CTAs):",
                  "| step (softmax thread 0) | cycles |", "|---|---|"]
        for k, name in enumerate(STEP_NAMES):
            lines.append(f"| {name} | {np.median(per[:, k]):.0f} |")
        lines.append(f"| total | {np.median(per.sum(axis=1)):.0f} |")
        mma = rows[busy, 22:25].astype(np.float64) / np.maximum(chunks[busy], 1)[:, None]
        prod = rows[busy, 25:27].astype(np.float64) / np.maximum(chunks[busy], 1)[:, None]
        lines += [f"MMA thread per chunk: waiting for K {np.median(mma[:, 0]):.0f}, for P/V "
                  f"{np.median(mma[:, 1]):.0f}, loop total {np.median(mma[:, 2]):.0f} cycles",
                  f"producer per chunk: waiting for a free buffer {np.median(prod[:, 0]):.0f}, loop total "
                  f"{np.median(prod[:, 1]):.0f} cycles"]
    ex = rel[busy, 6]
    span = np.nanmax(rel[:, 6])
    ramp = np.nanmedian(rel[busy, 4])
    tail = span - np.nanmedian(ex)
    blocks = (info >> 32)[busy].astype(np.int64)
    pieces = ((info >> 16) & 0xFFFF)[busy].astype(np.int64)
    stream = np.nanmedian(rel[busy, 5] - rel[busy, 4])
    lines += ["",
              f"span (first entry to last exit): {span:.2f} us"
              + (f"; mean time per launch, graph of back-to-back launches (same build): {event_us:.2f} us"
                 if event_us else ""),
              f"ramp (median first data): {ramp:.2f} us; tail (last exit - median exit): {tail:.2f} us",
              f"median streaming time per CTA (first data to last data): {stream:.2f} us",
              f"median epilogue after the last block (exit - last data): "
              f"{np.nanmedian(rel[busy, 6] - rel[busy, 5]):.2f} us",
              f"blocks per CTA: min {blocks.min()}, median {int(np.median(blocks))}, max {blocks.max()}; "
              f"pieces per CTA: min {pieces.min()}, median {int(np.median(pieces))}, max {pieces.max()}",
              f"exit spread among CTAs with work: p10 {np.nanpercentile(ex, 10):.2f}, "
              f"p90 {np.nanpercentile(ex, 90):.2f} us"]
    return "\n".join(lines)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="8b", choices=list(wl.NAMED))
    ap.add_argument("--num-seqs", type=int, default=0)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--raw", default="", help="write the per-CTA rows to this CSV file")
    args = ap.parse_args(argv)
    w, rows, event_us = run(args.config, args.num_seqs, args.iters)
    print(summarize(w, rows, event_us))
    if args.raw:
        hdr = ",".join(EVENTS + ["sm", "pieces", "blocks"] + LATE + [f"w{k}" for k in range(12, 27)])
        t0 = rows[:, :7][rows[:, :7] > 0].min()
        with open(args.raw, "w") as f:
            f.write(hdr + "\n")
            for r in rows:
                ev = [f"{(int(x) - int(t0)) / 1e3:.3f}" if x else "" for x in r[:7]]
                late = [f"{(int(x) - int(t0)) / 1e3:.3f}" if x else "" for x in r[8:11]]
                f.write(",".join(ev + [str(int(r[7]) & 0xFFFF), str((int(r[7]) >> 16) & 0xFFFF),
                                       str(int(r[7]) >> 32)] + late + [str(int(x)) for x in r[12:27]]) + "\n")


if __name__ == "__main__":
    main()
