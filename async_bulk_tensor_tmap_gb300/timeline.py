"""Per-CTA timelines of the streaming kernels on one GPU, from the tracing build of the library.

    python async_bulk_tensor_tmap_gb300/timeline.py [--out FILE.json] [--reps N]

Builds libtmap_gb300_trace.so (the library compiled with -DTM_TRACE: each CTA of the tensor-map
streaming kernel and of the ring writes %globaltimer stamps at entry, after its first loads are
issued, as each stage completes and at exit) and loads it in place of the library.  Every launch
is timed as bench.py times it: after a 512 MiB device write that flushes L2, between two CUDA
events on the launching stream.  For each workload it prints the event time and, from the stamps
of the median launch, where that time goes:

  outside   event time minus the kernel's span (first CTA entry to last CTA exit): launch and
            event overhead, which the kernel cannot touch; the same flush and events with nothing
            between them, or around one trivial torch kernel, give the floor of this figure on the
            machine, and a one-box copy with a trivial kernel between the flush and the first
            event shows what of it the flush leaves behind
  issue     entry to the first S stages issued (median CTA)
  first     entry to the first stage complete (median CTA): the ramp
  steady    the stream's rate between the times 25 % and 75 % of all stages completed
  tail      from 90 % of the stages completed to the last CTA's exit
  spread    first to last CTA exit

and for the vector path's segment kernels, per CTA (medians): `sync` entry to the producer past
the CTA's barrier initialisation, `table` from there to its first item's row table written,
`loads` from there to that item's bulk copies issued.

The stamps sit in the tracing build only; the library itself compiles them to nothing.
"""
from __future__ import annotations

import argparse
import ctypes
import importlib.util
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SLOTS = 64
FLUSH_BYTES = 512 << 20


def _build_trace_library() -> str:
    spec = importlib.util.spec_from_file_location("tmap_gb300_build", os.path.join(HERE, "csrc", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build(trace=True)


def _stamps(lib, name: str) -> np.ndarray:
    buf = np.zeros((2048, SLOTS), np.uint64)
    rc = getattr(lib, f"tm_trace_fetch_{name}")(buf.ctypes.data_as(ctypes.c_void_p),
                                                ctypes.c_size_t(buf.nbytes))
    if rc != 0:
        raise RuntimeError(f"tm_trace_fetch_{name} failed ({rc})")
    return buf


def analyse(stamps: np.ndarray, event_us: float, nbytes: int, item_slots, spans=None) -> dict:
    """The decomposition above for one launch; nbytes: algorithmic bytes of the launch.  Each CTA
    stamps its first len(item_slots) stages and records its stage count in slot 61.  spans: name ->
    (slot a, slot b), reported as the median over CTAs of stamp b minus stamp a."""
    t = stamps[stamps[:, 0] > 0].astype(np.int64)
    counts = t[:, 61]
    share = float(np.minimum(counts, len(item_slots)).sum() / max(1, counts.sum()))
    t0 = t[:, 0].min()
    rel = np.where(t > 0, t - t0, -1) / 1000.0
    exit_ = rel[:, SLOTS - 1]
    items = rel[:, item_slots]
    done = np.sort(items[items >= 0])
    q = lambda f: float(done[min(len(done) - 1, int(f * len(done)))])
    span = float(exit_.max())
    per_item = nbytes * share / max(1, (items >= 0).sum())
    t25, t75 = q(0.25), q(0.75)
    steady = 0.5 * len(done) * per_item / max(1e-9, (t75 - t25) * 1e-6) / 1e9
    extra = {}
    for name, (sa, sb) in (spans or {}).items():
        ok = (t[:, sa] > 0) & (t[:, sb] > 0)
        extra[name] = round(float(np.median((t[ok, sb] - t[ok, sa]) / 1000.0)), 2) if ok.any() else None
    return {
        **extra,
        "event_us": round(event_us, 2), "span_us": round(span, 2),
        "outside_us": round(event_us - span, 2),
        "issue_us": round(float(np.median(rel[:, 1])), 2),
        "first_us": round(float(np.median(rel[:, item_slots[0]])), 2),
        "steady_GBps": round(steady),
        "tail_us": round(span - q(0.9), 2) if share >= 1.0 else None,  # needs every stage stamped
        "spread_us": round(float(exit_.max() - exit_[exit_ >= 0].min()), 2),
        "ctas": int(len(t)),
        "GBps": round(nbytes / (event_us * 1e-6) / 1e9),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=None)
    ap.add_argument("--reps", type=int, default=7)
    args = ap.parse_args()

    _build_trace_library()
    os.environ["TMAP_GB300_TRACE"] = "1"
    sys.path.insert(0, ROOT)
    import torch

    import async_bulk_tensor_tmap_gb300 as tm
    import workloads
    assert tm.library_path.endswith("libtmap_gb300_trace.so"), tm.library_path
    torch.cuda.set_device(0)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.uint8)).cuda()

    def timed(fn, kname, nbytes, item_slots, reps, pre=None, spans=None):
        for _ in range(3):
            flush.fill_(1)
            fn()
        torch.cuda.synchronize()
        runs = []
        for _ in range(reps):
            flush.fill_(1)
            if pre is not None:
                pre()
            if kname:
                assert getattr(tm._L, f"tm_trace_clear_{kname}")() == 0
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ev = e0.elapsed_time(e1) * 1000.0
            runs.append((ev, _stamps(tm._L, kname) if kname else None))
        if tm.tm_stream_check() != tm.TM_OK:
            raise RuntimeError(tm.tm_last_error())
        runs.sort(key=lambda r: r[0])
        ev, st = runs[len(runs) // 2]
        out = analyse(st, ev, nbytes, item_slots, spans) if kname else {"event_us": round(ev, 2)}
        out["event_us_all"] = [round(r[0], 2) for r in runs]
        return out

    stream_items = list(range(2, 60))
    ring_items = list(range(2, 58))
    res = {}
    tiny = torch.zeros(1, device="cuda")
    res["events alone (floor)"] = timed(lambda: None, None, 0, None, args.reps)
    res["torch trivial kernel (floor)"] = timed(lambda: tiny.add_(1), None, 0, None, args.reps)

    x = workloads.w3_tensor()
    r3 = workloads.w3_map()
    xd = dev(x)
    sw = tm.TM_SWIZZLE_128B
    m3 = tm.tmap_encode(tm.TM_BF16, xd, r3["dims"], r3["strides"], r3["box"], swizzle=sw)
    out3 = torch.empty_like(xd)
    m3o = tm.tmap_encode(tm.TM_BF16, out3, r3["dims"], r3["strides"], r3["box"], swizzle=sw)
    img3 = torch.empty(m3.num_boxes * m3.box_bytes, dtype=torch.uint8, device="cuda")
    nb3 = 2 * xd.numel()
    res["w3.copy one box"] = timed(lambda: tm.tiled_copy(m3, [[0, 0]], img3), "stream",
                                   2 * m3.box_bytes, stream_items, args.reps)
    res["w3.copy one box, a kernel after the flush"] = timed(
        lambda: tm.tiled_copy(m3, [[0, 0]], img3), "stream", 2 * m3.box_bytes, stream_items,
        args.reps, pre=lambda: tiny.add_(1))
    res["w3.copy"] = timed(lambda: tm.tiled_copy(m3, None, img3), "stream", nb3, stream_items, args.reps)
    res["w3.roundtrip"] = timed(lambda: tm.tiled_roundtrip(m3o, None, img3), "stream", nb3,
                                stream_items, args.reps)
    del xd, out3, img3

    x4 = workloads.w4_tensor()
    r4 = workloads.w4_rank3_map(64, span=128)
    x4d = dev(x4)
    m4 = tm.tmap_encode(tm.TM_BF16, x4d, r4["dims"], r4["strides"], r4["box"], swizzle=sw)
    img4 = torch.empty(m4.num_boxes * m4.box_bytes, dtype=torch.uint8, device="cuda")
    nb4 = 2 * 16 * 4095 * 1000 * 2
    res["w4r3.copy"] = timed(lambda: tm.tiled_copy(m4, None, img4), "stream", nb4, stream_items, args.reps)
    # the rank-5 view (200-byte stride): the vector path's segment kernels
    r5 = workloads.w4_rank5_map(span=128)
    m5 = tm.tmap_encode(tm.TM_BF16, x4d, r5["dims"], r5["strides"], r5["box"], swizzle=sw)
    out4 = x4d.clone()
    m5o = tm.tmap_encode(tm.TM_BF16, out4, r5["dims"], r5["strides"], r5["box"], swizzle=sw)
    img5 = torch.empty(m5.num_boxes * m5.box_bytes, dtype=torch.uint8, device="cuda")
    nb5 = 16 * 4095 * 1000 * 2 + m5.num_boxes * m5.box_bytes
    seg_items = list(range(2, 60))
    seg_spans = {"sync_us": (0, 62), "table_us": (62, 60), "loads_us": (60, 1)}
    res["w4r5.copy"] = timed(lambda: tm.tiled_copy(m5, None, img5), "seg", nb5, seg_items, args.reps,
                             spans=seg_spans)
    res["w4r5.roundtrip"] = timed(lambda: tm.tiled_roundtrip(m5o, None, img5), "seg", nb5, seg_items,
                                  args.reps, spans=seg_spans)
    del x4d, img4, out4, img5

    a, b = workloads.w5b_tensors()
    ra, rb = workloads.w5b_maps()
    ad, bd = dev(a), dev(b)
    ma = tm.tmap_encode(tm.TM_BF16, ad, ra["dims"], ra["strides"], ra["box"], swizzle=sw)
    mb = tm.tmap_encode(tm.TM_BF16, bd, rb["dims"], rb["strides"], rb["box"], swizzle=sw)
    n = ma.num_boxes
    cs = [torch.zeros(n, dtype=dt, device="cuda") for dt in (torch.float32, torch.float32,
                                                              torch.int64, torch.int64)]
    res["w5b.ring"] = timed(lambda: tm.stream_tiles(ma, mb, 4, *cs), "ring", ad.numel() + bd.numel(),
                            ring_items, args.reps)
    del ad, bd

    d, s = workloads.w5a_tensors()
    r5 = workloads.w5a_map()
    dd, sd = dev(d), dev(s)
    md = tm.tmap_encode(tm.TM_F32, dd, r5["dims"], r5["strides"], r5["box"], swizzle=sw)
    ms = tm.tmap_encode(tm.TM_F32, sd, r5["dims"], r5["strides"], r5["box"], swizzle=sw)
    res["w5a.reduce"] = timed(lambda: tm.tile_reduce_add(md, ms), "stream", 3 * 4 * d.size,
                              stream_items, max(3, args.reps // 2))

    cols = ["event_us", "outside_us", "span_us", "issue_us", "first_us", "steady_GBps", "tail_us",
            "spread_us", "GBps", "sync_us", "table_us", "loads_us"]
    print("| launch | " + " | ".join(cols) + " |")
    print("|---" * (len(cols) + 1) + "|")
    for k, v in res.items():
        print(f"| {k} | " + " | ".join(str(v.get(c, "")) for c in cols) + " |")
    if args.out:
        with open(args.out, "w") as f:
            json.dump(res, f, indent=1)


if __name__ == "__main__":
    main()
