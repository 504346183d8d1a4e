"""Benchmark of the tiled tensor movement hot path on one GB300 (or N, one process per GPU).

One step = one pass of every kernel of the path over one batch of synthetic input, each kernel
preceded by an L2 flush (a 512 MiB device write, not timed):
  w3.copy       bf16 8192 x 8192, 128 x 64 boxes, 128B swizzle -> 8192 tile-major images
  w3.roundtrip  the images stored back through the map into a second tensor
  w4r3.copy / .roundtrip      bf16 16 x 4095 x 1000 (row pitch 1024), 1 x 64 x 64 boxes, 128B
  w4r3n.copy / .roundtrip     same tensor, 1 x 64 x 32 boxes, 64B
  w4r5.copy / .roundtrip      rank-5 view 4 x 4 x 4095 x 10 x 100, box 1 x 1 x 32 x 10 x 64,
                              200-byte stride: the vector fallback path
  w5a.reduce    fp32 16384 x 16384: dst += src, 128 x 32 boxes, 128B swizzle
  w5b.ring      bf16 A 8192 x 4096 and B 4096 x 8192, 128 x 64 tiles, 4-stage ring + checksums

value = algorithmic bytes of the step / device time of its kernels (CUDA events on the launching
stream), in GB/s; under torchrun every rank runs the same per-GPU workload (weak scaling) and the
step time is the max over ranks.  The JSON line also carries the roofline of the dominant kernel
(the reduce-add), an end-to-end figure with host buffers, the CPU oracle baseline, clocks sampled
during the timed region, and a per-kernel breakdown.

--impl reference times the CPU oracle (the reference of this build) on a bounded sample of the
same workload on the host's cores and prints the same kind of line.
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

import workloads  # noqa: E402

METRIC = "tiled copy / round-trip / reduce-add HBM GB/s on 1 GB300 and % of HBM peak"
GB = 1e9
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e nominal bandwidth (about 8 TB/s), beside the measured peak
FLUSH_BYTES = 512 << 20
WORKLOAD = ("tmap hot path: W3 bf16 8192x8192 copy+roundtrip (128x64, 128B); W4 bf16 "
            "16x4095x1000 pitch 1024 rank-3 (1x64x64 128B, 1x64x32 64B) and rank-5 fallback view "
            "copy+roundtrip; W5a fp32 16384x16384 reduce-add (128x32, 128B); W5b bf16 "
            "8192x4096 + 4096x8192 4-stage ring")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="tmap", choices=["tmap", "reference"])
    p.add_argument("--e2e-steps", type=int, default=None,
                   help="steps of the end-to-end leg (default: --steps, the same K as the device "
                        "timing; 0 skips the leg)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--ops", default="", help="comma list of op names to run (default: all)")
    p.add_argument("--scale", type=float, default=1.0,
                   help="divide every workload's row count by this (small cases for profiling, "
                        "below 1 for larger ones)")
    p.add_argument("--ring-stages", type=int, default=4, help="stages of the W5b ring")
    p.add_argument("--gemm-stages", type=int, default=7, help="ring stages of the W7 GEMM")
    p.add_argument("--ring-swizzle", default="128", choices=["128", "none", "ungrouped"],
                   help="swizzle of the ring's tiles (none = the 8-way bank-conflict control; "
                        "ungrouped = 128B tiles read in the order of an ungrouped 256-byte row, "
                        "the 2-way control)")
    args = p.parse_args()
    if args.ring_swizzle == "ungrouped":
        os.environ["TM_RING_ROW_PAIRS"] = "1"  # read by the library at each ring call
    return args


def max_over_ranks(x: float, world: int) -> float:
    """The largest of every rank's x (the step time is the slowest rank's); the identity at N=1."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(step_bytes: int, step_ms: float, world: int) -> float:
    """Whole-job GB/s: every rank moves step_bytes per step; the step lasts the slowest rank's time."""
    return world * step_bytes / (step_ms * 1e-3) / GB


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


# ------------------------------------------------------------------------------------------------
# Workload: host arrays (numpy, the bytes both the GPU and the oracle see) and maps
# ------------------------------------------------------------------------------------------------
class HostWorkload:
    def __init__(self, scale: float = 1.0, ops=None, ring_span: int = 128):
        t0 = time.time()
        need = lambda prefix: ops is None or any(o.startswith(prefix) for o in ops)
        r3, r4, r5a, m5b = (int(8192 / scale), int(4095 / scale), int(16384 / scale),
                            int(8192 / scale))
        self.w3 = workloads.w3_tensor(r3, 8192) if need("w3") or need("w6") else None
        self.w4 = workloads.w4_tensor(rows=r4) if need("w4") or need("w6") else None
        self.w5a_dst, self.w5a_src = workloads.w5a_tensors(r5a) if need("w5a") else (None, None)
        self.w5b_a, self.w5b_b = workloads.w5b_tensors(m5b, 4096, m5b) if need("w5b") else (None, None)
        # widened reduce ops (not in the default step): bf16 add on its own tensors; s32 min and
        # f32 max over the W5a buffers
        # the ring in GEMM order with its tensor-core consumer (not in the default step)
        self.w7_a, self.w7_b = (workloads.w7_operands(int(8192 / scale), int(8192 / scale))
                                if ops is not None and need("w7") else (None, None))
        if ops is not None and need("w5c"):
            if self.w5a_dst is None:
                self.w5a_dst, self.w5a_src = workloads.w5a_tensors(r5a)
            self.w5c_dst = workloads.normal_bf16((r5a, 16384), 55)
            self.w5c_src = workloads.normal_bf16((r5a, 16384), 56)
            # bf16 add through the W4 rank-5 view (a 200-byte stride: the vector path)
            self.w5c_r5_dst = workloads.w4_tensor(rows=r4, seed=57)
            self.w5c_r5_src = workloads.w4_tensor(rows=r4, seed=58)
        else:
            self.w5c_dst = self.w5c_src = None
            self.w5c_r5_dst = self.w5c_r5_src = None
        self.gen_s = time.time() - t0
        self.r3 = workloads.w3_map(r3, 8192)
        self.r4_128 = workloads.w4_rank3_map(64, rows=r4, span=128)
        self.r4_64 = workloads.w4_rank3_map(32, rows=r4, span=64)
        self.r4_r5 = workloads.w4_rank5_map(rows=r4, span=128)
        self.r5a = workloads.w5a_map(r5a, 16384)
        self.r5b_a, self.r5b_b = workloads.w5b_maps(m5b, 4096, m5b, span=ring_span)
        self.r5c = dict(self.r5a, box=[64, 128], esize=2, strides=[self.r5a["dims"][0] * 2])
        # descriptor features over the W3 and W4 tensors: every other row, every other column,
        # NaN out-of-bounds fill
        self.r6_rows2 = workloads.w6_rows2_map(r3, 8192)
        self.r6_cols2 = workloads.w6_cols2_map(r3, 8192)
        self.r6_nan = dict(self.r4_128, nan=True)
        self.r6_box512 = dict(self.r3, box=[64, 4])  # 512-byte boxes, 128B swizzle


def box_count(r):
    n = 1
    for d, b in zip(r["dims"], r["box"]):
        n *= -(-d // b)
    return n


def box_bytes(r):
    """Image bytes: esize * prod(ceil(box / elementStrides))."""
    n = r["esize"]
    for i, b in enumerate(r["box"]):
        n *= -(-b // r.get("estrides", [1] * len(r["box"]))[i])
    return n


def inbounds_bytes(r):
    n = r["esize"]
    for d in r["dims"]:
        n *= d
    return n


def op_table(h: HostWorkload):
    """(name, algorithmic bytes) per op: bytes read + bytes written, counting in-bounds tensor bytes
    and whole images."""
    t = []
    for name, r in (("w3", h.r3), ("w4r3", h.r4_128), ("w4r3n", h.r4_64), ("w4r5", h.r4_r5)):
        img = box_count(r) * box_bytes(r)
        ten = inbounds_bytes(r)
        t.append((f"{name}.copy", ten + img))
        t.append((f"{name}.roundtrip", img + ten))
    t.append(("w5a.reduce", 3 * inbounds_bytes(h.r5a)))
    t.append(("w5b.ring", inbounds_bytes(h.r5b_a) + inbounds_bytes(h.r5b_b)))
    return t


# Widened ops, timed only when named with --ops: (name, algorithmic bytes per call).
#   w5c: reduces of other types and ops: dst read + src read + dst written (add_bf16_r5: through
#     the W4 rank-5 view, whose 200-byte stride puts it on the vector path).
#   w6.rows2: the image takes every other row: the taken rows are read, the images written.
#   w6.cols2: every other column (vector path: an innermost step above 1); the taken elements
#     are 4 bytes apart, so every 32-byte sector of the tensor holds some and the whole tensor is
#     read.
#   w6.cols2_rt: those images stored back: images read, every sector of the tensor written.
#   w6.nan: the W4 rank-3 copy with NaN out-of-bounds fill (bytes as w4r3.copy).
#   w6.box512: the W3 copy through 64 x 4 boxes (512-byte images, 128B swizzle; bytes as w3.copy).
#   w7.gemm: C = A * B^T on the tensor cores, A and B 8192 x 4096 bf16, C 8192 x 8192 fp32 (bytes:
#     A + B read once, C written; its figure of merit is TFLOP/s, 2 * M * N * K per call).
def gemm_flops(h: HostWorkload) -> int:
    return 2 * h.w7_a.shape[0] * h.w7_b.shape[0] * h.w7_a.shape[1] if h.w7_a is not None else 0


def extra_ops(h: HostWorkload):
    n = inbounds_bytes(h.r5a) // 4  # elements
    rows2_img = box_count(h.r6_rows2) * box_bytes(h.r6_rows2)
    cols2_img = box_count(h.r6_cols2) * box_bytes(h.r6_cols2)
    w3 = inbounds_bytes(h.r3)
    return [("w5c.add_bf16", 3 * 2 * n), ("w5c.min_s32", 3 * 4 * n), ("w5c.max_f32", 3 * 4 * n),
            ("w5c.add_bf16_r5", 3 * inbounds_bytes(h.r4_r5)),
            ("w6.rows2", 2 * rows2_img), ("w6.cols2", w3 + cols2_img),
            ("w6.cols2_rt", cols2_img + w3),
            ("w6.nan", inbounds_bytes(h.r6_nan) + box_count(h.r6_nan) * box_bytes(h.r6_nan)),
            ("w6.box512", w3 + box_count(h.r6_box512) * box_bytes(h.r6_box512))] + \
        ([("w7.gemm", h.w7_a.nbytes + h.w7_b.nbytes + 4 * h.w7_a.shape[0] * h.w7_b.shape[0])]
         if h.w7_a is not None else [])


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------
def bind_device(world: int, local: int):
    """The one device this process uses: cuda:LOCAL_RANK under torchrun (one rank per GPU), cuda:0
    alone.  Every buffer of the workload is allocated on it, and no rank touches another's."""
    import torch
    index = local if world > 1 else 0
    torch.cuda.set_device(index)
    return torch.device("cuda", index)


class GpuWorkload:
    def __init__(self, h: HostWorkload, stream, ring_stages: int = 4, gemm_stages: int = 7,
                 device=None, tm=None):
        import torch

        if tm is None:
            import async_bulk_tensor_tmap_gb300 as tm
        self.tm, self.torch, self.stream = tm, torch, stream
        self.device = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.ring_stages = ring_stages
        self.gemm_stages = gemm_stages
        on = self.device
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.uint8)).to(on)
        self.t = {k: dev(getattr(h, k)) for k in ("w3", "w4", "w5a_dst", "w5a_src", "w5b_a",
                                                  "w5b_b") if getattr(h, k) is not None}
        sw = {0: 0, 32: 1, 64: 2, 128: 3}

        def enc(dtype, buf, r):
            return tm.tmap_encode(dtype, buf, r["dims"], r["strides"], r["box"],
                                  element_strides=r.get("estrides"), swizzle=sw[r["span"]],
                                  oob=tm.TM_OOB_NAN if r.get("nan") else tm.TM_OOB_ZERO)

        bf, f32 = tm.TM_BF16, tm.TM_F32
        self.maps = {}
        if "w3" in self.t:
            self.t["w3_out"] = torch.empty_like(self.t["w3"])
            self.maps["w3"] = enc(bf, self.t["w3"], h.r3)
            self.maps["w3_out"] = enc(bf, self.t["w3_out"], h.r3)
        if "w4" in self.t:
            self.t["w4_out"] = self.t["w4"].clone()
            for k, r in (("w4r3", h.r4_128), ("w4r3n", h.r4_64), ("w4r5", h.r4_r5)):
                self.maps[k] = enc(bf, self.t["w4"], r)
                self.maps[f"{k}_out"] = enc(bf, self.t["w4_out"], r)
        if "w5a_dst" in self.t:
            self.maps["w5a_dst"] = enc(f32, self.t["w5a_dst"], h.r5a)
            self.maps["w5a_src"] = enc(f32, self.t["w5a_src"], h.r5a)
        if "w5b_a" in self.t:
            self.maps["w5b_a"] = enc(bf, self.t["w5b_a"], h.r5b_a)
            self.maps["w5b_b"] = enc(bf, self.t["w5b_b"], h.r5b_b)
            n = self.maps["w5b_a"].num_boxes
            self.t["cs_a"] = torch.zeros(n, dtype=torch.float32, device=on)
            self.t["cs_b"] = torch.zeros(n, dtype=torch.float32, device=on)
            self.t["bits_a"] = torch.zeros(n, dtype=torch.int64, device=on)
            self.t["bits_b"] = torch.zeros(n, dtype=torch.int64, device=on)
        if h.w7_a is not None:
            (M, K), N = h.w7_a.shape, h.w7_b.shape[0]
            self.t["w7_a"], self.t["w7_b"] = dev(h.w7_a), dev(h.w7_b)
            self.t["w7_c"] = torch.empty(M * N, dtype=torch.float32, device=on)
            self.maps["w7_a"] = tm.tmap_encode(bf, self.t["w7_a"], [K, M], [K * 2], [64, 128],
                                               swizzle=tm.TM_SWIZZLE_128B)
            self.maps["w7_b"] = tm.tmap_encode(bf, self.t["w7_b"], [K, N], [K * 2], [64, 256],
                                               swizzle=tm.TM_SWIZZLE_128B)
        if h.w5c_dst is not None:
            self.t["w5c_dst"], self.t["w5c_src"] = dev(h.w5c_dst), dev(h.w5c_src)
            self.maps["w5c_dst"] = enc(tm.TM_BF16, self.t["w5c_dst"], h.r5c)
            self.maps["w5c_src"] = enc(tm.TM_BF16, self.t["w5c_src"], h.r5c)
            self.t["w5c_r5_dst"], self.t["w5c_r5_src"] = dev(h.w5c_r5_dst), dev(h.w5c_r5_src)
            self.maps["w5c_r5_dst"] = enc(tm.TM_BF16, self.t["w5c_r5_dst"], h.r4_r5)
            self.maps["w5c_r5_src"] = enc(tm.TM_BF16, self.t["w5c_r5_src"], h.r4_r5)
            self.maps["w5a_dst_s32"] = enc(tm.TM_S32, self.t["w5a_dst"], h.r5a)
            self.maps["w5a_src_s32"] = enc(tm.TM_S32, self.t["w5a_src"], h.r5a)
        if "w3" in self.t and "w4" in self.t:
            self.maps["w6_rows2"] = enc(bf, self.t["w3"], h.r6_rows2)
            self.maps["w6_cols2"] = enc(bf, self.t["w3"], h.r6_cols2)
            self.maps["w6_cols2_out"] = enc(bf, self.t["w3_out"], h.r6_cols2)
            self.maps["w6_nan"] = enc(bf, self.t["w4"], h.r6_nan)
            self.maps["w6_box512"] = enc(bf, self.t["w3"], h.r6_box512)
        for k in ("w3", "w4r3", "w4r3n", "w4r5", "w6_rows2", "w6_cols2", "w6_nan", "w6_box512"):
            if k in self.maps:
                m = self.maps[k]
                self.t[f"{k}_img"] = torch.empty(m.num_boxes * m.box_bytes, dtype=torch.uint8,
                                                 device=on)
        self.flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=on)
        self.paths = {k: m.path for k, m in self.maps.items()}
        self.check_rank_local()

    def check_rank_local(self):
        """Every tensor of the workload lives on this process's device and every map describes
        one of them: a kernel of this rank is never given another GPU's memory (no peer
        operands; the ranks share nothing but the timing reduction)."""
        spans = []
        for k, t in self.t.items():
            if t.device != self.device:
                raise RuntimeError(f"buffer {k} is on {t.device}, not on this rank's {self.device}")
            spans.append((t.data_ptr(), t.data_ptr() + t.numel() * t.element_size()))
        for k, m in self.maps.items():
            if not any(lo <= m.base < hi for lo, hi in spans):
                raise RuntimeError(f"map {k} does not describe a buffer of this rank")

    def run_op(self, name, stream=None):
        tm, t, m = self.tm, self.t, self.maps
        s = self.stream if stream is None else stream
        base, kind = name.split(".")
        if kind == "copy":
            tm.tiled_copy(m[base], None, t[f"{base}_img"], s)
        elif kind == "roundtrip":
            tm.tiled_roundtrip(m[f"{base}_out"], None, t[f"{base}_img"], s)
        elif kind == "reduce":
            tm.tile_reduce_add(m["w5a_dst"], m["w5a_src"], s)
        elif kind == "add_bf16":
            tm.tile_reduce(m["w5c_dst"], m["w5c_src"], tm.TM_RED_ADD, s)
        elif kind == "add_bf16_r5":
            tm.tile_reduce(m["w5c_r5_dst"], m["w5c_r5_src"], tm.TM_RED_ADD, s)
        elif kind == "min_s32":
            tm.tile_reduce(m["w5a_dst_s32"], m["w5a_src_s32"], tm.TM_RED_MIN, s)
        elif kind == "max_f32":
            tm.tile_reduce(m["w5a_dst"], m["w5a_src"], tm.TM_RED_MAX, s)
        elif kind == "ring":
            tm.stream_tiles(m["w5b_a"], m["w5b_b"], self.ring_stages, t["cs_a"], t["cs_b"],
                            t["bits_a"], t["bits_b"], s)
        elif kind == "gemm":
            tm.stream_gemm(m["w7_a"], m["w7_b"], t["w7_c"], stages=self.gemm_stages, stream=s)
        elif kind in ("rows2", "cols2", "nan", "box512"):
            tm.tiled_copy(m[f"w6_{kind}"], None, t[f"w6_{kind}_img"], s)
        elif kind == "cols2_rt":
            tm.tiled_roundtrip(m["w6_cols2_out"], None, t["w6_cols2_img"], s)
        else:
            raise ValueError(f"unknown op {name}")

    def flush_l2(self):
        with self.torch.cuda.stream(self.stream):
            self.flush.fill_(1)


class ClockSampler:
    """nvidia-smi samples (every 100 ms) from the first warm-up step to the end of the timed
    steps."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu, self.rows, self.proc = gpu_index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in self.rows for n, v in zip(names, r[4:8]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


def time_steps(g: GpuWorkload, ops, steps, warmup):
    """Per-op device ms for each timed step (events on the launching stream)."""
    torch = g.torch
    t0, done = time.time(), 0
    while done < warmup or time.time() - t0 < 1.0:
        for name, _ in ops:
            g.flush_l2()
            g.run_op(name)
        done += 1
        if done >= warmup:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    rc = g.tm.tm_stream_check(g.stream)
    if rc != g.tm.TM_OK:
        raise RuntimeError(g.tm.tm_last_error())
    per = {name: [] for name, _ in ops}
    ev = []
    for _ in range(steps):
        for name, _ in ops:
            g.flush_l2()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(g.stream)
            g.run_op(name)
            e1.record(g.stream)
            ev.append((name, e0, e1))
    return per, ev


def collect(per, ev):
    for name, e0, e1 in ev:
        per[name].append(e0.elapsed_time(e1))
    return per


# End-to-end groups: the ops that share input tensors, the tensors copied in, the results read back.
E2E_GROUPS = (
    ("w3", ("w3",), ("w3_out",)),
    ("w4", ("w4",), ("w4_out",)),
    ("w5a", ("w5a_dst", "w5a_src"), ("w5a_dst",)),
    ("w5b", ("w5b_a", "w5b_b"), ("cs_a", "cs_b", "bits_a", "bits_b")),
)


# maps over each device buffer of the step (all start at the buffer's base)
E2E_MAPS = {
    "w3": ("w3",), "w3_out": ("w3_out",),
    "w4": ("w4r3", "w4r3n", "w4r5"), "w4_out": ("w4r3_out", "w4r3n_out", "w4r5_out"),
    "w5a_dst": ("w5a_dst",), "w5a_src": ("w5a_src",),
    "w5b_a": ("w5b_a",), "w5b_b": ("w5b_b",),
}


def e2e_run(g: GpuWorkload, h: HostWorkload, ops, steps, warmup=1):
    """Same step through the public API with HOST buffers: every step copies its inputs from
    pinned host memory and its results back, inside the timed region.  Three streams pipeline the
    work group by group (inputs of group k+1 go in while group k computes and group k-1's results
    come out).  Every input and result has two device buffers used by alternate steps (the maps
    over them moved with tmap_replace_address), so that a step's uploads wait only for the kernels
    (or read-out) of the step before last, and its kernels only for that step's read-out: the
    host link is the only thing that orders consecutive steps."""
    torch = g.torch
    names = [n for n, _ in ops]
    groups = [(gn, ins, outs, [n for n in names if n.split(".")[0].startswith(gn)])
              for gn, ins, outs in E2E_GROUPS]
    assert sum(len(x[3]) for x in groups) == len(names), "every op belongs to one group"
    groups = [x for x in groups if x[3]]
    src = {"w3": h.w3, "w4": h.w4, "w5a_dst": h.w5a_dst, "w5a_src": h.w5a_src,
           "w5b_a": h.w5b_a, "w5b_b": h.w5b_b}
    pin_in, pin_out = {}, {}
    for _, ins, outs, _ in groups:
        for k in ins:
            pin_in[k] = torch.empty_like(g.t[k], device="cpu").pin_memory()
            pin_in[k].copy_(torch.from_numpy(np.ascontiguousarray(src[k]).reshape(-1).view(np.uint8)))
        for k in outs:
            pin_out[k] = torch.empty_like(g.t[k], device="cpu").pin_memory()
    bi = sum(v.numel() * v.element_size() for v in pin_in.values())
    bo = sum(v.numel() * v.element_size() for v in pin_out.values())
    s_in, s_out, s_run = torch.cuda.Stream(), torch.cuda.Stream(), g.stream
    keys = {k for _, ins, outs, _ in groups for k in ins + outs}
    # the second buffer of a result starts as a copy of the first, so that bytes a round trip
    # does not write (padding) match on both
    bufs = {k: [g.t[k], g.t[k].clone()] for k in keys}
    free = {k: [None, None] for k in keys}  # the event after which buffer [par] may be rewritten
    nstep = [0]

    def use(k, par):
        g.t[k] = bufs[k][par]
        for mk in E2E_MAPS.get(k, ()):
            g.tm.tmap_replace_address(g.maps[mk], g.t[k])

    def step():
        par = nstep[0] & 1
        for gn, ins, outs, gops in groups:
            ev_in = torch.cuda.Event()
            with torch.cuda.stream(s_in):
                for k in ins:
                    if free[k][par] is not None:
                        s_in.wait_event(free[k][par])  # the step before last is done with it
                    bufs[k][par].copy_(pin_in[k], non_blocking=True)
                ev_in.record(s_in)
            for k in set(ins) | set(outs):
                use(k, par)
            s_run.wait_event(ev_in)
            for k in outs:
                if k not in ins and free[k][par] is not None:
                    s_run.wait_event(free[k][par])  # its result of the step before last is out
            for name in gops:
                g.run_op(name, s_run)
            ev_done = torch.cuda.Event()
            ev_done.record(s_run)
            ev_out = torch.cuda.Event()
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done)
                for k in outs:
                    pin_out[k].copy_(g.t[k], non_blocking=True)
                ev_out.record(s_out)
            for k in ins:
                free[k][par] = ev_out if k in outs else ev_done
            for k in outs:
                free[k][par] = ev_out
        nstep[0] += 1

    for _ in range(max(warmup, 1)):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_run)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for _ in range(steps):
        step()
    for st in (s_in, s_out):
        ev = torch.cuda.Event()
        ev.record(st)
        s_run.wait_event(ev)
    e1.record(s_run)
    torch.cuda.synchronize()
    if g.tm.tm_stream_check(g.stream) != g.tm.TM_OK:
        raise RuntimeError(g.tm.tm_last_error())
    e2e_verify(h, pin_out)
    return e0.elapsed_time(e1) / steps, bi, bo


def e2e_verify(h: HostWorkload, pin_out):
    """The results the end-to-end leg read back are right: the round trips restored their tensors
    byte for byte and the reduce destination holds dst + src (each step uploads dst afresh)."""
    for k, src in (("w3_out", h.w3), ("w4_out", h.w4)):
        if k in pin_out and not np.array_equal(pin_out[k].numpy(),
                                                np.ascontiguousarray(src).reshape(-1).view(np.uint8)):
            raise RuntimeError(f"end-to-end result {k} differs from its input")
    if "w5a_dst" in pin_out:
        got = pin_out["w5a_dst"].numpy().view(np.float32)
        want = (h.w5a_dst.reshape(-1) + h.w5a_src.reshape(-1)).astype(np.float32)
        if not np.array_equal(got.view(np.uint32), want.view(np.uint32)):
            raise RuntimeError("end-to-end reduce result differs from dst + src")


# ------------------------------------------------------------------------------------------------
# CPU arm: the oracle as it stands, on a bounded sample of the same workload
# ------------------------------------------------------------------------------------------------
def oracle_sample(h: HostWorkload, ops, fraction: float, threads: int):
    """Runs the oracle over the first `fraction` of the boxes of every op; returns (seconds,
    algorithmic bytes covered)."""
    import oracle

    def om(arr, r):
        fill = oracle.FILL_NAN_BF16 if r.get("nan") else oracle.FILL_ZERO
        return oracle.Map(arr, r["esize"], r["dims"], r["strides"], r["box"], r["span"],
                          estrides=r.get("estrides"), fill=fill)

    def sample(fn, r, nbytes):
        """fn(k): oracle work over the first k boxes of map r; returns the seconds it took."""
        n = box_count(r)
        k = max(1, int(n * fraction))
        return fn(k), nbytes * k // n

    def timed(f, *a, **kw):
        t0 = time.perf_counter()
        f(*a, **kw)
        return time.perf_counter() - t0

    spent, covered = 0.0, 0
    if not hasattr(h, "scratch3"):  # destinations of the sampled round trips, made once
        h.scratch3 = np.empty_like(h.w3) if h.w3 is not None else None
        h.scratch4 = h.w4.copy() if h.w4 is not None else None
    scratch3, scratch4 = h.scratch3, h.scratch4
    for name, nbytes in ops:
        base, kind = name.split(".")
        if base in ("w3", "w4r3", "w4r3n", "w4r5"):
            r = {"w3": h.r3, "w4r3": h.r4_128, "w4r3n": h.r4_64, "w4r5": h.r4_r5}[base]
            src = h.w3 if base == "w3" else h.w4
            dst = scratch3 if base == "w3" else scratch4
            n = box_count(r)
            k = max(1, int(n * fraction))
            imgs = np.empty(k * box_bytes(r), np.uint8)
            if kind == "copy":
                t0 = time.perf_counter()
                oracle.tiled_copy(om(src, r), threads=threads, b0=0, b1=k, out=imgs, nbox=k)
                spent += time.perf_counter() - t0
            else:
                oracle.tiled_copy(om(src, r), threads=threads, b0=0, b1=k, out=imgs, nbox=k)
                t0 = time.perf_counter()
                oracle.tiled_roundtrip(om(dst, r), imgs, threads=threads, b0=0, b1=k)
                spent += time.perf_counter() - t0
            covered += nbytes * k // n
        elif kind == "reduce":
            n = box_count(h.r5a)
            k = max(1, int(n * fraction))
            d = h.w5a_dst  # the oracle adds in place into the host copy (a sample of boxes)
            t0 = time.perf_counter()
            oracle.tile_reduce_add(om(d, h.r5a), om(h.w5a_src, h.r5a), threads=threads, b0=0, b1=k)
            spent += time.perf_counter() - t0
            covered += nbytes * k // n
        elif base == "w5c":
            if kind == "add_bf16":
                d, sr, r, ty, op = h.w5c_dst, h.w5c_src, h.r5c, oracle.BF16, oracle.ADD
            elif kind == "add_bf16_r5":
                d, sr, r, ty, op = h.w5c_r5_dst, h.w5c_r5_src, h.r4_r5, oracle.BF16, oracle.ADD
            else:
                d, sr, r = h.w5a_dst, h.w5a_src, h.r5a
                ty, op = (oracle.S32, oracle.MIN) if kind == "min_s32" else (oracle.F32, oracle.MAX)
            sec, cov = sample(lambda k: timed(oracle.tile_reduce, om(d, r), om(sr, r), ty, op,
                                              threads=threads, b0=0, b1=k), r, nbytes)
            spent, covered = spent + sec, covered + cov
        elif base == "w6":
            r = {"rows2": h.r6_rows2, "nan": h.r6_nan, "box512": h.r6_box512}.get(kind, h.r6_cols2)
            src = h.w4 if kind == "nan" else h.w3

            def run(k):
                imgs = np.empty(k * box_bytes(r), np.uint8)
                sec = timed(oracle.tiled_copy, om(src, r), threads=threads, b0=0, b1=k, out=imgs,
                            nbox=k)
                if kind == "cols2_rt":
                    sec = timed(oracle.tiled_roundtrip, om(scratch3, r), imgs, threads=threads,
                                b0=0, b1=k)
                return sec
            sec, cov = sample(run, r, nbytes)
            spent, covered = spent + sec, covered + cov
        elif kind == "gemm":
            rows = h.w7_a.shape[0]
            k = max(1, int(rows * fraction))
            t0 = time.perf_counter()
            oracle_gemm_rows(h.w7_a, h.w7_b, k, threads)
            spent += time.perf_counter() - t0
            covered += nbytes * k // rows
        elif kind == "ring":
            n = box_count(h.r5b_a)
            k = max(1, int(n * fraction))
            t0 = time.perf_counter()
            oracle.stream_checksums(om(h.w5b_a, h.r5b_a), om(h.w5b_b, h.r5b_b), threads=threads,
                                    t0=0, t1=k)
            spent += time.perf_counter() - t0
            covered += nbytes * k // n
    return spent, covered


def oracle_gemm_rows(a, b, rows: int, threads: int):
    """The oracle's C = A * B^T for the first `rows` rows of A, rows split over threads (ctypes
    releases the GIL)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    step = -(-rows // threads)
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda r0: oracle.gemm(a, b, r0, min(rows, r0 + step)),
                    range(0, rows, step)))


def calibrated_fraction(h: HostWorkload, ops, threads: int, target_s: float) -> float:
    """Fraction of every op's boxes that keeps one oracle sample near `target_s` seconds."""
    frac = 0.005
    oracle_sample(h, ops, frac, threads)
    spent, _ = oracle_sample(h, ops, frac, threads)
    return min(1.0, frac * target_s / max(spent, 1e-3))


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------------------------------------
def measured_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def measured_bf16_peak():
    """Dense bf16 TFLOP/s of a cuBLAS GEMM timed alone (burst) on the GB300s."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def tma_kernel_source() -> bytes:
    """What defines the tensor-map streaming kernels: k_tma.cu, tm_ptx.cuh and, of tm_internal.h,
    everything from the BoxWalk struct to the end of stream_plan (the arguments, the work split,
    the default L2 policies and the launch shape).  Comments, blank lines and trailing blanks are
    left out, so that only a change of the code itself makes the recorded counters stale (none of
    these files holds "//" or "/*" inside a string)."""
    import re
    csrc = os.path.join(ROOT, "async_bulk_tensor_tmap_gb300", "csrc")
    out = b""
    for f in ("k_tma.cu", "tm_ptx.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            out += fh.read()
    with open(os.path.join(csrc, "tm_internal.h"), "rb") as fh:
        hdr = fh.read()
    i = hdr.index(b"struct BoxWalk")
    j = hdr.index(b"\n}\n", hdr.index(b"inline void stream_plan(")) + 3
    code = re.sub(rb"/\*.*?\*/", b"", out + hdr[i:j], flags=re.S)
    lines = (re.sub(rb"//.*", b"", ln).rstrip() for ln in code.split(b"\n"))
    return b"\n".join(ln for ln in lines if ln)


def recorded_traffic(kernel: str):
    """Per-launch DRAM traffic of `kernel` from profiles/roofline_traffic.txt, or None when the
    kernel's source changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "roofline_traffic.txt")
    try:
        fields = dict(ln.split(":", 1) for ln in open(path) if ":" in ln and not ln.startswith("#"))
    except OSError:
        return None
    fields = {k.strip(): v.strip() for k, v in fields.items()}
    h = hashlib.sha256()
    h.update(tma_kernel_source())
    if fields.get("kernel") != kernel or fields.get("source_sha256") != h.hexdigest():
        return None
    return int(fields["traffic_bytes"])


def select_ops(h, spec):
    ops = op_table(h)
    if spec:
        keep = set(spec.split(","))
        ops = [o for o in ops + extra_ops(h) if o[0] in keep]
    return ops


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    h = HostWorkload(args.scale, args.ops.split(",") if args.ops else None,
                     0 if args.ring_swizzle == "none" else 128)
    ops = select_ops(h, args.ops)
    cores = cpu_cores()
    frac = calibrated_fraction(h, ops, cores, target_s=2.0)
    for _ in range(args.warmup):
        oracle_sample(h, ops, frac / 4, cores)
    spent, covered = 0.0, 0
    for _ in range(args.steps):
        s, c = oracle_sample(h, ops, frac, cores)
        spent += s
        covered += c
    value = covered / spent / GB
    sample = (f"first {frac:.2%} of the boxes of every op per step "
              f"({covered // max(args.steps, 1)} algorithmic bytes)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": spent / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    rank, world, local = dist_env()
    device = bind_device(world, local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    h = HostWorkload(args.scale, args.ops.split(",") if args.ops else None,
                     0 if args.ring_swizzle == "none" else 128)
    ops = select_ops(h, args.ops)
    stream = torch.cuda.Stream()
    g = GpuWorkload(h, stream, args.ring_stages, args.gemm_stages, device=device)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    barrier()
    with ClockSampler(local) as clk:
        per, ev = time_steps(g, ops, args.steps, args.warmup)
        torch.cuda.synchronize()
    per = collect(per, ev)
    barrier()
    rc = g.tm.tm_stream_check(stream)
    if rc != g.tm.TM_OK:
        raise RuntimeError(g.tm.tm_last_error())
    step_ms = max_over_ranks(sum(sum(v) for v in per.values()) / args.steps, world)
    step_bytes = sum(b for _, b in ops)
    value = weak_scaling_value(step_bytes, step_ms, world)
    peak, peak_kind = measured_hbm_peak()
    breakdown = {}
    tpeak, tpeak_kind = measured_bf16_peak()
    for name, nbytes in ops:
        ms = statistics.mean(per[name])
        breakdown[name] = {"ms": round(ms, 4), "ms_median": round(statistics.median(per[name]), 4),
                           "ms_best": round(min(per[name]), 4),
                           "GB/s": round(nbytes / ms / 1e6, 1),
                           "frac_of_peak": round(nbytes / ms / 1e6 / peak, 3),
                           "frac_of_nominal": round(nbytes / ms / 1e6 / NOMINAL_HBM_GBS, 3),
                           "bytes": nbytes}
        if name == "w7.gemm":
            tflops = gemm_flops(h) / ms / 1e9
            breakdown[name].update({"TFLOP/s": round(tflops, 1),
                                    "frac_of_bf16_peak": round(tflops / tpeak, 3)})
    dom = max(ops, key=lambda o: statistics.mean(per[o[0]]))
    dom_name, dom_bytes = dom
    dom_ms = statistics.mean(per[dom_name])
    achieved = dom_bytes / dom_ms / 1e6
    roofline = {"kernel": dom_name, "bound": "hbm", "achieved": achieved, "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                "traffic": recorded_traffic(dom_name) if args.scale == 1 else None}
    if dom_name == "w7.gemm":  # a dense contraction: against the measured bf16 tensor peak
        tflops = gemm_flops(h) / dom_ms / 1e9
        roofline = {"kernel": dom_name, "bound": "tensor", "achieved": tflops, "peak": tpeak,
                    "peak_kind": tpeak_kind, "unit": "TFLOP/s", "frac": tflops / tpeak,
                    "traffic": None}
    if any(n.startswith(("w5c", "w6", "w7")) for n, _ in ops):
        args.e2e_steps = 0  # the widened ops have no end-to-end leg
    if args.e2e_steps is None:
        args.e2e_steps = args.steps
    if args.e2e_steps > 0:
        e2e_ms, bi, bo = e2e_run(g, h, ops, args.e2e_steps, args.warmup)
        e2e_ms = max_over_ranks(e2e_ms, world)  # the whole job lasts as long as its slowest rank
        e2e = {"value": world * step_bytes / (e2e_ms * 1e-3) / GB, "unit": "GB/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo}
    else:
        e2e = None
    if rank != 0:
        return
    if args.scale != 1 or world > 1:
        args.no_cpu_baseline = True  # the oracle is timed at N = 1 on the full-size workload only
    cpu = None
    if not args.no_cpu_baseline:
        cores = cpu_cores()
        frac = calibrated_fraction(h, ops, cores, target_s=2.0)
        spent, covered = oracle_sample(h, ops, frac, cores)
        cpu = None if covered == 0 else {"value": covered / spent / GB, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"first {frac:.2%} of the boxes of every op ({covered} algorithmic "
                         f"bytes, {spent:.1f} s on {cores} threads)"}
        if cpu is not None:  # the same oracle on one thread, beside the box-parallel figure
            frac1 = calibrated_fraction(h, ops, 1, target_s=1.5)
            spent1, covered1 = oracle_sample(h, ops, frac1, 1)
            if covered1:
                cpu["single_thread"] = {
                    "value": covered1 / spent1 / GB, "cores": 1,
                    "sample": f"first {frac1:.3%} of the boxes of every op ({covered1} algorithmic "
                              f"bytes, {spent1:.1f} s on 1 thread)"}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "step_bytes": step_bytes,
                   "l2": "flushed by a 512 MiB device write before every kernel (not timed)",
                   "hbm_frac_of_peak": round(value / world / peak, 3),
                   "hbm_frac_of_nominal": round(value / world / NOMINAL_HBM_GBS, 3),
                   "paths": {k: ("tma" if p == 1 else "fallback") for k, p in g.paths.items()
                             if not k.endswith("_out")}},
        "roofline": roofline,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "gpu_launches": len(ops) * args.steps,
        "clocks": clk.summary(),
        "breakdown": breakdown,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
