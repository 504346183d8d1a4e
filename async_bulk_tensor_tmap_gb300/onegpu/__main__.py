"""Times stream_gemm_multicast against the library's stream_gemm (CTA-pair form and one-SM form)
on one GPU: C = A * B^T, bf16 in, fp32 out, each call after a 512 MiB L2 flush, CUDA events on the
launching stream, median of the timed calls.

    python -m async_bulk_tensor_tmap_gb300.onegpu [M N K] [--reps R]
"""
import argparse
import json
import os
import statistics

import numpy as np
import torch

import async_bulk_tensor_tmap_gb300 as tm
from async_bulk_tensor_tmap_gb300 import onegpu


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("shape", nargs="*", type=int, default=[8192, 8192, 4096])
    ap.add_argument("--reps", type=int, default=10)
    args = ap.parse_args()
    M, N, K = args.shape
    torch.cuda.set_device(0)
    g = torch.Generator(device="cpu").manual_seed(7)
    a = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    b = torch.randn(N, K, generator=g).to(torch.bfloat16).cuda()
    c = torch.empty(M, N, dtype=torch.float32, device="cuda")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    sw = tm.TM_SWIZZLE_128B
    ma = tm.tmap_encode(tm.TM_BF16, a, [K, M], [K * 2], [64, 128], swizzle=sw)
    mb = tm.tmap_encode(tm.TM_BF16, b, [K, N], [K * 2], [64, 256], swizzle=sw)
    mbh = tm.tmap_encode(tm.TM_BF16, b, [K, N], [K * 2], [64, 128], swizzle=sw)
    forms = {
        "multicast (one-SM CTAs, B shared by a cluster of two)":
            lambda: onegpu.stream_gemm_multicast(ma, mbh, c, stages=4),
        "library stream_gemm, CTA pairs (default)": lambda: tm.stream_gemm(ma, mb, c, stages=7),
        "library stream_gemm, one SM per tile (TM_GEMM_PAIR=0)": lambda: tm.stream_gemm(ma, mb, c, stages=4),
    }
    out = {}
    for name, fn in forms.items():
        os.environ["TM_GEMM_PAIR"] = "0" if "one SM" in name else "1"
        ms = []
        for i in range(args.reps + 3):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if i >= 3:
                ms.append(e0.elapsed_time(e1))
        assert onegpu.tm_onegpu_check() == tm.TM_OK, onegpu.last_error()
        assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()
        med = statistics.median(ms)
        out[name] = {"ms": round(med, 4), "TFLOP/s": round(2 * M * N * K / med / 1e9, 1)}
        print(f"{name:56s} {med * 1e3:8.1f} us  {2 * M * N * K / med / 1e9:7.1f} TFLOP/s", flush=True)
    os.environ.pop("TM_GEMM_PAIR", None)
    # the three forms agree within the fp32 summation bound on a sample of rows
    ref = (a[:64].float() @ b.float().T)
    onegpu.stream_gemm_multicast(ma, mbh, c, stages=4)
    torch.cuda.synchronize()
    bound = K * 2.0 ** -23 * (a[:64].float().abs() @ b.float().abs().T)
    assert bool(((c[:64] - ref).abs() <= bound + 1e-30).all())
    print(json.dumps({"shape": [M, N, K], "forms": out}))


if __name__ == "__main__":
    main()
