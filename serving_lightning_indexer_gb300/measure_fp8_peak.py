"""Dense FP8 (e4m3) tensor-core throughput of this GPU, measured with cuBLASLt
through torch._scaled_mm on 8192^3 (2*N^3 flop): best of 10 (burst) and a
4-second back-to-back loop (sustained).  Prints one JSON line.

  python -m serving_lightning_indexer_gb300.measure_fp8_peak
"""
from __future__ import annotations

import json
import time

import torch


def main():
    n = 8192
    dev = torch.device("cuda:0")
    a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()   # column-major operand
    one = torch.tensor(1.0, device=dev)

    def mm():
        return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

    for _ in range(3):
        mm()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mm()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    flop = 2.0 * n ** 3
    t_end = time.time() + 4.0
    iters = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    while time.time() < t_end:
        for _ in range(20):
            mm()
        iters += 20
        torch.cuda.synchronize()
    e1.record()
    torch.cuda.synchronize()
    sustained = flop * iters / (e0.elapsed_time(e1) / 1e3) / 1e12
    print(json.dumps({"fp8_e4m3_tflops": flop / (best / 1e3) / 1e12, "fp8_e4m3_tflops_sustained": sustained,
                      "how": "torch._scaled_mm e4m3 8192^3, bf16 out: best of 10, and back to back for 4 s",
                      "gpu": torch.cuda.get_device_name(dev), "torch": torch.__version__}), flush=True)


if __name__ == "__main__":
    main()
