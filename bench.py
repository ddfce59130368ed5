"""Benchmark of the CSA2 global-attention decode step on GB300.

Workload: one 38-layer CSA2 decode step (encoder layers 2..19 at m=2 with Full
layers 2/8/14, decoder layers 20..39 at m=1 with Full layer 20 and Reindex
layers 24/28/32/36), batch 8 with context lengths {32K, 256K, 1M, 1M} x 2, four
resident main-KV / index-K cache copies, per-layer q, w, SWA and sink drawn
independently.  A step = the Full layers' entry build, Lightning-Indexer scan,
top-512 (+ candidate pool at layer 20), the Reindex layers' pool rescoring and
top-512, and sparse attention in all 38 layers.

Metric: indexer keys scored per second (every visible entry of the Full layers
plus the 16,384 pool candidates of each Reindex row); sparse-attention
query-layers per second is reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: W eager warm-up steps, then K steps captured in one CUDA graph and
replayed once between two device synchronisations (max over ranks).  Every
step streams ~1.6 GB of index-K cache, far above the 129 MB L2, so no L2
flush is inserted.  CUDA events recorded inside the graph (on a side branch,
so that the kernels keep their programmatic-launch overlap) around each
indexer-scan launch give the dominant kernel's duration for the roofline.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "indexer keys scored/s + sparse-attn queries/s at 1M ctx; % of GB300 roofline"
LENGTHS = [32768, 262144, 1 << 20, 1 << 20] * 2
WORKLOAD = "csa2-decode-38layer-b8-ctx{32K,256K,1M,1M}x2"
INDEX_KEY_BYTES = 132   # 128 e4m3 codes + one fp32 scale per key
# one attention row (query-layer): q 64 x 512 bf16, 128 SWA records of 528 B,
# 512 main-KV entries of 272 B (256 B codes + 16 scales), bf16 output, slots
ATTN_ROW_BYTES = 65536 + 128 * 528 + 512 * 272 + 65536 + 640 * 4
ATTN_ROW_FLOP = 2 * 2 * 64 * 640 * 512   # S = q K^T and O = P V


def _scan_traffic_per_key():
    """DRAM bytes per key of the decode scan from the committed ncu capture
    (profiles/index_scan_decode_b8x262k.md), or None when the kernel source has
    changed since that capture was taken."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "serving_lightning_indexer_gb300", "csrc")
    src = b"".join(open(os.path.join(csrc, f), "rb").read() for f in ("index_score.cu", "csa2_device.cuh"))
    digest = hashlib.sha256(src).hexdigest()[:16]
    try:
        text = open(os.path.join(ROOT, "profiles", "index_scan_decode_b8x262k.md")).read()
    except OSError:
        return None
    per_key = re.search(r"dram_bytes_per_key:\s*([0-9.]+)", text)
    sha = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    if not per_key or not sha or sha.group(1) != digest:
        return None
    return float(per_key.group(1))


def max_over_ranks(value: float, device) -> float:
    """The largest of a per-rank value over all ranks of the process group
    (the value itself when there is none or it has one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step: float, steps: int, world: int, ms_max: float) -> float:
    """Units per second of the whole job: every rank processes units_per_rank_step
    each step (weak scaling), over the slowest rank's time."""
    return units_per_rank_step * steps * world / (ms_max / 1e3)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        return 1700.0


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        time.sleep(0.1)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        inside = [r for r in rows if self.t0 and self.t1 and self.t0 <= r[0] <= self.t1]
        if not inside:   # region shorter than the sampling period: nearest samples
            mid = (self.t0 + self.t1) / 2 if self.t0 and self.t1 else rows[-1][0]
            inside = sorted(rows, key=lambda r: abs(r[0] - mid))[:3]
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names[1:], r[3][1:]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


def cpu_baseline(step, budget_s: float, device_copy):
    """The oracle, as it stands, on a bounded sample of the same workload:
    decoder Full-layer rows (score every visible entry, top-512, pool) until the
    time budget is spent.  Returns keys/s, threads used and the sample."""
    from oracle import csa2_oracle as o
    c = step.caches[3]
    li = step.inputs[20]
    cache, pt = device_copy(c.pc.index_k), device_copy(c.pc.page_table)
    q8, qs, w = device_copy(li.iq.q_fp8), device_copy(li.iq.q_scale), device_copy(li.iq.w)
    keys = 0
    rows = 0
    t0 = time.perf_counter()
    chunk = 131072
    b = 0
    while time.perf_counter() - t0 < budget_s and rows < 64:
        n = min(c.entries[b], chunk)
        s = o.index_scores_row(q8[b], qs[b], w[b], cache, pt[b], n)
        o.topk_positions(s, 512)
        o.candidate_pool(o.block_maxima(s, n), 2048)
        keys += n
        rows += 1
        b = (b + 1) % len(c.entries)
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return keys / dt, cores, f"{rows} decoder Full-layer row prefixes of {chunk} entries: score + top-512 + pool"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    import torch

    if args.impl == "reference":
        return reference_arm(args, rank, world)

    import __graft_entry__
    __graft_entry__.build()
    from serving_lightning_indexer_gb300 import csa2
    from serving_lightning_indexer_gb300.decode_step import DecodeStep

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    step = DecodeStep(LENGTHS, seed=4 + rank, device=dev)
    keys_per_step = step.keys_scored_per_step()
    attn_per_step = step.attn_query_layers_per_step()
    scan_bytes_per_step = step.index_bytes_per_step()
    stream = torch.cuda.Stream(device=dev)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step.run(stream)
    stream.synchronize()
    rc = csa2.check_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device error status {rc} during warm-up")

    # ---- K steps in one graph, events around every indexer scan.  The timing
    # events are recorded on a side stream that forks from the step's stream,
    # so they hang off the kernel chain instead of sitting between two kernels
    # (a node between them would cut the programmatic-launch overlap).
    K = args.steps
    ev_pairs = []
    side = torch.cuda.Stream(device=dev)

    def side_event():
        fork = torch.cuda.Event()
        fork.record(stream)
        side.wait_event(fork)
        e = torch.cuda.Event(enable_timing=True, external=True)  # an event node inside the graph
        e.record(side)
        return e

    def on_scan(layer):
        ev_pairs.append([layer, side_event(), None])

    def after_scan(layer):
        ev_pairs[-1][2] = side_event()

    attn_pairs = []

    def on_attn(layer):
        attn_pairs.append([side_event(), None])

    def after_attn(layer):
        attn_pairs[-1][1] = side_event()

    g = torch.cuda.CUDAGraph()
    step.on_index_score, step.after_index_score = on_scan, after_scan
    step.on_attn, step.after_attn = on_attn, after_attn
    with torch.cuda.graph(g, stream=stream):
        for _ in range(K):
            step.run(stream)
        join = torch.cuda.Event()
        join.record(side)
        stream.wait_event(join)
    step.on_index_score = step.after_index_score = None
    step.on_attn = step.after_attn = None
    with torch.cuda.stream(stream):
        g.replay()                   # untimed: first replay of the instantiated graph
    stream.synchronize()

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler.mark(True)
    with torch.cuda.stream(stream):  # the graph replays on the current stream
        t_start.record(stream)
        g.replay()
        t_end.record(stream)
    stream.synchronize()
    sampler.mark(False)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms_total = t_start.elapsed_time(t_end)
    if rank == 0:
        sampler.stop()
    rc = csa2.check_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device error status {rc} in the timed region")
    scan_ms = [a.elapsed_time(b) for _, a, b in ev_pairs]
    per_layer = {}
    for (l, _, _), ms in zip(ev_pairs, scan_ms):
        per_layer.setdefault(l, []).append(ms)
    scan_ms_total = sum(scan_ms)
    attn_ms = [a.elapsed_time(b) for a, b in attn_pairs]
    ms_total = max_over_ranks(ms_total, dev)

    # ---- end to end: pinned host inputs -> device, step, outputs -> pinned host.
    # Every step copies all of its query-side inputs in and all 38 attention
    # outputs out.  The copies run on two copy streams: layer l waits only for
    # its own inputs, and its output is read back while later layers compute;
    # the next step starts after the last read-back.
    in_by_layer, h2d, host_out = {}, 0, {}
    for l in step.layers:
        li = step.inputs[l]
        ts = [li.attn.q]
        if li.iq is not None:
            ts += [li.iq.q_fp8, li.iq.q_scale, li.iq.w]
        if li.C is not None:
            ts += [li.C] + ([li.Z] if li.Z is not None else [])
        in_by_layer[l] = [(t.detach().cpu().pin_memory(), t) for t in ts]
        h2d += sum(t.numel() * t.element_size() for t in ts)
        host_out[l] = step.buf.out[l].detach().cpu().pin_memory()
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    cp_in = torch.cuda.Stream(device=dev)
    cp_out = torch.cuda.Stream(device=dev)
    Ke = max(1, min(K, 20))
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        for _ in range(Ke):
            begin = torch.cuda.Event()
            begin.record(stream)
            cp_in.wait_event(begin)
            ready = {}
            with torch.cuda.stream(cp_in):
                for l in step.layers:
                    for h, d in in_by_layer[l]:
                        d.copy_(h, non_blocking=True)
                    ready[l] = torch.cuda.Event()
                    ready[l].record(cp_in)

            def before(l, ready=ready):
                stream.wait_event(ready[l])

            def after(l):
                done = torch.cuda.Event()
                done.record(stream)
                cp_out.wait_event(done)
                with torch.cuda.stream(cp_out):
                    host_out[l].copy_(step.buf.out[l], non_blocking=True)

            step.before_layer, step.after_layer = before, after
            step.run(stream)
            finished = torch.cuda.Event()
            finished.record(cp_out)
            stream.wait_event(finished)
        step.before_layer = step.after_layer = None
    with torch.cuda.stream(stream):
        g2.replay()
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        g2.replay()
        e1.record(stream)
    stream.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, dev)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = _peaks()
    bf16_peak = _bf16_peak()
    traffic_per_key = _scan_traffic_per_key()
    ms_per_step = ms_total / K
    value = whole_job_rate(keys_per_step, K, world, ms_total)
    scan_launches = len(scan_ms)
    scan_bytes_per_launch = scan_bytes_per_step * K / scan_launches
    achieved = scan_bytes_per_step * K / (scan_ms_total / 1e3) / 1e9
    # our kernels launched per step: a Full layer runs compress, the scan and the
    # two select passes (filter, final); a Reindex layer the pool gather and the
    # final select; every layer one clustered attention launch (the histogram
    # memsets are not kernels)
    from serving_lightning_indexer_gb300 import decode_step as ds
    n_full = sum(1 for l in step.layers if ds.role_of(l) == "full")
    n_reidx = sum(1 for l in step.layers if ds.role_of(l) == "reindex")
    launches_per_step = n_full * 4 + n_reidx * 2 + len(step.layers)
    cpu = None
    if not args.no_cpu_baseline:
        v, cores, sample = cpu_baseline(step, args.cpu_budget, lambda t: t.detach().cpu().numpy())
        cpu = {"value": v, "unit": "keys/s", "cores": cores, "kind": "oracle", "sample": sample}
    out = {
        "metric": METRIC, "value": value, "unit": "keys/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 (indexer, fp32 accumulate) + bf16 (attention)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": len(LENGTHS), "context_lengths": LENGTHS, "layers": 38,
                   "keys_scored_per_step": keys_per_step, "attn_query_layers_per_step": attn_per_step,
                   "timing": "K steps in one CUDA graph; inputs larger than L2 (no flush)",
                   "parallelism": f"replicas x{world}"},
        "attn_query_layers_per_s": whole_job_rate(attn_per_step, K, world, ms_total),
        "roofline": {"bound": "hbm", "kernel": "index_tiles_kernel<1,scan> (decode Lightning-Indexer scan)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_kind,
                     "traffic": (None if traffic_per_key is None
                                 else traffic_per_key * scan_bytes_per_launch / INDEX_KEY_BYTES),
                     "traffic_source": "ncu dram bytes per key of the committed scan capture, scaled to the "
                                       "keys of an average launch",
                     "algorithmic_bytes_per_launch": scan_bytes_per_launch,
                     "avg_launch_ms": scan_ms_total / scan_launches, "launches_timed": scan_launches,
                     "per_layer_ms": {str(l): statistics.mean(v) for l, v in per_layer.items()}},
        # the sparse attention, the step's largest time share: latency-bound at
        # 8 rows a launch, reported beside the scan against both rooflines
        "roofline_attention": {
            "bound": "latency", "kernel": "sparse_attn_tc_kernel (8 rows x 64 heads x 640 keys)",
            "avg_launch_ms": statistics.mean(attn_ms), "launches_timed": len(attn_ms),
            "share_of_step": sum(attn_ms) / ms_total,
            "algorithmic_bytes_per_launch": ATTN_ROW_BYTES * len(LENGTHS),
            "hbm_frac": ATTN_ROW_BYTES * len(LENGTHS) / (statistics.mean(attn_ms) / 1e3) / 1e9 / peak,
            "flop_per_launch": ATTN_ROW_FLOP * len(LENGTHS),
            "bf16_tensor_frac": ATTN_ROW_FLOP * len(LENGTHS) / (statistics.mean(attn_ms) / 1e3) / 1e12 / bf16_peak,
            "peaks": {"hbm_gbs": peak, "bf16_tflops": bf16_peak, "source": peak_kind}},
        "cpu_baseline": cpu,
        "e2e": {"value": whole_job_rate(keys_per_step, Ke, world, e2e_ms), "unit": "keys/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": Ke},
        "gpu_launches": launches_per_step * K,
        "clocks": sampler.summary(),
    }
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def reference_arm(args, rank, world):
    """The oracle, as it stands, on the host cores: each step scores a bounded
    sample of the workload (one decoder Full-layer row prefix of 131072 entries,
    with its top-512 and pool)."""
    if rank != 0:
        return
    import torch

    from oracle import csa2_oracle as o
    from serving_lightning_indexer_gb300 import workloads as W
    n = 131072
    pc = W.make_paged_cache([n] * 2, seed=4, device="cpu")
    iq = W.make_indexer_query(2, seed=5, device="cpu")
    cache, pt = pc.index_k.numpy(), pc.page_table.numpy()

    def one(b):
        s = o.index_scores_row(iq.q_fp8[b].numpy(), iq.q_scale[b].numpy(), iq.w[b].numpy(), cache, pt[b], n)
        o.topk_positions(s, 512)
        o.candidate_pool(o.block_maxima(s, n), 2048)

    for i in range(args.warmup):
        one(i % 2)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i % 2)
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    v = n * args.steps / dt
    sample = f"per step one decoder Full-layer row prefix of {n} entries: score + top-512 + pool"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "keys/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_entries_per_step": n},
        "cpu_baseline": {"value": v, "unit": "keys/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "keys/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


if __name__ == "__main__":
    main()
