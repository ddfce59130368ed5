"""Benchmark of the CSA2 global-attention step on GB300.

Headline workload: one 38-layer CSA2 decode step (encoder layers 2..19 at m=2
with Full layers 2/8/14, decoder layers 20..39 at m=1 with Full layer 20 and
Reindex layers 24/28/32/36), batch 8 with context lengths {32K, 256K, 1M, 1M}
x 2, four resident main-KV / index-K cache copies, per-layer q, w, SWA and sink
drawn independently.  A step = the Full layers' entry build, Lightning-Indexer
scan, top-512 (+ candidate pool at layer 20), the Reindex layers' pool
rescoring and top-512, and sparse attention in all 38 layers.

Metric: indexer keys scored per second (every visible entry of the Full layers
plus the 16,384 pool candidates of each Reindex row); sparse-attention
query-layers per second is reported beside it.  The same run also measures
  * the 4096-query prefill chunk after a 256K-token prefix (m = 2): entry
    build, the prefill indexer GEMM (roofline against the FP8 tensor peak),
    top-512 of every query and sparse attention of the 4096 queries;
  * the decode Reindex at 1M context (batch 16, 16,384 pool candidates per
    row, 10 % planted blocks) and the attention of its four layers.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --case scan|topk|reindex|attn|prefill|prefill_chunk|project [--iters N]   (for profilers)

Timing: W eager warm-up steps, then K steps captured in one CUDA graph; the
graph is replayed (each replay timed with CUDA events between two device
synchronisations) until at least --min-seconds have passed, and the median
replay gives the step time (max over ranks).  Every step streams ~1.6 GB of
index-K cache, far above the 129 MB L2, so no L2 flush is inserted.  CUDA
events recorded inside the graph (on a side branch, so that the kernels keep
their programmatic-launch overlap) around each indexer scan and attention
launch give those kernels' durations for the rooflines.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import tempfile
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
INDEX_PAIR_FLOP = 2 * 32 * 128           # one (query, entry) pair of the indexer: 32 heads x 128 dims
# prefill chunk: 4096 new tokens after a 256K-token prefix, m = 2
PREFILL_PREFIX, PREFILL_T, PREFILL_M = 1 << 18, 4096, 2
# decode Reindex: batch 16 at 1M context, 2048-block x 8 pools
REINDEX_B, REINDEX_N = 16, 1 << 20
REINDEX_POOLS = 6


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
    """(HBM GB/s, bf16 burst TFLOP/s, bf16 sustained TFLOP/s, source)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


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
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
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


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on the host cores, in worker processes whose BLAS
# thread count is set before numpy loads
# ---------------------------------------------------------------------------

def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


def _cpu_worker(path: str, budget: float) -> dict:
    """Runs in a child process: the oracle on the saved sample until the time
    budget is spent; reports the rates, wall time and CPU time of the process."""
    import numpy as np

    from oracle import csa2_oracle as o
    d = np.load(path)
    n = int(d["n"])
    res = {}
    # indexer: score every visible entry of a row prefix, top-512 and the pool
    t0, c0 = time.perf_counter(), time.process_time()
    rows = 0
    while rows < 1 or (time.perf_counter() - t0 < 0.6 * budget and rows < 64):
        s = o.index_scores_row(d["q8"], d["qs"], d["w"], d["cache"], d["pt"], n)
        o.topk_positions(s, 512)
        o.candidate_pool(o.block_maxima(s, n), 2048)
        rows += 1
    wall, cpu = time.perf_counter() - t0, time.process_time() - c0
    res.update(keys_per_s=n * rows / wall, index_rows=rows, index_wall_s=wall, index_cpu_s=cpu)
    # attention: one query-layer (64 heads over 128 SWA + 512 main entries, sink)
    t0, c0 = time.perf_counter(), time.process_time()
    qa = 0
    while qa < 1 or (time.perf_counter() - t0 < 0.4 * budget and qa < 400):
        o.attention_row(d["aq"], d["main"], d["mslot"], d["swa"], d["sslot"], d["sink"], 1 / math.sqrt(512))
        qa += 1
    awall, acpu = time.perf_counter() - t0, time.process_time() - c0
    res.update(attn_query_layers_per_s=qa / awall, attn_rows=qa, attn_wall_s=awall, attn_cpu_s=acpu)
    res["threads_busy"] = (cpu + acpu) / (wall + awall)
    return res


def _save_cpu_sample(step, device_copy, n=131072) -> str:
    """One decoder Full-layer row prefix of n entries (its pages remapped to
    0..n/64-1) and one attention query-layer of layer 21, saved for the CPU
    workers."""
    import numpy as np
    import torch
    c = step.caches[3]
    li = step.inputs[20]
    b = 2                                   # a 1M-entry sequence
    cache = device_copy(c.pc.index_k[c.pc.page_table[b, : n // 64].long()])
    al = step.inputs[21].attn
    slots = device_copy(step.buf.topk_slot[3][b]).astype(np.int64)
    ok = slots >= 0
    mslot = np.full(slots.shape, -1, dtype=np.int64)
    mslot[ok] = np.arange(ok.sum())
    main = device_copy(c.pc.main_kv[step.buf.topk_slot[3][b][torch.as_tensor(ok, device=c.pc.main_kv.device)].long()])
    ss = device_copy(al.swa_slot[b]).astype(np.int64)
    sok = ss >= 0
    sslot = np.full(ss.shape, -1, dtype=np.int64)
    sslot[sok] = np.arange(sok.sum())
    swa = device_copy(al.swa_kv[al.swa_slot[b][torch.as_tensor(sok, device=al.swa_kv.device)].long()])
    fd, path = tempfile.mkstemp(suffix=".npz", prefix="csa2_cpu_sample_")
    os.close(fd)
    np.savez(path, n=n, q8=device_copy(li.iq.q_fp8[b]), qs=device_copy(li.iq.q_scale[b]), w=device_copy(li.iq.w[b]),
             cache=cache, pt=np.arange(n // 64, dtype=np.int64),
             aq=al.q[b].float().cpu().numpy().astype(np.float64), main=main, mslot=mslot, swa=swa, sslot=sslot,
             sink=device_copy(al.sink).astype(np.float64))
    return path


def _run_cpu_worker(path: str, threads: int, budget: float) -> dict:
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
              "NUMEXPR_NUM_THREADS", "VECLIB_MAXIMUM_THREADS"):
        env[k] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", path, "--cpu-budget", str(budget)],
                       capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        raise RuntimeError(f"CPU worker failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(path: str, budget: float) -> dict:
    """The oracle, as it stands, on the host cores: once with its BLAS on every
    core the process may use, once on one thread."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    multi = _run_cpu_worker(path, cores, budget)
    one = _run_cpu_worker(path, 1, budget * 0.5)
    return {
        "value": multi["keys_per_s"], "unit": "keys/s", "cores": cores, "kind": "oracle",
        "threads": round(multi["threads_busy"], 2),
        "threads_note": "process CPU time / wall time of the worker, BLAS threads set to `cores`",
        "model": cpu_model(), "value_1thread": one["keys_per_s"],
        "attn_query_layers_per_s": multi["attn_query_layers_per_s"],
        "attn_query_layers_per_s_1thread": one["attn_query_layers_per_s"],
        # a query of the 4096-query prefill chunk scores 131,072..133,120 entries
        # (132,096 on average), the same work per entry as the decode row sampled
        "prefill_query_rows_per_s": multi["keys_per_s"] / 132096,
        "prefill_chunk_s_extrapolated": 4096 * 132096 / multi["keys_per_s"],
        "sample": (f"{multi['index_rows']} x one decoder Full-layer row prefix of 131072 entries (score + top-512 + "
                   f"pool) and {multi['attn_rows']} x one attention query-layer (64 heads, 128 SWA + 512 main keys, "
                   f"sink), float64 numpy oracle"),
    }


# ---------------------------------------------------------------------------
# GPU measurement helpers
# ---------------------------------------------------------------------------

def _time_calls(fn, iters: int, stream, warm: int = 2, replays: int = 7) -> float:
    """Device time in ms of one fn() call: iters back-to-back calls captured in
    one CUDA graph (so host launch overhead does not starve the GPU), replayed
    `replays` times, median replay over iters (CUDA events on the stream)."""
    import torch
    torch.cuda.synchronize()   # inputs made on other streams are complete
    with torch.cuda.stream(stream):
        for _ in range(warm):
            fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(iters):
            fn()
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    runs = []
    for _ in range(replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        stream.synchronize()
        runs.append(e0.elapsed_time(e1) / iters)
    del g
    return statistics.median(runs)


def prefill_case(dev, seed=300):
    """The 4096-query prefill chunk after a 256K-token prefix (m = 2): inputs
    and the calls of one chunk, in step order."""
    import torch

    from serving_lightning_indexer_gb300 import csa2
    from serving_lightning_indexer_gb300 import workloads as W
    m, prefix, T = PREFILL_M, PREFILL_PREFIX, PREFILL_T
    n_tok = prefix + T
    n_ent = n_tok // m
    pc = W.make_paged_cache([n_ent], seed=seed, device=dev)
    # the same entries' index keys as FP4 pages (scored on the per-row scan)
    pc4 = W.make_paged_cache([n_ent], seed=seed, device=dev, with_main=False, index_fp4=True)
    Cm, Z, gamma = W.make_compress_inputs(n_tok, seed=seed + 1, device=dev)
    iq = W.make_indexer_query(T, seed=seed + 2, device=dev)
    row_pos = torch.arange(prefix, n_tok, dtype=torch.int32, device=dev)
    r = csa2.rows(T, 1, row_seq=torch.zeros(T, dtype=torch.int32, device=dev), row_pos=row_pos, ratio_m=m)
    ld = (n_ent + 127) // 128 * 128
    scores = torch.empty(T, ld, dtype=torch.float32, device=dev)
    pos = torch.empty(T, 512, dtype=torch.int32, device=dev)
    slot = torch.empty_like(pos)
    al = W.make_attn_layer(T, seed=seed + 3, device=dev, swa_positions=[(t, 128) for t in range(T)],
                           n_swa_records=T + 127)
    out = torch.empty(T, 64, 512, dtype=torch.bfloat16, device=dev)
    pt0 = pc.page_table[0].contiguous()
    calls = {
        "compress": lambda: csa2.compress_m2(Cm, Z, m, gamma, pc.main_kv, page_table=pt0, first_entry=0),
        "index_score": lambda: csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores),
        "topk": lambda: csa2.topk_with_candidates(scores, r, 512, pos, slot, pc.page_table),
        "attn": lambda: csa2.sparse_attn(al.q, pc.main_kv, slot, al.swa_kv, al.swa_slot, al.sink, out),
        "index_score_fp4": lambda: csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc4.index_k, pc4.page_table, r,
                                                    scores),
    }
    pairs = float(sum((p + 1) // m for p in range(prefix, n_tok)))
    return calls, dict(n_entries=n_ent, tokens=n_tok, queries=T, flop=pairs * INDEX_PAIR_FLOP, pairs=pairs)


def reindex_case(dev, seed=200):
    """The decode Reindex at 1M context: batch 16, a given 2048-block pool per
    row, 10 % of the blocks shifted by +3 sigma along the Reindex query's
    weighted direction, then the attention of the Reindex layer and 3 Reuse
    layers."""
    import torch

    from serving_lightning_indexer_gb300 import csa2
    from serving_lightning_indexer_gb300 import workloads as W
    B, n = REINDEX_B, REINDEX_N
    lengths = [n] * B
    iq = W.make_indexer_query(B, seed=seed + 1, device=dev)
    dirs = (iq.w[:, :, None] * iq.q_float).sum(dim=1)
    pc = W.make_paged_cache(lengths, seed=seed, device=dev, plant_dirs=dirs, plant_frac=0.1, plant_shift=3.0)
    # REINDEX_POOLS different pools (and their selections) are cycled through,
    # so that the candidate blocks one call reads (34.6 MB) were last read
    # REINDEX_POOLS - 1 calls earlier and L2 (129 MB) no longer holds them
    pools = [W.make_pool(lengths, seed=seed + 2 + 97 * j, device=dev) for j in range(REINDEX_POOLS)]
    layers = [W.make_attn_layer(B, seed=seed + 10 + i, device=dev) for i in range(4)]
    r = csa2.rows(B, B, n_visible=pc.n_entries)
    pos = [torch.empty(B, 512, dtype=torch.int32, device=dev) for _ in pools]
    slot = [torch.empty_like(p_) for p_ in pos]
    outs = [torch.empty(B, 64, 512, dtype=torch.bfloat16, device=dev) for _ in layers]
    turn = {"reindex": 0, **{f"attn{i}": 0 for i in range(4)}}

    def nxt(name):
        j = turn[name] % REINDEX_POOLS
        turn[name] += 1
        return j

    calls = {"reindex": lambda: (lambda j: csa2.reindex(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r,
                                                        pools[j], 512, pos[j], slot[j]))(nxt("reindex"))}
    for i, (al, o_) in enumerate(zip(layers, outs)):
        calls[f"attn{i}"] = (lambda al=al, o_=o_, i=i: (lambda j: csa2.sparse_attn(
            al.q, pc.main_kv, slot[j], al.swa_kv, al.swa_slot, al.sink, o_, kv_ready=i > 0))(nxt(f"attn{i}")))
    keys = int(sum(min(n, W.POOL_BLOCKS * W.POOL_BLOCK) for _ in range(B)))
    return calls, dict(rows=B, keys=keys)


def measure_prefill(dev, stream, iters: int, peak_fp8: float, peak_fp8_sust: float) -> dict:
    """Per-call times of the prefill chunk and the prefill indexer's roofline."""
    import torch
    calls, info = prefill_case(dev)
    for name in ("compress", "index_score", "topk", "attn"):   # one pass in order: inputs of each call
        with torch.cuda.stream(stream):
            calls[name]()
    stream.synchronize()
    ms = {name: _time_calls(calls[name], iters if name == "index_score" else max(3, iters // 4), stream)
          for name in ("compress", "index_score", "topk", "attn")}
    # FP4 pages last (they overwrite the scores the top-k above read)
    fp4_ms = _time_calls(calls["index_score_fp4"], 3, stream)
    achieved = info["flop"] / (ms["index_score"] / 1e3) / 1e12
    del calls
    torch.cuda.empty_cache()
    return {
        "roofline_prefill": {
            "bound": "tensor", "kernel": "index_tiles_kernel (prefill: 8 queries x 32 heads per MMA tile)",
            "workload": f"4096 queries at positions 262144..266239, m=2, {info['n_entries']} entries (causal)",
            "achieved": achieved, "peak": peak_fp8, "unit": "TFLOP/s", "frac": achieved / peak_fp8,
            "frac_vs_sustained": achieved / peak_fp8_sust,
            "peak_source": "FP8 dense = 2 x the measured bf16 burst (nominal FP8:BF16 ratio); sustained likewise",
            "flop_per_launch": info["flop"], "avg_launch_ms": ms["index_score"], "launches_timed": iters * 7,
            "traffic": None},
        "prefill_chunk": {
            "workload": "prefill chunk: 4096 queries after a 256K-token prefix, m=2",
            "call_ms": ms, "chunk_ms": sum(ms.values()),
            "attn_query_layers_per_s": PREFILL_T / (ms["attn"] / 1e3),
            "entries_built_per_s": info["n_entries"] / (ms["compress"] / 1e3),
            "topk_rows_per_s": PREFILL_T / (ms["topk"] / 1e3)},
        "prefill_index_fp4": {
            "workload": "the same 4096 queries over FP4 index-K pages of the 133120 entries",
            "path": "per-row scan (M = 128 keys x 32 heads a tile, 4 block accumulators; each query reads the "
                    "keys again, from L2)",
            "avg_launch_ms": fp4_ms, "pairs_per_s": info["pairs"] / (fp4_ms / 1e3),
            "vs_fp8_gemm": ms["index_score"] / fp4_ms},
    }


def measure_reindex(dev, stream, iters: int, hbm_peak: float) -> dict:
    """Reindex at 1M context, batch 16: the call (gather + selection) and the
    attention of its four layers."""
    import torch
    calls, info = reindex_case(dev)
    with torch.cuda.stream(stream):
        for _ in range(REINDEX_POOLS):   # every pool's selection, before any attention reads it
            calls["reindex"]()
        for name, fn in calls.items():
            if name != "reindex":
                fn()
    stream.synchronize()
    ms = {name: _time_calls(fn, iters, stream) for name, fn in calls.items()}
    attn = statistics.mean(ms[f"attn{i}"] for i in range(4))
    del calls
    torch.cuda.empty_cache()
    gbs = info["keys"] * INDEX_KEY_BYTES / (ms["reindex"] / 1e3) / 1e9
    return {"roofline_reindex": {
        "bound": "hbm", "kernel": "index_tiles_kernel<gather> + sel_final_kernel (csa2_reindex)",
        "workload": "decode Reindex at 1M context, batch 16 x 16384 pool candidates, 10% planted blocks",
        "keys_per_s": info["keys"] / (ms["reindex"] / 1e3), "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
        "frac": gbs / hbm_peak, "frac_vs_nominal_8tbs": gbs / 8000.0,
        "algorithmic_bytes_per_launch": info["keys"] * INDEX_KEY_BYTES,
        "avg_launch_ms": ms["reindex"], "launches_timed": iters * 7, "traffic": None,
        "timing": (f"CUDA graph of {iters} calls replayed 7 times, median; {REINDEX_POOLS} pools cycled so the "
                   "candidate blocks are not L2-resident"),
        "attn_avg_launch_ms": attn, "attn_query_layers_per_s": REINDEX_B / (attn / 1e3),
        "attn_hbm_frac": ATTN_ROW_BYTES * REINDEX_B / (attn / 1e3) / 1e9 / hbm_peak}}


def measure_kv_project(dev, stream, iters: int, hbm_peak: float) -> dict:
    """The hidden-state projection C = H W of a Full layer's new tokens (the
    entry build's input; outside the step, which takes C as given): 16 rows
    rows, batch 8: 8 (decoder, m = 1) and 16 (encoder, m = 2, two tokens a
    sequence), hidden width 7168, weight 7168 x 512 bf16."""
    import torch

    from serving_lightning_indexer_gb300 import csa2
    from serving_lightning_indexer_gb300 import workloads as W
    res = {}
    for T in (8, 16):
        H, w = W.make_hidden_projection(T, seed=400 + T, device=dev)
        out = torch.empty(T, 512, dtype=torch.bfloat16, device=dev)
        # 24 weight copies (176 MB, more than L2) cycled so that each call reads
        # its weight from HBM
        ws = [w] + [w.clone() for _ in range(23)]
        k = [0]

        def call():
            csa2.kv_project(H, ws[k[0] % 24], out)
            k[0] += 1
        ms = _time_calls(call, iters * 24, stream)
        nbytes = w.numel() * 2 + H.numel() * 2 + out.numel() * 2
        gbs = nbytes / (ms / 1e3) / 1e9
        res[f"rows_{T}"] = {"avg_launch_ms": ms, "algorithmic_bytes_per_launch": nbytes, "achieved": gbs,
                            "frac": gbs / hbm_peak}
        del ws, H, w, out
    torch.cuda.empty_cache()
    return {"roofline_kv_project": {"bound": "hbm", "kernel": "kv_project_kernel (csa2_kv_project)",
                                    "hidden": W.HIDDEN, "peak": hbm_peak, "unit": "GB/s", **res}}


# ---------------------------------------------------------------------------
# single-call cases for profilers
# ---------------------------------------------------------------------------

def run_case(args):
    """One call of the library on a small input, timed with CUDA events (for
    ncu captures: a few GB on the device at most)."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from serving_lightning_indexer_gb300 import csa2
    from serving_lightning_indexer_gb300 import workloads as W
    dev = torch.device("cuda:0")
    st = torch.cuda.Stream(device=dev)   # graph capture needs a non-default stream
    B, n = args.batch, args.entries
    res = {"case": args.case}
    if args.case in ("scan", "topk", "reindex"):
        lengths = [n] * B
        pc = W.make_paged_cache(lengths, seed=1, device=dev, with_main=False, index_fp4=args.fp4)
        kb = 68 if args.fp4 else INDEX_KEY_BYTES
        iq = W.make_indexer_query(B, seed=2, device=dev)
        r = csa2.rows(B, B, n_visible=pc.n_entries)
        ld = (n + 127) // 128 * 128
        scores = torch.empty(B, ld, dtype=torch.float32, device=dev)
        bm = torch.empty(B, ld // 8, dtype=torch.float32, device=dev)
        hist = torch.zeros(2, B, 2048, dtype=torch.int32, device=dev)
        if args.case == "scan":
            ms = _time_calls(lambda: csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores,
                                                      bm, hist=hist), args.iters, st)
            res.update(ms=ms, keys=B * n, GBps=B * n * kb / ms / 1e6, fp4=args.fp4)
        elif args.case == "topk":
            pos = torch.empty(B, 512, dtype=torch.int32, device=dev)
            slot = torch.empty_like(pos)
            pool = torch.empty(B, 2048, dtype=torch.int32, device=dev)

            def both():
                csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores, bm, hist=hist)
                csa2.topk_with_candidates(scores, r, 512, pos, slot, pc.page_table, bm, pool, hist=hist)
            ms = _time_calls(both, args.iters, st)
            res.update(ms_scan_and_select=ms, rows=B, entries=n)
        else:
            pool = W.make_pool(lengths, seed=3, device=dev)
            pos = torch.empty(B, 512, dtype=torch.int32, device=dev)
            slot = torch.empty_like(pos)
            ms = _time_calls(lambda: csa2.reindex(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, pool, 512,
                                                  pos, slot), args.iters, st)
            res.update(ms=ms, keys=B * 16384, GBps=B * 16384 * kb / ms / 1e6, fp4=args.fp4)
    elif args.case == "attn":
        pc = W.make_paged_cache([n], seed=4, device=dev)
        al = W.make_attn_layer(B, seed=5, device=dev)
        slot = torch.randint(0, n, (B, 512), dtype=torch.int32, device=dev)
        out = torch.empty(B, 64, 512, dtype=torch.bfloat16, device=dev)
        ms = _time_calls(lambda: csa2.sparse_attn(al.q, pc.main_kv, slot, al.swa_kv, al.swa_slot, al.sink, out),
                         args.iters, st)
        res.update(ms=ms, query_layers=B)
    elif args.case == "prefill_chunk":
        # the 4,096-query prefill chunk after a 256K-token prefix, its four calls
        # in order, args.iters times (for an ncu launch list of the chunk)
        calls, info = prefill_case(dev)
        order = ("compress", "index_score", "topk", "attn")
        ms = {}
        for name in order:
            ms[name] = _time_calls(calls[name], args.iters, st, warm=1, replays=1)
        res.update(call_ms=ms, queries=info["queries"], entries=info["n_entries"])
    elif args.case == "project":
        H, w = W.make_hidden_projection(B, seed=8, device=dev)
        out = torch.empty(B, 512, dtype=torch.bfloat16, device=dev)
        ms = _time_calls(lambda: csa2.kv_project(H, w, out), args.iters, st)
        res.update(ms=ms, rows=B, hidden=W.HIDDEN)
    else:  # prefill: the query-blocked indexer over one sequence, m = 2, T queries at the end of n entries
        T = args.queries
        pc = W.make_paged_cache([n], seed=6, device=dev, with_main=False)
        iq = W.make_indexer_query(T, seed=7, device=dev)
        row_pos = torch.arange(2 * n - T, 2 * n, dtype=torch.int32, device=dev)
        r = csa2.rows(T, 1, row_seq=torch.zeros(T, dtype=torch.int32, device=dev), row_pos=row_pos, ratio_m=2)
        ld = (n + 127) // 128 * 128
        scores = torch.empty(T, ld, dtype=torch.float32, device=dev)
        ms = _time_calls(lambda: csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores),
                         args.iters, st)
        flop = float(sum((p + 1) // 2 for p in range(2 * n - T, 2 * n))) * INDEX_PAIR_FLOP
        res.update(ms=ms, queries=T, entries=n, TFLOPs=flop / ms / 1e9)
    rc = csa2.check_device_error()
    if rc != 0:
        raise RuntimeError(f"device error status {rc}")
    print(json.dumps(res), flush=True)


# ---------------------------------------------------------------------------
# the benchmark
# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--min-seconds", type=float, default=0.6, help="replay the K-step graph at least this long")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the prefill and Reindex workloads")
    ap.add_argument("--case", choices=["scan", "topk", "reindex", "attn", "prefill", "prefill_chunk", "project"])
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--batch", type=int, default=8)
    ap.add_argument("--entries", type=int, default=262144)
    ap.add_argument("--queries", type=int, default=1024)
    ap.add_argument("--fp4", action="store_true", help="FP4 index-K pages in --case scan/topk/reindex")
    ap.add_argument("--cpu-worker", help=argparse.SUPPRESS)
    args = ap.parse_args()

    if args.cpu_worker:
        print(json.dumps(_cpu_worker(args.cpu_worker, args.cpu_budget)), flush=True)
        return
    if args.case:
        return run_case(args)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    import torch

    if args.impl == "reference":
        return reference_arm(args, rank, world)

    import __graft_entry__
    __graft_entry__.build()
    from serving_lightning_indexer_gb300 import csa2
    from serving_lightning_indexer_gb300 import decode_step as ds
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

    # ---- K steps in one graph, events around every indexer scan and attention.
    # The timing events are recorded on a side stream that forks from the
    # step's stream, so they hang off the kernel chain instead of sitting
    # between two kernels (a node between them would cut the programmatic-launch
    # overlap).
    K = args.steps
    side = torch.cuda.Stream(device=dev)

    def side_event():
        fork = torch.cuda.Event()
        fork.record(stream)
        side.wait_event(fork)
        e = torch.cuda.Event(enable_timing=True, external=True)  # an event node inside the graph
        e.record(side)
        return e

    ev_pairs, attn_pairs = [], []
    step.on_index_score = lambda l: ev_pairs.append([l, side_event(), None])
    step.after_index_score = lambda l: ev_pairs[-1].__setitem__(2, side_event())
    step.on_attn = lambda l: attn_pairs.append([l, side_event(), None])
    step.after_attn = lambda l: attn_pairs[-1].__setitem__(2, side_event())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(K):
            step.run(stream)
        join = torch.cuda.Event()
        join.record(side)
        stream.wait_event(join)
    step.on_index_score = step.after_index_score = step.on_attn = step.after_attn = None
    # the same K steps without the timing events: the step time comes from this
    # graph (the event nodes of the other cost ~1 % of the step)
    g_plain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_plain, stream=stream):
        for _ in range(K):
            step.run(stream)
    with torch.cuda.stream(stream):
        g.replay()                   # untimed: first replays of the instantiated graphs
        g_plain.replay()
    stream.synchronize()

    # ---- timed region: replays of the K-step graph until min_seconds have
    # passed; each round replays the plain graph (the step time) and the graph
    # with the timing events (the scan and attention launch times)
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    replay_ms, marked_ms, scan_ms, attn_ms, per_layer, attn_role = [], [], [], [], {}, {}
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler.mark(True)
    t_wall = time.time()
    while len(replay_ms) < 3 or time.time() - t_wall < args.min_seconds:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):  # the graph replays on the current stream
            t_start.record(stream)
            g_plain.replay()
            t_end.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        replay_ms.append(t_start.elapsed_time(t_end))
        with torch.cuda.stream(stream):
            t_start.record(stream)
            g.replay()
            t_end.record(stream)
        stream.synchronize()
        marked_ms.append(t_start.elapsed_time(t_end))
        for l, a, b in ev_pairs:
            ms = a.elapsed_time(b)
            scan_ms.append(ms)
            per_layer.setdefault(l, []).append(ms)
        for l, a, b in attn_pairs:
            ms = a.elapsed_time(b)
            attn_ms.append(ms)
            attn_role.setdefault(ds.role_of(l), []).append(ms)
    sampler.mark(False)
    if world > 1:
        dist.barrier()
    if rank == 0:
        sampler.stop()
    rc = csa2.check_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device error status {rc} in the timed region")
    ms_replay = max_over_ranks(statistics.median(replay_ms), dev)
    ms_per_step = ms_replay / K

    # ---- end to end: pinned host inputs -> device, step, outputs -> pinned host.
    # Every step copies all of its query-side inputs in and all 38 attention
    # outputs out.  The inputs of all layers sit in one pinned host buffer; on
    # the device there are two such buffers, and the step's input tensors are
    # views into the one of the current step.  While step k computes, step
    # k + 1's inputs are copied into the other buffer, so no layer of a step
    # waits on a copy (a wait or an event between two kernels of the step would
    # cut their programmatic overlap); the first step's copy runs before it.
    # Likewise the outputs go to one of two device buffers and a step's are
    # read back in one copy while the next step computes; the last step's
    # read-back ends the timed replay.
    layout, off = [], 0
    for l in step.layers:
        li = step.inputs[l]
        fields = [(li.attn, "q")]
        if li.iq is not None:
            fields += [(li.iq, "q_fp8"), (li.iq, "q_scale"), (li.iq, "w")]
        if li.C is not None:
            fields += [(li, "C")] + ([(li, "Z")] if li.Z is not None else [])
        for obj, name in fields:
            t = getattr(obj, name)
            nb = t.numel() * t.element_size()
            layout.append((obj, name, t, off, nb))
            off = (off + nb + 255) // 256 * 256
    dbufs = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]
    hbuf = torch.empty(off, dtype=torch.uint8).pin_memory()
    views = [[], []]
    for obj, name, t, o, nb in layout:
        hbuf[o:o + nb].copy_(t.detach().contiguous().cpu().view(torch.uint8).reshape(-1))
        for k in range(2):
            view = dbufs[k][o:o + nb].view(t.dtype).view(t.shape)
            view.copy_(t)
            views[k].append((obj, name, view))
    h2d = off
    # the 38 outputs of a step in one buffer (two, alternating by step): a
    # step's outputs are read back in one copy while the next step computes
    o0 = step.buf.out[step.layers[0]]
    obufs = [torch.empty((len(step.layers),) + tuple(o0.shape), dtype=o0.dtype, device=dev) for _ in range(2)]
    oviews = [{l: ob[i] for i, l in enumerate(step.layers)} for ob in obufs]
    host_obuf = torch.empty(tuple(obufs[0].shape), dtype=o0.dtype).pin_memory()
    d2h = obufs[0].numel() * obufs[0].element_size()
    out_orig = step.buf.out
    cp_in = torch.cuda.Stream(device=dev)
    cp_out = torch.cuda.Stream(device=dev)
    Ke = max(1, min(K, 20))

    def load_inputs(k):
        """Copy a step's inputs into buffer k % 2 on cp_in, after the work so far on the stream."""
        mark = torch.cuda.Event()
        mark.record(stream)
        cp_in.wait_event(mark)
        with torch.cuda.stream(cp_in):
            dbufs[k % 2].copy_(hbuf, non_blocking=True)
            done = torch.cuda.Event()
            done.record(cp_in)
        return done

    g2 = torch.cuda.CUDAGraph()
    read_back = [None, None]
    with torch.cuda.graph(g2, stream=stream):
        ready = load_inputs(0)
        for k in range(Ke):
            stream.wait_event(ready)             # this step's inputs are in its buffer
            if read_back[k % 2] is not None:     # its output buffer has been read back
                stream.wait_event(read_back[k % 2])
            if k + 1 < Ke:
                ready = load_inputs(k + 1)       # the next step's, while this one computes
            for obj, name, view in views[k % 2]:
                setattr(obj, name, view)
            step.buf.out = oviews[k % 2]
            step.run(stream)
            end = torch.cuda.Event()
            end.record(stream)
            cp_out.wait_event(end)
            with torch.cuda.stream(cp_out):      # this step's outputs, while the next one computes
                host_obuf.copy_(obufs[k % 2], non_blocking=True)
                read_back[k % 2] = torch.cuda.Event()
                read_back[k % 2].record(cp_out)
        stream.wait_event(read_back[(Ke - 1) % 2])   # the last step's outputs are on the host
    step.buf.out = out_orig
    with torch.cuda.stream(stream):
        g2.replay()
    stream.synchronize()
    e2e_runs = []
    for _ in range(3):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g2.replay()
            e1.record(stream)
        stream.synchronize()
        e2e_runs.append(e0.elapsed_time(e1))
    e2e_ms = max_over_ranks(statistics.median(e2e_runs), dev)

    hbm_peak, bf16_peak, bf16_sust, peak_kind = _peaks()
    cpu_path = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu_path = _save_cpu_sample(step, lambda t: t.detach().cpu().numpy())
    del g, g2
    n_full = sum(1 for l in step.layers if ds.role_of(l) == "full")
    n_reidx = sum(1 for l in step.layers if ds.role_of(l) == "reindex")
    n_layers = len(step.layers)
    del step
    torch.cuda.empty_cache()

    # ---- the prefill chunk and the decode Reindex at 1M, measured in the same run
    extra = {}
    if not args.no_workloads:
        extra.update(measure_prefill(dev, stream, 20, 2 * bf16_peak, 2 * bf16_sust))
        extra.update(measure_reindex(dev, stream, 20, hbm_peak))
        extra.update(measure_kv_project(dev, stream, 20, hbm_peak))

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    traffic_per_key = _scan_traffic_per_key()
    value = whole_job_rate(keys_per_step, K, world, ms_replay)
    scan_bytes_per_launch = scan_bytes_per_step * K / (len(ev_pairs))
    scan_avg = statistics.mean(scan_ms)
    achieved = scan_bytes_per_launch / (scan_avg / 1e3) / 1e9
    attn_avg = statistics.mean(attn_ms)
    # our kernels launched per step: a Full layer runs compress, the scan and the
    # two select passes (filter, final); a Reindex layer the pool gather and the
    # final select; every layer one clustered attention launch (the histogram
    # memsets are not kernels)
    launches_per_step = n_full * 4 + n_reidx * 2 + n_layers
    cpu = None
    if cpu_path:
        try:
            cpu = cpu_baseline(cpu_path, args.cpu_budget)
        finally:
            os.remove(cpu_path)
    out = {
        "metric": METRIC, "value": value, "unit": "keys/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 (indexer, fp32 accumulate) + bf16 (attention)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": len(LENGTHS), "context_lengths": LENGTHS, "layers": n_layers,
                   "keys_scored_per_step": keys_per_step, "attn_query_layers_per_step": attn_per_step,
                   "timing": (f"K steps in one CUDA graph, replayed {len(replay_ms)} times over >= "
                              f"{args.min_seconds} s, median replay; inputs larger than L2 (no flush); "
                              "each replay followed by one of the same steps with side-stream timing events, "
                              "which give the per-launch scan and attention times"),
                   "parallelism": f"replicas x{world}"},
        "replays": len(replay_ms), "replay_ms": {"median": statistics.median(replay_ms), "min": min(replay_ms),
                                                 "max": max(replay_ms),
                                                 "with_timing_events_median": statistics.median(marked_ms)},
        "attn_query_layers_per_s": whole_job_rate(attn_per_step, K, world, ms_replay),
        "roofline": {"bound": "hbm", "kernel": "index_tiles_kernel<1,scan> (decode Lightning-Indexer scan)",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "frac_vs_nominal_8tbs": achieved / 8000.0,
                     "peak_source": peak_kind,
                     "traffic": (None if traffic_per_key is None
                                 else traffic_per_key * scan_bytes_per_launch / INDEX_KEY_BYTES),
                     "traffic_source": "ncu dram bytes per key of the committed scan capture, scaled to the "
                                       "keys of an average launch",
                     "algorithmic_bytes_per_launch": scan_bytes_per_launch,
                     "avg_launch_ms": scan_avg, "launches_timed": len(scan_ms),
                     "per_layer_ms": {str(l): statistics.mean(v) for l, v in per_layer.items()}},
        # the sparse attention: latency-bound at 8 rows a launch, reported
        # beside the scan against both rooflines
        "roofline_attention": {
            "bound": "latency", "kernel": "sparse_attn_tc_kernel (8 rows x 64 heads x 640 keys)",
            "avg_launch_ms": attn_avg, "launches_timed": len(attn_ms),
            # Reuse layers gather their keys before the dependency wait; Full and
            # Reindex layers read slots written by the launch just before
            "avg_launch_ms_by_role": {r: statistics.mean(v) for r, v in attn_role.items()},
            "share_of_step": attn_avg * n_layers / ms_per_step,
            "algorithmic_bytes_per_launch": ATTN_ROW_BYTES * len(LENGTHS),
            "hbm_frac": ATTN_ROW_BYTES * len(LENGTHS) / (attn_avg / 1e3) / 1e9 / hbm_peak,
            "flop_per_launch": ATTN_ROW_FLOP * len(LENGTHS),
            "bf16_tensor_frac": ATTN_ROW_FLOP * len(LENGTHS) / (attn_avg / 1e3) / 1e12 / bf16_sust,
            "peaks": {"hbm_gbs": hbm_peak, "bf16_tflops_sustained": bf16_sust, "source": peak_kind}},
        **extra,
        "cpu_baseline": cpu,
        "e2e": {"value": whole_job_rate(keys_per_step, Ke, world, e2e_ms), "unit": "keys/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": Ke, "replays": len(e2e_runs)},
        "gpu_launches": launches_per_step * K * (len(replay_ms) + len(marked_ms)),
        "gpu_launches_per_step": launches_per_step,
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
    t0, c0 = time.perf_counter(), time.process_time()
    for i in range(args.steps):
        one(i % 2)
    dt, cpu_s = time.perf_counter() - t0, time.process_time() - c0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    v = n * args.steps / dt
    sample = f"per step one decoder Full-layer row prefix of {n} entries: score + top-512 + pool"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "keys/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_entries_per_step": n},
        "cpu_baseline": {"value": v, "unit": "keys/s", "cores": cores, "kind": "oracle", "sample": sample,
                         "threads": round(cpu_s / dt, 2), "model": cpu_model()},
        "e2e": {"value": v, "unit": "keys/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


if __name__ == "__main__":
    main()
