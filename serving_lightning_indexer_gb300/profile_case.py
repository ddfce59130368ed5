"""Small, self-contained invocations of one CSA2 call, for kernel profiling.

  python -m serving_lightning_indexer_gb300.profile_case --case scan   [--iters N]
  python -m serving_lightning_indexer_gb300.profile_case --case topk
  python -m serving_lightning_indexer_gb300.profile_case --case reindex
  python -m serving_lightning_indexer_gb300.profile_case --case attn
  python -m serving_lightning_indexer_gb300.profile_case --case prefill

--fp4 stores the index keys of the scan / topk / reindex cases as FP4 pages.

Each case holds well under 2 GB on the device, reads more than the 129 MB L2
per launch where the call is HBM-bound, runs a few warm-up launches and then
`--iters` timed launches (CUDA events), and prints one line per case.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import csa2
from . import workloads as W


def _time(fn, iters, stream):
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", default="scan", choices=["scan", "topk", "reindex", "attn", "prefill"])
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--batch", type=int, default=8)
    ap.add_argument("--entries", type=int, default=262144)
    ap.add_argument("--fp4", action="store_true", help="FP4 index-K pages (68 B per key)")
    a = ap.parse_args()
    csa2.load(build_if_missing=True)
    dev = torch.device("cuda:0")
    st = torch.cuda.current_stream()
    B, n = a.batch, a.entries
    res = {"case": a.case}
    if a.case in ("scan", "topk", "reindex"):
        lengths = [n] * B
        pc = W.make_paged_cache(lengths, seed=1, device=dev, with_main=False, index_fp4=a.fp4)
        kb = 68 if a.fp4 else 132  # index-K bytes per key
        iq = W.make_indexer_query(B, seed=2, device=dev)
        r = csa2.rows(B, B, n_visible=pc.n_entries)
        ld = (n + 127) // 128 * 128
        scores = torch.empty(B, ld, dtype=torch.float32, device=dev)
        bm = torch.empty(B, ld // 8, dtype=torch.float32, device=dev)
        if a.case == "scan":
            ms = _time(lambda: csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores, bm),
                       a.iters, st)
            res.update(ms=ms, keys=B * n, GBps=B * n * kb / ms / 1e6, fp4=a.fp4)
        elif a.case == "topk":
            csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores, bm)
            pos = torch.empty(B, 512, dtype=torch.int32, device=dev)
            slot = torch.empty_like(pos)
            pool = torch.empty(B, 2048, dtype=torch.int32, device=dev)
            ms = _time(lambda: csa2.topk_with_candidates(scores, r, 512, pos, slot, pc.page_table, bm, pool),
                       a.iters, st)
            res.update(ms=ms, rows=B, entries=n)
        else:
            pool = W.make_pool(lengths, seed=3, device=dev)
            pos = torch.empty(B, 512, dtype=torch.int32, device=dev)
            slot = torch.empty_like(pos)
            ms = _time(lambda: csa2.reindex(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, pool, 512, pos,
                                            slot), a.iters, st)
            res.update(ms=ms, keys=B * 16384, GBps=B * 16384 * kb / ms / 1e6, fp4=a.fp4)
    elif a.case == "attn":
        pc = W.make_paged_cache([n], seed=4, device=dev)
        al = W.make_attn_layer(B, seed=5, device=dev)
        slot = torch.randint(0, n, (B, 512), dtype=torch.int32, device=dev)
        out = torch.empty(B, 64, 512, dtype=torch.bfloat16, device=dev)
        ms = _time(lambda: csa2.sparse_attn(al.q, pc.main_kv, slot, al.swa_kv, al.swa_slot, al.sink, out), a.iters, st)
        res.update(ms=ms, query_layers=B)
    else:  # prefill: query-blocked indexer over one sequence, m = 2
        T = 1024
        pc = W.make_paged_cache([n], seed=6, device=dev, with_main=False)
        iq = W.make_indexer_query(T, seed=7, device=dev)
        row_pos = torch.arange(2 * n - T, 2 * n, dtype=torch.int32, device=dev)
        r = csa2.rows(T, 1, row_seq=torch.zeros(T, dtype=torch.int32, device=dev), row_pos=row_pos, ratio_m=2)
        ld = (n + 127) // 128 * 128
        scores = torch.empty(T, ld, dtype=torch.float32, device=dev)
        ms = _time(lambda: csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores),
                   a.iters, st)
        flops = 2.0 * T * n * 32 * 128
        res.update(ms=ms, TFLOPs=flops / ms / 1e9)
    assert csa2.check_device_error() == 0
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
