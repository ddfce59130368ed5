"""The multi-rank path of bench.py on CPU: two gloo ranks (the GPU runs use one
process per GPU over NCCL with the same code; decode shards by sequence with
no collective on the data path, so the only exchange is the timing)."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout
from types import SimpleNamespace

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [10.0, 12.5][rank]          # rank 1 is the slow one
    m = bench.max_over_ranks(ms, "cpu")
    dist.barrier()
    q.put((rank, m, bench.whole_job_rate(1000, 4, world, m)))
    dist.destroy_process_group()


def test_two_gloo_ranks_time_the_slowest_rank_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    assert all(m == 12.5 for _, m, _ in res)                  # max over ranks, seen by every rank
    assert all(v == 1000 * 4 * 2 / 12.5e-3 for _, _, v in res)  # whole-job units over the slowest time


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.whole_job_rate(10, 2, 1, 1000.0) == 20.0


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.reference_arm(SimpleNamespace(steps=1, warmup=0), rank=1, world=2)
    assert buf.getvalue() == ""      # the other ranks exit without work or output


def test_reference_arm_prints_the_contract_line_on_rank_zero():
    # the oracle on the host cores: one JSON line with the metric, its unit,
    # the CPU record and an e2e object without host-device copies
    sys.path.insert(0, ROOT)
    import json
    import bench
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.reference_arm(SimpleNamespace(steps=1, warmup=0), rank=0, world=1)
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "keys/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 1 and d["n_gpus"] == 1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "keys/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"]
