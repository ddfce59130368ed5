"""Context-parallel prefill split and all-gather (DSA page, "并行：为什么 DSA
偏爱 CP"): the split rules on CPU, and the all-gather on two gloo ranks."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
from serving_lightning_indexer_gb300 import cp  # noqa: E402


@pytest.mark.parametrize("strategy", cp.STRATEGIES)
@pytest.mark.parametrize("n,world", [(8000, 4), (1001, 2), (7, 3), (0, 2), (5, 8)])
def test_shares_partition_the_units(strategy, n, world):
    shares = [cp.cp_units(n, world, r, strategy) for r in range(world)]
    allu = torch.cat(shares)
    assert sorted(allu.tolist()) == list(range(n))
    for s in shares:
        assert s.tolist() == sorted(s.tolist())
    assert max(s.numel() for s in shares) - min(s.numel() for s in shares) <= 2


def test_interleave_is_round_robin():
    assert cp.cp_units(10, 3, 1, "interleave").tolist() == [1, 4, 7]


def test_zigzag_worked_example_from_the_page():
    """8000 tokens, p = 4, blocks of 1000: rank 0 takes b0 (about 500 keys seen
    on average) and b7 (about 7500), rank 3 takes b3 (about 3500) and b4 (about
    4500), and every rank's total is about 1000 x 8000 = 8M query-key pairs."""
    n, p = 8000, 4
    r0 = cp.cp_units(n, p, 0, "zigzag")
    assert r0[:1000].tolist() == list(range(1000)) and r0[1000:].tolist() == list(range(7000, 8000))
    r3 = cp.cp_units(n, p, 3, "zigzag")
    assert r3.tolist() == list(range(3000, 5000))
    seen = lambda ids: (ids + 1).double()              # m = 1: query i sees i + 1 keys
    assert abs(seen(r0[:1000]).mean() - 500) < 1 and abs(seen(r0[1000:]).mean() - 7500) < 1
    assert abs(seen(r3[:1000]).mean() - 3500) < 1 and abs(seen(r3[1000:]).mean() - 4500) < 1
    pairs = [cp.cp_causal_pairs(n, 1, p, r, "zigzag") for r in range(p)]
    assert len(set(pairs)) == 1                         # exactly balanced: 1000 x 8001
    assert pairs[0] == 1000 * 8001 and abs(pairs[0] - 8_000_000) / 8e6 < 1e-3
    # a plain split into p consecutive segments leaves the last rank about 2p - 1 times the first
    seg = [int((torch.arange(r * 2000, (r + 1) * 2000) + 1).sum()) for r in range(p)]
    assert abs(seg[-1] / seg[0] - (2 * p - 1)) < 0.01


def test_entry_units_keep_the_m_tokens_of_an_entry_together():
    toks = [cp.cp_tokens(301, 2, 2, r, "interleave") for r in range(2)]
    assert sorted(torch.cat(toks).tolist()) == list(range(602))
    for t in toks:
        assert ((t[0::2] % 2) == 0).all() and (t[1::2] == t[0::2] + 1).all()


def test_bad_arguments():
    with pytest.raises(ValueError):
        cp.cp_units(10, 2, 0, "ring")
    with pytest.raises(ValueError):
        cp.cp_units(10, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from serving_lightning_indexer_gb300 import cp as cpr
    ok = []
    for strategy in cpr.STRATEGIES:
        for n in (1, 5, 300, 1001):
            g = torch.Generator().manual_seed(n)
            # every rank knows the whole sequence's rows only to check the result:
            # main-KV records (288 B) and index-K entries (132 B), as bytes
            full_kv = torch.randint(0, 256, (n, 288), generator=g, dtype=torch.uint8)
            full_ik = torch.randint(0, 256, (n, 132), generator=g, dtype=torch.uint8)
            mine = cpr.cp_units(n, world, rank, strategy)
            got_kv = cpr.cp_all_gather(full_kv[mine].clone(), n, world, rank, strategy)
            got_ik = cpr.cp_all_gather(full_ik[mine].clone(), n, world, rank, strategy)
            ok.append((strategy, n, torch.equal(got_kv, full_kv) and torch.equal(got_ik, full_ik)))
    # a wrong share size is refused before any exchange
    try:
        cpr.cp_all_gather(torch.zeros(3, 4), 100, world, rank)
        refused = False
    except ValueError:
        refused = True
    dist.barrier()
    q.put((rank, ok, refused))
    dist.destroy_process_group()


def test_all_gather_on_two_gloo_ranks_returns_the_sequence_in_order():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ok, refused in res:
        assert refused
        assert all(good for _, _, good in ok), [(s, n) for s, n, good in ok if not good]


def test_gather_volume_is_linear_in_the_sequence():
    """O(S) per rank: (p - 1) padded shares of the record size."""
    assert cp.cp_gather_bytes_per_rank(8000, 132, 4) == 3 * 2000 * 132
    assert cp.cp_gather_bytes_per_rank(8001, 132, 4) == 3 * 2001 * 132
