"""Pins of the oracle's indexer score, top-k, slot translation, candidate pool
and Reindex against hand-computed values, the pages' worked example,
brute force and invariants the pages state."""
import itertools

import numpy as np

from conftest import read_golden
from oracle import csa2_oracle as o
from serving_lightning_indexer_gb300 import workloads as W


def _golden_score():
    rows = read_golden("index_score_hand.txt")
    q = np.array([[float(v) for v in r] for k, r in rows if k == "q"])
    keys = np.array([[float(v) for v in r] for k, r in rows if k == "k"])
    ks = np.array([float(v) for v in [r for k, r in rows if k == "kscale"][0]])
    ws = [np.array([float(v) for v in r]) for k, r in rows if k == "w"]
    Is = [np.array([float(v) for v in r]) for k, r in rows if k == "I"]
    return q, keys * ks[:, None], ws, Is


def test_index_score_hand_values():
    q, keys, ws, Is = _golden_score()
    for w, I in zip(ws, Is):
        assert np.array_equal(o.index_score_values(q, w, keys), I)


def test_index_score_bruteforce_loops():
    rng = np.random.default_rng(0)
    H, d, n = 3, 5, 7
    q = rng.normal(size=(H, d))
    k = rng.normal(size=(n, d))
    w = rng.normal(size=H)
    want = []
    for s in range(n):
        tot = 0.0
        for h in range(H):
            dot = sum(q[h, j] * k[s, j] for j in range(d))
            tot += w[h] * (dot if dot > 0 else 0.0)
        want.append(tot)
    assert np.allclose(o.index_score_values(q, w, k), want, rtol=1e-14, atol=1e-14)


def test_scale_folding_identity():
    # DSA page, "fp8 与 scale 的吸收": a positive per-head q scale moves through
    # ReLU into the head weight; a positive per-key scale moves out of the head sum
    rng = np.random.default_rng(1)
    q8 = rng.integers(0, 0x7E, size=(32, 128))
    q8 = np.where(rng.random((32, 128)) < 0.5, q8, q8 | 0x80)
    qs = rng.uniform(0.01, 2.0, size=32)
    w = rng.normal(size=32)
    kraw = o.FP8[rng.integers(0, 0x7E, size=(50, 128))]
    ksc = rng.uniform(0.01, 2.0, size=50)
    direct = o.index_score_values(o.dequant_q(q8, qs), w, kraw * ksc[:, None])
    folded = ksc * o.index_score_values(o.FP8[q8], w * qs, kraw)
    assert np.allclose(direct, folded, rtol=1e-12, atol=1e-12)


def test_visible_entries():
    # CSA2 page, "候选池不减少存储": (pos + 1) // ratio
    assert [o.visible_entries(p, 2) for p in range(6)] == [0, 1, 1, 2, 2, 3]
    assert [o.visible_entries(p, 1) for p in range(3)] == [1, 2, 3]


def _pool_golden():
    return {k: v for k, v in read_golden("pool_worked_example.txt")}


def test_worked_example_block_max_topk_pool():
    g = _pool_golden()
    s = np.array([float(v) for v in g["scores"]])
    assert np.array_equal(o.block_maxima(s, len(s)), [float(v) for v in g["block_max"]])
    assert o.topk_positions(s, 6).tolist() == [int(v) for v in g["topk6"]]
    bm = o.block_maxima(s, len(s))
    for n in (1, 2, 3):
        want = [int(v) for v in g[f"pool{n}"]]
        assert o.candidate_pool(bm, n).tolist() == want
    s2 = np.array([float(v) for v in g["scores_maxmean"]])
    assert o.candidate_pool(o.block_maxima(s2, len(s2)), 2).tolist() == [int(v) for v in g["pool2_maxmean"]]


def test_topk_bruteforce_and_fill():
    rng = np.random.default_rng(2)
    for n in (0, 1, 5, 20, 33):
        s = np.round(rng.normal(size=n), 1)        # many exact ties
        s[rng.random(n) < 0.2] = -np.inf
        k = 8
        want = sorted([(-s[i], i) for i in range(n) if np.isfinite(s[i])])[:k]
        want = sorted(i for _, i in want) + [-1] * (k - len(want))
        assert o.topk_positions(s, k).tolist() == want


def test_topk_all_selected_when_short():
    s = np.random.default_rng(3).normal(size=300)
    got = o.topk_positions(s, 512)
    assert sorted(got[:300].tolist()) == list(range(300)) and (got[300:] == -1).all()


def test_slot_translation_golden():
    g = {k: v for k, v in read_golden("slot_translation.txt")}
    table = np.array([int(v) for v in g["table"]])
    pos = np.array([int(v) for v in g["pos"]])
    assert o.slots_of(pos, table).tolist() == [int(v) for v in g["slot"]]


def test_pool_contains_own_topk_without_ties():
    # CSA2 page, "分块不是压缩": without ties the pool holds the layer's own top-512
    rng = np.random.default_rng(4)
    for n in (20000, 33333):
        s = rng.normal(size=n)
        pool = o.candidate_pool(o.block_maxima(s, n), 2048)
        top = o.topk_positions(s, 512)
        assert set((top // 8).tolist()) <= set(pool[pool >= 0].tolist())
        assert (pool >= 0).sum() == 2048 and (n - 1) // 8 in set(pool.tolist())


def test_pool_is_everything_when_short():
    # CSA2 page, "池里的 16384 个位置是哪些": ceil(N/8) <= 2048 -> every block
    s = np.random.default_rng(5).normal(size=16381)
    pool = o.candidate_pool(o.block_maxima(s, 16381), 2048)
    assert pool.tolist() == list(range(2048))


def test_pool_bruteforce_small():
    rng = np.random.default_rng(6)
    for nblk, npool in itertools.product((1, 3, 9), (1, 2, 4)):
        bm = np.round(rng.normal(size=nblk), 1)
        key = [(-(np.inf if j == nblk - 1 else bm[j]), j) for j in range(nblk)]
        want = sorted(j for _, j in sorted(key)[:npool])
        got = o.candidate_pool(bm, npool)
        assert got[: len(want)].tolist() == want and (got[len(want):] == -1).all()


def _small_cache(n, seed):
    pc = W.make_paged_cache([n], seed=seed, with_main=False)
    iq = W.make_indexer_query(1, seed=seed + 100)
    return pc, iq


def test_reindex_equals_full_topk_when_pool_covers_everything():
    n = 3000
    pc, iq = _small_cache(n, 7)
    cache, pt = pc.index_k.numpy(), pc.page_table[0].numpy()
    full = o.index_scores_row(iq.q_fp8[0].numpy(), iq.q_scale[0].numpy(), iq.w[0].numpy(), cache, pt, n)
    pool = o.candidate_pool(o.block_maxima(full, n), 2048)
    assert (pool >= 0).sum() == -(-n // 8)
    got = o.reindex_topk(iq.q_fp8[0].numpy(), iq.q_scale[0].numpy(), iq.w[0].numpy(), cache, pt, n, pool, 512)
    assert got.tolist() == o.topk_positions(full, 512).tolist()


def test_reindex_result_inside_pool_and_scores_match_full():
    n = 40000
    pc, iq = _small_cache(n, 8)
    cache, pt = pc.index_k.numpy(), pc.page_table[0].numpy()
    args = (iq.q_fp8[0].numpy(), iq.q_scale[0].numpy(), iq.w[0].numpy(), cache, pt, n)
    full = o.index_scores_row(*args)
    pool = W.make_pool([n], seed=9)[0].numpy()
    got = o.reindex_topk(*args, pool, 512)
    assert set((got[got >= 0] // 8).tolist()) <= set(pool.tolist())
    # rescoring inside the pool reproduces the Full layer's scores at those positions
    sc = o.reindex_scores(*args, pool)
    pos = o.pool_positions(pool, n)
    assert np.array_equal(sc[pos >= 0], full[pos[pos >= 0]])
    # and the selection equals the top-k of the full row restricted to the pool
    masked = np.full(n, -np.inf)
    masked[pos[pos >= 0]] = full[pos[pos >= 0]]
    assert got.tolist() == o.topk_positions(masked, 512).tolist()


def test_pool_positions_mask_invisible_tail():
    pos = o.pool_positions(np.array([0, 2, -1]), 19)
    assert pos.tolist() == list(range(8)) + [16, 17, 18] + [-1] * 5 + [-1] * 8


def test_index_k_at_matches_whole_row_decode():
    # keys at arbitrary positions are the rows of the whole-sequence decode
    pc = W.make_paged_cache([300, 1000], seed=11, device="cpu")
    cache = pc.index_k.numpy()
    for b, n in enumerate([300, 1000]):
        pt = pc.page_table[b].numpy()
        full = o.index_k_entries(cache, pt, n)
        pos = np.random.default_rng(b).choice(n, size=min(n, 97), replace=False)
        assert np.array_equal(o.index_k_at(cache, pt, pos), full[pos])
        assert np.array_equal(o.index_k_at(cache, pt, np.arange(n)), full)
