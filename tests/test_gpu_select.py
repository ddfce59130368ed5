"""GPU parity of csa2_topk_with_candidates and csa2_reindex.

Selection on given fp32 scores is bit-exact against the oracle run on the same
fp32 values (both sides decide in fp32); end-to-end selection from the FP8
cache follows the near-tie rule."""
import numpy as np
import pytest
import torch

from gpu_util import assert_scores_close, assert_selection_ok, need_gpu, np_
from oracle import csa2_oracle as o
from serving_lightning_indexer_gb300 import csa2
from serving_lightning_indexer_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run_topk(scores_np, lengths, k=512, pool_n=2048, pt=None):
    dev = need_gpu()
    T, ld = scores_np.shape
    scores = torch.tensor(scores_np, dtype=torch.float32, device=dev)
    # block maxima of the given scores over the visible part, as the scorer writes them
    nbld = (ld + 7) // 8 + 3 & ~3
    bm_np = np.full((T, nbld), -np.inf, dtype=np.float32)
    for t, n in enumerate(lengths):
        for j in range((n + 7) // 8):
            bm_np[t, j] = scores_np[t, 8 * j:min(8 * j + 8, n)].max()
    bm = torch.tensor(bm_np, device=dev)
    if pt is None:
        pt_np = np.stack([np.random.default_rng(t).permutation(4096 * 4)[: (ld + 63) // 64] for t in range(T)])
    else:
        pt_np = pt
    ptab = torch.tensor(pt_np, dtype=torch.int32, device=dev)
    nvis = torch.tensor(lengths, dtype=torch.int32, device=dev)
    pos = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    slot = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    pool = torch.full((T, pool_n), -7, dtype=torch.int32, device=dev)
    csa2.topk_with_candidates(scores, csa2.rows(T, T, n_visible=nvis), k, pos, slot, ptab, bm, pool)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    return np_(pos), np_(slot), np_(pool), bm_np, pt_np


def _check_exact(scores_np, lengths, k=512, pool_n=2048):
    pos, slot, pool, bm_np, pt = _run_topk(scores_np, lengths, k, pool_n)
    for t, n in enumerate(lengths):
        s = scores_np[t, :n]
        want = o.topk_positions(s, k)
        assert pos[t].tolist() == want.tolist(), f"row {t}: positions differ"
        assert slot[t].tolist() == o.slots_of(want, pt[t]).tolist(), f"row {t}: slots differ"
        wpool = o.candidate_pool(bm_np[t, :(n + 7) // 8].astype(np.float64), pool_n)
        assert pool[t].tolist() == wpool.tolist(), f"row {t}: pool differs"


def test_exact_short_and_ragged_rows():
    rng = np.random.default_rng(0)
    lengths = [0, 1, 7, 300, 511, 512, 513, 4000, 16384]
    ld = 16384
    s = rng.normal(size=(len(lengths), ld)).astype(np.float32)
    _check_exact(s, lengths)


def test_exact_with_many_ties():
    rng = np.random.default_rng(1)
    lengths = [5000, 12000]
    s = np.round(rng.normal(size=(2, 12000)), 1).astype(np.float32)
    _check_exact(s, lengths)


def test_exact_long_rows_streaming_passes():
    rng = np.random.default_rng(2)
    lengths = [300_000, 65_537, 200_003]
    ld = 300_032
    s = rng.normal(size=(3, ld)).astype(np.float32)
    _check_exact(s, lengths)


def test_exact_crowded_threshold_bin_refines():
    # a narrow distribution far from zero puts thousands of scores in one 11-bit bin
    rng = np.random.default_rng(3)
    lengths = [400_000, 150_000]
    s = (100.0 + 0.01 * rng.normal(size=(2, 400_000))).astype(np.float32)
    _check_exact(s, lengths)


def test_exact_massive_ties_fall_back_to_streaming_select():
    lengths = [100_000, 40_000]
    s = np.full((2, 100_000), 3.5, dtype=np.float32)
    s[0, 99_000] = 4.0
    pos, slot, pool, bm_np, pt = _run_topk(s, lengths)
    # the best score and the 511 lowest tied positions, in ascending position order
    assert pos[0].tolist() == list(range(511)) + [99_000]
    assert pos[0].tolist() == o.topk_positions(s[0, :100_000].astype(np.float64), 512).tolist()
    assert pos[1].tolist() == list(range(512))
    assert pool[0].tolist() == o.candidate_pool(bm_np[0, :12_500].astype(np.float64), 2048).tolist()


@pytest.mark.parametrize("T,ld,kind", [
    (2500, 20000, "normal"),    # many long rows: hist CTAs of 65,536 scores, filter
                                # CTAs of several 4096-score chunks, the threshold
                                # bin found once per row
    (2500, 20000, "ties"),      # crowded threshold bin, ties broken by position
    (400, 20000, "equal"),      # every score equal: the candidate lists overflow
                                # and the streaming radix select takes over
    (400, 20000, "sparse"),     # 300 selectable scores a row: all of them
    (300, 280000, "normal"),    # fewer, longer rows, the same multi-chunk passes
])
def test_exact_many_long_rows(T, ld, kind):
    # long rows without histograms (the hist, filter and final passes)
    dev = need_gpu()
    rng = np.random.default_rng(T + ld + len(kind))
    lengths = rng.integers(ld * 4 // 5, ld + 1, size=T)
    lengths[::97] = ld
    s = rng.normal(size=(T, ld)).astype(np.float32)
    if kind == "ties":
        s = (np.round(s * 2) / 2).astype(np.float32)
    elif kind == "equal":
        s[:] = 1.0
    elif kind == "sparse":
        keep = np.zeros((T, ld), dtype=bool)
        for t in range(T):
            keep[t, rng.choice(int(lengths[t]), size=300, replace=False)] = True
        s[~keep] = -np.inf
    scores = torch.tensor(s, device=dev)
    pos = torch.full((T, 512), -7, dtype=torch.int32, device=dev)
    nvis = torch.tensor(lengths, dtype=torch.int32, device=dev)
    csa2.topk_with_candidates(scores, csa2.rows(T, T, n_visible=nvis), 512, pos)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    got = np_(pos)
    step = max(1, T // 100)
    for t in sorted(set(range(0, T, step)) | {1, T - 1}):
        want = o.topk_positions(s[t, :lengths[t]], 512)
        assert got[t].tolist() == want.tolist(), f"row {t} ({kind}): positions differ"


def test_exact_all_excluded_rows():
    s = np.full((2, 1024), -np.inf, dtype=np.float32)
    s[1, 5] = 1.0
    pos, slot, pool, _, _ = _run_topk(s, [1000, 1000])
    assert (pos[0] == -1).all() and (slot[0] == -1).all()
    assert pos[1].tolist() == [5] + [-1] * 511


def test_end_to_end_selection_from_cache():
    dev = need_gpu()
    lengths = [20000, 17000]
    pc = W.make_paged_cache(lengths, seed=11, device=dev, with_main=False)
    iq = W.make_indexer_query(2, seed=12, device=dev)
    nvis = torch.tensor(lengths, dtype=torch.int32, device=dev)
    r = csa2.rows(2, 2, n_visible=nvis)
    scores = torch.empty(2, 20096, dtype=torch.float32, device=dev)
    bm = torch.empty(2, 2512, dtype=torch.float32, device=dev)
    csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores, bm)
    pos = torch.empty(2, 512, dtype=torch.int32, device=dev)
    pool = torch.empty(2, 2048, dtype=torch.int32, device=dev)
    csa2.topk_with_candidates(scores, r, 512, pos, None, None, bm, pool)
    torch.cuda.synchronize()
    cache, pt = np_(pc.index_k), np_(pc.page_table)
    for b, n in enumerate(lengths):
        ref = o.index_scores_row(np_(iq.q_fp8[b]), np_(iq.q_scale[b]), np_(iq.w[b]), cache, pt[b], n)
        assert_selection_ok(np_(pos[b]), ref, 512)
        # the newest block is forced: give it a value above every block maximum
        bmx = o.block_maxima(ref, n)
        bmx[-1] = bmx.max() + 1.0
        assert_selection_ok(np_(pool[b]), bmx, 2048, "pool")
        p = np_(pool[b])
        assert np.all(np.diff(p[p >= 0]) > 0)
        assert set((np_(pos[b]) // 8).tolist()) <= set(p.tolist())


@pytest.mark.parametrize("lengths", [[3000, 16384], [40000, 1_000_003]])
def test_reindex_matches_oracle(lengths):
    dev = need_gpu()
    B = len(lengths)
    pc = W.make_paged_cache(lengths, seed=13, device=dev, with_main=False)
    iq = W.make_indexer_query(B, seed=14, device=dev)
    pool = W.make_pool(lengths, seed=15, device=dev)
    nvis = torch.tensor(lengths, dtype=torch.int32, device=dev)
    r = csa2.rows(B, B, n_visible=nvis)
    pos = torch.empty(B, 512, dtype=torch.int32, device=dev)
    slot = torch.empty(B, 512, dtype=torch.int32, device=dev)
    ps = torch.empty(B, 2048 * 8, dtype=torch.float32, device=dev)
    csa2.reindex(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, pool, 512, pos, slot, ps)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    cache, pt = np_(pc.index_k), np_(pc.page_table)
    for b, n in enumerate(lengths):
        args = (np_(iq.q_fp8[b]), np_(iq.q_scale[b]), np_(iq.w[b]), cache, pt[b], n)
        ref = o.reindex_scores(*args, np_(pool[b]))
        assert_scores_close(np_(ps[b]), ref, f"pool scores {b}")
        # selection on the kernel's own fp32 pool scores is exact
        full = np.full(n, -np.inf, dtype=np.float32)
        pp = o.pool_positions(np_(pool[b]), n)
        full[pp[pp >= 0]] = np_(ps[b])[pp >= 0]
        want = o.topk_positions(full, 512)
        assert np_(pos[b]).tolist() == want.tolist()
        assert np_(slot[b]).tolist() == o.slots_of(want, pt[b]).tolist()
        # and against the float64 oracle under the near-tie rule
        reff = np.full(n, -np.inf)
        reff[pp[pp >= 0]] = ref[pp >= 0]
        assert_selection_ok(np_(pos[b]), reff, 512, "reindex")


def test_reindex_equals_full_topk_when_pool_covers_all():
    dev = need_gpu()
    n = 12000
    pc = W.make_paged_cache([n], seed=16, device=dev, with_main=False)
    iq = W.make_indexer_query(1, seed=17, device=dev)
    nvis = torch.tensor([n], dtype=torch.int32, device=dev)
    r = csa2.rows(1, 1, n_visible=nvis)
    scores = torch.empty(1, 12032, dtype=torch.float32, device=dev)
    bm = torch.empty(1, 1504, dtype=torch.float32, device=dev)
    csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores, bm)
    pos = torch.empty(1, 512, dtype=torch.int32, device=dev)
    pool = torch.empty(1, 2048, dtype=torch.int32, device=dev)
    csa2.topk_with_candidates(scores, r, 512, pos, None, None, bm, pool)
    rpos = torch.empty(1, 512, dtype=torch.int32, device=dev)
    csa2.reindex(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, pool, 512, rpos)
    torch.cuda.synchronize()
    assert (np_(pool[0])[:1500] == np.arange(1500)).all()
    assert np_(rpos[0]).tolist() == np_(pos[0]).tolist()


def test_fused_histograms_give_identical_selection():
    # the decode scan's key histograms, passed on to the top-k, must not change
    # any result; the top-k returns them to zero, so the same buffer serves the
    # next layer's scan without a memset
    dev = need_gpu()
    lengths = [70000, 140001, 20000]
    B = len(lengths)
    pc = W.make_paged_cache(lengths, seed=21, device=dev, with_main=False)
    iq = W.make_indexer_query(B, seed=22, device=dev)
    r = csa2.rows(B, B, n_visible=torch.tensor(lengths, dtype=torch.int32, device=dev))
    ld = 140032
    scores = torch.empty(B, ld, dtype=torch.float32, device=dev)
    bm = torch.empty(B, ld // 8, dtype=torch.float32, device=dev)
    hist = torch.zeros((2, B, 2048), dtype=torch.int32, device=dev)
    runs = []
    for rep in range(2):
        csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores, bm, hist=hist)
        h = np_(hist).astype(np.int64)
        outs = []
        for hh in (None, hist):
            pos = torch.empty(B, 512, dtype=torch.int32, device=dev)
            slot = torch.empty_like(pos)
            pool = torch.empty(B, 2048, dtype=torch.int32, device=dev)
            csa2.topk_with_candidates(scores, r, 512, pos, slot, pc.page_table, bm, pool, hist=hh)
            outs.append((np_(pos), np_(slot), np_(pool)))
        torch.cuda.synchronize()
        assert csa2.check_device_error() == 0
        for a, b in zip(*outs):
            assert np.array_equal(a, b)
        assert not np_(hist).any(), "the top-k call leaves the histograms at zero"
        runs.append(outs[1])
        # the histograms count exactly the visible scores and block maxima, in their top-11-bit bins
        for b_, n in enumerate(lengths):
            s = np_(scores[b_, :n])
            key = s.view(np.uint32).astype(np.int64)
            key = np.where(key & 0x80000000, ~key & 0xFFFFFFFF, key | 0x80000000)
            assert np.array_equal(h[0, b_], np.bincount(key >> 21, minlength=2048))
            nb = (n + 7) // 8
            bmk = np_(bm[b_, :nb]).view(np.uint32).astype(np.int64)
            bmk = np.where(bmk & 0x80000000, ~bmk & 0xFFFFFFFF, bmk | 0x80000000)
            bmk[-1] = 0xFFFFFFFF
            assert np.array_equal(h[1, b_], np.bincount(bmk >> 21, minlength=2048))
    for a, b in zip(*runs):
        assert np.array_equal(a, b), "a second scan + top-k on the returned buffer gives the same selection"
    # without a pool the top-k also clears the block-maximum half
    csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores, bm, hist=hist)
    pos = torch.empty(B, 512, dtype=torch.int32, device=dev)
    csa2.topk_with_candidates(scores, r, 512, pos, None, None, hist=hist)
    torch.cuda.synchronize()
    assert not np_(hist).any()


def test_reindex_fp4_index_keys_match_oracle():
    dev = need_gpu()
    lengths = [30000, 16384 * 8 + 5, 700]
    B = len(lengths)
    pc = W.make_paged_cache(lengths, seed=23, device=dev, with_main=False, index_fp4=True)
    iq = W.make_indexer_query(B, seed=24, device=dev)
    pool = W.make_pool(lengths, seed=25, device=dev)
    r = csa2.rows(B, B, n_visible=torch.tensor(lengths, dtype=torch.int32, device=dev))
    pos = torch.empty(B, 512, dtype=torch.int32, device=dev)
    slot = torch.empty(B, 512, dtype=torch.int32, device=dev)
    ps = torch.empty(B, 2048 * 8, dtype=torch.float32, device=dev)
    csa2.reindex(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, pool, 512, pos, slot, ps)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    cache, pt = np_(pc.index_k), np_(pc.page_table)
    for b, n in enumerate(lengths):
        ref = o.reindex_scores(np_(iq.q_fp8[b]), np_(iq.q_scale[b]), np_(iq.w[b]), cache, pt[b], n,
                               np_(pool[b]), fp4=True)
        assert_scores_close(np_(ps[b]), ref, f"fp4 pool scores {b}")
        full = np.full(n, -np.inf, dtype=np.float32)
        pp = o.pool_positions(np_(pool[b]), n)
        full[pp[pp >= 0]] = np_(ps[b])[pp >= 0]
        want = o.topk_positions(full, 512)
        assert np_(pos[b]).tolist() == want.tolist()
        assert np_(slot[b]).tolist() == o.slots_of(want, pt[b]).tolist()


@pytest.mark.parametrize("lengths", [[300, 511, 5000, 16384], [70_001, 200_000, 16_385]])
def test_best_first_order(lengths):
    # order = 1 (CSA2_ORDER_SCORE): the same top-k set, reported score
    # descending with ties to the lower position, so every prefix k' of the row
    # is the row's top-k'; slots follow their positions; the pool is unchanged
    dev = need_gpu()
    rng = np.random.default_rng(len(lengths))
    T, ld = len(lengths), (max(lengths) + 3) & ~3
    s = rng.normal(size=(T, ld)).astype(np.float32)
    s[:, 100:140] = 0.25                                 # ties inside the selection
    scores = torch.tensor(s, device=dev)
    nbld = (ld + 7) // 8 + 3 & ~3
    bm_np = np.full((T, nbld), -np.inf, dtype=np.float32)
    for t, n in enumerate(lengths):
        v = s[t, :n]
        bm_np[t, :(n + 7) // 8] = np.pad(v, (0, -n % 8), constant_values=-np.inf).reshape(-1, 8).max(1)
    bm = torch.tensor(bm_np, device=dev)
    pt_np = np.stack([rng.permutation(1 << 16)[: (ld + 63) // 64] for _ in range(T)]).astype(np.int32)
    pt = torch.tensor(pt_np, device=dev)
    r = csa2.rows(T, T, n_visible=torch.tensor(lengths, dtype=torch.int32, device=dev))
    outs = []
    for order in (0, 1):
        pos = torch.full((T, 512), -7, dtype=torch.int32, device=dev)
        slot = torch.full((T, 512), -7, dtype=torch.int32, device=dev)
        pool = torch.full((T, 2048), -7, dtype=torch.int32, device=dev)
        csa2.topk_with_candidates(scores, r, 512, pos, slot, pt, bm, pool, order=order)
        outs.append((np_(pos), np_(slot), np_(pool)))
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    (p0, s0, q0), (p1, s1, q1) = outs
    assert np.array_equal(q0, q1)
    for t, n in enumerate(lengths):
        want = o.topk_positions(s[t, :n], 512)
        assert p0[t].tolist() == want.tolist()
        sel = want[want >= 0]
        best = sel[np.lexsort((sel, -s[t, sel].astype(np.float64)))]   # score desc, position asc
        got = p1[t]
        assert got[:len(best)].tolist() == best.tolist() and (got[len(best):] == -1).all(), f"row {t}"
        assert s1[t].tolist() == o.slots_of(got, pt_np[t]).tolist()


def test_reindex_best_first_order():
    dev = need_gpu()
    lengths = [30000, 16384 * 8 + 5, 700]
    B = len(lengths)
    pc = W.make_paged_cache(lengths, seed=41, device=dev, with_main=False)
    iq = W.make_indexer_query(B, seed=42, device=dev)
    pool = W.make_pool(lengths, seed=43, device=dev)
    r = csa2.rows(B, B, n_visible=torch.tensor(lengths, dtype=torch.int32, device=dev))
    res = []
    for order in (0, 1):
        pos = torch.empty(B, 512, dtype=torch.int32, device=dev)
        ps = torch.empty(B, 2048 * 8, dtype=torch.float32, device=dev)
        csa2.reindex(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, pool, 512, pos, None, ps, order=order)
        res.append((np_(pos), np_(ps)))
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    (p0, ps0), (p1, ps1) = res
    for b, n in enumerate(lengths):
        full = np.full(n, -np.inf, dtype=np.float32)
        pp = o.pool_positions(np_(pool[b]), n)
        full[pp[pp >= 0]] = ps0[b][pp >= 0]
        sel = p0[b][p0[b] >= 0]
        best = sel[np.lexsort((sel, -full[sel].astype(np.float64)))]
        assert p1[b][:len(best)].tolist() == best.tolist(), f"row {b}"

