"""GPU parity of csa2_index_score (decode scan and prefill query-blocked path)."""
import numpy as np
import pytest
import torch

from gpu_util import assert_scores_close, need_gpu, np_
from oracle import csa2_oracle as o
from serving_lightning_indexer_gb300 import csa2
from serving_lightning_indexer_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _decode(lengths, seed, ld=None, with_bm=True, fp4=False, hist=None):
    dev = need_gpu()
    B = len(lengths)
    pc = W.make_paged_cache(lengths, seed=seed, device=dev, with_main=False, index_fp4=fp4)
    iq = W.make_indexer_query(B, seed=seed + 1, device=dev)
    nvis = torch.tensor(lengths, dtype=torch.int32, device=dev)
    ld = ld or ((max(lengths) + 127) // 128 * 128)
    scores = torch.full((B, ld), 7.0, dtype=torch.float32, device=dev)
    bm = torch.full((B, (ld + 7) // 8 + 4), 7.0, dtype=torch.float32, device=dev) if with_bm else None
    r = csa2.rows(B, B, n_visible=nvis)
    csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores, bm, hist=hist)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    return pc, iq, scores, bm


@pytest.mark.parametrize("lengths", [[1], [127, 128, 129], [4096], [100, 1000, 4133, 64, 65, 8191]])
def test_decode_scores_match_oracle(lengths):
    pc, iq, scores, bm = _decode(lengths, seed=len(lengths))
    cache, pt = np_(pc.index_k), np_(pc.page_table)
    for b, n in enumerate(lengths):
        ref = o.index_scores_row(np_(iq.q_fp8[b]), np_(iq.q_scale[b]), np_(iq.w[b]), cache, pt[b], n)
        got = np_(scores[b])
        assert_scores_close(got[:n], ref, f"row {b}")
        tail = got[n:(n + 127) // 128 * 128]
        assert np.all(np.isneginf(tail)), "positions past E must hold -inf inside the last tile"
        # block maxima are exactly the max of the kernel's own scores over visible positions
        nb = (n + 7) // 8
        want = [got[8 * j:min(8 * j + 8, n)].max() for j in range(nb)]
        assert np.array_equal(np_(bm[b, :nb]), np.array(want, dtype=np.float32))
        assert np.all(np_(bm[b, nb:]) == 7.0) or nb * 8 >= bm.shape[1] * 8


def test_decode_row_seq_and_clipped_ld():
    dev = need_gpu()
    lengths = [300, 700]
    pc = W.make_paged_cache(lengths, seed=5, device=dev, with_main=False)
    iq = W.make_indexer_query(3, seed=6, device=dev)
    row_seq = torch.tensor([1, 0, 1], dtype=torch.int32, device=dev)
    nvis = torch.tensor(lengths, dtype=torch.int32, device=dev)
    ld = 512                                  # shorter than sequence 1: written up to ld only
    scores = torch.full((3, ld), 7.0, dtype=torch.float32, device=dev)
    csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table,
                     csa2.rows(3, 2, row_seq=row_seq, n_visible=nvis), scores)
    torch.cuda.synchronize()
    cache, pt = np_(pc.index_k), np_(pc.page_table)
    for t, b in enumerate([1, 0, 1]):
        n = lengths[b]
        ref = o.index_scores_row(np_(iq.q_fp8[t]), np_(iq.q_scale[t]), np_(iq.w[t]), cache, pt[b], n)
        m = min(n, ld)
        assert_scores_close(np_(scores[t, :m]), ref[:m], f"row {t}")


def test_bad_page_id_is_reported_not_faulted():
    dev = need_gpu()
    lengths = [256]
    pc = W.make_paged_cache(lengths, seed=7, device=dev, with_main=False)
    iq = W.make_indexer_query(1, seed=8, device=dev)
    pt = pc.page_table.clone()
    pt[0, 2] = 10_000                         # beyond the cache
    scores = torch.empty(1, 256, dtype=torch.float32, device=dev)
    csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pt,
                     csa2.rows(1, 1, n_visible=torch.tensor([256], dtype=torch.int32, device=dev)), scores)
    assert csa2.check_device_error() == 6
    assert csa2.check_device_error() == 0     # the record is cleared


@pytest.mark.parametrize("T,ratio,n_entries", [(64, 2, 3000), (100, 1, 3000), (203, 2, 20000)])
def test_prefill_query_blocked_path(T, ratio, n_entries):
    dev = need_gpu()
    pc = W.make_paged_cache([n_entries], seed=9, device=dev, with_main=False)
    iq = W.make_indexer_query(T, seed=10, device=dev)
    # queries at the end of the context, causal visibility (pos + 1) // m
    first = n_entries * ratio - T
    row_pos = torch.arange(first, first + T, dtype=torch.int32, device=dev)
    ld = (n_entries + 127) // 128 * 128
    scores = torch.full((T, ld), 7.0, dtype=torch.float32, device=dev)
    bm = torch.full((T, ld // 8), 7.0, dtype=torch.float32, device=dev)
    r = csa2.rows(T, 1, row_seq=torch.zeros(T, dtype=torch.int32, device=dev), row_pos=row_pos, ratio_m=ratio)
    csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores, bm)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    cache, pt = np_(pc.index_k), np_(pc.page_table)
    keys = o.index_k_entries(cache, pt[0], n_entries)
    for t in list(range(0, T, 7)) + [T - 1]:
        e = o.visible_entries(first + t, ratio)
        ref = o.index_score_values(o.dequant_q(np_(iq.q_fp8[t]), np_(iq.q_scale[t])), np_(iq.w[t]), keys[:e])
        got = np_(scores[t])
        assert_scores_close(got[:e], ref, f"row {t}")
        assert np.all(np.isneginf(got[e:min(ld, (e + 127) // 128 * 128)]))
    # block maxima: exactly the max of the kernel's own scores over each block of
    # 8 visible entries; blocks past the visible ones are not written
    s_all, bm_all = np_(scores), np_(bm)
    for t in range(T):
        e = o.visible_entries(first + t, ratio)
        nb = (e + 7) // 8
        want = np.maximum.reduceat(np.where(np.arange(nb * 8) < e, s_all[t, :nb * 8], -np.inf), np.arange(0, nb * 8, 8))
        assert np.array_equal(bm_all[t, :nb], want.astype(np.float32)), f"block maxima of row {t}"
        assert np.all(bm_all[t, nb:] == 7.0), f"row {t}: block maxima written past the visible blocks"


def _check_rows(scores, bm, iq, cache, pt_rows, visible, rows_to_check, fp4, what):
    """Scores of the given rows against the oracle, -inf up to the row's last
    128-entry tile, block maxima equal to the max over the kernel's own scores."""
    ld = scores.shape[1]
    for t in rows_to_check:
        e = visible[t]
        got = np_(scores[t])
        if e:
            ref = o.index_scores_row(np_(iq.q_fp8[t]), np_(iq.q_scale[t]), np_(iq.w[t]), cache, pt_rows[t], e,
                                     fp4=fp4)
            assert_scores_close(got[:e], ref, f"{what} row {t}")
        assert np.all(np.isneginf(got[e:min(ld, (e + 127) // 128 * 128)])), f"{what} row {t}: tail"
        assert np.all(got[(e + 127) // 128 * 128:] == 7.0), f"{what} row {t}: written past its last tile"
        nb = (e + 7) // 8
        want = [got[8 * j:min(8 * j + 8, e)].max() for j in range(nb)]
        assert np.array_equal(np_(bm[t, :nb]), np.array(want, dtype=np.float32)), f"{what} row {t}: block maxima"
        assert np.all(np_(bm[t, nb:]) == 7.0)


@pytest.mark.parametrize("T,ratio,n_entries", [(100, 2, 3000), (2100, 1, 2500)])
def test_prefill_fp4_index_keys_take_the_per_row_scan(T, ratio, n_entries):
    # FP4 pages at a prefill shape (row_pos, one sequence, T >= 64) are scored
    # by the per-row scan, in launches of 2048 rows
    dev = need_gpu()
    pc = W.make_paged_cache([n_entries], seed=31, device=dev, with_main=False, index_fp4=True)
    iq = W.make_indexer_query(T, seed=32, device=dev)
    first = n_entries * ratio - T
    row_pos = torch.arange(first, first + T, dtype=torch.int32, device=dev)
    ld = (n_entries + 127) // 128 * 128 + 128
    scores = torch.full((T, ld), 7.0, dtype=torch.float32, device=dev)
    bm = torch.full((T, ld // 8), 7.0, dtype=torch.float32, device=dev)
    r = csa2.rows(T, 1, row_seq=torch.zeros(T, dtype=torch.int32, device=dev), row_pos=row_pos, ratio_m=ratio)
    csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores, bm)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    pt = np_(pc.page_table)
    visible = [o.visible_entries(first + t, ratio) for t in range(T)]
    rows = sorted(set([0, 1, T // 2, T - 1] + ([2047, 2048] if T > 2048 else [])))
    _check_rows(scores, bm, iq, np_(pc.index_k), [pt[0]] * T, visible, rows, True, "fp4 prefill")


@pytest.mark.parametrize("with_row_seq", [True, False])
def test_per_row_scan_takes_more_than_2048_rows_in_launches(with_row_seq):
    # 2100 rows: launches of rows 0..2047 and 2048..2099.  With row_seq, three
    # sequences shared by the rows; without, every row is its own sequence
    # (page-table rows and n_visible follow the row)
    dev = need_gpu()
    T = 2100
    rng = np.random.default_rng(41)
    lengths = [300, 1000, 129] if with_row_seq else [int(x) for x in rng.integers(1, 300, size=T)]
    pc = W.make_paged_cache(lengths, seed=42, device=dev, with_main=False)
    iq = W.make_indexer_query(T, seed=43, device=dev)
    ld = (max(lengths) + 127) // 128 * 128 + 128
    scores = torch.full((T, ld), 7.0, dtype=torch.float32, device=dev)
    bm = torch.full((T, ld // 8), 7.0, dtype=torch.float32, device=dev)
    nvis = torch.tensor(lengths, dtype=torch.int32, device=dev)
    if with_row_seq:
        seq = rng.integers(0, 3, size=T)
        r = csa2.rows(T, 3, row_seq=torch.tensor(seq, dtype=torch.int32, device=dev), n_visible=nvis)
    else:
        seq = np.arange(T)
        r = csa2.rows(T, T, n_visible=nvis)
    csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores, bm)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    pt = np_(pc.page_table)
    visible = [lengths[seq[t]] for t in range(T)]
    _check_rows(scores, bm, iq, np_(pc.index_k), [pt[seq[t]] for t in range(T)], visible,
                [0, 1, 1000, 2046, 2047, 2048, 2049, 2099], False, "split")


@pytest.mark.parametrize("lengths", [[1], [127, 128, 129], [4096], [100, 1000, 4133, 64, 65, 8191]])
def test_decode_fp4_index_keys_match_oracle(lengths):
    # FP4 index-K pages (e2m1 + ue8m0 per 32 dims): the same scan, the e2m1 keys
    # fed to the tensor cores as 4-bit operands, one accumulator per 32-dim block
    dev = need_gpu()
    hist = torch.zeros(2, len(lengths), 2048, dtype=torch.int32, device=dev)
    pc, iq, scores, bm = _decode(lengths, seed=20 + len(lengths), fp4=True, hist=hist)
    assert pc.index_k.shape[1] == 4352
    cache, pt = np_(pc.index_k), np_(pc.page_table)
    for b, n in enumerate(lengths):
        ref = o.index_scores_row(np_(iq.q_fp8[b]), np_(iq.q_scale[b]), np_(iq.w[b]), cache, pt[b], n, fp4=True)
        got = np_(scores[b])
        assert_scores_close(got[:n], ref, f"fp4 row {b}")
        assert np.all(np.isneginf(got[n:(n + 127) // 128 * 128]))
        nb = (n + 7) // 8
        want = [got[8 * j:min(8 * j + 8, n)].max() for j in range(nb)]
        assert np.array_equal(np_(bm[b, :nb]), np.array(want, dtype=np.float32))
        # the score histogram counts every visible score once
        assert int(np_(hist[0, b]).sum()) == n
