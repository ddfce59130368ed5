"""Parity at the full sizes of the five benchmark workloads.

Each test runs the calls at the workload's full size and in the order the
decode / prefill step issues them, then checks sampled rows against the oracle
(which evaluates them one by one, reading only the pages and records those
rows use) and properties that hold for every row:

  tiny single Full layer (1 query, 4096 keys) ........ everything checked
  decode Full + 3 Reuse, batch 32, 64K..128K ......... rows 0, 13, 31
  decode Reindex at 1M context, batch 16 ............. rows 0, 9, 15
  prefill chunk, 4096 queries after a 256K prefix .... queries 0, 1, 2047, 4095
  38-layer decode step, batch 8, {32K, 256K, 1M x2} .. layers 2, 3, 20, 21, 24, 25
"""
import math

import numpy as np
import pytest
import torch

from gpu_util import (NEAR_TIE_RTOL, assert_attention_close, assert_pool_ok, assert_records_match_except_near_boundaries,
                      assert_scores_close, assert_selection_ok, need_gpu, np_)
from oracle import csa2_oracle as o
from serving_lightning_indexer_gb300 import csa2
from serving_lightning_indexer_gb300 import decode_step as ds
from serving_lightning_indexer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
SCALE = 1 / math.sqrt(512)


# ---------------------------------------------------------------- oracle on sampled rows
def _q(iq, t):
    return o.dequant_q(np_(iq.q_fp8[t]), np_(iq.q_scale[t])), np_(iq.w[t])


def _scores_at(iq, t, pc, b, positions, fp4=False):
    """Oracle scores of indexer row t (sequence b) at the given positions,
    reading only the pages holding them (FP8 or, with fp4, FP4 pages)."""
    pos = np.asarray(positions, dtype=np.int64)
    if len(pos) == 0:
        return np.zeros(0)
    lp = np.unique(pos // 64)
    pages = pc.page_table[b, torch.as_tensor(lp, device=pc.page_table.device)].long()
    sub = np_(pc.index_k[pages])
    remap = np.full(int(lp.max()) + 1, -1, dtype=np.int64)
    remap[lp] = np.arange(len(lp))
    q, w = _q(iq, t)
    return o.index_score_values(q, w, (o.index_k_fp4_at if fp4 else o.index_k_at)(sub, remap, pos))


def _row_scores(iq, t, pc, b, n):
    return _scores_at(iq, t, pc, b, np.arange(n))


def _attn_ref(al, t, main_kv, slot_row):
    """Oracle attention of row t from the records it uses (main and SWA)."""
    def compact(cache, sl):
        sl = np.asarray(sl, dtype=np.int64)
        v = sl[sl >= 0]
        rec = np_(cache[torch.as_tensor(v, device=cache.device)]) if len(v) else np.zeros((0, cache.shape[1]), np.uint8)
        idx = np.full(sl.shape, -1, dtype=np.int64)
        idx[sl >= 0] = np.arange(len(v))
        return rec, idx
    mrec, midx = compact(main_kv, slot_row)
    srec, sidx = compact(al.swa_kv, np_(al.swa_slot[t]))
    q = al.q[t].float().cpu().numpy().astype(np.float64)
    return o.attention_row(q, mrec, midx, srec, sidx, np_(al.sink).astype(np.float64), SCALE)


def _check_attention(al, out, rows, main_kv, slots):
    for t in rows:
        ref, _ = _attn_ref(al, t, main_kv, slots[t])
        assert_attention_close(out[t].double().cpu().numpy(), ref, f"attention row {t}")


def _check_topk_sampled(iq, t, pc, b, n, got_pos, k=512, n_sample=4096, seed=0, fp4=False):
    """Selection check for rows too long for the oracle's full score row: the
    selected positions against a random sample of the others."""
    sel = got_pos[got_pos >= 0]
    assert len(sel) == min(k, n) and len(np.unique(sel)) == len(sel)
    assert sel.min() >= 0 and sel.max() < n
    rng = np.random.default_rng(seed)
    oth = np.setdiff1d(rng.choice(n, size=min(n, n_sample), replace=False), sel)
    s_sel, s_oth = _scores_at(iq, t, pc, b, sel, fp4), _scores_at(iq, t, pc, b, oth, fp4)
    thr = s_sel.min()
    assert s_oth.max() <= thr + NEAR_TIE_RTOL * abs(thr), \
        f"row {t}: an unselected key scores {s_oth.max()} above the selection's minimum {thr}"


def _check_slots(pos, slot, pt_row):
    assert np.array_equal(slot, o.slots_of(pos, np_(pt_row)))


def _all_rows_valid(pos, slot, n_vis, k=512):
    """Every row: min(k, n) distinct positions inside [0, n), then -1; slot -1 exactly where pos is."""
    pos, slot, n_vis = np_(pos), np_(slot), np_(n_vis)
    for t in range(pos.shape[0]):
        m = min(k, int(n_vis[t]))
        p = pos[t]
        assert (p[:m] >= 0).all() and (p[m:] == -1).all()
        assert len(np.unique(p[:m])) == m and p[:m].max() < n_vis[t]
        assert np.array_equal(slot[t] < 0, p < 0)


# ---------------------------------------------------------------- tiny single Full layer
def test_tiny_single_full_layer_everything():
    dev = need_gpu()
    n = 4096
    pc = W.make_paged_cache([n], seed=0, device=dev)
    iq = W.make_indexer_query(1, seed=1, device=dev)
    al = W.make_attn_layer(1, seed=2, device=dev)
    scores = torch.empty(1, n, dtype=torch.float32, device=dev)
    r = csa2.rows(1, 1, n_visible=pc.n_entries)
    csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores)
    pos = torch.empty(1, 512, dtype=torch.int32, device=dev)
    slot = torch.empty_like(pos)
    csa2.topk_with_candidates(scores, r, 512, pos, slot, pc.page_table)
    out = torch.empty(1, 64, 512, dtype=torch.float32, device=dev)
    lse = torch.empty(1, 64, dtype=torch.float32, device=dev)
    csa2.sparse_attn(al.q, pc.main_kv, slot, al.swa_kv, al.swa_slot, al.sink, out, lse)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    ref = _row_scores(iq, 0, pc, 0, n)
    assert_scores_close(np_(scores[0]), ref, "scores")
    assert_selection_ok(np_(pos[0]), ref, 512)
    _check_slots(np_(pos[0]), np_(slot[0]), pc.page_table[0])
    ref_o, ref_l = _attn_ref(al, 0, pc.main_kv, np_(slot[0]))
    assert_attention_close(np_(out[0]).astype(np.float64), ref_o)
    assert np.abs(np_(lse[0]) - ref_l).max() < 2e-3


# ---------------------------------------------------------------- decode Full + 3 Reuse, batch 32
def test_decode_full_and_reuse_batch32_64k_128k():
    dev = need_gpu()
    lengths = W.config_lengths(1)
    B = len(lengths)
    pc = W.make_paged_cache(lengths, seed=100, device=dev)
    iq = W.make_indexer_query(B, seed=101, device=dev)
    layers = [W.make_attn_layer(B, seed=110 + i, device=dev) for i in range(4)]   # Full + 3 Reuse
    ld = (max(lengths) + 127) // 128 * 128
    scores = torch.empty(B, ld, dtype=torch.float32, device=dev)
    bm = torch.empty(B, ld // 8, dtype=torch.float32, device=dev)
    hist = torch.zeros(2, B, 2048, dtype=torch.int32, device=dev)
    r = csa2.rows(B, B, n_visible=pc.n_entries)
    pos = torch.empty(B, 512, dtype=torch.int32, device=dev)
    slot = torch.empty_like(pos)
    pool = torch.empty(B, 2048, dtype=torch.int32, device=dev)
    csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores, bm, hist=hist)
    csa2.topk_with_candidates(scores, r, 512, pos, slot, pc.page_table, bm, pool, hist=hist)
    outs = []
    for al in layers:
        outs.append(torch.empty(B, 64, 512, dtype=torch.bfloat16, device=dev))
        csa2.sparse_attn(al.q, pc.main_kv, slot, al.swa_kv, al.swa_slot, al.sink, outs[-1])
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    _all_rows_valid(pos, slot, pc.n_entries)
    sc_np, pos_np, slot_np, pool_np = np_(scores), np_(pos), np_(slot), np_(pool)
    rows = [0, 13, 31]
    for b in rows:
        n = lengths[b]
        ref = _row_scores(iq, b, pc, b, n)
        assert_scores_close(sc_np[b, :n], ref, f"scores row {b}")
        assert_selection_ok(pos_np[b], ref, 512, f"top-k row {b}")
        _check_slots(pos_np[b], slot_np[b], pc.page_table[b])
        # the pool is exactly the oracle's pool of the kernel's own block maxima,
        # and the float64 oracle's pool up to near-ties
        bmax = o.block_maxima(sc_np[b, :n].astype(np.float64), n)
        assert np.array_equal(pool_np[b], o.candidate_pool(bmax)), f"pool row {b}"
        assert_pool_ok(pool_np[b], o.block_maxima(ref, n), what=f"pool row {b} (float64)")
    for al, out in zip(layers, outs):
        _check_attention(al, out, rows, pc.main_kv, slot_np)


# ---------------------------------------------------------------- decode Reindex at 1M, batch 16
def test_decode_reindex_1m_batch16_planted():
    dev = need_gpu()
    lengths = W.config_lengths(2)
    B = len(lengths)
    iq = W.make_indexer_query(B, seed=201, device=dev)
    # 10% of the blocks get a +3 sigma shift along the Reindex query's weighted direction
    qd = o.FP8[np_(iq.q_fp8).astype(np.int64)] * np_(iq.q_scale)[:, :, None]
    dirs = torch.tensor((np_(iq.w)[:, :, None] * qd).sum(axis=1), dtype=torch.float32, device=dev)
    pc = W.make_paged_cache(lengths, seed=200, device=dev, plant_dirs=dirs, plant_frac=0.1, plant_shift=3.0)
    pool = W.make_pool(lengths, seed=202, device=dev)
    layers = [W.make_attn_layer(B, seed=210 + i, device=dev) for i in range(4)]   # Reindex + 3 Reuse
    r = csa2.rows(B, B, n_visible=pc.n_entries)
    pos = torch.empty(B, 512, dtype=torch.int32, device=dev)
    slot = torch.empty_like(pos)
    ps = torch.empty(B, 2048 * 8, dtype=torch.float32, device=dev)
    csa2.reindex(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, pool, 512, pos, slot, ps)
    outs = []
    for al in layers:
        outs.append(torch.empty(B, 64, 512, dtype=torch.bfloat16, device=dev))
        csa2.sparse_attn(al.q, pc.main_kv, slot, al.swa_kv, al.swa_slot, al.sink, outs[-1])
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    _all_rows_valid(pos, slot, pc.n_entries)
    pos_np, slot_np, ps_np, pool_np = np_(pos), np_(slot), np_(ps), np_(pool)
    rows = [0, 9, 15]
    for b in rows:
        n = lengths[b]
        cand = o.pool_positions(pool_np[b], n)
        ok = cand >= 0
        ref = np.full(len(cand), -np.inf)
        ref[ok] = _scores_at(iq, b, pc, b, cand[ok])
        assert_scores_close(ps_np[b], ref, f"candidate scores row {b}")
        full = np.full(n, -np.inf)
        full[cand[ok]] = ref[ok]
        assert_selection_ok(pos_np[b], full, 512, f"reindex top-k row {b}")
        _check_slots(pos_np[b], slot_np[b], pc.page_table[b])
        assert np.isin(pos_np[b][pos_np[b] >= 0] // 8, pool_np[b]).all()
        # the planted shift makes the selection non-trivial: many picks are planted blocks
        planted = np.isin(pos_np[b] // 8, np_(pc.planted[b]))
        assert planted.mean() > 0.3
    for al, out in zip(layers, outs):
        _check_attention(al, out, rows, pc.main_kv, slot_np)


# ---------------------------------------------------------------- prefill chunk after a 256K prefix
def test_prefill_chunk_4096_after_256k_prefix():
    dev = need_gpu()
    m, prefix, T = 2, 1 << 18, 4096
    n_tok = prefix + T
    n_ent = n_tok // m                                     # 128K + 2K entries
    pc = W.make_paged_cache([n_ent], seed=300, device=dev)
    # main-KV entries of the whole context built by the 2-token compression
    Cm, Z, gamma = W.make_compress_inputs(n_tok, seed=301, device=dev)
    csa2.compress_m2(Cm, Z, m, gamma, pc.main_kv, page_table=pc.page_table[0].contiguous(), first_entry=0)
    iq = W.make_indexer_query(T, seed=302, device=dev)
    row_pos = torch.arange(prefix, n_tok, dtype=torch.int32, device=dev)
    r = csa2.rows(T, 1, row_seq=torch.zeros(T, dtype=torch.int32, device=dev), row_pos=row_pos, ratio_m=m)
    ld = (n_ent + 127) // 128 * 128
    scores = torch.empty(T, ld, dtype=torch.float32, device=dev)
    csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores)
    pos = torch.empty(T, 512, dtype=torch.int32, device=dev)
    slot = torch.empty_like(pos)
    csa2.topk_with_candidates(scores, r, 512, pos, slot, pc.page_table)
    # SWA window of query t: the 128 raw tokens ending at it (records t .. t+127)
    al = W.make_attn_layer(T, seed=303, device=dev, swa_positions=[(t, 128) for t in range(T)],
                           n_swa_records=T + 127)
    out = torch.empty(T, 64, 512, dtype=torch.bfloat16, device=dev)
    csa2.sparse_attn(al.q, pc.main_kv, slot, al.swa_kv, al.swa_slot, al.sink, out)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    vis = torch.tensor([o.visible_entries(p, m) for p in range(prefix, n_tok)], dtype=torch.int32)
    _all_rows_valid(pos, slot, vis)
    # compression: every one of the n_ent entry records against the float64 oracle's
    # entry build, in chunks (bit-exact except next to a rounding boundary)
    C_all, Z_all, g64 = np_(Cm.float()), np_(Z.float()), np_(gamma).astype(np.float64)
    kv_all = np_(pc.main_kv)
    slots_all = o.slots_of(np.arange(n_ent), np_(pc.page_table[0]))
    for e0 in range(0, n_ent, 8192):
        es = np.arange(e0, min(n_ent, e0 + 8192))
        lat = o.compress_latent(C_all[e0 * m:(es[-1] + 1) * m].astype(np.float64),
                                Z_all[e0 * m:(es[-1] + 1) * m].astype(np.float64), m, g64, 1e-6, es * m, 10000.0)
        assert_records_match_except_near_boundaries(kv_all[slots_all[es]], lat)
    # indexer, selection and attention of sampled queries
    sc_np, pos_np, slot_np = np_(scores), np_(pos), np_(slot)
    rows = [0, 1, T // 2 - 1, T - 1]
    for t in rows:
        e = int(vis[t])
        ref = _row_scores(iq, t, pc, 0, e)
        assert_scores_close(sc_np[t, :e], ref, f"scores query {t}")
        assert np.all(np.isneginf(sc_np[t, e:min(ld, (e + 127) // 128 * 128)]))
        assert_selection_ok(pos_np[t], ref, 512, f"top-k query {t}")
        _check_slots(pos_np[t], slot_np[t], pc.page_table[0])
    _check_attention(al, out, rows, pc.main_kv, slot_np)


# ---------------------------------------------------------------- the 38-layer decode step
def test_decode_step_38_layers_sampled():
    dev = need_gpu()
    step = ds.DecodeStep(W.config_lengths(4), seed=7, device=dev)
    b = step.buf
    cap = {}

    def grab(l):
        ci = ds.cache_of(l)
        if ds.role_of(l) == "full":
            cap[l] = dict(scores=np_(b.scores).copy(), pos=np_(b.topk_pos).copy(), slot=np_(b.topk_slot[ci]).copy(),
                          pool=np_(b.pool).copy() if ci == 3 else None)
        elif ds.role_of(l) == "reindex":
            cap[l] = dict(pos=np_(b.topk_pos).copy(), slot=np_(b.topk_slot[ci]).copy())
        else:
            cap[l] = dict(slot=np_(b.topk_slot[ci]).copy())

    step.after_layer = grab
    step.run()
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0

    # Full layers 2 (encoder, m=2; rows of 16K, 128K and 512K entries) and 20
    # (decoder, m=1, with the pool; rows of 32K and 1M entries): every score of
    # the row against the float64 oracle, the top-512 and the pool under the
    # near-tie rule
    for l, rows in ((2, [0, 1, 3]), (20, [0, 2])):
        c = step.caches[ds.cache_of(l)]
        li = step.inputs[l]
        k = cap[l]
        for t in rows:
            n = c.entries[t]
            ref = _row_scores(li.iq, t, c.pc, t, n)
            assert_scores_close(k["scores"][t, :n], ref, f"layer {l} scores row {t}")
            assert_selection_ok(k["pos"][t], ref, 512, f"layer {l} top-k row {t}")
            _check_slots(k["pos"][t], k["slot"][t], c.pc.page_table[t])
            if k["pool"] is not None:
                bmax = o.block_maxima(k["scores"][t, :n].astype(np.float64), n)
                assert np.array_equal(k["pool"][t], o.candidate_pool(bmax)), f"pool row {t}"
                assert_pool_ok(k["pool"][t], o.block_maxima(ref, n), what=f"layer {l} pool row {t} (float64)")
            del ref
        # the Full layer wrote each sequence's newest main-KV entry
        m = c.ratio_m
        lat = o.compress_latent(li.C.float().cpu().numpy().astype(np.float64),
                                li.Z.float().cpu().numpy().astype(np.float64) if m == 2 else None, m,
                                np_(li.gamma).astype(np.float64), 1e-6, np_(c.entry_pos_new).astype(np.float64),
                                10000.0)
        want = o.fp4_encode_records(lat)
        got = np_(c.pc.main_kv[c.entry_slot_new.long()])
        stp = np.repeat(o.ue8m0(want[:, 256:272]), 32, axis=1)
        assert np.all(np.abs(o.main_kv_records(got, np.arange(step.B)) - o.main_kv_records(want, np.arange(step.B)))
                      <= 0.5 * stp + 1e-12)

    # Reindex layer 24 over layer 20's pool
    c = step.caches[3]
    li = step.inputs[24]
    for t in (1, 3):
        n = c.entries[t]
        cand = o.pool_positions(cap[20]["pool"][t], n)
        ok = cand >= 0
        full = np.full(n, -np.inf)
        full[cand[ok]] = _scores_at(li.iq, t, c.pc, t, cand[ok])
        assert_selection_ok(cap[24]["pos"][t], full, 512, f"layer 24 row {t}")
        _check_slots(cap[24]["pos"][t], cap[24]["slot"][t], c.pc.page_table[t])

    # attention of Full, Reuse and Reindex layers with the slots they used
    for l, rows in ((2, [0]), (3, [1]), (20, [2]), (21, [3]), (24, [1]), (25, [6])):
        c = step.caches[ds.cache_of(l)]
        _check_attention(step.inputs[l].attn, b.out[l], rows, c.pc.main_kv, cap[l]["slot"])


# ---------------------------------------------------------------- FP4 index keys, 1M context
def test_decode_fp4_index_keys_batch8_1m():
    """The decoder Full layer of the 38-layer step (batch 8, {32K, 256K, 1M x2} x 2)
    with FP4 index-K pages: scan with block maxima and histograms, then top-512
    and the candidate pool, checked on sampled rows."""
    dev = need_gpu()
    lengths = [32768, 262144, 1 << 20, 1 << 20] * 2
    B = len(lengths)
    pc = W.make_paged_cache(lengths, seed=31, device=dev, with_main=False, index_fp4=True)
    iq = W.make_indexer_query(B, seed=32, device=dev)
    nvis = torch.tensor(lengths, dtype=torch.int32, device=dev)
    r = csa2.rows(B, B, n_visible=nvis)
    ld = max(lengths)
    scores = torch.empty(B, ld, dtype=torch.float32, device=dev)
    bm = torch.empty(B, ld // 8, dtype=torch.float32, device=dev)
    hist = torch.zeros(2, B, 2048, dtype=torch.int32, device=dev)
    pos = torch.empty(B, 512, dtype=torch.int32, device=dev)
    slot = torch.empty(B, 512, dtype=torch.int32, device=dev)
    pool = torch.empty(B, 2048, dtype=torch.int32, device=dev)
    csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores, bm, hist=hist)
    csa2.topk_with_candidates(scores, r, 512, pos, slot, pc.page_table, bm, pool, hist=hist)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    _all_rows_valid(pos, slot, nvis)
    rng = np.random.default_rng(33)
    for b in (0, 3, 6):
        n = lengths[b]
        sample = np.sort(rng.choice(n, size=min(n, 8192), replace=False))
        got = np_(scores[b])[sample]
        assert_scores_close(got, _scores_at(iq, b, pc, b, sample, fp4=True), f"fp4 row {b}")
        p = np_(pos[b])
        _check_topk_sampled(iq, b, pc, b, n, p, seed=b, fp4=True)
        _check_slots(p, np_(slot[b]), pc.page_table[b])
        # the pool: 2048 ascending distinct blocks with the newest block, ⊇ the top-k blocks
        pb = np_(pool[b])
        assert len(pb) == 2048 and (np.diff(pb) > 0).all() and pb[-1] == (n - 1) // 8
        assert set((p // 8).tolist()) <= set(pb.tolist())
