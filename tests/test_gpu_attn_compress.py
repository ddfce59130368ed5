"""GPU parity of csa2_sparse_attn and csa2_compress_m2."""
import math

import numpy as np
import pytest
import torch

from gpu_util import assert_attention_close, assert_records_match_except_near_boundaries, need_gpu, np_
from oracle import csa2_oracle as o
from serving_lightning_indexer_gb300 import csa2
from serving_lightning_indexer_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _attn_case(T, k, n_swa, seed, holes=0.0, out_bf16=False, n_entries=5000, inv_rope=False, replay=False):
    dev = need_gpu()
    pc = W.make_paged_cache([n_entries], seed=seed, device=dev)
    al = W.make_attn_layer(T, seed=seed + 1, device=dev)
    rng = np.random.default_rng(seed)
    slots = np.stack([o.slots_of(rng.choice(n_entries, size=k, replace=False), np_(pc.page_table[0]))
                      for _ in range(T)]) if k else np.zeros((T, 0), dtype=np.int64)
    if holes:
        slots[rng.random(slots.shape) < holes] = -1
    tks = torch.tensor(slots, dtype=torch.int32, device=dev) if k else None
    swa = al.swa_slot[:, :n_swa].contiguous() if n_swa else None
    if n_swa and holes:
        swa = swa.clone()
        swa[torch.tensor(rng.random(tuple(swa.shape)) < holes, device=dev)] = -1
    qp_np = sg_np = None
    qp = sg = None
    if inv_rope or replay:   # query positions up to 1M: RoPE angles up to 1e6 rad
        qp_np = rng.integers(n_swa + 1000, 1 << 20, size=T)
        qp = torch.tensor(qp_np, dtype=torch.int32, device=dev)
    if replay:               # segment starts from the query itself to before its window
        sg_np = qp_np - rng.integers(0, n_swa + 20, size=T)
        sg_np[0] = qp_np[0]
        sg = torch.tensor(sg_np, dtype=torch.int32, device=dev)
    out = torch.empty(T, 64, 512, dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dev)
    lse = torch.empty(T, 64, dtype=torch.float32, device=dev)
    csa2.sparse_attn(al.q, pc.main_kv if k else None, tks, al.swa_kv if n_swa else None, swa, al.sink, out, lse,
                     q_pos=qp, out_inv_rope=inv_rope, swa_seg_start=sg)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    main_np, swa_np = np_(pc.main_kv), np_(al.swa_kv)
    for t in range(T):
        ref, rl = o.attention_row(al.q[t].float().cpu().numpy().astype(np.float64), main_np,
                                  slots[t] if k else np.zeros(0, dtype=np.int64), swa_np,
                                  np_(swa[t]) if n_swa else np.zeros(0, dtype=np.int64),
                                  np_(al.sink).astype(np.float64), 1 / math.sqrt(512),
                                  q_pos=None if qp_np is None else int(qp_np[t]),
                                  swa_seg_start=None if sg_np is None else int(sg_np[t]),
                                  inv_rope_theta=10000.0 if inv_rope else None)
        assert_attention_close(out[t].double().cpu().numpy(), ref, f"row {t}")
        assert np.abs(np_(lse[t]) - rl).max() < 2e-3


@pytest.mark.parametrize("T,k,n_swa", [(1, 512, 128), (3, 512, 128), (16, 512, 128), (200, 512, 128),
                                       (2, 100, 0), (2, 0, 37), (5, 2048, 128), (1, 1, 0),
                                       (2, 1152, 128), (2, 1153, 128), (3, 33, 48),
                                       # 19 rows x 8 chunks = 152 CTAs: the last launch of the
                                       # cluster kernel on 152 SMs; 20 rows: the split-K kernel
                                       (19, 512, 128), (20, 512, 128)])
def test_attention_matches_oracle(T, k, n_swa):
    _attn_case(T, k, n_swa, seed=T * 7 + k + n_swa)


def test_attention_with_empty_slots_and_bf16_out():
    _attn_case(4, 512, 128, seed=99, holes=0.3, out_bf16=True)


@pytest.mark.parametrize("T,k,n_swa,inv_rope,replay,out_bf16", [
    (3, 512, 128, True, False, False), (8, 512, 128, True, True, False), (16, 512, 128, False, True, True),
    (2, 2048, 128, True, True, False),      # split-K kernel, merged over the cluster
    (160, 2048, 128, True, True, True),     # split-K kernel, one CTA per row
    (4, 100, 37, True, True, False)])
def test_attention_inverse_rope_and_bounded_replay(T, k, n_swa, inv_rope, replay, out_bf16):
    # output inverse RoPE at the query position and the SWA window cut to the
    # replayed segment (CSA2 page: attention section; "Decoder SWA Bounded Replay")
    _attn_case(T, k, n_swa, seed=300 + T + k, out_bf16=out_bf16, inv_rope=inv_rope, replay=replay)


def test_attention_no_keys_at_all_gives_zero():
    dev = need_gpu()
    al = W.make_attn_layer(2, seed=5, device=dev)
    swa = torch.full((2, 128), -1, dtype=torch.int32, device=dev)
    out = torch.full((2, 64, 512), 7.0, dtype=torch.float32, device=dev)
    lse = torch.empty(2, 64, dtype=torch.float32, device=dev)
    csa2.sparse_attn(al.q, None, None, al.swa_kv, swa, al.sink, out, lse)
    torch.cuda.synchronize()
    assert (np_(out) == 0).all()
    assert np.allclose(np_(lse), np.repeat(np_(al.sink)[None], 2, 0), atol=1e-6)   # only the sink remains


def test_attention_bad_slot_is_reported():
    dev = need_gpu()
    pc = W.make_paged_cache([256], seed=6, device=dev)
    al = W.make_attn_layer(1, seed=7, device=dev)
    tks = torch.arange(512, dtype=torch.int32, device=dev)[None].contiguous()
    tks[0, 3] = pc.main_kv.shape[0] + 5
    out = torch.empty(1, 64, 512, dtype=torch.float32, device=dev)
    csa2.sparse_attn(al.q, pc.main_kv, tks[:, :256].contiguous(), al.swa_kv, al.swa_slot, al.sink, out)
    assert csa2.check_device_error() == 6


@pytest.mark.parametrize("ratio", [1, 2])
def test_compress_matches_oracle(ratio):
    dev = need_gpu()
    n_tok = 4096 + ratio
    Cm, Z, gamma = W.make_compress_inputs(n_tok, seed=20 + ratio, device=dev)
    n_ent = n_tok // ratio
    first = 1000
    pt = torch.randperm(96, device=dev).to(torch.int32)           # 96 pages hold entries < 6144
    kv = torch.zeros(96 * 64, 288, dtype=torch.uint8, device=dev)
    lat = torch.empty(n_ent, 512, dtype=torch.float32, device=dev)
    csa2.compress_m2(Cm, Z if ratio == 2 else None, ratio, gamma, kv, page_table=pt, first_entry=first,
                     latent_out=lat)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    pos = (first + np.arange(n_ent)) * ratio
    ref = o.compress_latent(Cm.float().cpu().numpy().astype(np.float64), Z.float().cpu().numpy().astype(np.float64),
                            ratio, np_(gamma).astype(np.float64), 1e-6, pos, 10000.0)
    got_lat = np_(lat).astype(np.float64)
    assert np.abs(got_lat - ref).max() <= 1e-4 * np.abs(ref).max()
    slots = o.slots_of(first + np.arange(n_ent), np_(pt))
    got = np_(kv)[slots]
    # the kernel's FP4 decisions equal the oracle's encoder applied to the kernel's own fp32 latent
    assert np.array_equal(got, o.fp4_encode_records(got_lat.astype(np.float32).astype(np.float64)))
    # against the float64 oracle: codes may differ only next to a rounding boundary
    assert_records_match_except_near_boundaries(got, ref)


def test_compress_entry_slots_and_no_rope():
    dev = need_gpu()
    Cm, Z, gamma = W.make_compress_inputs(64, seed=30, device=dev)
    es = torch.tensor(np.random.default_rng(0).permutation(100)[:32], dtype=torch.int32, device=dev)
    kv = torch.zeros(100, 288, dtype=torch.uint8, device=dev)
    lat = torch.empty(32, 512, dtype=torch.float32, device=dev)
    csa2.compress_m2(Cm, Z, 2, gamma, kv, entry_slot=es, apply_rope=False, latent_out=lat)
    torch.cuda.synchronize()
    ref = o.compress_latent(Cm.float().cpu().numpy().astype(np.float64), Z.float().cpu().numpy().astype(np.float64),
                            2, np_(gamma).astype(np.float64), 1e-6, np.zeros(32), 10000.0, apply_rope=False)
    assert np.abs(np_(lat) - ref).max() <= 1e-4 * np.abs(ref).max()
    assert np.array_equal(np_(kv)[np_(es)], o.fp4_encode_records(np_(lat).astype(np.float64)))
    untouched = np.setdiff1d(np.arange(100), np_(es))
    assert (np_(kv)[untouched] == 0).all()


def test_attention_main_kv_with_varied_block_scales():
    # e2m1 records whose 32-element groups carry scales 2^(u-127) with u spread
    # over a wide range (the table-lookup dequantisation) and at the ends of the
    # ue8m0 range (the exact float path); compared relative to the output scale.
    dev = need_gpu()
    rng = np.random.default_rng(7)
    n = 600
    rec = np.zeros((n, 288), dtype=np.uint8)
    rec[:, :256] = rng.integers(0, 256, size=(n, 256), dtype=np.uint8)
    u = rng.integers(118, 137, size=(n, 16))
    u[::7, 3] = 0
    u[::11, 5] = 1
    u[::13, 9] = 2
    rec[:, 256:272] = u.astype(np.uint8)
    main = torch.tensor(rec, device=dev)
    al = W.make_attn_layer(2, seed=8, device=dev)
    slots = np.stack([rng.choice(n, size=512, replace=False) for _ in range(2)])
    tks = torch.tensor(slots, dtype=torch.int32, device=dev)
    out = torch.empty(2, 64, 512, dtype=torch.float32, device=dev)
    csa2.sparse_attn(al.q, main, tks, al.swa_kv, al.swa_slot, al.sink, out, softmax_scale=1e-3)
    torch.cuda.synchronize()
    for t in range(2):
        ref, _ = o.attention_row(al.q[t].float().cpu().numpy().astype(np.float64), rec, slots[t], np_(al.swa_kv),
                                 np_(al.swa_slot[t]), np_(al.sink).astype(np.float64), 1e-3)
        err = np.abs(np_(out[t]).astype(np.float64) - ref).max() / np.abs(ref).max()
        assert err < 1e-2, err


def test_attention_keys_gathered_early_give_identical_results():
    # kv_ready lets the kernel gather slots and records before the dependency
    # wait; with slots and caches written long before, the result is the same
    dev = need_gpu()
    pc = W.make_paged_cache([20000], seed=41, device=dev)
    al = W.make_attn_layer(8, seed=42, device=dev)
    rng = np.random.default_rng(43)
    slots = torch.tensor(np.stack([o.slots_of(rng.choice(20000, size=512, replace=False), np_(pc.page_table[0]))
                                   for _ in range(8)]), dtype=torch.int32, device=dev)
    outs = []
    for ready in (False, True, True):
        out = torch.empty(8, 64, 512, dtype=torch.bfloat16, device=dev)
        csa2.sparse_attn(al.q, pc.main_kv, slots, al.swa_kv, al.swa_slot, al.sink, out, kv_ready=ready)
        outs.append(out)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


@pytest.mark.parametrize("ratio,fp4,n_ent", [(2, False, 1001), (1, False, 1001), (2, True, 1001), (1, True, 1001),
                                              (2, False, 7), (1, True, 152)])
def test_compress_builds_index_keys(ratio, fp4, n_ent):
    # Full layer's index key from the main-KV latent before RoPE (V4.1 Q&A page):
    # k = RMSNorm(y W^IK) * k_gamma, RoPE on dims 64..127, FP8 or FP4 entry;
    # up to one entry per SM takes the one-entry-per-CTA launch, beyond it eight
    dev = need_gpu()
    n_tok = n_ent * ratio
    Cm, Z, gamma = W.make_compress_inputs(n_tok, seed=40 + ratio, device=dev)
    w_ik, k_gamma = W.make_index_projection(seed=41, device=dev)
    n_ent = n_tok // ratio
    first = 300
    pt = torch.randperm(40, device=dev).to(torch.int32)            # 40 pages hold entries < 2560
    kv = torch.zeros(40 * 64, 288, dtype=torch.uint8, device=dev)
    kv_plain = torch.zeros_like(kv)
    ik = torch.zeros(40, 4352 if fp4 else 8448, dtype=torch.uint8, device=dev)
    klat = torch.empty(n_ent, 128, dtype=torch.float32, device=dev)
    csa2.compress_m2(Cm, Z if ratio == 2 else None, ratio, gamma, kv, page_table=pt, first_entry=first,
                     w_ik=w_ik, k_gamma=k_gamma, index_k=ik, index_latent_out=klat)
    csa2.compress_m2(Cm, Z if ratio == 2 else None, ratio, gamma, kv_plain, page_table=pt, first_entry=first)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    assert torch.equal(kv, kv_plain)                                # the main-KV records are unchanged
    pos = (first + np.arange(n_ent)) * ratio
    y_pre = o.compress_latent(Cm.float().cpu().numpy().astype(np.float64),
                              Z.float().cpu().numpy().astype(np.float64) if ratio == 2 else None,
                              ratio, np_(gamma).astype(np.float64), 1e-6, pos, 10000.0, apply_rope=False)
    ref = o.index_key_latent(y_pre, w_ik.float().cpu().numpy().astype(np.float64), np_(k_gamma).astype(np.float64),
                             1e-6, pos, 10000.0)
    got = np_(klat)
    assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max()
    # the entry bytes equal the oracle's encoder applied to the kernel's own fp32 key
    slots = o.slots_of(first + np.arange(n_ent), np_(pt))
    page, row = slots // 64, slots % 64
    pages = np_(ik)
    if fp4:
        c4, u4 = o.index_key_fp4_bytes(got.astype(np.float64))
        assert np.array_equal(pages[page[:, None], row[:, None] * 64 + np.arange(64)[None, :]], c4)
        assert np.array_equal(pages[page[:, None], 4096 + row[:, None] * 4 + np.arange(4)[None, :]], u4)
        dec = o.index_k_fp4_at(pages, np_(pt), first + np.arange(n_ent))
        assert np.all(np.abs(dec - ref) <= np.repeat(o.ue8m0(u4), 32, axis=1) + 1e-4 * np.abs(ref).max())
    else:
        c8, s8 = o.index_key_fp8_bytes(got)
        assert np.array_equal(pages[page[:, None], row[:, None] * 128 + np.arange(128)[None, :]], c8)
        sb = pages[page[:, None], 8192 + row[:, None] * 4 + np.arange(4)[None, :]]
        assert np.array_equal(np.ascontiguousarray(sb).view(np.float32).reshape(-1), s8)
        dec = o.index_k_at(pages, np_(pt), first + np.arange(n_ent))
        assert np.all(np.abs(dec - ref) <= np.abs(ref) * 2.0 ** -4 + s8[:, None] * 2.0 ** -9 + 1e-4 * np.abs(ref).max())
