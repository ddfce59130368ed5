"""Pins of the oracle's storage-format decoders and encoders against things
other than themselves: a library decoder, a public spec table, brute force."""
import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import csa2_oracle as o
from serving_lightning_indexer_gb300 import workloads as W


def test_fp8_table_matches_torch_decoder():
    # library routine: torch's own float8_e4m3fn -> float64 conversion
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    ours = o.FP8
    assert np.array_equal(np.isnan(lib), np.isnan(ours))
    ok = ~np.isnan(lib)
    assert np.array_equal(lib[ok], ours[ok])
    # the report reading's bound uses 448 as the e4m3 maximum
    assert np.nanmax(ours) == 448.0 and np.nanmin(ours) == -448.0
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])


def test_fp4_table_matches_ocp_mx_spec():
    rows = read_golden("fp4_e2m1_ocp_mx.txt")
    for code, (val,) in rows:
        v = float(val)
        assert o.FP4[int(code)] == v
        assert np.signbit(o.FP4[int(code)]) == np.signbit(v)
    assert o.FP4.max() * 448.0 == 2688.0   # the report reading's "448 x 6 = 2688"


def test_ue8m0():
    assert o.ue8m0(127) == 1.0 and o.ue8m0(128) == 2.0 and o.ue8m0(125) == 0.25
    assert np.isnan(o.ue8m0(255))


def test_fp4_scale_exponent_is_minimal():
    rng = np.random.default_rng(0)
    amax = np.concatenate([rng.lognormal(0, 3, 2000), [6.0, 3.0, 12.0, 6 * 2.0 ** -5, 1e-30]])
    u = o.fp4_scale_exponent(amax)
    k = u - 127
    assert np.all(6.0 * np.exp2(k) >= amax)
    assert np.all(6.0 * np.exp2(k - 1) < amax)
    assert o.fp4_scale_exponent(0.0) == 127


def test_fp4_codes_nearest_with_even_ties_bruteforce():
    mags = o.FP4[:8]
    vals = np.concatenate([np.linspace(-7, 7, 2801), (mags[:-1] + mags[1:]) / 2, -(mags[:-1] + mags[1:]) / 2])
    codes = o.fp4_codes(vals)
    for v, c in zip(vals, codes):
        a = min(abs(v), 6.0)
        d = [abs(a - m) for m in mags]
        best = min(d)
        cands = [i for i in range(8) if d[i] == best]
        want = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
        assert (c & 7) == want, (v, c, want)
        assert (c >> 3) == (1 if v < 0 else 0)


def test_generator_fp8_roundtrip_through_oracle_decoder():
    g = torch.Generator().manual_seed(1)
    x = torch.randn(50, 128, generator=g)
    codes, scale = W.fp8_encode(x)
    dec = o.FP8[codes.numpy().astype(np.int64)] * scale.numpy().astype(np.float64)[:, None]
    # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 of the value, plus the
    # subnormal step 2^-9 * scale
    err = np.abs(dec - x.numpy())
    bound = np.abs(x.numpy()) * 2.0 ** -4 + scale.numpy()[:, None] * 2.0 ** -9
    assert np.all(err <= bound + 1e-12)
    assert np.all(np.abs(dec).max(axis=1) == pytest.approx(np.abs(x.numpy()).max(axis=1), rel=1e-6))


def test_generator_fp4_encoder_agrees_with_oracle_encoder():
    # two independent encoders of the same format (generator: threshold counting,
    # oracle: nearest-magnitude search) must produce identical records
    g = torch.Generator().manual_seed(2)
    x = torch.randn(64, 512, generator=g) * torch.exp(torch.randn(64, 1, generator=g))
    x[0, :32] = 0.0                          # all-zero group -> u = 127
    x[1, :32] = torch.tensor([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] * 4)   # exact ties
    rec_gen = W.fp4_encode_records(x).numpy()
    rec_orc = o.fp4_encode_records(x.numpy().astype(np.float64))
    assert np.array_equal(rec_gen, rec_orc)
    dec = o.main_kv_records(rec_orc, np.arange(64))
    assert np.all(np.abs(dec - x.numpy()) <= np.repeat(o.ue8m0(rec_orc[:, 256:272]), 32, axis=1) + 1e-12)


def test_swa_record_roundtrip():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(10, 512, generator=g)
    rec = W.swa_encode_records(x).numpy()
    dec = o.swa_records(rec, np.arange(10))
    assert np.allclose(dec, x.numpy(), rtol=2.0 ** -4, atol=1e-2)


def test_index_page_layout_roundtrip():
    pc = W.make_paged_cache([100, 70], seed=4, with_main=False)
    e0 = o.index_k_entries(pc.index_k.numpy(), pc.page_table[0].numpy(), 100)
    e1 = o.index_k_entries(pc.index_k.numpy(), pc.page_table[1].numpy(), 70)
    assert e0.shape == (100, 128) and e1.shape == (70, 128)
    # page size 64 and 8448-B pages (DSA page: 64 x 132 = 8448)
    assert pc.index_k.shape[1] == 8448 == 64 * 132
    # distinct sequences land on distinct physical pages
    p0 = set(pc.page_table[0, :2].tolist())
    p1 = set(pc.page_table[1, :2].tolist())
    assert not (p0 & p1)
    # byte-level check of one key: codes at row*128, scale at 8192 + row*4
    page = int(pc.page_table[1, 1])
    row = 70 - 64 - 1
    codes = pc.index_k[page, row * 128:(row + 1) * 128].numpy()
    scale = pc.index_k[page, 8192 + row * 4:8192 + row * 4 + 4].numpy().view(np.float32)[0]
    assert np.array_equal(e1[69], o.FP8[codes.astype(np.int64)] * np.float64(scale))


def _fp4_page_by_hand(codes, u):
    """One FP4 index-K page [4352] from codes [64,128] (0..15) and scales [64,4]."""
    codes = np.asarray(codes, dtype=np.uint8)
    page = np.zeros(4352, dtype=np.uint8)
    page[:4096] = (codes[:, 0::2] | (codes[:, 1::2] << 4)).reshape(-1)
    page[4096:] = np.asarray(u, dtype=np.uint8).reshape(-1)
    return page


def test_fp4_index_page_hand_values():
    # key 5: dims 0..31 scale 2^0, 32..63 scale 2^-1, 64..95 scale 2^2, 96..127 scale 2^-3;
    # codes: dim 0 -> +6 (0x7), dim 1 -> -0.5 (0x9), dim 32 -> +3 (0x5), dim 127 -> -4 (0xE)
    codes = np.zeros((64, 128), dtype=np.uint8)
    u = np.full((64, 4), 127, dtype=np.uint8)
    codes[5, 0], codes[5, 1], codes[5, 32], codes[5, 127] = 0x7, 0x9, 0x5, 0xE
    u[5] = [127, 126, 129, 124]
    page = _fp4_page_by_hand(codes, u)
    # byte-level layout: byte 5*64 holds dims 0 (low nibble) and 1 (high nibble)
    assert page[5 * 64] == 0x97 and page[4096 + 5 * 4 + 2] == 129
    k = o.index_k_fp4_at(page, np.array([0]), np.array([5]))[0]
    want = np.zeros(128)
    want[0], want[1], want[32], want[127] = 6.0, -0.5, 3.0 * 0.5, -4.0 * 0.125
    assert np.array_equal(k, want)
    assert o.INDEX_FP4_PAGE_BYTES == 4352 == 64 * 68   # 68 B per entry (report reading: 890 = 2.5 x (288 + 68))


def test_fp4_index_keys_equal_fp8_index_keys_for_common_values():
    # keys whose values are exact in both formats, written once as an FP4 page and
    # once as an FP8 page (e4m3 codes times an fp32 scale of 2^-2): both decoders
    # (the FP8 one pinned against torch) must return the same keys
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 16, size=(64, 128)).astype(np.uint8)
    u = rng.integers(124, 130, size=(64, 4)).astype(np.uint8)          # 2^-3 .. 2^2
    fp4_page = _fp4_page_by_hand(codes, u)
    vals = o.FP4[codes.astype(np.int64)] * np.repeat(o.ue8m0(u), 32, axis=1)   # in [-24, 24]
    fp8_scale = np.float32(0.25)
    e4m3 = torch.tensor(vals / 0.25, dtype=torch.float64).to(torch.float8_e4m3fn)
    assert np.array_equal(e4m3.double().numpy() * 0.25, vals)           # exact in e4m3 too
    fp8_page = np.zeros(8448, dtype=np.uint8)
    fp8_page[:8192] = e4m3.view(torch.uint8).numpy().reshape(-1)
    fp8_page[8192:] = np.full(64, fp8_scale, dtype=np.float32).view(np.uint8)
    pt = np.array([0])
    assert np.array_equal(o.index_k_fp4_entries(fp4_page, pt, 64), o.index_k_entries(fp8_page, pt, 64))
    # and so the scores of both formats agree
    q8 = rng.integers(0, 0x7E, size=(32, 128))
    qs = rng.random(32) + 0.5
    w = rng.standard_normal(32)
    assert np.array_equal(o.index_scores_row(q8, qs, w, fp4_page, pt, 64, fp4=True),
                          o.index_scores_row(q8, qs, w, fp8_page, pt, 64))


def test_generator_fp4_index_pages_decode_near_the_fp8_keys():
    # the same seeded keys written in both formats: the FP4 decode is within half
    # an e2m1 grid step (x block scale) of the finer FP8 decode
    pc8 = W.make_paged_cache([300], seed=5, with_main=False)
    pc4 = W.make_paged_cache([300], seed=5, with_main=False, index_fp4=True)
    assert pc4.index_k.shape[1] == 4352
    assert torch.equal(pc8.page_table, pc4.page_table)
    k8 = o.index_k_entries(pc8.index_k.numpy(), pc8.page_table[0].numpy(), 300)
    k4 = o.index_k_fp4_entries(pc4.index_k.numpy(), pc4.page_table[0].numpy(), 300)
    pages = pc4.index_k.numpy()[pc4.page_table[0].numpy()[np.arange(300) // 64]]
    u = pages[np.arange(300)[:, None], 4096 + (np.arange(300) % 64)[:, None] * 4 + np.arange(4)[None, :]]
    step = np.repeat(o.ue8m0(u), 32, axis=1)          # the widest e2m1 gap (4 -> 6) is 2 x scale
    assert np.all(np.abs(k4 - k8) <= step + np.abs(k8) * 2.0 ** -4 + 1e-9)
    assert np.abs(k4 - k8).mean() < 0.2
