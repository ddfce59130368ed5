"""Pins of the oracle's main-KV entry build (compression, RMSNorm, RoPE, FP4)
against closed forms, library routines and the invariants the pages state."""
import numpy as np
import torch

from oracle import csa2_oracle as o
from serving_lightning_indexer_gb300 import workloads as W


def _inputs(n_tok, seed):
    C, Z, gamma = W.make_compress_inputs(n_tok, seed)
    return (C.float().numpy().astype(np.float64), Z.float().numpy().astype(np.float64),
            gamma.numpy().astype(np.float64))


def test_m1_weight_is_identically_one():
    # V4.1 Q&A page: for m=1 the softmax weight is identically 1 (no Z at all)
    C, Z, gamma = _inputs(6, 0)
    pos = np.arange(6)
    a = o.compress_latent(C, None, 1, gamma, 1e-6, pos, 10000.0, apply_rope=False)
    b = o.compress_latent(C, Z, 1, gamma, 1e-6, pos, 10000.0, apply_rope=False)
    ref = torch.nn.functional.rms_norm(torch.tensor(C), (512,), torch.tensor(gamma), eps=1e-6).numpy()
    assert np.allclose(a, ref, rtol=1e-12) and np.array_equal(a, b)


def test_m2_equal_gates_give_the_mean_and_library_rmsnorm():
    C, Z, gamma = _inputs(8, 1)
    Z[:] = 0.3
    lat = o.compress_latent(C, Z, 2, gamma, 1e-6, np.zeros(4), 10000.0, apply_rope=False)
    mean = (C[0::2] + C[1::2]) / 2
    ref = torch.nn.functional.rms_norm(torch.tensor(mean), (512,), torch.tensor(gamma), eps=1e-6).numpy()
    assert np.allclose(lat, ref, rtol=1e-12)


def test_m2_is_per_channel_softmax_over_two_tokens():
    C, Z, gamma = _inputs(2, 2)
    lat = o.compress_latent(C, Z, 2, np.ones(512), 0.0, np.zeros(1), 10000.0, apply_rope=False)
    wts = torch.softmax(torch.tensor(Z), dim=0).numpy()       # library softmax over the 2 tokens
    x = (wts * C).sum(0)
    assert np.allclose(lat[0], x / np.sqrt((x * x).mean()), rtol=1e-12)


def test_m2_entries_depend_only_on_their_own_pair():
    # non-overlapping windows: perturbing tokens outside a pair leaves its entry unchanged
    C, Z, gamma = _inputs(12, 3)
    pos = np.arange(6) * 2
    base = o.compress_latent(C, Z, 2, gamma, 1e-6, pos, 10000.0)
    C2, Z2 = C.copy(), Z.copy()
    C2[[0, 1, 4, 5, 10, 11]] += 5.0
    Z2[[0, 1, 4, 5, 10, 11]] -= 2.0
    pert = o.compress_latent(C2, Z2, 2, gamma, 1e-6, pos, 10000.0)
    assert np.array_equal(base[[1, 3, 4]], pert[[1, 3, 4]])
    assert not np.allclose(base[[0, 2, 5]], pert[[0, 2, 5]])


def test_rope_matches_complex_rotation_and_keeps_norm():
    rng = np.random.default_rng(4)
    y = rng.normal(size=(5, 512))
    pos = np.array([0, 1, 7, 1000, 1 << 20])
    r = o.rope_interleaved(y, pos, 10000.0)
    assert np.array_equal(r[:, :448], y[:, :448])
    assert np.array_equal(r[0], y[0])                            # position 0: identity
    z = y[:, 448::2] + 1j * y[:, 449::2]
    freq = 10000.0 ** (-np.arange(32) / 32.0)
    zr = z * np.exp(1j * pos[:, None] * freq[None, :])
    assert np.allclose(r[:, 448::2], zr.real, atol=1e-12) and np.allclose(r[:, 449::2], zr.imag, atol=1e-12)
    assert np.allclose(np.linalg.norm(r, axis=1), np.linalg.norm(y, axis=1), rtol=1e-13)   # RoPE keeps the norm


def test_records_decode_close_to_latent():
    C, Z, gamma = _inputs(64, 5)
    rec, lat = o.compress_records(C, Z, 2, gamma, 1e-6, np.arange(32) * 2, 10000.0)
    dec = o.main_kv_records(rec, np.arange(32))
    step = np.repeat(o.ue8m0(rec[:, 256:272]), 32, axis=1)      # e2m1 spacing is <= 2 x 2^k
    assert np.all(np.abs(dec - lat) <= step + 1e-12)
    assert rec.shape == (32, 288) and (rec[:, 272:] == 0).all()
    # the report reading's bound: a unit-RMS 512-vector has |x| <= sqrt(512) << 2688
    assert np.abs(lat).max() < np.sqrt(512) * 1.5


# ---------------------------------------------------------------- index-key build
def _ik_inputs(n, seed):
    rng = np.random.default_rng(seed)
    y_pre = rng.standard_normal((n, 512))
    w_ik = rng.standard_normal((512, 128)) / np.sqrt(512)
    k_gamma = 1.0 + 0.1 * rng.standard_normal(128)
    return y_pre, w_ik, k_gamma


def test_index_key_is_library_rmsnorm_of_the_projection_at_position_zero():
    # V4.1 Q&A page: k = RMSNorm(y_pre W^IK); position 0 rotates nothing
    y_pre, w_ik, k_gamma = _ik_inputs(5, 3)
    k = o.index_key_latent(y_pre, w_ik, k_gamma, 1e-6, np.zeros(5), 10000.0)
    proj = torch.tensor(y_pre) @ torch.tensor(w_ik)               # library matmul
    ref = torch.nn.functional.rms_norm(proj, (128,), torch.tensor(k_gamma), eps=1e-6).numpy()
    assert np.allclose(k, ref, rtol=1e-10, atol=1e-12)
    # a selector projection picks input dims: k = RMSNorm of the first 128 latent dims
    sel = np.zeros((512, 128))
    sel[np.arange(128), np.arange(128)] = 1.0
    k2 = o.index_key_latent(y_pre, sel, np.ones(128), 0.0, np.zeros(5), 10000.0)
    x = y_pre[:, :128]
    assert np.allclose(k2, x / np.sqrt((x * x).mean(axis=1, keepdims=True)), rtol=1e-12)


def test_index_key_rope_turns_only_the_last_64_dims():
    # V4.1 Q&A page: after the projection the last 64 dims get their own RoPE
    y_pre, w_ik, k_gamma = _ik_inputs(4, 4)
    pos = np.array([0, 1, 77, 131071])
    k0 = o.index_key_latent(y_pre, w_ik, k_gamma, 1e-6, np.zeros(4), 10000.0)
    k = o.index_key_latent(y_pre, w_ik, k_gamma, 1e-6, pos, 10000.0)
    assert np.array_equal(k[:, :64], k0[:, :64])
    assert np.allclose(np.linalg.norm(k, axis=1), np.linalg.norm(k0, axis=1), rtol=1e-12)   # rotation
    # the same rotation as complex multiplication of the pairs (64+2i, 65+2i)
    z = torch.complex(torch.tensor(k0[:, 64::2]), torch.tensor(k0[:, 65::2]))
    ang = torch.tensor(pos, dtype=torch.float64)[:, None] * (10000.0 ** (-2.0 * torch.arange(32, dtype=torch.float64) / 64))
    zr = z * torch.polar(torch.ones_like(ang), ang)
    assert np.allclose(k[:, 64::2], zr.real.numpy(), atol=1e-9) and np.allclose(k[:, 65::2], zr.imag.numpy(), atol=1e-9)


def test_fp8_e4m3_codes_match_torch_conversion():
    # library routine: torch's float32 -> float8_e4m3fn conversion (round to nearest even)
    v = np.concatenate([np.linspace(-447, 447, 40001), o.FP8[:0x7F], -o.FP8[1:0x7F],
                        (o.FP8[1:0x7F] + o.FP8[:0x7E]) / 2, [448.0, -448.0, 1e-4, -1e-4]])
    ref = torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(o.fp8_e4m3_codes(v.astype(np.float32)).astype(np.uint8), ref)
    assert o.fp8_e4m3_codes(np.array([1e9]))[0] == 0x7E and o.fp8_e4m3_codes(np.array([-1e9]))[0] == 0xFE


def test_index_key_bytes_decode_through_the_page_readers():
    y_pre, w_ik, k_gamma = _ik_inputs(64, 5)
    k = o.index_key_latent(y_pre, w_ik, k_gamma, 1e-6, np.arange(64), 10000.0)
    k32 = k.astype(np.float32)
    codes, scale = o.index_key_fp8_bytes(k32)
    page8 = np.zeros(8448, dtype=np.uint8)
    page8[:8192] = codes.reshape(-1)
    page8[8192:] = scale.view(np.uint8)
    dec8 = o.index_k_entries(page8, np.array([0]), 64)
    assert np.all(np.abs(dec8 - k32) <= np.abs(k32) * 2.0 ** -4 + scale[:, None] * 2.0 ** -9 + 1e-12)
    c4, u4 = o.index_key_fp4_bytes(k)
    page4 = np.zeros(4352, dtype=np.uint8)
    page4[:4096] = c4.reshape(-1)
    page4[4096:] = u4.reshape(-1)
    dec4 = o.index_k_fp4_entries(page4, np.array([0]), 64)
    assert np.all(np.abs(dec4 - k) <= np.repeat(o.ue8m0(u4), 32, axis=1) + 1e-12)
    # the generator's independent FP4 encoder writes the same bytes
    gc, gu = W.fp4_encode_blocks(torch.tensor(k))
    assert np.array_equal(gc.numpy(), c4) and np.array_equal(gu.numpy(), u4)


def test_record_comparison_rule_accepts_the_oracle_and_catches_planted_errors():
    """The FP4 record comparison the GPU tests use (boundary rule, then every
    decoded value within half its local grid spacing of the float64 latent)
    accepts the oracle's own encoding and rejects a flipped code or scale."""
    import pytest as _pytest
    from gpu_util import assert_records_match_except_near_boundaries
    rng = np.random.default_rng(0)
    lat = rng.normal(size=(500, 512))
    rec = o.fp4_encode_records(lat)
    assert_records_match_except_near_boundaries(rec, lat)
    bad = rec.copy()
    bad[5, 10] ^= 0x11
    with _pytest.raises(AssertionError):
        assert_records_match_except_near_boundaries(bad, lat)
    bad = rec.copy()
    bad[7, 256] += 1
    with _pytest.raises(AssertionError):
        assert_records_match_except_near_boundaries(bad, lat)


def test_kv_project_brute_force_and_selector():
    """C = H W written out as a triple loop on a tiny case; a selector W (the
    identity on the first 512 input dims) returns those dims of H; a scaled
    hidden state scales C (linearity)."""
    rng = np.random.default_rng(3)
    H = rng.normal(size=(3, 40))
    Wt = rng.normal(size=(40, 7))
    want = np.zeros((3, 7))
    for t in range(3):
        for n in range(7):
            for k in range(40):
                want[t, n] += H[t, k] * Wt[k, n]
    assert np.allclose(o.kv_project(H, Wt), want, rtol=1e-13, atol=1e-13)
    H2 = rng.normal(size=(2, 7168))
    sel = np.zeros((7168, 512))
    sel[np.arange(512), np.arange(512)] = 1.0
    assert np.array_equal(o.kv_project(H2, sel), H2[:, :512])
    W2 = rng.normal(size=(7168, 512))
    assert np.allclose(o.kv_project(2.5 * H2, W2), 2.5 * o.kv_project(H2, W2), rtol=1e-12)
