"""Pins of the oracle's sparse MQA attention with sink: closed forms, the
dense-equals-sparse identity, and a library attention routine."""
import math

import numpy as np
import torch

from oracle import csa2_oracle as o
from serving_lightning_indexer_gb300 import workloads as W


def test_closed_form_two_keys_with_sink():
    # 1 head, keys (1,0),(0,1), q=(1,0), scale 1, sink 0:
    # o = (e*(1,0) + 1*(0,1)) / (e + 1 + 1)
    out, lse = o.sparse_attention(np.array([[1.0, 0.0]]), np.eye(2), np.array([0.0]), 1.0)
    e = math.e
    assert np.allclose(out[0], [e / (e + 2), 1 / (e + 2)], rtol=1e-15)
    assert np.isclose(lse[0], math.log(e + 2))


def test_single_key_gives_v_when_sink_vanishes():
    v = np.random.default_rng(0).normal(size=(1, 512))
    q = np.random.default_rng(1).normal(size=(64, 512))
    out, _ = o.sparse_attention(q, v, np.full(64, -np.inf), 0.1)
    assert np.allclose(out, np.repeat(v, 64, axis=0), rtol=1e-14)


def test_sink_share_closes_the_simplex():
    # softmax weights plus the sink share sum to 1: with V = all-ones columns the
    # output equals 1 - sink share
    rng = np.random.default_rng(2)
    q = rng.normal(size=(64, 512))
    kv = rng.normal(size=(40, 512))
    sink = rng.normal(size=64)
    scale = 1 / math.sqrt(512)
    _, lse = o.sparse_attention(q, kv, sink, scale)
    logits = q @ kv.T * scale
    share = np.exp(sink - lse)
    assert np.allclose(np.exp(logits - lse[:, None]).sum(1) + share, 1.0, rtol=1e-13)


def test_matches_torch_sdpa_with_sink_as_extra_key():
    # library routine: torch scaled_dot_product_attention (float64).  The sink is
    # an extra key whose logit is s_i for head i and whose value is 0.
    rng = np.random.default_rng(3)
    H, d, n = 64, 512, 37
    q = rng.normal(size=(H, d))
    kv = rng.normal(size=(n, d))
    sink = rng.normal(size=H)
    scale = 1 / math.sqrt(d)
    ours, _ = o.sparse_attention(q, kv, sink, scale)
    for h in (0, 17, 63):
        ks = q[h] * (sink[h] / (scale * (q[h] @ q[h])))
        K = np.vstack([kv, ks])
        V = np.vstack([kv, np.zeros(d)])
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.tensor(q[h][None, None, None]), torch.tensor(K[None, None]), torch.tensor(V[None, None]),
            scale=scale)[0, 0, 0].numpy()
        assert np.allclose(ours[h], ref, rtol=1e-10, atol=1e-12)


def test_sparse_equals_dense_when_everything_selected():
    # DSA page: when S <= k the top-k holds every position and sparse = dense.
    # Build the attention from the caches through slot tables and compare with
    # plain softmax attention over all decoded vectors.
    n = 200
    pc = W.make_paged_cache([n], seed=11)
    al = W.make_attn_layer(1, seed=12)
    pt = pc.page_table[0].numpy()
    slots = o.slots_of(np.arange(n), pt)
    tk = np.full(512, -1)
    tk[:n] = np.random.default_rng(0).permutation(slots)
    q = al.q[0].float().numpy().astype(np.float64)
    sink = al.sink.numpy().astype(np.float64)
    out, _ = o.attention_row(q, pc.main_kv.numpy(), tk, al.swa_kv.numpy(), al.swa_slot[0].numpy(), sink,
                             1 / math.sqrt(512))
    allkv = np.vstack([o.swa_records(al.swa_kv.numpy(), al.swa_slot[0].numpy()),
                       o.main_kv_records(pc.main_kv.numpy(), slots)])
    logits = np.hstack([q @ allkv.T / math.sqrt(512), sink[:, None]])
    p = torch.softmax(torch.tensor(logits), dim=1).numpy()
    dense = p[:, :-1] @ allkv
    assert np.allclose(out, dense, rtol=1e-11, atol=1e-13)


def test_empty_slots_ignored_and_order_free():
    n = 50
    pc = W.make_paged_cache([n], seed=13)
    al = W.make_attn_layer(1, seed=14)
    slots = o.slots_of(np.arange(n), pc.page_table[0].numpy())
    q = al.q[0].float().numpy().astype(np.float64)
    sink = al.sink.numpy().astype(np.float64)
    a = np.full(512, -1)
    a[:n] = slots
    b = np.full(512, -1)
    b[100:100 + n] = slots[::-1]
    oa, la = o.attention_row(q, pc.main_kv.numpy(), a, al.swa_kv.numpy(), al.swa_slot[0].numpy(), sink, 0.05)
    ob, lb = o.attention_row(q, pc.main_kv.numpy(), b, al.swa_kv.numpy(), al.swa_slot[0].numpy(), sink, 0.05)
    assert np.allclose(oa, ob, rtol=1e-12) and np.allclose(la, lb, rtol=1e-13)


# ---- Decoder SWA Bounded Replay (CSA2 page, "Decoder SWA Bounded Replay") ----

def test_replay_visible_counts_close_the_triangle():
    # a replayed tail of W tokens: query k of the segment (0-based) sees k + 1 SWA
    # keys, so the segment holds 1 + 2 + ... + W = W (W + 1) / 2 query-key pairs
    W, s = 128, 5000
    counts = [int(o.swa_replay_visible(s + k, s, W).sum()) for k in range(W)]
    assert counts == list(range(1, W + 1))
    assert sum(counts) == W * (W + 1) // 2 == 8256
    # a longer segment: every query after the first W sees the full window
    L = 300
    total = sum(int(o.swa_replay_visible(s + k, s, W).sum()) for k in range(L))
    assert total == W * (W + 1) // 2 + (L - W) * W


def test_replay_visible_special_cases():
    W = 128
    # the first query of a segment sees only its own key, the newest slot
    v = o.swa_replay_visible(777, 777, W)
    assert v.sum() == 1 and v[-1]
    # a segment start at or before the window's first position cuts nothing
    for s in (0, 777 - W + 1, 777 - 5000):
        assert o.swa_replay_visible(777, s, W).all()
    # one position inside: the oldest slot alone drops out
    v = o.swa_replay_visible(777, 777 - W + 2, W)
    assert not v[0] and v[1:].all()
    # the visible keys are a contiguous run that ends at the query's own key
    for s in range(700, 778):
        v = o.swa_replay_visible(777, s, W)
        first = int(np.argmax(v))
        assert v[first:].all() and not v[:first].any()


def test_replay_row_equals_attention_over_the_segment_keys_only():
    # brute force: attend over exactly the keys whose positions lie in the
    # segment and the window, built position by position
    rng = np.random.default_rng(11)
    W, s, i = 16, 40, 47
    kv_by_pos = {p: rng.normal(size=512) for p in range(i - W + 1, i + 1)}
    q = rng.normal(size=(64, 512))
    sink = rng.normal(size=64)
    keys = np.array([kv_by_pos[p] for p in range(i - W + 1, i + 1) if p >= s])
    ref, _ = o.sparse_attention(q, keys, sink, 0.05)
    vis = o.swa_replay_visible(i, s, W)
    window = np.array([kv_by_pos[p] for p in range(i - W + 1, i + 1)])
    got, _ = o.sparse_attention(q, window[vis], sink, 0.05)
    assert len(keys) == i - s + 1 == int(vis.sum())
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-15)


# ---- Output inverse RoPE (CSA2 page, attention section) ----

def _rope_rows(x, pos, theta=10000.0):
    return o.rope_interleaved(x, np.full(x.shape[0], float(pos)), theta)


def test_inverse_rope_makes_the_output_relative():
    # keys carry RoPE at their own positions, the query at its position; after the
    # output's inverse RoPE only relative positions remain: shifting every
    # position by the same amount leaves the output unchanged.  Without the
    # inverse (or with the rotation's sign flipped) the shift shows.
    rng = np.random.default_rng(12)
    x = rng.normal(size=(20, 512))
    kpos = np.sort(rng.choice(5000, size=20, replace=False))
    qx = rng.normal(size=(64, 512)) * 0.05
    qpos = 5000
    sink = rng.normal(size=64)

    def run(shift, inverse=True, sign=1.0):
        K = o.rope_interleaved(x, kpos + shift, 10000.0)
        q = _rope_rows(qx, qpos + shift)
        out, lse = o.sparse_attention(q, K, sink, 1 / math.sqrt(512))
        if inverse:
            out = o.output_inverse_rope(out, sign * (qpos + shift), 10000.0)
        return out, lse

    a, la = run(0)
    b, lb = run(123457)
    assert np.allclose(la, lb, rtol=1e-9)             # logits depend on relative positions only
    assert np.allclose(a, b, rtol=1e-8, atol=1e-10)
    c, _ = run(123457, inverse=False)
    assert not np.allclose(a[:, 448:], c[:, 448:], atol=1e-3)
    d, _ = run(123457, sign=-1.0)
    assert not np.allclose(a[:, 448:], d[:, 448:], atol=1e-3)
    assert np.array_equal(b[:, :448], c[:, :448])     # the first 448 dims are not rotated


def test_inverse_rope_of_a_single_key_returns_its_latent():
    # one key at the query's own position and no sink mass: the output is that
    # key, and its inverse RoPE at the same position is the latent before RoPE
    rng = np.random.default_rng(13)
    lat = rng.normal(size=(1, 512))
    pos = 987654
    out, _ = o.sparse_attention(rng.normal(size=(64, 512)), _rope_rows(lat, pos), np.full(64, -np.inf), 0.1)
    back = o.output_inverse_rope(out, pos, 10000.0)
    assert np.allclose(back, np.repeat(lat, 64, axis=0), rtol=1e-9, atol=1e-12)


def test_inverse_rope_is_a_complex_rotation_by_minus_the_angle():
    # torch complex arithmetic: pair (2p, 2p+1) of the last 64 dims times
    # exp(-i * pos * theta^(-2p/64)); position 0 is the identity
    rng = np.random.default_rng(14)
    y = rng.normal(size=(64, 512))
    pos, theta = 31337, 10000.0
    got = o.output_inverse_rope(y, pos, theta)
    z = torch.view_as_complex(torch.tensor(y[:, 448:]).reshape(64, 32, 2).contiguous())
    ang = -pos * theta ** (-2.0 * torch.arange(32, dtype=torch.float64) / 64)
    ref = torch.view_as_real(z * torch.polar(torch.ones(32, dtype=torch.float64), ang)).reshape(64, 64).numpy()
    assert np.abs(got[:, 448:] - ref).max() <= 1e-10 * np.abs(ref).max()   # angles ~3e4 rad
    assert np.array_equal(got[:, :448], y[:, :448])
    assert np.array_equal(o.output_inverse_rope(y, 0, theta), y)
