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
