"""Helpers of the GPU parity tests: acceptance rules and device plumbing."""
import numpy as np
import pytest
import torch

# Acceptance rules of the CSA2 parity contract.
SCORE_RTOL = 1e-3          # scores: |d| <= 1e-3 * max(|ref|, 1e-2 * rms(row))
NEAR_TIE_RTOL = 1e-3       # selection: symmetric difference only within 1e-3 of the threshold score
ATTN_MAX_ABS = 2e-2
ATTN_MEAN_ABS = 5e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from serving_lightning_indexer_gb300 import _build, csa2
    _build.build()
    csa2.load()
    return torch.device("cuda:0")


def assert_scores_close(got, ref, what="scores"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: -inf pattern differs"
    if not fin.any():
        return
    rms = np.sqrt((ref[fin] ** 2).mean())
    tol = SCORE_RTOL * np.maximum(np.abs(ref[fin]), 1e-2 * rms)
    err = np.abs(got[fin] - ref[fin])
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} of {fin.sum()} beyond tolerance, worst {err.max():.3e}"


def assert_selection_ok(got_ids, ref_values, k, what="top-k"):
    """got_ids: selected ids (-1 padded); ref_values: oracle values over all ids
    (-inf excluded).  The selected set equals the oracle's top-k except for
    elements whose oracle value is within NEAR_TIE_RTOL of the threshold."""
    from oracle import csa2_oracle as o
    ref_values = np.asarray(ref_values, dtype=np.float64)
    want = o.topk_positions(ref_values, k)
    want_set = set(int(x) for x in want if x >= 0)
    got = [int(x) for x in np.asarray(got_ids) if x >= 0]
    assert len(got) == len(set(got)), f"{what}: duplicate ids"
    got_set = set(got)
    assert len(got_set) == len(want_set), f"{what}: {len(got_set)} selected, oracle {len(want_set)}"
    diff = got_set ^ want_set
    if diff:
        thr = ref_values[want[len(want_set) - 1]]
        for x in diff:
            assert np.isfinite(ref_values[x]), f"{what}: selected an excluded id {x}"
            assert abs(ref_values[x] - thr) <= NEAR_TIE_RTOL * abs(thr), \
                f"{what}: id {x} (value {ref_values[x]}) differs from the oracle away from the threshold {thr}"


def assert_pool_ok(got_blocks, bmax_ref, n_pool=2048, what="pool"):
    """got_blocks: the kernel's pool (ascending block ids, -1 padded); bmax_ref:
    float64 oracle block maxima of the row.  The pool holds the newest block
    and otherwise equals the oracle's pool except for blocks whose oracle
    maximum is within NEAR_TIE_RTOL of the pool's threshold (the n_pool-th
    largest block maximum, the newest block counted as +inf)."""
    from oracle import csa2_oracle as o
    got_blocks = np.asarray(got_blocks)
    bmax_ref = np.asarray(bmax_ref, dtype=np.float64)
    nb = len(bmax_ref)
    sel = got_blocks[got_blocks >= 0]
    assert np.array_equal(got_blocks[len(sel):], np.full(len(got_blocks) - len(sel), -1)), f"{what}: -1 padding"
    assert (np.diff(sel) > 0).all() and sel.max() < nb, f"{what}: not ascending distinct block ids"
    assert len(sel) == min(n_pool, nb), f"{what}: {len(sel)} blocks"
    assert sel[-1] == nb - 1, f"{what}: the newest block is missing"
    want = o.candidate_pool(bmax_ref, n_pool)
    diff = set(sel.tolist()) ^ set(want[want >= 0].tolist())
    if diff:
        b = bmax_ref.copy()
        b[-1] = np.inf
        thr = np.sort(b)[::-1][n_pool - 1]
        for x in diff:
            assert abs(b[x] - thr) <= NEAR_TIE_RTOL * abs(thr), \
                f"{what}: block {x} (max {b[x]}) differs from the oracle away from the threshold {thr}"


def assert_attention_close(got, ref, what="attention"):
    d = np.abs(np.asarray(got, dtype=np.float64) - np.asarray(ref, dtype=np.float64))
    assert d.max() <= ATTN_MAX_ABS, f"{what}: max abs {d.max():.3e}"
    assert d.mean() <= ATTN_MEAN_ABS, f"{what}: mean abs {d.mean():.3e}"


FP4_MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def assert_records_match_except_near_boundaries(got, ref_latent, rtol=1e-5):
    """FP4 records of the kernel against the float64 oracle's encoding of the
    float64 latent.  The fp32 latent differs from the float64 one by rounding
    only, so a code may differ only where the float64 value sits within rtol of
    a decision boundary: a ue8m0 scale only where a group's amax / 6 is within
    rtol of a power of two (the exponent rule flips there), an e2m1 code (of a
    group whose scale agrees) only where value / scale is within rtol of an
    e2m1 rounding midpoint.  Everything else is bit-exact, and every decoded
    value is the float64 latent rounded to its record's grid."""
    n = ref_latent.shape[0]
    want = _o().fp4_encode_records(ref_latent)
    g = np.abs(ref_latent).reshape(n, 16, 32)
    amax = g.max(axis=2)
    t = amax / 6.0
    with np.errstate(divide="ignore"):
        near_pow2 = (amax > 0) & (np.abs(t / np.exp2(np.round(np.log2(np.where(t > 0, t, 1.0)))) - 1.0) < rtol)
    scale_diff = got[:, 256:272] != want[:, 256:272]
    assert not (scale_diff & ~near_pow2).any(), "a scale code differs away from a power-of-two boundary"
    y = g / _o().ue8m0(want[:, 256:272])[:, :, None]
    near_mid = (np.abs(y[..., None] - FP4_MIDPOINTS) < rtol * FP4_MIDPOINTS).any(axis=-1)
    codes_got = np.stack([got[:, :256] & 15, got[:, :256] >> 4], axis=-1).reshape(n, 16, 32)
    codes_want = np.stack([want[:, :256] & 15, want[:, :256] >> 4], axis=-1).reshape(n, 16, 32)
    code_diff = (codes_got != codes_want) & ~scale_diff[:, :, None]
    assert not (code_diff & ~near_mid).any(), "an e2m1 code differs away from a rounding midpoint"
    assert np.array_equal(got[:, 272:], want[:, 272:])
    # every decoded value is the float64 latent rounded to the e2m1 grid of its
    # record's scale: within half the local grid spacing (0.5, 1 or 2 scale
    # units below 2, 4, 6), saturating at 6 units
    dec_got = _o().main_kv_records(got, np.arange(n))
    s_got = np.repeat(_o().ue8m0(got[:, 256:272]), 32, axis=1)
    ax = np.abs(ref_latent) / s_got
    spacing = np.where(ax < 2, 0.5, np.where(ax < 4, 1.0, 2.0)) * s_got
    over = np.maximum(np.abs(ref_latent) - 6 * s_got, 0.0)
    assert np.all(np.abs(dec_got - ref_latent) <= 0.5 * spacing * (1 + 1e-4) + over + 1e-12), \
        "a decoded value is not the latent rounded to its record's grid"


def _o():
    from oracle import csa2_oracle
    return csa2_oracle


def np_(t):
    return t.detach().cpu().numpy()
