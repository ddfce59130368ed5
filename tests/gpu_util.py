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


def assert_attention_close(got, ref, what="attention"):
    d = np.abs(np.asarray(got, dtype=np.float64) - np.asarray(ref, dtype=np.float64))
    assert d.max() <= ATTN_MAX_ABS, f"{what}: max abs {d.max():.3e}"
    assert d.mean() <= ATTN_MEAN_ABS, f"{what}: mean abs {d.mean():.3e}"


def np_(t):
    return t.detach().cpu().numpy()
