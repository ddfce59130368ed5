"""GPU parity of csa2_kv_project (C = H W, the entry build's per-token input)
against the oracle's float64 product."""
import ctypes as C

import numpy as np
import pytest
import torch

from gpu_util import need_gpu, np_
from oracle import csa2_oracle as o
from serving_lightning_indexer_gb300 import csa2
from serving_lightning_indexer_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _check(T, hidden, seed):
    """Tolerance from the arithmetic: bf16 x bf16 products are exact in fp32;
    the fp32 sum runs through fewer than 2^6 additions in a chain (at most 32
    rows a thread, three shuffle steps, eight warps, two batches, eight
    cluster slices for hidden <= 16384), so its error is below
    2^-17 sum_k |h_k w_k|; the bf16 result
    adds at most 2^-8 of its magnitude (bf16 keeps 8 significant bits)."""
    dev = need_gpu()
    H, w = W.make_hidden_projection(T, seed=seed, device=dev, hidden=hidden)
    out = torch.full((T, 512), float("nan"), dtype=torch.bfloat16, device=dev)
    csa2.kv_project(H, w, out)
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    h, wv = np_(H.float()).astype(np.float64), np_(w.float()).astype(np.float64)
    ref = o.kv_project(h, wv)
    e_sum = 2.0 ** -17 * (np.abs(h) @ np.abs(wv))
    got = np_(out.float()).astype(np.float64)
    tol = 2.0 ** -8 * (np.abs(ref) + e_sum) + e_sum
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"T={T} hidden={hidden}: {bad.sum()} outside, worst {np.abs(got - ref).max()}"


@pytest.mark.parametrize("T,hidden", [(1, 7168), (8, 7168), (16, 7168), (17, 7168), (32, 7168), (64, 7168),
                                      (33, 512), (5, 4608), (48, 16384), (3, 9216)])
def test_kv_project_matches_oracle(T, hidden):
    _check(T, hidden, seed=T * 131 + hidden)


def test_kv_project_rejects_bad_shapes():
    dev = need_gpu()
    H, w = W.make_hidden_projection(4, seed=1, device=dev, hidden=512)
    out = torch.empty(4, 512, dtype=torch.bfloat16, device=dev)
    lib = csa2.load()
    for T, hd in ((0, 512), (65, 512), (4, 256), (4, 768), (4, 16896)):
        a = csa2.KvProjectArgs(H.data_ptr(), w.data_ptr(), T, hd, out.data_ptr())
        assert lib.csa2_kv_project(C.byref(a), None) == 2
        assert lib.csa2_last_error_detail().startswith(b"csa2_kv_project:")
