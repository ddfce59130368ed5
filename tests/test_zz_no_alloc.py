"""The no-allocation top-k entry point, called through the C ABI.

csa2_topk_with_candidates_noalloc serves callers that cannot give the library
device scratch memory (operator interfaces that pass only inputs and outputs,
allocators without a scratch hook, paths that must not call cudaMalloc): its
scratch is a static device array inside the library.  This file is collected
last so that a run stopping at the first failure has run every other test."""
import ctypes as C

import numpy as np
import pytest
import torch

from gpu_util import need_gpu, np_
from serving_lightning_indexer_gb300 import csa2

pytestmark = pytest.mark.gpu


def _inputs(seed, lengths, dev):
    rng = np.random.default_rng(seed)
    T, ld = len(lengths), max(lengths) + 3 & ~3
    s = rng.normal(size=(T, ld)).astype(np.float32)
    nb = (ld + 7) // 8 + 3 & ~3
    bm = np.full((T, nb), -np.inf, dtype=np.float32)
    for t, n in enumerate(lengths):
        v = s[t, :n]
        bm[t, :(n + 7) // 8] = np.pad(v, (0, -n % 8), constant_values=-np.inf).reshape(-1, 8).max(1)
    pt = np.stack([rng.permutation(1 << 16)[: (ld + 63) // 64] for _ in range(T)]).astype(np.int32)
    t_ = lambda a: torch.tensor(a, device=dev)
    return t_(s), t_(bm), t_(pt), torch.tensor(lengths, dtype=torch.int32, device=dev)


def _outputs(T, dev):
    return (torch.full((T, 512), -7, dtype=torch.int32, device=dev),
            torch.full((T, 512), -7, dtype=torch.int32, device=dev),
            torch.full((T, 2048), -7, dtype=torch.int32, device=dev))


def test_noalloc_topk_matches_workspace_topk_on_two_calls_in_a_row():
    dev = need_gpu()
    lib = csa2.load()
    stream = torch.cuda.current_stream()
    for call, lengths in enumerate(([150_000, 40_000, 16_385], [70_001, 300_000, 20_000, 5_000])):
        scores, bm, pt, nvis = _inputs(call, lengths, dev)
        T = len(lengths)
        r = csa2.rows(T, T, n_visible=nvis)
        want = _outputs(T, dev)
        csa2.topk_with_candidates(scores, r, 512, want[0], want[1], pt, bm, want[2])
        got = _outputs(T, dev)
        a = csa2.TopkArgs(scores.data_ptr(), scores.shape[1], bm.data_ptr(), bm.shape[1], pt.data_ptr(),
                          pt.shape[1], r, 512, got[0].data_ptr(), got[1].data_ptr(), 512, got[2].data_ptr(), 2048,
                          None)
        assert lib.csa2_topk_with_candidates_noalloc(C.byref(a), stream.cuda_stream) == 0
        torch.cuda.synchronize()
        assert csa2.check_device_error() == 0
        for w, g in zip(want, got):
            assert np.array_equal(np_(w), np_(g)), f"call {call}"


def test_noalloc_topk_rejects_rows_beyond_the_static_scratch():
    dev = need_gpu()
    lib = csa2.load()
    T = 80                                   # 160 rows of 100,000 with pools: ~17 MB, more than the static scratch
    scores = torch.zeros(T, 100_000, dtype=torch.float32, device=dev)
    bm = torch.zeros(T, 12_500, dtype=torch.float32, device=dev)
    pt = torch.zeros(T, 1_563, dtype=torch.int32, device=dev)
    nvis = torch.full((T,), 100_000, dtype=torch.int32, device=dev)
    out = torch.empty(T, 512, dtype=torch.int32, device=dev)
    pool = torch.empty(T, 2048, dtype=torch.int32, device=dev)
    a = csa2.TopkArgs(scores.data_ptr(), 100_000, bm.data_ptr(), 12_500, pt.data_ptr(), 1_563,
                      csa2.rows(T, T, n_visible=nvis), 512, out.data_ptr(), None, 512, pool.data_ptr(), 2048, None)
    assert lib.csa2_topk_with_candidates_noalloc(C.byref(a), torch.cuda.current_stream().cuda_stream) == 7
    assert b"static scratch" in lib.csa2_last_error_detail()
