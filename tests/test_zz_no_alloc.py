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
from serving_lightning_indexer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
LIMIT = 8 << 20          # CSA2_TOPK_NOALLOC_SCRATCH_BYTES


def _scratch_bytes(T, L, pool, hist_given=False):
    """The scratch rule stated in include/csa2.h."""
    if L <= 16384:
        return 0
    V = T * (2 if pool else 1)
    c = -(-L // 4096)
    return (0 if hist_given else V * 8192 + (V * 8 + 255) // 256 * 256) + (V * c * 4 + 255) // 256 * 256 + V * c * 8192


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


def _args(scores, bm, pt, r, out, hist=None):
    return csa2.TopkArgs(scores.data_ptr(), scores.shape[1], bm.data_ptr(), bm.shape[1], pt.data_ptr(), pt.shape[1],
                         r, 512, out[0].data_ptr(), out[1].data_ptr(), 512, out[2].data_ptr(), 2048,
                         hist.data_ptr() if hist is not None else None)


def _compare(lib, scores, bm, pt, nvis, hist=None, what="", before=None):
    """The no-allocation call against the workspace call on the same inputs: bit-exact.
    `before` (if given) runs ahead of each of the two calls: a top-k call that
    is given the scan's histograms returns them to zero, so the scan writes
    them again for the next one."""
    dev = scores.device
    T = scores.shape[0]
    r = csa2.rows(T, T, n_visible=nvis)
    want = _outputs(T, dev)
    if before:
        before()
    csa2.topk_with_candidates(scores, r, 512, want[0], want[1], pt, bm, want[2], hist=hist)
    got = _outputs(T, dev)
    if before:
        before()
    a = _args(scores, bm, pt, r, got, hist)
    assert lib.csa2_topk_with_candidates_noalloc(C.byref(a), torch.cuda.current_stream().cuda_stream) == 0, \
        lib.csa2_last_error_detail()
    torch.cuda.synchronize()
    assert csa2.check_device_error() == 0
    for w, g in zip(want, got):
        assert np.array_equal(np_(w), np_(g)), what


def test_noalloc_topk_matches_workspace_topk_on_two_calls_in_a_row():
    dev = need_gpu()
    lib = csa2.load()
    for call, lengths in enumerate(([150_000, 40_000, 16_385], [70_001, 300_000, 20_000, 5_000])):
        _compare(lib, *_inputs(call, lengths, dev), what=f"call {call}")


def test_noalloc_topk_short_rows_use_no_scratch():
    """Rows of at most 16,384 entries are selected directly (no scratch)."""
    dev = need_gpu()
    lib = csa2.load()
    lengths = [16_384, 5_000, 100, 12_345]
    assert _scratch_bytes(len(lengths), max(lengths) + 3 & ~3, True) == 0
    for call in range(2):
        _compare(lib, *_inputs(10 + call, lengths, dev), what=f"short rows, call {call}")


def test_noalloc_topk_with_the_scan_histograms():
    """With the scan's histograms the scratch holds no histogram part."""
    dev = need_gpu()
    lib = csa2.load()
    lengths = [40_000, 100_000, 70_000]
    B = len(lengths)
    pc = W.make_paged_cache(lengths, seed=21, device=dev, with_main=False)
    iq = W.make_indexer_query(B, seed=22, device=dev)
    r = csa2.rows(B, B, n_visible=pc.n_entries)
    ld = (max(lengths) + 127) // 128 * 128
    scores = torch.empty(B, ld, dtype=torch.float32, device=dev)
    bm = torch.empty(B, ld // 8, dtype=torch.float32, device=dev)
    hist = torch.zeros(2, B, 2048, dtype=torch.int32, device=dev)

    def scan():
        csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, r, scores, bm, hist=hist)
    for call in range(2):
        _compare(lib, scores, bm, pc.page_table, pc.n_entries, hist=hist, what=f"with histograms, call {call}",
                 before=scan)
        assert not np_(hist).any(), "the call returns the histograms to zero"


def test_noalloc_topk_just_under_and_just_over_the_static_scratch():
    """Seven rows of 262,144 entries with pools fit the 8 MiB array (7,458,560 B);
    eight (8,524,032 B) are rejected before any launch."""
    dev = need_gpu()
    lib = csa2.load()
    n = 262_144
    assert _scratch_bytes(7, n, True) <= LIMIT < _scratch_bytes(8, n, True)
    _compare(lib, *_inputs(30, [n] * 7, dev), what="7 rows of 262,144 with pools")
    scores, bm, pt, nvis = _inputs(31, [n] * 8, dev)
    r = csa2.rows(8, 8, n_visible=nvis)
    out = _outputs(8, dev)
    a = _args(scores, bm, pt, r, out)
    need = C.c_size_t(0)
    assert lib.csa2_workspace_size(csa2.CALL_TOPK, C.cast(C.byref(a), C.c_void_p), C.byref(need)) == 0
    assert need.value == _scratch_bytes(8, n, True) > LIMIT
    assert lib.csa2_topk_with_candidates_noalloc(C.byref(a), torch.cuda.current_stream().cuda_stream) == 7
    detail = lib.csa2_last_error_detail()
    assert b"static scratch" in detail and b"csa2_topk_with_candidates_noalloc" in detail
    torch.cuda.synchronize()
    assert (np_(out[0]) == -7).all()      # nothing was launched


def test_noalloc_topk_argument_errors_name_the_called_function():
    need_gpu()
    lib = csa2.load()
    a = csa2.TopkArgs()                  # everything NULL / zero
    assert lib.csa2_topk_with_candidates_noalloc(C.byref(a), None) != 0
    assert lib.csa2_last_error_detail().startswith(b"csa2_topk_with_candidates_noalloc:")
