"""Host-side checks of the C ABI that need no GPU: the library builds, loads and
exports every symbol include/csa2.h declares, the ctypes structs match the C
layout, and argument validation returns status codes without launching."""
import ctypes as C
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "csa2.h")


@pytest.fixture(scope="module")
def lib():
    from serving_lightning_indexer_gb300 import _build, csa2
    _build.build()
    return csa2.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CSA2_API\s+[\w\s\*]+?\b(csa2_\w+)\s*\(", text)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("csa2_index_score", "csa2_topk_with_candidates", "csa2_reindex", "csa2_sparse_attn",
              "csa2_compress_m2"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from serving_lightning_indexer_gb300 import _build
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(csa2_\w+)", out))
    assert set(declared_functions()) <= exported
    from serving_lightning_indexer_gb300 import csa2
    assert set(csa2.EXPORTED) == set(declared_functions())
    # nothing but the ABI is exported
    assert all(s.startswith("csa2_") for s in exported)


def _struct_sizes_from_c():
    src = r"""
#include <stdio.h>
#include <stddef.h>
#include "csa2.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu\n", sizeof(csa2_rows), sizeof(csa2_index_score_args), sizeof(csa2_topk_args),
         sizeof(csa2_reindex_args), sizeof(csa2_sparse_attn_args), sizeof(csa2_compress_args));
  printf("%zu %zu %zu %zu\n", offsetof(csa2_index_score_args, rows), offsetof(csa2_topk_args, k),
         offsetof(csa2_sparse_attn_args, softmax_scale), offsetof(csa2_compress_args, latent_out));
  return 0;
}
"""
    import tempfile
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "s.c")
        open(c, "w").write(src)
        exe = os.path.join(d, "s")
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        return [list(map(int, l.split())) for l in subprocess.run([exe], capture_output=True, text=True).stdout.split("\n") if l]


def test_ctypes_structs_match_c_layout():
    from serving_lightning_indexer_gb300 import csa2
    sizes, offs = _struct_sizes_from_c()
    assert sizes == [C.sizeof(csa2.Rows), C.sizeof(csa2.IndexScoreArgs), C.sizeof(csa2.TopkArgs),
                     C.sizeof(csa2.ReindexArgs), C.sizeof(csa2.SparseAttnArgs), C.sizeof(csa2.CompressArgs)]
    assert offs == [csa2.IndexScoreArgs.rows.offset, csa2.TopkArgs.k.offset, csa2.SparseAttnArgs.softmax_scale.offset,
                    csa2.CompressArgs.latent_out.offset]


FAKE = 0x10000  # a non-null, 16-B aligned address that is never dereferenced


def test_validation_returns_codes_without_launch(lib):
    from serving_lightning_indexer_gb300 import csa2
    r = csa2.Rows(2, 2, None, None, FAKE, 1)
    a = csa2.IndexScoreArgs(FAKE, FAKE, FAKE, None, 10, FAKE, 4, r, FAKE, 128, None, 0)
    assert lib.csa2_index_score(C.byref(a), None, 0, None) == 1                  # NULL index_k
    a.index_k = FAKE + 8
    assert lib.csa2_index_score(C.byref(a), None, 0, None) == 3                  # misaligned
    a.index_k = FAKE
    a.ld_scores = 130
    assert lib.csa2_index_score(C.byref(a), None, 0, None) == 3                  # ld not a multiple of 4
    a.ld_scores = 128
    a.rows = csa2.Rows(3, 2, None, None, FAKE, 1)
    assert lib.csa2_index_score(C.byref(a), None, 0, None) == 2                  # T != B without row_seq
    a.rows = csa2.Rows(2, 2, None, FAKE, None, 3)
    assert lib.csa2_index_score(C.byref(a), None, 0, None) == 4                  # ratio_m = 3
    assert b"ratio_m" in lib.csa2_last_error_detail()
    a.rows = csa2.Rows(2, 2, None, None, FAKE, 1)
    a.index_k_format = 2
    assert lib.csa2_index_score(C.byref(a), None, 0, None) == 4                  # unknown page format
    a.index_k_format = csa2.INDEX_FP4
    a.index_k = FAKE + 16
    assert lib.csa2_index_score(C.byref(a), None, 0, None) == 3                  # FP4 pages need 32-B alignment
    a.index_k = FAKE
    a.rows = csa2.Rows(2049, 1, FAKE, FAKE, None, 2)
    a.hist = FAKE
    assert lib.csa2_index_score(C.byref(a), None, 0, None) == 2                  # FP4 prefill rows: per-row scan,
    assert b"hist" in lib.csa2_last_error_detail()                               # whose hist takes <= 2048 rows
    a.index_k_format = csa2.INDEX_FP8
    assert lib.csa2_index_score(C.byref(a), None, 0, None) == 4                  # FP8 prefill path: no hist
    a.hist = None
    a.rows = csa2.Rows(16385, 1, FAKE, FAKE, None, 2)
    assert lib.csa2_index_score(C.byref(a), None, 0, None) == 2                  # prefill path: <= 16384 rows

    t = csa2.TopkArgs(FAKE, 128, None, 0, None, 0, csa2.Rows(2, 2, None, None, FAKE, 1), 4096, FAKE, None, 4096,
                      None, 0)
    assert lib.csa2_topk_with_candidates(C.byref(t), None, 0, None) == 2         # k > 2048
    t.k, t.ld_topk = 512, 512
    t.pool_blocks, t.pool_n = FAKE, 2048
    assert lib.csa2_topk_with_candidates(C.byref(t), None, 0, None) == 1         # pool needs block_max
    t.block_max, t.ld_block_max = FAKE, 16
    n = C.c_size_t(0)
    assert lib.csa2_workspace_size(2, C.cast(C.byref(t), C.c_void_p), C.byref(n)) == 0 and n.value == 0
    t.ld_scores, t.ld_block_max = 32768, 4096                                    # rows past the direct path
    assert lib.csa2_workspace_size(2, C.cast(C.byref(t), C.c_void_p), C.byref(n)) == 0 and n.value > 0
    assert lib.csa2_topk_with_candidates(C.byref(t), None, 0, None) == 7         # workspace missing
    t.order = 2
    assert lib.csa2_topk_with_candidates(C.byref(t), None, 0, None) == 2         # order is 0 or 1
    assert b"order" in lib.csa2_last_error_detail()
    t.order = 0

    s = csa2.SparseAttnArgs(FAKE, FAKE, 10, FAKE, 512, 512, FAKE, 10, FAKE, 129, 129, FAKE, 0.0, 1, 0, FAKE, None)
    assert lib.csa2_sparse_attn(C.byref(s), None, 0, None) == 2                  # n_swa > 128
    s.n_swa, s.softmax_scale = 128, -1.0
    assert lib.csa2_sparse_attn(C.byref(s), None, 0, None) == 2                  # negative scale
    s.softmax_scale, s.out_inv_rope = 0.0, 1
    assert lib.csa2_sparse_attn(C.byref(s), None, 0, None) == 1                  # inverse RoPE needs q_pos
    s.out_inv_rope, s.swa_seg_start = 0, FAKE
    assert lib.csa2_sparse_attn(C.byref(s), None, 0, None) == 1                  # bounded replay needs q_pos
    s.q_pos, s.out_inv_rope = FAKE, 2
    assert lib.csa2_sparse_attn(C.byref(s), None, 0, None) == 2                  # flag is 0 or 1
    s.out_inv_rope, s.rope_theta = 1, -5.0
    assert lib.csa2_sparse_attn(C.byref(s), None, 0, None) == 2                  # negative theta

    ca = csa2.CompressArgs(FAKE, None, 64, 2, FAKE, 1e-6, 1, 10000.0, 0, None, FAKE, 64, FAKE, 1, None, None)
    assert lib.csa2_compress_m2(C.byref(ca), None) == 1                          # m=2 needs Z
    ca.ratio_m = 4
    assert lib.csa2_compress_m2(C.byref(ca), None) == 4
    ca.ratio_m = 1
    ca.gamma = FAKE + 4                                                          # weights read as 16-B vectors
    assert lib.csa2_compress_m2(C.byref(ca), None) == 3
    ca.gamma, ca.w_ik, ca.k_gamma, ca.index_k, ca.index_k_pages = FAKE, FAKE, FAKE + 8, FAKE, 1
    assert lib.csa2_compress_m2(C.byref(ca), None) == 3
    for code in range(9):
        assert lib.csa2_status_string(code)
    assert lib.csa2_debug_bounded_wait(0, None) == 2                             # polls out of range: no launch


def test_binding_refuses_cpu_tensors(lib):
    import torch

    from serving_lightning_indexer_gb300 import csa2
    x = torch.zeros(4, 32, 128, dtype=torch.uint8)
    with pytest.raises(ValueError):
        csa2.index_score(x, x, x, x, x, csa2.Rows(1, 1, None, None, None, 1), x)


def _topk_scratch_rule(T, L, pool, hist_given):
    """The top-k scratch rule include/csa2.h states for the no-allocation call
    (and that csa2_workspace_size reports for the workspace call)."""
    if L <= 16384:
        return 0
    V = T * (2 if pool else 1)
    c = -(-L // 4096)
    return (0 if hist_given else V * 8192 + (V * 8 + 255) // 256 * 256) + (V * c * 4 + 255) // 256 * 256 + V * c * 8192


@pytest.mark.parametrize("T,ld_scores,ld_bm,pool,hist", [
    (1, 1 << 20, 1 << 17, True, False),     # a 1M row with its pool: 4,212,992 B
    (1, 1 << 20, 1 << 17, False, False),    # without the pool: 2.1 MB
    (3, 1 << 20, 1 << 17, False, False),    # three 1M rows fit the 8 MiB array
    (7, 262144, 32768, True, False),        # seven 262,144-entry rows with pools fit
    (8, 262144, 32768, True, False),        # eight do not
    (5, 100000, 12500, True, True),         # histograms given: no histogram part
    (4, 16384, 2048, True, False),          # direct path: no scratch
    (2, 20000, 40000, True, False),         # the pool row is the longer one
])
def test_topk_workspace_size_follows_the_documented_rule(lib, T, ld_scores, ld_bm, pool, hist):
    from serving_lightning_indexer_gb300 import csa2
    t = csa2.TopkArgs(FAKE, ld_scores, FAKE, ld_bm, FAKE, 8, csa2.Rows(T, T, None, None, FAKE, 1), 512, FAKE, FAKE,
                      512, FAKE if pool else None, 2048, FAKE if hist else None)
    n = C.c_size_t(0)
    assert lib.csa2_workspace_size(csa2.CALL_TOPK, C.cast(C.byref(t), C.c_void_p), C.byref(n)) == 0
    L = max(ld_scores, ld_bm) if pool else ld_scores
    assert n.value == _topk_scratch_rule(T, L, pool, hist)
    limit = 8 << 20
    if (T, ld_scores, pool) == (1, 1 << 20, True):
        assert n.value == 4_212_992
    if (T, ld_scores, pool) == (7, 262144, True):
        assert n.value == 7_458_560 <= limit
    if (T, ld_scores, pool) == (8, 262144, True):
        assert n.value == 8_524_032 > limit
