"""Thin Python binding of the CSA2 C ABI (``include/csa2.h``).

Argument marshalling only: every step runs in the CUDA kernels of
``libcsa2.so``.  Tensors are torch CUDA tensors (their device pointers are
passed); there is no CPU fallback -- a missing library or a CPU tensor raises.
Workspace is allocated by torch on first use and cached per device.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import _build

_P = C.c_void_p
_I32 = C.c_int32
_I64 = C.c_int64


class Csa2Error(RuntimeError):
    def __init__(self, code: int, where: str, detail: str):
        super().__init__(f"{where}: status {code} ({detail})")
        self.code = code


# ---------------------------------------------------------------- C structs
class Rows(C.Structure):
    _fields_ = [("T", _I32), ("B", _I32), ("row_seq", _P), ("row_pos", _P), ("n_visible", _P), ("ratio_m", _I32)]


class IndexScoreArgs(C.Structure):
    _fields_ = [("q_fp8", _P), ("q_scale", _P), ("w", _P), ("index_k", _P), ("index_k_pages", _I64),
                ("page_table", _P), ("pt_stride", _I32), ("rows", Rows), ("scores", _P), ("ld_scores", _I64),
                ("block_max", _P), ("ld_block_max", _I64), ("hist", _P), ("index_k_format", _I32)]


class TopkArgs(C.Structure):
    _fields_ = [("scores", _P), ("ld_scores", _I64), ("block_max", _P), ("ld_block_max", _I64),
                ("page_table", _P), ("pt_stride", _I32), ("rows", Rows), ("k", _I32), ("topk_pos", _P),
                ("topk_slot", _P), ("ld_topk", _I64), ("pool_blocks", _P), ("pool_n", _I32), ("hist", _P),
                ("order", _I32)]


class ReindexArgs(C.Structure):
    _fields_ = [("q_fp8", _P), ("q_scale", _P), ("w", _P), ("index_k", _P), ("index_k_pages", _I64),
                ("page_table", _P), ("pt_stride", _I32), ("rows", Rows), ("pool_blocks", _P), ("pool_n", _I32),
                ("k", _I32), ("topk_pos", _P), ("topk_slot", _P), ("ld_topk", _I64), ("pool_scores", _P),
                ("index_k_format", _I32), ("order", _I32)]


class SparseAttnArgs(C.Structure):
    _fields_ = [("q", _P), ("main_kv", _P), ("main_kv_slots", _I64), ("topk_slot", _P), ("k", _I32),
                ("ld_topk", _I64), ("swa_kv", _P), ("swa_slots", _I64), ("swa_slot", _P), ("n_swa", _I32),
                ("ld_swa", _I64), ("sink", _P), ("softmax_scale", C.c_float), ("T", _I32), ("out_bf16", _I32),
                ("out", _P), ("lse", _P), ("kv_ready", _I32), ("q_pos", _P), ("out_inv_rope", _I32),
                ("rope_theta", C.c_float), ("swa_seg_start", _P)]


class CompressArgs(C.Structure):
    _fields_ = [("C", _P), ("Z", _P), ("n_tokens", _I64), ("ratio_m", _I32), ("gamma", _P), ("eps", C.c_float),
                ("apply_rope", _I32), ("rope_theta", C.c_float), ("first_entry", _I64), ("entry_pos", _P),
                ("main_kv", _P), ("main_kv_slots", _I64), ("page_table", _P), ("pt_len", _I64),
                ("entry_slot", _P), ("latent_out", _P), ("w_ik", _P), ("k_gamma", _P), ("index_k", _P),
                ("index_k_pages", _I64), ("index_k_format", _I32), ("index_latent_out", _P)]


class KvProjectArgs(C.Structure):
    _fields_ = [("hidden", _P), ("w", _P), ("T", _I32), ("hidden_dim", _I32), ("out", _P)]


CALL_INDEX_SCORE, CALL_TOPK, CALL_REINDEX, CALL_SPARSE_ATTN = 1, 2, 3, 4
EXPORTED = ("csa2_status_string", "csa2_last_error_detail", "csa2_index_score", "csa2_topk_with_candidates",
            "csa2_reindex", "csa2_sparse_attn", "csa2_compress_m2", "csa2_workspace_size",
            "csa2_check_device_error", "csa2_version", "csa2_topk_with_candidates_noalloc",
            "csa2_debug_bounded_wait", "csa2_kv_project")

_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> C.CDLL:
    """Load libcsa2.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"libcsa2.so is not built ({path}); run __graft_entry__.build()")
        _build.build()
    lib = C.CDLL(path)
    lib.csa2_status_string.restype = C.c_char_p
    lib.csa2_status_string.argtypes = [C.c_int]
    lib.csa2_last_error_detail.restype = C.c_char_p
    lib.csa2_version.restype = C.c_char_p
    for name, st in (("csa2_index_score", IndexScoreArgs), ("csa2_topk_with_candidates", TopkArgs),
                     ("csa2_reindex", ReindexArgs), ("csa2_sparse_attn", SparseAttnArgs)):
        f = getattr(lib, name)
        f.restype = C.c_int
        f.argtypes = [C.POINTER(st), _P, C.c_size_t, _P]
    lib.csa2_topk_with_candidates_noalloc.restype = C.c_int
    lib.csa2_topk_with_candidates_noalloc.argtypes = [C.POINTER(TopkArgs), _P]
    lib.csa2_compress_m2.restype = C.c_int
    lib.csa2_compress_m2.argtypes = [C.POINTER(CompressArgs), _P]
    lib.csa2_workspace_size.restype = C.c_int
    lib.csa2_workspace_size.argtypes = [C.c_int, _P, C.POINTER(C.c_size_t)]
    lib.csa2_check_device_error.restype = C.c_int
    lib.csa2_check_device_error.argtypes = [_P]
    lib.csa2_kv_project.restype = C.c_int
    lib.csa2_kv_project.argtypes = [C.POINTER(KvProjectArgs), _P]
    lib.csa2_debug_bounded_wait.restype = C.c_int
    lib.csa2_debug_bounded_wait.argtypes = [C.c_uint32, _P]
    _lib = lib
    return lib


def _check(rc: int, where: str):
    if rc != 0:
        lib = load()
        raise Csa2Error(rc, where, (lib.csa2_last_error_detail() or b"").decode())


# ---------------------------------------------------------------- helpers
def _ptr(t) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("CSA2 calls take CUDA tensors (no CPU path)")
    if not t.is_contiguous():
        raise ValueError("CSA2 calls take contiguous tensors")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


_ws_cache: dict = {}


def workspace(nbytes: int, device, tag: str = "main") -> torch.Tensor | None:
    """A cached device buffer of at least nbytes (16-B aligned), or None."""
    if nbytes == 0:
        return None
    key = (str(device), tag)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


INDEX_FP8, INDEX_FP4 = 0, 1
INDEX_PAGE_BYTES = {8448: INDEX_FP8, 4352: INDEX_FP4}


def index_format(index_k) -> int:
    """Page format of an index-K cache [n_pages, page bytes]: FP8 (8448 B) or FP4 (4352 B)."""
    fmt = INDEX_PAGE_BYTES.get(int(index_k.shape[-1]))
    if fmt is None:
        raise ValueError(f"index-K pages of {index_k.shape[-1]} B: expected 8448 (FP8) or 4352 (FP4)")
    return fmt


def rows(T, B, row_seq=None, row_pos=None, n_visible=None, ratio_m=1) -> Rows:
    """Row description of a call.  The struct holds device pointers; it also
    keeps the tensors themselves, so that they stay allocated as long as the
    struct is in use."""
    r = Rows(T, B, _ptr(row_seq), _ptr(row_pos), _ptr(n_visible), ratio_m)
    r._tensors = (row_seq, row_pos, n_visible)
    return r


# ---------------------------------------------------------------- calls
def index_score(q_fp8, q_scale, w, index_k, page_table, r: Rows, scores, block_max=None, stream=None, hist=None):
    """Lightning-Indexer scores (csa2_index_score); `hist` ([2,T,2048] int32) optionally
    receives the key histograms that csa2_topk_with_candidates can reuse."""
    lib = load()
    a = IndexScoreArgs(_ptr(q_fp8), _ptr(q_scale), _ptr(w), _ptr(index_k), index_k.shape[0], _ptr(page_table),
                       page_table.shape[-1], r, _ptr(scores), scores.shape[-1], _ptr(block_max),
                       block_max.shape[-1] if block_max is not None else 0, _ptr(hist), index_format(index_k))
    _check(lib.csa2_index_score(C.byref(a), None, 0, _stream(stream)), "csa2_index_score")


def topk_with_candidates(scores, r: Rows, k, topk_pos, topk_slot=None, page_table=None, block_max=None,
                         pool_blocks=None, stream=None, ws=None, hist=None, order=0):
    """Top-k positions / slots and the optional candidate pool (csa2_topk_with_candidates)."""
    lib = load()
    a = TopkArgs(_ptr(scores), scores.shape[-1], _ptr(block_max), block_max.shape[-1] if block_max is not None else 0,
                 _ptr(page_table), page_table.shape[-1] if page_table is not None else 0, r, k, _ptr(topk_pos),
                 _ptr(topk_slot), topk_pos.shape[-1], _ptr(pool_blocks),
                 pool_blocks.shape[-1] if pool_blocks is not None else 0, _ptr(hist), order)
    need = C.c_size_t(0)
    _check(lib.csa2_workspace_size(CALL_TOPK, C.cast(C.byref(a), _P), C.byref(need)), "csa2_workspace_size")
    buf = ws if ws is not None else workspace(need.value, scores.device, "topk")
    _check(lib.csa2_topk_with_candidates(C.byref(a), _ptr(buf), buf.numel() if buf is not None else 0,
                                         _stream(stream)), "csa2_topk_with_candidates")


def topk_with_candidates_noalloc(scores, r: Rows, k, topk_pos, topk_slot=None, page_table=None, block_max=None,
                                 pool_blocks=None, stream=None, hist=None, order=0):
    """csa2_topk_with_candidates_noalloc: the same selection without a workspace; its
    scratch is a static device array inside the library (for callers that cannot
    allocate device memory)."""
    lib = load()
    a = TopkArgs(_ptr(scores), scores.shape[-1], _ptr(block_max), block_max.shape[-1] if block_max is not None else 0,
                 _ptr(page_table), page_table.shape[-1] if page_table is not None else 0, r, k, _ptr(topk_pos),
                 _ptr(topk_slot), topk_pos.shape[-1], _ptr(pool_blocks),
                 pool_blocks.shape[-1] if pool_blocks is not None else 0, _ptr(hist), order)
    _check(lib.csa2_topk_with_candidates_noalloc(C.byref(a), _stream(stream)), "csa2_topk_with_candidates_noalloc")


def reindex(q_fp8, q_scale, w, index_k, page_table, r: Rows, pool_blocks, k, topk_pos, topk_slot=None,
            pool_scores=None, stream=None, ws=None, order=0):
    """Pool-only rescoring and top-k of a Reindex layer (csa2_reindex)."""
    lib = load()
    a = ReindexArgs(_ptr(q_fp8), _ptr(q_scale), _ptr(w), _ptr(index_k), index_k.shape[0], _ptr(page_table),
                    page_table.shape[-1], r, _ptr(pool_blocks), pool_blocks.shape[-1], k, _ptr(topk_pos),
                    _ptr(topk_slot), topk_pos.shape[-1], _ptr(pool_scores), index_format(index_k), order)
    need = C.c_size_t(0)
    _check(lib.csa2_workspace_size(CALL_REINDEX, C.cast(C.byref(a), _P), C.byref(need)), "csa2_workspace_size")
    buf = ws if ws is not None else workspace(need.value, q_fp8.device, "reindex")
    _check(lib.csa2_reindex(C.byref(a), _ptr(buf), buf.numel() if buf is not None else 0, _stream(stream)),
           "csa2_reindex")


def sparse_attn(q, main_kv, topk_slot, swa_kv, swa_slot, sink, out, lse=None, softmax_scale=0.0, k=None,
                n_swa=None, stream=None, ws=None, kv_ready=False, q_pos=None, out_inv_rope=False, rope_theta=0.0,
                swa_seg_start=None):
    """MQA sparse attention with SWA keys and sink (csa2_sparse_attn); with q_pos
    ([T] int32) optionally the output's inverse RoPE and the SWA bounded-replay
    mask (swa_seg_start, [T] int32)."""
    lib = load()
    T = q.shape[0]
    kk = topk_slot.shape[-1] if (k is None and topk_slot is not None) else (k or 0)
    ns = swa_slot.shape[-1] if (n_swa is None and swa_slot is not None) else (n_swa or 0)
    a = SparseAttnArgs(_ptr(q), _ptr(main_kv), main_kv.shape[0] if main_kv is not None else 0, _ptr(topk_slot), kk,
                       topk_slot.shape[-1] if topk_slot is not None else 0, _ptr(swa_kv),
                       swa_kv.shape[0] if swa_kv is not None else 0, _ptr(swa_slot), ns,
                       swa_slot.shape[-1] if swa_slot is not None else 0, _ptr(sink), float(softmax_scale), T,
                       1 if out.dtype == torch.bfloat16 else 0, _ptr(out), _ptr(lse), 1 if kv_ready else 0,
                       _ptr(q_pos), 1 if out_inv_rope else 0, float(rope_theta), _ptr(swa_seg_start))
    need = C.c_size_t(0)
    _check(lib.csa2_workspace_size(CALL_SPARSE_ATTN, C.cast(C.byref(a), _P), C.byref(need)), "csa2_workspace_size")
    buf = ws if ws is not None else workspace(need.value, q.device, "attn")
    _check(lib.csa2_sparse_attn(C.byref(a), _ptr(buf), buf.numel() if buf is not None else 0, _stream(stream)),
           "csa2_sparse_attn")


def compress_m2(Cm, Z, ratio_m, gamma, main_kv, page_table=None, entry_slot=None, eps=1e-6, rope_theta=10000.0,
                apply_rope=True, first_entry=0, entry_pos=None, latent_out=None, stream=None,
                w_ik=None, k_gamma=None, index_k=None, index_latent_out=None):
    """Main-KV entry build: m=2 softmax pooling (or m=1), RMSNorm, RoPE, FP4 (csa2_compress_m2);
    with w_ik ([512,128] bf16), k_gamma and index_k also the entries' index keys."""
    lib = load()
    a = CompressArgs(_ptr(Cm), _ptr(Z), Cm.shape[0], ratio_m, _ptr(gamma), eps, 1 if apply_rope else 0, rope_theta,
                     first_entry, _ptr(entry_pos), _ptr(main_kv), main_kv.shape[0], _ptr(page_table),
                     page_table.numel() if page_table is not None else 0, _ptr(entry_slot), _ptr(latent_out),
                     _ptr(w_ik), _ptr(k_gamma), _ptr(index_k), index_k.shape[0] if index_k is not None else 0,
                     index_format(index_k) if index_k is not None else 0, _ptr(index_latent_out))
    _check(lib.csa2_compress_m2(C.byref(a), _stream(stream)), "csa2_compress_m2")


def kv_project(hidden, w, out, stream=None):
    """out [T,512] bf16 = hidden [T,H] bf16 @ w [H,512] bf16 (csa2_kv_project)."""
    lib = load()
    a = KvProjectArgs(_ptr(hidden), _ptr(w), hidden.shape[0], hidden.shape[1], _ptr(out))
    _check(lib.csa2_kv_project(C.byref(a), _stream(stream)), "csa2_kv_project")


def check_device_error(stream=None) -> int:
    """Synchronise the stream and return the device error status (0 = ok)."""
    lib = load()
    return lib.csa2_check_device_error(_stream(stream))


def version() -> str:
    return load().csa2_version().decode()
