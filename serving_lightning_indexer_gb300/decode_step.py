"""One CSA2 decode step over a layer stack, driven through the C ABI.

Layer roles and cache sharing follow the CSA2 page ("三种模式", "V4.1-Flash 的
实际配置") and the V4.1 Q&A page (SharedAttentionRuntime):
  * encoder layers 2..19, m = 2, three groups of six: a Full layer (2, 8, 14)
    builds its group's main-KV entry for the new token pair, scores every
    visible entry and selects top-512; the five Reuse layers reuse its
    top-512 slots.
  * decoder layers 20..39, m = 1, five groups of four: the Full layer 20 builds
    the entry, scores, selects top-512 and the 2048-block candidate pool;
    Reindex layers 24, 28, 32, 36 rescore only that pool with their own
    indexer query; Reuse layers reuse the latest slots.
  * every layer runs sparse attention with its own q, SWA keys and sink.
Four resident cache copies exist: three encoder copies (N/2 entries each) and
one decoder copy (N entries).  Everything on the path runs in the library's
kernels; this module only allocates buffers and issues the calls in order.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import csa2
from . import workloads as W

ENCODER_FULL = (2, 8, 14)
DECODER_FULL = 20
REINDEX = (24, 28, 32, 36)
LAYERS = tuple(range(2, 40))


def role_of(layer: int) -> str:
    if layer in ENCODER_FULL or layer == DECODER_FULL:
        return "full"
    if layer in REINDEX:
        return "reindex"
    return "reuse"


def cache_of(layer: int) -> int:
    """Index of the resident cache copy a layer reads (0..2 encoder, 3 decoder)."""
    return (layer - 2) // 6 if layer < 20 else 3


def ratio_of(cache: int) -> int:
    """Compression ratio m of a cache copy: 2 in the encoder, 1 in the decoder."""
    return 2 if cache < 3 else 1


def keys_scored(lengths, layers=LAYERS) -> int:
    """Index keys one decode step scores: every visible entry (N // m) of each
    sequence for a Full layer, the pool positions (at most 2048 blocks of 8)
    for a Reindex layer, none for a Reuse layer."""
    n = 0
    for l in layers:
        ents = [length // ratio_of(cache_of(l)) for length in lengths]
        if role_of(l) == "full":
            n += sum(ents)
        elif role_of(l) == "reindex":
            n += sum(min(e, W.POOL_BLOCKS * W.POOL_BLOCK) for e in ents)
    return n


@dataclass
class CacheCopy:
    ratio_m: int
    entries: list
    pc: W.PagedCache
    n_visible: torch.Tensor
    ld: int
    entry_slot_new: torch.Tensor     # slot of each sequence's newest entry
    entry_pos_new: torch.Tensor      # its RoPE position


@dataclass
class LayerInputs:
    layer: int
    attn: W.AttnLayer
    iq: W.IndexerQuery | None = None
    C: torch.Tensor | None = None    # bf16 [B*m, 512] tokens of the new entry (Full layers)
    Z: torch.Tensor | None = None
    gamma: torch.Tensor | None = None
    w_ik: torch.Tensor | None = None  # bf16 [512,128] index-key projection of a Full layer (weights)
    k_gamma: torch.Tensor | None = None


@dataclass
class StepBuffers:
    scores: torch.Tensor
    block_max: torch.Tensor
    topk_pos: torch.Tensor
    topk_slot: dict = field(default_factory=dict)   # cache copy -> latest [B,512] slots (topk_idxs slot)
    pool: torch.Tensor | None = None                 # candidates slot
    out: dict = field(default_factory=dict)          # layer -> [B,64,512] bf16
    hist: torch.Tensor | None = None


class DecodeStep:
    """The 38-layer decode step of one batch of sequences with the given context lengths."""

    def __init__(self, lengths: list[int], seed: int, device, layers=LAYERS, out_bf16=True):
        self.lengths = list(lengths)
        self.B = len(lengths)
        self.device = device
        self.layers = tuple(layers)
        dev = device
        self.caches: list[CacheCopy] = []
        for ci in range(4):
            m = ratio_of(ci)
            ents = [n // m for n in lengths]
            if not any(cache_of(l) == ci for l in self.layers):
                self.caches.append(None)
                continue
            pc = W.make_paged_cache(ents, seed=seed * 100 + ci, device=dev)
            ld = (max(ents) + 127) // 128 * 128
            newest = torch.tensor([e - 1 for e in ents], dtype=torch.int64, device=dev)
            slot = (pc.page_table.gather(1, (newest // 64)[:, None]).squeeze(1).long() * 64 + newest % 64).to(torch.int32)
            pos = torch.tensor([(e - 1) * m for e in ents], dtype=torch.int32, device=dev)
            self.caches.append(CacheCopy(m, ents, pc, pc.n_entries, ld, slot, pos))
        self.inputs: dict[int, LayerInputs] = {}
        for l in self.layers:
            li = LayerInputs(l, W.make_attn_layer(self.B, seed=seed * 1000 + l, device=dev))
            if role_of(l) in ("full", "reindex"):
                li.iq = W.make_indexer_query(self.B, seed=seed * 1000 + 500 + l, device=dev)
            if role_of(l) == "full":
                m = self.caches[cache_of(l)].ratio_m
                Cm, Z, gamma = W.make_compress_inputs(self.B * m, seed=seed * 1000 + 700 + l, device=dev)
                li.C, li.Z, li.gamma = Cm, (Z if m == 2 else None), gamma
                li.w_ik, li.k_gamma = W.make_index_projection(seed=seed * 1000 + 800 + l, device=dev)
            self.inputs[l] = li
        ld = max(c.ld for c in self.caches if c is not None)
        self.buf = StepBuffers(
            scores=torch.empty(self.B, ld, dtype=torch.float32, device=dev),
            block_max=torch.empty(self.B, ld // 8, dtype=torch.float32, device=dev),
            topk_pos=torch.empty(self.B, W.TOPK, dtype=torch.int32, device=dev),
        )
        # key histograms produced by the scan and reused by the top-k of the same layer
        self.buf.hist = torch.zeros(2, self.B, 2048, dtype=torch.int32, device=dev)
        for ci, c in enumerate(self.caches):
            if c is not None:
                self.buf.topk_slot[ci] = torch.empty(self.B, W.TOPK, dtype=torch.int32, device=dev)
        if any(cache_of(l) == 3 for l in self.layers):
            self.buf.pool = torch.empty(self.B, W.POOL_BLOCKS, dtype=torch.int32, device=dev)
        for l in self.layers:
            self.buf.out[l] = torch.empty(self.B, W.ATT_HEADS, W.ATT_DIM,
                                          dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dev)
        self.rows = {ci: csa2.rows(self.B, self.B, n_visible=c.n_visible) for ci, c in enumerate(self.caches)
                     if c is not None}
        self.on_index_score = None   # optional hooks (event recording around the indexer scan)
        self.after_index_score = None
        self.on_attn = None          # optional hooks around the sparse attention call
        self.after_attn = None
        self.before_layer = None     # optional hook called with the layer number before its first call
        self.after_layer = None      # optional hook called with the layer number after its last call

    # ---------------------------------------------------------------- per-step work
    def keys_scored_per_step(self) -> int:
        return keys_scored(self.lengths, self.layers)

    def attn_query_layers_per_step(self) -> int:
        return len(self.layers) * self.B

    def index_bytes_per_step(self) -> int:
        return sum(sum(self.caches[cache_of(l)].entries) for l in self.layers if role_of(l) == "full") * 132

    def run(self, stream=None):
        b = self.buf
        for l in self.layers:
            if self.before_layer:
                self.before_layer(l)
            li = self.inputs[l]
            ci = cache_of(l)
            c = self.caches[ci]
            role = role_of(l)
            if role == "full":
                # the Full layer writes its group's newest main-KV entry and index key,
                # then scores and selects
                csa2.compress_m2(li.C, li.Z, c.ratio_m, li.gamma, c.pc.main_kv, entry_slot=c.entry_slot_new,
                                 entry_pos=c.entry_pos_new, stream=stream, w_ik=li.w_ik, k_gamma=li.k_gamma,
                                 index_k=c.pc.index_k)
                sc = b.scores[:, :c.ld]
                bm = b.block_max[:, :c.ld // 8]
                if self.on_index_score:
                    self.on_index_score(l)
                csa2.index_score(li.iq.q_fp8, li.iq.q_scale, li.iq.w, c.pc.index_k, c.pc.page_table,
                                 self.rows[ci], b.scores, b.block_max if ci == 3 else None, stream=stream,
                                 hist=b.hist)
                if self.after_index_score:
                    self.after_index_score(l)
                csa2.topk_with_candidates(b.scores, self.rows[ci], W.TOPK, b.topk_pos, b.topk_slot[ci],
                                          c.pc.page_table, b.block_max if ci == 3 else None,
                                          b.pool if ci == 3 else None, stream=stream, hist=b.hist)
                del sc, bm
            elif role == "reindex":
                csa2.reindex(li.iq.q_fp8, li.iq.q_scale, li.iq.w, c.pc.index_k, c.pc.page_table, self.rows[ci],
                             b.pool, W.TOPK, b.topk_pos, b.topk_slot[ci], stream=stream)
            at = li.attn
            # a Reuse layer's slots and caches were written by its Full or Reindex
            # layer's calls, at least two launches back: its keys are gathered early
            if self.on_attn:
                self.on_attn(l)
            csa2.sparse_attn(at.q, c.pc.main_kv, b.topk_slot[ci], at.swa_kv, at.swa_slot, at.sink, b.out[l],
                             stream=stream, kv_ready=(role == "reuse"))
            if self.after_attn:
                self.after_attn(l)
            if self.after_layer:
                self.after_layer(l)
