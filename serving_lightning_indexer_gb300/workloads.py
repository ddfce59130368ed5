"""Seeded synthetic inputs for the CSA2 global-attention step.

This module only draws random tensors and writes them in the cache storage
formats (FP8 e4m3 with an fp32 scale, FP4 e2m1 with ue8m0 block scales, paged
layouts with a random page permutation).  It computes no step of the method:
no score, selection, attention, compression, normalisation or rotation.  Both
the CUDA path (tests, benchmark) and the CPU oracle consume the bytes it
produces.

Shapes and distributions follow the workloads of the CSA2 / DSA pages:
32 indexer heads x 128 dims, 64 attention heads x 512 dims, 128 SWA keys,
top-512, 2048-block x 8 candidate pools, page size 64.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

PAGE = 64
IDX_HEADS, IDX_DIM = 32, 128
ATT_HEADS, ATT_DIM = 64, 512
INDEX_PAGE_BYTES = PAGE * (IDX_DIM + 4)
INDEX_FP4_PAGE_BYTES = PAGE * (IDX_DIM // 2 + 4)   # 64 x 64 B e2m1 codes, then 64 x 4 ue8m0 scales
MAIN_RECORD_BYTES = 288
SWA_RECORD_BYTES = 528
SWA_WINDOW = 128
TOPK = 512
POOL_BLOCKS = 2048
POOL_BLOCK = 8


# ---------------------------------------------------------------------------
# storage-format encoders (input encoding only)
# ---------------------------------------------------------------------------

def fp8_encode(x: torch.Tensor):
    """e4m3 codes of x [..., n] with one fp32 scale per row (amax / 448; 1 for an
    all-zero row).  Returns (codes uint8 [..., n], scale float32 [...])."""
    x = x.float()
    amax = x.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (x / scale.unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


# e2m1 magnitudes 0,.5,1,1.5,2,3,4,6; a value exactly between two neighbours goes
# to the even code, so the comparison is '>' below an even code and '>=' below
# an odd one.
_FP4_MIDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def fp4_encode_blocks(x: torch.Tensor):
    """e2m1 codes of x [n,d] (d a multiple of 32) with one ue8m0 scale per 32
    elements: the smallest power of two 2^k with 6 * 2^k >= amax, 127 for an
    all-zero block.  Returns (codes uint8 [n,d//2], element 2i in the low nibble
    of byte i; scales uint8 [n,d//32])."""
    x = x.float()
    n, d = x.shape
    g = x.reshape(n, d // 32, 32)
    amax = g.abs().amax(dim=-1)
    safe = torch.where(amax > 0, amax, torch.full_like(amax, 6.0))
    k = torch.ceil(torch.log2(safe / 6.0))
    for _ in range(2):
        k = torch.where(6.0 * torch.exp2(k) < safe, k + 1, k)
        k = torch.where(6.0 * torch.exp2(k - 1) >= safe, k - 1, k)
    u = torch.where(amax > 0, k + 127, torch.full_like(k, 127.0)).clamp(0, 254)
    y = g / torch.exp2(u - 127).unsqueeze(-1)
    mag = y.abs()
    code = torch.zeros_like(mag, dtype=torch.int32)
    for i, m in enumerate(_FP4_MIDS):
        code += (mag > m).int() if i % 2 == 0 else (mag >= m).int()
    code = code.clamp(max=7) | ((y < 0).int() << 3)
    code = code.reshape(n, d)
    return (code[:, 0::2] | (code[:, 1::2] << 4)).to(torch.uint8), u.to(torch.uint8)


def fp4_encode_records(x: torch.Tensor) -> torch.Tensor:
    """288-byte main-KV records of x [n,512]: 512 e2m1 codes (element 2i in the
    low nibble of byte i), 16 ue8m0 scales (one per 32 elements), 16 zero
    bytes."""
    x = x.float().reshape(-1, ATT_DIM)
    codes, u = fp4_encode_blocks(x)
    rec = torch.zeros(x.shape[0], MAIN_RECORD_BYTES, dtype=torch.uint8, device=x.device)
    rec[:, :256] = codes
    rec[:, 256:272] = u
    return rec


def swa_encode_records(x: torch.Tensor) -> torch.Tensor:
    """528-byte SWA records of x [n,512]: 512 e4m3 codes, then 4 fp32 scales (one
    per 128 channels)."""
    x = x.float().reshape(-1, 4, 128)
    codes, scale = fp8_encode(x)                                 # [n,4,128], [n,4]
    n = x.shape[0]
    rec = torch.empty(n, SWA_RECORD_BYTES, dtype=torch.uint8, device=x.device)
    rec[:, :512] = codes.reshape(n, 512)
    rec[:, 512:] = scale.contiguous().view(torch.uint8).reshape(n, 16)
    return rec


# ---------------------------------------------------------------------------
# paged caches
# ---------------------------------------------------------------------------

@dataclass
class PagedCache:
    """One shared cache pair of a Full layer: the index-K pages and the main-KV
    records, addressed through the same page table (entry e of sequence b is
    slot page_table[b, e // 64] * 64 + e % 64 in both)."""
    index_k: torch.Tensor          # uint8 [n_pages, 8448] (FP8 keys) or [n_pages, 4352] (FP4 keys)
    main_kv: torch.Tensor          # uint8 [n_pages * 64, 288]
    page_table: torch.Tensor       # int32 [B, pt_stride], -1 past the sequence
    n_entries: torch.Tensor        # int32 [B]
    n_entries_host: list = field(default_factory=list)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_paged_cache(entries: list[int], seed: int, device="cpu", permute=True,
                     plant_dirs: torch.Tensor | None = None, plant_frac: float = 0.0,
                     plant_shift: float = 3.0, with_main=True, chunk_pages=4096,
                     index_fp4=False) -> PagedCache:
    """Index-K pages (keys ~ N(0,1) -> e4m3 + fp32 scale per key, or with
    index_fp4 e2m1 + one ue8m0 scale per 32 dims) and main-KV records (~ N(0,1)
    -> e2m1 + ue8m0/32) for sequences with the given entry counts, pages of 64
    in a random physical permutation.

    plant_dirs [B,128] (optional): for a random plant_frac of the 8-entry blocks
    of sequence b, plant_shift * unit(plant_dirs[b]) is added to the key before
    quantisation (a +3 sigma shift of the key's projection on that direction).
    """
    g = _gen(seed, device)
    B = len(entries)
    pages = [max(1, math.ceil(e / PAGE)) for e in entries]
    P = sum(pages)
    phys = torch.randperm(P, generator=g, device=device) if permute else torch.arange(P, device=device)
    pt_stride = max(pages)
    page_table = torch.full((B, pt_stride), -1, dtype=torch.int32, device=device)
    owner = torch.empty(P, dtype=torch.int64, device=device)      # physical page -> sequence
    lpage = torch.empty(P, dtype=torch.int64, device=device)      # physical page -> logical page
    off = 0
    for b, np_ in enumerate(pages):
        ids = phys[off:off + np_]
        page_table[b, :np_] = ids.to(torch.int32)
        owner[ids] = b
        lpage[ids] = torch.arange(np_, device=device)
        off += np_
    planted = None
    if plant_dirs is not None and plant_frac > 0:
        planted = []
        for b, e in enumerate(entries):
            nblk = math.ceil(e / POOL_BLOCK)
            cnt = int(round(plant_frac * nblk))
            planted.append(torch.randperm(nblk, generator=g, device=device)[:cnt])
        units = plant_dirs.float() / plant_dirs.float().norm(dim=-1, keepdim=True)
        # per (physical page, row) shift mask
        mask = torch.zeros(P, PAGE, dtype=torch.bool, device=device)
        for b, blks in enumerate(planted):
            pos = (blks[:, None] * POOL_BLOCK + torch.arange(POOL_BLOCK, device=device)[None]).reshape(-1)
            pos = pos[pos < entries[b]]
            pp = page_table[b, (pos // PAGE)].long()
            mask[pp, pos % PAGE] = True
    index_k = torch.empty(P, INDEX_FP4_PAGE_BYTES if index_fp4 else INDEX_PAGE_BYTES, dtype=torch.uint8,
                          device=device)
    main_kv = torch.empty(P * PAGE, MAIN_RECORD_BYTES, dtype=torch.uint8, device=device) if with_main else None
    for p0 in range(0, P, chunk_pages):
        p1 = min(P, p0 + chunk_pages)
        k = torch.randn(p1 - p0, PAGE, IDX_DIM, generator=g, device=device)
        if planted is not None:
            shift = units[owner[p0:p1]][:, None, :] * plant_shift           # [n,1,128]
            k = k + shift * mask[p0:p1, :, None].float()
        if index_fp4:
            codes, u = fp4_encode_blocks(k.reshape(-1, IDX_DIM))
            index_k[p0:p1, :PAGE * IDX_DIM // 2] = codes.reshape(p1 - p0, -1)
            index_k[p0:p1, PAGE * IDX_DIM // 2:] = u.reshape(p1 - p0, -1)
        else:
            codes, scale = fp8_encode(k)
            index_k[p0:p1, :PAGE * IDX_DIM] = codes.reshape(p1 - p0, -1)
            index_k[p0:p1, PAGE * IDX_DIM:] = scale.contiguous().view(torch.uint8).reshape(p1 - p0, -1)
        if with_main:
            x = torch.randn((p1 - p0) * PAGE, ATT_DIM, generator=g, device=device)
            main_kv[p0 * PAGE:p1 * PAGE] = fp4_encode_records(x)
    n_entries = torch.tensor(entries, dtype=torch.int32, device=device)
    pc = PagedCache(index_k, main_kv, page_table, n_entries, list(entries))
    pc.planted = planted
    return pc


# ---------------------------------------------------------------------------
# per-layer query-side inputs
# ---------------------------------------------------------------------------

@dataclass
class IndexerQuery:
    q_fp8: torch.Tensor     # uint8 [T,32,128]
    q_scale: torch.Tensor   # float32 [T,32]
    w: torch.Tensor         # float32 [T,32]
    q_float: torch.Tensor   # float32 [T,32,128] (pre-quantisation, for planting only)


def make_indexer_query(T: int, seed: int, device="cpu") -> IndexerQuery:
    """q ~ N(0,1) -> e4m3 with one fp32 scale per head; w ~ N(0,1)/sqrt(32)."""
    g = _gen(seed, device)
    q = torch.randn(T, IDX_HEADS, IDX_DIM, generator=g, device=device)
    codes, scale = fp8_encode(q)
    w = torch.randn(T, IDX_HEADS, generator=g, device=device) / math.sqrt(IDX_HEADS)
    return IndexerQuery(codes.contiguous(), scale.contiguous(), w.contiguous(), q)


@dataclass
class AttnLayer:
    q: torch.Tensor          # bf16 [T,64,512]
    swa_kv: torch.Tensor     # uint8 [n_swa_slots, 528]
    swa_slot: torch.Tensor   # int32 [T,128], -1 pad
    sink: torch.Tensor       # float32 [64]


def make_attn_layer(T: int, seed: int, device="cpu", swa_positions: list | None = None,
                    n_swa_records: int | None = None) -> AttnLayer:
    """Attention inputs of one layer: q bf16 ~ N(0,1), sink ~ N(0,1), and an SWA
    cache of FP8 records ~ N(0,1).

    Decode (swa_positions None): row t owns the ring slots t*128 .. t*128+127.
    Prefill: swa_positions[t] = (first, count) gives the window's first record
    index and length; the layer's SWA cache holds n_swa_records records.
    """
    g = _gen(seed, device)
    q = torch.randn(T, ATT_HEADS, ATT_DIM, generator=g, device=device).to(torch.bfloat16)
    sink = torch.randn(ATT_HEADS, generator=g, device=device)
    if swa_positions is None:
        n_rec = T * SWA_WINDOW
        slot = (torch.arange(T, device=device)[:, None] * SWA_WINDOW
                + torch.randperm(SWA_WINDOW, generator=g, device=device)[None, :]).to(torch.int32)
    else:
        n_rec = n_swa_records
        slot = torch.full((T, SWA_WINDOW), -1, dtype=torch.int32, device=device)
        for t, (first, cnt) in enumerate(swa_positions):
            slot[t, :cnt] = torch.arange(first, first + cnt, device=device, dtype=torch.int32)
    x = torch.randn(n_rec, ATT_DIM, generator=g, device=device)
    swa = swa_encode_records(x)
    return AttnLayer(q.contiguous(), swa, slot.contiguous(), sink)


def make_pool(entries: list[int], seed: int, device="cpu", n_pool=POOL_BLOCKS) -> torch.Tensor:
    """A given candidate pool per sequence: n_pool-1 distinct blocks drawn
    uniformly from all but the newest block, plus the newest block; ascending,
    -1 padded when the sequence has fewer blocks."""
    g = _gen(seed, device)
    out = torch.full((len(entries), n_pool), -1, dtype=torch.int32, device=device)
    for b, e in enumerate(entries):
        nblk = math.ceil(e / POOL_BLOCK)
        if nblk <= n_pool:
            out[b, :nblk] = torch.arange(nblk, device=device, dtype=torch.int32)
            continue
        pick = torch.randperm(nblk - 1, generator=g, device=device)[:n_pool - 1]
        allb = torch.cat([pick, torch.tensor([nblk - 1], device=device)])
        out[b] = torch.sort(allb).values.to(torch.int32)
    return out


def make_compress_inputs(n_tokens: int, seed: int, device="cpu"):
    """C, Z ~ N(0,1) in bf16 [n_tokens,512]; gamma = 1 + 0.1 N(0,1)."""
    g = _gen(seed, device)
    C = torch.randn(n_tokens, ATT_DIM, generator=g, device=device).to(torch.bfloat16)
    Z = torch.randn(n_tokens, ATT_DIM, generator=g, device=device).to(torch.bfloat16)
    gamma = 1.0 + 0.1 * torch.randn(ATT_DIM, generator=g, device=device)
    return C.contiguous(), Z.contiguous(), gamma.contiguous()


def make_index_projection(seed: int, device="cpu"):
    """W^IK [512,128] bf16 ~ N(0,1)/sqrt(512) (a random initialisation: no
    trained weights) and the k_norm weight k_gamma = 1 + 0.1 N(0,1)."""
    g = _gen(seed, device)
    w = (torch.randn(ATT_DIM, IDX_DIM, generator=g, device=device) / math.sqrt(ATT_DIM)).to(torch.bfloat16)
    k_gamma = 1.0 + 0.1 * torch.randn(IDX_DIM, generator=g, device=device)
    return w.contiguous(), k_gamma.contiguous()


HIDDEN = 7168   # model width of the hidden states (the DSA page's figure; no V4.1 width is given)


def make_hidden_projection(n_tokens: int, seed: int, device="cpu", hidden: int = HIDDEN):
    """Hidden states H [n_tokens,hidden] bf16 ~ N(0,1) and W^KV [hidden,512]
    bf16 ~ N(0,1)/sqrt(hidden) (a random initialisation: no trained weights)."""
    g = _gen(seed, device)
    H = torch.randn(n_tokens, hidden, generator=g, device=device).to(torch.bfloat16)
    w = (torch.randn(hidden, ATT_DIM, generator=g, device=device) / math.sqrt(hidden)).to(torch.bfloat16)
    return H.contiguous(), w.contiguous()


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

DECODE_LAYOUT_38 = (
    # (layer, role, group source); 0-based layer ids 2..39
    [(l, "full" if l in (2, 8, 14) else "reuse", 2 + 6 * ((l - 2) // 6)) for l in range(2, 20)]
    + [(l, "full" if l == 20 else ("reindex" if l in (24, 28, 32, 36) else "reuse"), 20 + 4 * ((l - 20) // 4))
       for l in range(20, 40)]
)


def config_lengths(cfg: int, seed: int = None) -> list[int]:
    """Context lengths (tokens) of the sequences of a workload."""
    if cfg == 0:
        return [4096]
    if cfg == 1:
        g = _gen(1000 + (seed or 1), "cpu")
        return [int(x) for x in torch.randint(65536, 131072 + 1, (32,), generator=g)]
    if cfg == 2:
        return [1 << 20] * 16
    if cfg == 4:
        return [32768, 262144, 1 << 20, 1 << 20] * 2
    raise ValueError(cfg)
