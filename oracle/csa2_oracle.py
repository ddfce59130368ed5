"""Plain CPU oracle for the CSA2 global-attention step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the test-suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.  It shares no code,
table or constant generator with the CUDA library; the two meet only at the
byte images of their inputs.

Every function is the plain definition of one step, evaluated in float64 on
the dequantised bytes that the GPU path also reads.  Sources (web pages on
DeepSeek-V4.1 CSA2 / V3.2 DSA):

* CSA2 page  -- "CSA2 = 会跨层复用的 CSA + 两级稀疏检索" (zdszero.github.io/csa2.html)
* V4.1 Q&A page -- "DeepSeek-V4.1 模型结构（2）" (xhh.club)
* V4.1-Flash report reading -- "把 KV Cache 压缩推到极限" (10100.com)
* DSA page   -- "DSA（DeepSeek Sparse Attention）" (zdszero.github.io/dsa.html)

Where the pages leave a step open the reading taken is stated at the
function.  Every function here is pinned by tests in ``tests/test_oracle*.py``
against hand-computed values, closed forms, library routines or brute force.
"""
from __future__ import annotations

import math

import numpy as np

# Fixed sizes of the method (CSA2 page, "一层 CSA2 的 attention 具体怎么算":
# 32 indexer heads x 128 dims, top-512; 64 attention heads x 512-dim K=V).
IDX_HEADS = 32
IDX_DIM = 128
ATT_HEADS = 64
ATT_DIM = 512
ROPE_DIMS = 64
PAGE = 64                      # entries per page (DSA page, "KV pool")
INDEX_PAGE_BYTES = PAGE * (IDX_DIM + 4)   # 64 x 128 B FP8 keys, then 64 x 4 B fp32 scales
INDEX_FP4_PAGE_BYTES = PAGE * (IDX_DIM // 2 + 4)   # 64 x 64 B FP4 keys, then 64 x 4 ue8m0 scales
MAIN_RECORD_BYTES = 288        # 256 B e2m1 codes + 16 B ue8m0 scales + 16 B pad
SWA_RECORD_BYTES = 528         # 512 B e4m3 codes + 4 x fp32 scales (one per 128 channels)
POOL_BLOCK = 8                 # candidate-pool block size (CSA2 page, "Hierarchical Sparse Indexer")


# ---------------------------------------------------------------------------
# Storage formats
# ---------------------------------------------------------------------------

def fp8_e4m3_table() -> np.ndarray:
    """Value of each of the 256 e4m3 codes.

    OCP 8-bit floating point: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
    bits, subnormals at exponent 0, no infinities, S.1111.111 is NaN.  The
    largest finite magnitude is 448 (the V4.1-Flash report reading, section 六,
    quotes 448 as the e4m3 maximum).
    """
    t = np.empty(256, dtype=np.float64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            t[c] = np.nan
        elif e == 0:
            t[c] = sign * (m / 8.0) * 2.0 ** (1 - 7)
        else:
            t[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return t


def fp4_e2m1_table() -> np.ndarray:
    """Value of each of the 16 e2m1 codes (OCP MX: 1 sign, 2 exponent bits with
    bias 1, 1 mantissa bit; largest magnitude 6, as the V4.1-Flash report
    reading's bound 448 x 6 = 2688 uses)."""
    t = np.empty(16, dtype=np.float64)
    for c in range(16):
        sign = -1.0 if c & 0x8 else 1.0
        e = (c >> 1) & 0x3
        m = c & 0x1
        if e == 0:
            t[c] = sign * (m * 0.5)
        else:
            t[c] = sign * (1.0 + m * 0.5) * 2.0 ** (e - 1)
    return t


FP8 = fp8_e4m3_table()
FP4 = fp4_e2m1_table()


def ue8m0(u) -> np.ndarray:
    """Power-of-two scale 2^(u-127) of a ue8m0 byte (255 is NaN)."""
    u = np.asarray(u, dtype=np.int64)
    v = np.ldexp(1.0, u - 127)
    return np.where(u == 255, np.nan, v)


def index_k_entries(cache: np.ndarray, page_table_row: np.ndarray, n: int) -> np.ndarray:
    """Dequantised index keys [n,128] of logical positions 0..n-1 of one sequence.

    Page layout (DSA page, "KV pool", IndexKeyCache): a page holds 64 keys; its
    first 64 x 128 bytes are the e4m3 codes of the keys in order, then
    64 x 4 bytes hold one fp32 scale per key.  A logical position p lives in
    physical page page_table_row[p // 64], row p % 64.
    """
    cache = np.asarray(cache, dtype=np.uint8).reshape(-1, INDEX_PAGE_BYTES)
    pos = np.arange(n)
    page = np.asarray(page_table_row, dtype=np.int64)[pos // PAGE]
    off = pos % PAGE
    codes = cache[page[:, None], off[:, None] * IDX_DIM + np.arange(IDX_DIM)[None, :]]
    sbytes = cache[page[:, None], PAGE * IDX_DIM + off[:, None] * 4 + np.arange(4)[None, :]]
    scale = np.ascontiguousarray(sbytes).view(np.float32).reshape(n).astype(np.float64)
    return FP8[codes] * scale[:, None]


def index_k_at(cache: np.ndarray, page_table_row: np.ndarray, positions: np.ndarray) -> np.ndarray:
    """Dequantised index keys [len(positions),128] at the given logical positions
    of one sequence (the page layout of ``index_k_entries``, for a subset)."""
    cache = np.asarray(cache, dtype=np.uint8).reshape(-1, INDEX_PAGE_BYTES)
    pos = np.asarray(positions, dtype=np.int64)
    page = np.asarray(page_table_row, dtype=np.int64)[pos // PAGE]
    off = pos % PAGE
    codes = cache[page[:, None], off[:, None] * IDX_DIM + np.arange(IDX_DIM)[None, :]]
    sbytes = cache[page[:, None], PAGE * IDX_DIM + off[:, None] * 4 + np.arange(4)[None, :]]
    scale = np.ascontiguousarray(sbytes).view(np.float32).reshape(len(pos)).astype(np.float64)
    return FP8[codes] * scale[:, None]


def index_k_fp4_at(cache: np.ndarray, page_table_row: np.ndarray, positions: np.ndarray) -> np.ndarray:
    """Dequantised FP4 index keys [len(positions),128] at the given logical
    positions of one sequence.

    The CSA2 page and the V4.1 Q&A page store the index K in FP4 (68 B per
    entry by the per-token byte count of the report reading: 890 B = 2.5 x
    (288 + 68)).  Reading taken: 128 e2m1 codes in 64 bytes (element 2i in the
    low nibble of byte i) and 4 ue8m0 scales, one per 32 dims (the MX block
    format of the main-KV records).  A page holds 64 keys: first their 64 x 64
    code bytes in order, then their 64 x 4 scale bytes.
    """
    cache = np.asarray(cache, dtype=np.uint8).reshape(-1, INDEX_FP4_PAGE_BYTES)
    pos = np.asarray(positions, dtype=np.int64)
    page = np.asarray(page_table_row, dtype=np.int64)[pos // PAGE]
    off = pos % PAGE
    data = cache[page[:, None], off[:, None] * (IDX_DIM // 2) + np.arange(IDX_DIM // 2)[None, :]]
    codes = np.empty((len(pos), IDX_DIM), dtype=np.int64)
    codes[:, 0::2] = data & 0xF
    codes[:, 1::2] = data >> 4
    u = cache[page[:, None], PAGE * (IDX_DIM // 2) + off[:, None] * 4 + np.arange(4)[None, :]]
    return FP4[codes] * np.repeat(ue8m0(u), 32, axis=1)


def index_k_fp4_entries(cache: np.ndarray, page_table_row: np.ndarray, n: int) -> np.ndarray:
    """Dequantised FP4 index keys [n,128] of logical positions 0..n-1."""
    return index_k_fp4_at(cache, page_table_row, np.arange(n))


def main_kv_records(cache: np.ndarray, slots: np.ndarray) -> np.ndarray:
    """Dequantised main-KV vectors [len(slots),512] of the given physical slots.

    Record (CSA2 page, "attention 计算的落点", KVLayout.V41_FP4 = 288 B): bytes
    0..255 hold 512 e2m1 codes, element 2i in the low nibble of byte i and
    element 2i+1 in the high nibble; bytes 256..271 hold 16 ue8m0 scales, one
    per 32 consecutive elements; bytes 272..287 are padding.
    """
    cache = np.asarray(cache, dtype=np.uint8).reshape(-1, MAIN_RECORD_BYTES)
    rec = cache[np.asarray(slots, dtype=np.int64)]
    data = rec[:, :256]
    codes = np.empty((len(rec), ATT_DIM), dtype=np.int64)
    codes[:, 0::2] = data & 0xF
    codes[:, 1::2] = data >> 4
    scale = ue8m0(rec[:, 256:272])                       # [n,16]
    return FP4[codes] * np.repeat(scale, 32, axis=1)


def swa_records(cache: np.ndarray, slots: np.ndarray) -> np.ndarray:
    """Dequantised SWA vectors [len(slots),512].

    Record (CSA2 page, KVLayout.V41 = 528 B FP8): 512 e4m3 codes, then four
    fp32 scales, scale j covering channels 128j..128j+127.
    """
    cache = np.asarray(cache, dtype=np.uint8).reshape(-1, SWA_RECORD_BYTES)
    rec = cache[np.asarray(slots, dtype=np.int64)]
    scale = np.ascontiguousarray(rec[:, 512:528]).view(np.float32).astype(np.float64)  # [n,4]
    return FP8[rec[:, :512]] * np.repeat(scale, 128, axis=1)


# ---------------------------------------------------------------------------
# Lightning-Indexer score
# ---------------------------------------------------------------------------

def index_score_values(q: np.ndarray, w: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """I[s] = sum_h w[h] * ReLU(q[h] . k[s]) for dequantised q [H,d] and keys [n,d].

    CSA2 page, "一层 CSA2 的 attention 具体怎么算" item 4; DSA page, "打分公式".
    No 1/sqrt(H) or 1/sqrt(d) factor is added (the CSA2 formula has none).
    """
    dots = np.asarray(keys, dtype=np.float64) @ np.asarray(q, dtype=np.float64).T   # [n,H]
    return np.maximum(dots, 0.0) @ np.asarray(w, dtype=np.float64)


def dequant_q(q8: np.ndarray, q_scale: np.ndarray) -> np.ndarray:
    """Indexer query [H,128]: e4m3 codes times one fp32 scale per head."""
    return FP8[np.asarray(q8, dtype=np.int64)] * np.asarray(q_scale, dtype=np.float64)[:, None]


def index_scores_row(q8, q_scale, w, cache, page_table_row, n_visible, fp4=False) -> np.ndarray:
    """Scores of one query row over its n_visible entries (Full layer); fp4
    selects the FP4 index-K page format."""
    keys = (index_k_fp4_entries if fp4 else index_k_entries)(cache, page_table_row, n_visible)
    return index_score_values(dequant_q(q8, q_scale), w, keys)


def visible_entries(pos: int, ratio_m: int) -> int:
    """Entries visible to the query at token position pos: (pos+1)//m.

    CSA2 page, "候选池不减少存储": an m=2 entry is written only once both of
    its tokens exist, so the visible count is (pos + 1) // ratio.
    """
    return (int(pos) + 1) // int(ratio_m)


# ---------------------------------------------------------------------------
# Top-k, slot translation, candidate pool
# ---------------------------------------------------------------------------

def topk_positions(scores: np.ndarray, k: int) -> np.ndarray:
    """Positions of the k best finite scores in ascending position order, -1 filled.

    DSA page, "Top-k：选的是 token，不是 block": token-level selection, -1 in
    empty slots.  Ties (left open by the pages) go to the lower position.  The
    pages leave the order of the reported positions open; they are reported in
    ascending position order.  -inf marks an excluded position and is never
    selected.
    """
    s = np.asarray(scores)
    cand = np.flatnonzero(np.isfinite(s))
    order = np.lexsort((cand, -s[cand]))
    sel = np.sort(cand[order[:k]])
    out = np.full(k, -1, dtype=np.int64)
    out[: len(sel)] = sel
    return out


def slots_of(positions: np.ndarray, page_table_row: np.ndarray) -> np.ndarray:
    """Physical slot of each logical position: table[p // 64] * 64 + p % 64, -1 kept.

    DSA page, "实现 / logits 与 top-k" (compact real_page_table, 64 slots/page).
    """
    p = np.asarray(positions, dtype=np.int64)
    pt = np.asarray(page_table_row, dtype=np.int64)
    out = np.full(p.shape, -1, dtype=np.int64)
    ok = p >= 0
    out[ok] = pt[p[ok] // PAGE] * PAGE + p[ok] % PAGE
    return out


def block_maxima(scores: np.ndarray, n_visible: int, block: int = POOL_BLOCK) -> np.ndarray:
    """Per-block maximum over the visible positions of each block of 8.

    CSA2 page, "分块不是压缩": the block score is the largest index score in
    the block (max, not mean); the last block may be partial and then uses only
    its visible positions.
    """
    n = int(n_visible)
    nblk = -(-n // block)
    out = np.empty(nblk, dtype=np.float64)
    s = np.asarray(scores, dtype=np.float64)
    for j in range(nblk):
        out[j] = s[j * block: min(j * block + block, n)].max()
    return out


def candidate_pool(bmax: np.ndarray, n_pool: int = 2048) -> np.ndarray:
    """Candidate blocks of one query: ascending block ids, -1 padded to n_pool.

    CSA2 page, "Hierarchical Sparse Indexer" and "池里的 16384 个位置是哪些";
    SGLang notes in "attention 计算的落点": keep the n_pool blocks with the
    highest block maxima and always keep the block of the newest position.
    Readings: the forced block takes one of the n_pool places; ties go to the
    lower block id; when there are at most n_pool blocks, all are kept.
    """
    b = np.asarray(bmax, dtype=np.float64).copy()
    nblk = len(b)
    out = np.full(n_pool, -1, dtype=np.int64)
    if nblk == 0:
        return out
    b[nblk - 1] = np.inf
    ids = np.arange(nblk)
    order = np.lexsort((ids, -b))
    sel = np.sort(ids[order[:n_pool]])
    out[: len(sel)] = sel
    return out


def pool_positions(pool_blocks: np.ndarray, n_visible: int, block: int = POOL_BLOCK) -> np.ndarray:
    """Positions covered by a pool, candidate i -> 8*pool[i//8] + i%8; -1 where the
    block is padding or the position is not visible."""
    pb = np.asarray(pool_blocks, dtype=np.int64)
    pos = (pb[:, None] * block + np.arange(block)[None, :]).reshape(-1)
    valid = (np.repeat(pb, block) >= 0) & (pos < n_visible)
    return np.where(valid, pos, -1)


def reindex_scores(q8, q_scale, w, cache, page_table_row, n_visible, pool_blocks, fp4=False) -> np.ndarray:
    """Scores over the candidate list of a Reindex layer: [8*len(pool)], -inf for
    padding and invisible positions.

    CSA2 page, "Hierarchical Sparse Indexer" item 2 and "attention 计算的落点":
    a Reindex layer scores only positions inside the pool; every other
    position counts as -inf.
    """
    pos = pool_positions(pool_blocks, n_visible)
    out = np.full(len(pos), -np.inf)
    ok = pos >= 0
    if ok.any():
        keys = (index_k_fp4_at if fp4 else index_k_at)(cache, page_table_row, pos[ok])
        out[ok] = index_score_values(dequant_q(q8, q_scale), w, keys)
    return out


def reindex_topk(q8, q_scale, w, cache, page_table_row, n_visible, pool_blocks, k=512, fp4=False):
    """Top-k positions of a Reindex layer: full-length score row with -inf outside
    the pool, then the ordinary top-k."""
    full = np.full(int(n_visible), -np.inf)
    pos = pool_positions(pool_blocks, n_visible)
    sc = reindex_scores(q8, q_scale, w, cache, page_table_row, n_visible, pool_blocks, fp4=fp4)
    ok = pos >= 0
    full[pos[ok]] = sc[ok]
    return topk_positions(full, k)


# ---------------------------------------------------------------------------
# Sparse MQA attention with SWA and sink
# ---------------------------------------------------------------------------

def sparse_attention(q: np.ndarray, kv: np.ndarray, sink: np.ndarray, scale: float):
    """o[i] = softmax([q_i K^T * scale || s_i]) . [V || 0], K = V = kv.

    CSA2 page, "一层 CSA2 的 attention 具体怎么算" (the attention equation):
    one joint softmax over the SWA keys and the selected main entries, the
    sink s_i entering only the denominator; MQA with K and V the same vector.
    The sink logit is not scaled.  Returns (o [H,512], lse [H]) with lse the
    natural log of the full denominator (sink included).
    """
    q = np.asarray(q, dtype=np.float64)
    kv = np.asarray(kv, dtype=np.float64)
    sink = np.asarray(sink, dtype=np.float64)
    logits = (q @ kv.T) * scale                             # [H,n]
    m = np.maximum(logits.max(axis=1) if kv.shape[0] else -np.inf, sink)
    p = np.exp(logits - m[:, None])
    ps = np.exp(sink - m)
    denom = p.sum(axis=1) + ps
    o = (p @ kv) / denom[:, None]
    return o, m + np.log(denom)


def swa_replay_visible(q_pos: int, seg_start: int, n_swa: int) -> np.ndarray:
    """Which keys of a query row's SWA window stay visible under Decoder SWA
    Bounded Replay (CSA2 page, "Decoder SWA Bounded Replay"): the query at
    position i of a replayed segment that starts at s sees the SWA keys at
    positions [max(s, i - W + 1), i] only.  Readings: the window W is the
    row's number of SWA slots, and slot j of the window holds position
    i - W + 1 + j (oldest first, the query's own key last).  Returns bool [W]."""
    i, W = int(q_pos), int(n_swa)
    key_pos = i - W + 1 + np.arange(W)
    lo = max(int(seg_start), i - W + 1)
    return (key_pos >= lo) & (key_pos <= i)


def output_inverse_rope(o: np.ndarray, q_pos: int, theta: float) -> np.ndarray:
    """The attention output of a query at position q_pos with its RoPE taken
    back off the last 64 dims, before the grouped output projection (CSA2 page,
    attention section: the output is un-RoPE'd first).  The inverse of the
    rotation by angle q_pos * f is the rotation by -q_pos * f, i.e. the
    same interleaved RoPE at position -q_pos."""
    o = np.asarray(o, dtype=np.float64)
    return rope_interleaved(o, np.full(o.shape[0], -float(q_pos)), theta)


def attention_row(q_bf16_values, main_cache, topk_slot_row, swa_cache, swa_slot_row, sink, scale,
                  q_pos=None, swa_seg_start=None, inv_rope_theta=None):
    """Attention of one query row from the caches: gathers the valid SWA and main
    slots (slot -1 is empty) and evaluates ``sparse_attention``.  With
    ``swa_seg_start`` the SWA window is cut to the replayed segment
    (``swa_replay_visible``); with ``inv_rope_theta`` the output is
    un-RoPE'd at ``q_pos`` (``output_inverse_rope``)."""
    ts = np.asarray(topk_slot_row, dtype=np.int64)
    ss = np.asarray(swa_slot_row, dtype=np.int64)
    if swa_seg_start is not None:
        ss = np.where(swa_replay_visible(q_pos, swa_seg_start, ss.shape[0]), ss, -1)
    parts = []
    if (ss >= 0).any():
        parts.append(swa_records(swa_cache, ss[ss >= 0]))
    if (ts >= 0).any():
        parts.append(main_kv_records(main_cache, ts[ts >= 0]))
    kv = np.concatenate(parts, axis=0) if parts else np.zeros((0, ATT_DIM))
    o, lse = sparse_attention(q_bf16_values, kv, sink, scale)
    if inv_rope_theta is not None:
        o = output_inverse_rope(o, q_pos, inv_rope_theta)
    return o, lse


# ---------------------------------------------------------------------------
# Main-KV entry build (m = 1 or 2)
# ---------------------------------------------------------------------------

def kv_project(hidden: np.ndarray, w_kv: np.ndarray) -> np.ndarray:
    """Per-token inputs of the entry build from the hidden states: C = H W.

    CSA2 page, "一层 CSA2 的 attention 具体怎么算" item 3: with m = 1 the
    main-KV entry is one linear projection of the token (weight identically 1
    in the compression); CSA2 page and report reading, CED: the decoder layers'
    C_l = H_{L/2} W^KV_l, the encoder layers' C and Z from their own hidden
    state.  H is [n_tokens, hidden], W is [hidden, 512] (row = input dim).
    Readings: the pages give no V4.1 hidden width; the DSA page's V3.2 figure,
    7168, is taken; the weights are random (no trained weights).
    """
    return np.asarray(hidden, dtype=np.float64) @ np.asarray(w_kv, dtype=np.float64)


def compress_latent(C: np.ndarray, Z, ratio_m: int, gamma: np.ndarray, eps: float,
                    positions: np.ndarray, rope_theta: float, apply_rope: bool = True) -> np.ndarray:
    """Latent [n_entries,512] of the main-KV entries, before quantisation.

    CSA2 page, "一层 CSA2 的 attention 具体怎么算" item 3, and the V4.1 Q&A page:
    m=1 is the projection itself (weight identically 1); m=2 is a per-channel
    softmax-weighted sum of two adjacent, non-overlapping tokens, no APE.  The
    result goes through RMSNorm, then RoPE on the last 64 dims.
    Readings: RMSNorm y = x / sqrt(mean(x^2) + eps) * gamma; RoPE rotates
    interleaved pairs (448+2i, 449+2i), i < 32, by angle pos * theta^(-2i/64).
    """
    C = np.asarray(C, dtype=np.float64)
    m = int(ratio_m)
    n = C.shape[0] // m
    Cg = C[: n * m].reshape(n, m, ATT_DIM)
    if m == 1:
        x = Cg[:, 0, :]
    else:
        Zg = np.asarray(Z, dtype=np.float64)[: n * m].reshape(n, m, ATT_DIM)
        zmax = Zg.max(axis=1, keepdims=True)
        e = np.exp(Zg - zmax)
        a = e / e.sum(axis=1, keepdims=True)
        x = (a * Cg).sum(axis=1)
    y = x / np.sqrt((x * x).mean(axis=1, keepdims=True) + eps) * np.asarray(gamma, dtype=np.float64)[None, :]
    if apply_rope:
        y = rope_interleaved(y, positions, rope_theta)
    return y


def rope_interleaved(y: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """RoPE on the last 64 dims of y [n,d], interleaved pairs (CSA2 page: RoPE
    only on the last 64 dims; pairing and base are readings)."""
    y = np.array(y, dtype=np.float64, copy=True)
    pos = np.asarray(positions, dtype=np.float64)
    half = ROPE_DIMS // 2
    inv = theta ** (-2.0 * np.arange(half) / ROPE_DIMS)
    ang = pos[:, None] * inv[None, :]
    c, s = np.cos(ang), np.sin(ang)
    base = y.shape[1] - ROPE_DIMS
    x0 = y[:, base + 0::2].copy()
    x1 = y[:, base + 1::2].copy()
    y[:, base + 0::2] = x0 * c - x1 * s
    y[:, base + 1::2] = x0 * s + x1 * c
    return y


def fp4_scale_exponent(amax) -> np.ndarray:
    """ue8m0 byte of 32-element groups: u = k + 127 with k the smallest integer
    such that 6 * 2^k >= amax (u = 127 when amax is 0), clamped to [0, 254].
    Reading of the V4.1-Flash report (section 六: e2m1 elements with a
    power-of-two block scale and no global scale)."""
    a = np.asarray(amax, dtype=np.float64)
    safe = np.where(a > 0, a, 6.0)
    k = np.ceil(np.log2(safe / 6.0))
    for _ in range(2):                                   # exact fix-up of log2 rounding
        k = np.where(6.0 * np.exp2(k) < safe, k + 1, k)
        k = np.where(6.0 * np.exp2(k - 1) >= safe, k - 1, k)
    u = np.where(a > 0, k + 127, 127)
    return np.clip(u, 0, 254).astype(np.int64)


_FP4_MAG = FP4[:8]


def fp4_codes(v) -> np.ndarray:
    """e2m1 codes of values already divided by their group scale: nearest
    magnitude, ties to the even code, saturating at 6; sign bit set for v < 0."""
    v = np.asarray(v, dtype=np.float64)
    d = np.abs(np.abs(v)[..., None] - _FP4_MAG)          # [..., 8]
    best = np.argmin(d, axis=-1)                          # lower code on ties
    nxt = np.minimum(best + 1, 7)
    dn = np.take_along_axis(d, nxt[..., None], -1)[..., 0]
    db = np.take_along_axis(d, best[..., None], -1)[..., 0]
    best = np.where((best & 1 == 1) & (nxt != best) & (dn == db), nxt, best)
    return best | np.where(v < 0, 8, 0)


def fp4_encode_records(y: np.ndarray) -> np.ndarray:
    """288-byte main-KV records [n,288] of 512-vectors y [n,512] (layout as in
    main_kv_records)."""
    y = np.asarray(y, dtype=np.float64).reshape(-1, ATT_DIM)
    n = y.shape[0]
    g = y.reshape(n, 16, 32)
    u = fp4_scale_exponent(np.abs(g).max(axis=2))        # [n,16]
    codes = fp4_codes(g / np.exp2(u - 127)[..., None]).reshape(n, ATT_DIM)
    rec = np.zeros((n, MAIN_RECORD_BYTES), dtype=np.uint8)
    rec[:, :256] = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    rec[:, 256:272] = u.astype(np.uint8)
    return rec


def compress_records(C, Z, ratio_m, gamma, eps, positions, rope_theta, apply_rope=True):
    """Records [n_entries,288] of the main-KV entries built from C (and Z)."""
    lat = compress_latent(C, Z, ratio_m, gamma, eps, positions, rope_theta, apply_rope)
    return fp4_encode_records(lat), lat


# ---------------------------------------------------------------------------
# Index-key build of a Full layer
# ---------------------------------------------------------------------------

def index_key_latent(y_pre: np.ndarray, w_ik: np.ndarray, k_gamma: np.ndarray, eps: float,
                     positions: np.ndarray, rope_theta: float) -> np.ndarray:
    """Index keys [n,128] before quantisation from the main-KV latents before
    RoPE y_pre [n,512].

    V4.1 Q&A page (indexer K from the main KV): k = RMSNorm(y_pre W^IK) with
    W^IK of 512 x 128, projected from the latent before its RoPE; the last 64
    dims of k then get their own RoPE.  CSA2 page item 3: latent -> wk -> k_norm
    -> RoPE -> quantisation.  Readings: k_norm is RMSNorm with a weight k_gamma
    and the eps of the main latent; the RoPE is the main latent's (interleaved
    pairs, base theta, the entry's position).
    """
    k = np.asarray(y_pre, dtype=np.float64) @ np.asarray(w_ik, dtype=np.float64)
    k = k / np.sqrt((k * k).mean(axis=1, keepdims=True) + eps) * np.asarray(k_gamma, dtype=np.float64)[None, :]
    return rope_interleaved(k, positions, rope_theta)


def fp8_e4m3_codes(v) -> np.ndarray:
    """e4m3 codes of v: the nearest finite e4m3 value, ties to the even code,
    saturating at +-448."""
    v = np.asarray(v, dtype=np.float64)
    mags = FP8[:0x7F]                                     # 0 .. 448 at codes 0 .. 0x7E
    a = np.minimum(np.abs(v), 448.0)
    best = np.clip(np.searchsorted(mags, a), 1, 0x7E)     # mags[best-1] < a <= mags[best]
    lo, hi = best - 1, best
    dlo, dhi = a - mags[lo], mags[hi] - a
    code = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(a == 0, 0, code)
    return (code | np.where(v < 0, 0x80, 0)).astype(np.int64)


def index_key_fp8_bytes(k32: np.ndarray):
    """FP8 index-K entry of fp32 keys k32 [n,128]: scale = amax / 448 in fp32 (1
    for an all-zero key), codes = e4m3 of the fp32 quotient k / scale.
    Returns (codes uint8 [n,128], scale float32 [n])."""
    k32 = np.asarray(k32, dtype=np.float32)
    amax = np.abs(k32).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = (k32 / scale[:, None]).astype(np.float32)
    return fp8_e4m3_codes(q).astype(np.uint8), scale


def index_key_fp4_bytes(k: np.ndarray):
    """FP4 index-K entry of keys k [n,128]: e2m1 codes (element 2i in the low
    nibble of byte i) and one ue8m0 scale per 32 dims, as the main-KV records.
    Returns (code bytes uint8 [n,64], scales uint8 [n,4])."""
    k = np.asarray(k, dtype=np.float64)
    n = k.shape[0]
    g = k.reshape(n, 4, 32)
    u = fp4_scale_exponent(np.abs(g).max(axis=2))
    codes = fp4_codes(g / np.exp2(u - 127)[..., None]).reshape(n, IDX_DIM)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8), u.astype(np.uint8)
