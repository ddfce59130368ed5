/*
 * csa2.h -- C ABI of the CSA2 global-attention step on one GB300 (sm_103a).
 *
 * The step, as the web pages on DeepSeek-V4.1 CSA2 describe it (CSA2 page,
 * zdszero.github.io/csa2.html, "一层 CSA2 的 attention 具体怎么算" and
 * "Hierarchical Sparse Indexer"; DSA page, zdszero.github.io/dsa.html,
 * "Lightning Indexer"):
 *
 *   1. Lightning-Indexer score  I[t,s] = sum_h w[t,h] * ReLU(q[t,h] . k[s])
 *      (32 heads x 128 dims, FP8 index-K cache)              -> csa2_index_score
 *   2. top-512 positions -> physical slots, and (Full layer of the decoder) a
 *      candidate pool of the 2048 blocks of 8 with the highest block maxima
 *                                                           -> csa2_topk_with_candidates
 *   3. Reindex: score only the pool, everything else -inf, top-512
 *                                                           -> csa2_reindex
 *   4. MQA sparse attention: 64 heads x 512-dim K=V, one joint softmax over
 *      128 SWA keys + <= 512 main-KV entries + a per-head sink in the
 *      denominator                                          -> csa2_sparse_attn
 *   5. main-KV entry build: m=2 per-channel softmax of two tokens (m=1:
 *      weight 1), RMSNorm, RoPE on the last 64 dims, FP4  -> csa2_compress_m2
 *
 * Conventions shared by every call
 *   - All pointers in the argument structs are DEVICE pointers to
 *     caller-owned memory (except the struct itself, which lives on the host
 *     and is read before the call returns).  The library never allocates or
 *     frees device memory; scratch comes from the caller's workspace, sized by
 *     csa2_workspace_size().
 *   - Every call is asynchronous on the given stream (a cudaStream_t passed
 *     as void*; NULL = legacy default stream) and never synchronises the host.
 *   - Arguments are validated on the host before any launch; an invalid
 *     argument returns a status code and launches nothing.  A failed launch
 *     returns CSA2_ERR_CUDA.
 *   - Kernels never trap.  An out-of-range page id or slot met on the device
 *     is skipped and recorded in a device-side error word that
 *     csa2_check_device_error() reads (it synchronises the stream).
 *   - Integer layouts are int32, row-major; "ld" arguments are row strides in
 *     elements.
 *
 * Storage formats (the same bytes the oracle decodes)
 *   index-K page : 8448 B = 64 keys x 128 e4m3 codes, then 64 fp32 scales
 *                  (DSA page, "KV pool").  Key s of a sequence is in physical
 *                  page page_table[b][s / 64], row s % 64.
 *   FP4 index-K page: 4352 B = 64 keys x 64 B of 128 e2m1 codes (element 2i
 *                  in the low nibble of byte i), then 64 x 4 ue8m0 scales (one
 *                  per 32 dims); 68 B per entry (CSA2 page and V4.1 Q&A page:
 *                  the index K is FP4; 890 B per token = 2.5 x (288 + 68)).
 *   main-KV record: 288 B at slot*288 = 256 B of 512 e2m1 codes (element 2i
 *                  in the low nibble of byte i), 16 ue8m0 scales (one per 32
 *                  elements, value 2^(u-127)), 16 B padding (CSA2 page,
 *                  "attention 计算的落点": 288 B per entry).
 *   SWA record   : 528 B at slot*528 = 512 e4m3 codes, then 4 fp32 scales, one
 *                  per 128 channels (CSA2 page: 528 B FP8 SWA entry).
 *   slot         : page_table[b][p / 64] * 64 + p % 64 (DSA page, "logits 与
 *                  top-k"); -1 marks an empty slot.
 */
#ifndef CSA2_H_
#define CSA2_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CSA2_API __attribute__((visibility("default")))
#else
#define CSA2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CSA2_OK = 0,
  CSA2_ERR_NULL = 1,          /* a required pointer is NULL */
  CSA2_ERR_SHAPE = 2,         /* a size or count is out of range */
  CSA2_ERR_ALIGN = 3,         /* a pointer or stride is not 16-byte aligned */
  CSA2_ERR_UNSUPPORTED = 4,   /* a valid but unsupported combination */
  CSA2_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
  CSA2_ERR_DEVICE_BOUNDS = 6, /* a kernel met an out-of-range page id or slot */
  CSA2_ERR_WORKSPACE = 7,     /* workspace missing or smaller than required */
  CSA2_ERR_DEVICE_TIMEOUT = 8 /* a kernel gave up a bounded wait (internal fault) */
} csa2_status;

/* Fixed sizes of the method. */
enum {
  CSA2_IDX_HEADS = 32, CSA2_IDX_DIM = 128,
  CSA2_ATT_HEADS = 64, CSA2_ATT_DIM = 512, CSA2_ROPE_DIMS = 64,
  CSA2_PAGE = 64, CSA2_INDEX_PAGE_BYTES = 8448, CSA2_INDEX_FP4_PAGE_BYTES = 4352,
  CSA2_MAIN_RECORD_BYTES = 288, CSA2_SWA_RECORD_BYTES = 528,
  CSA2_MAX_TOPK = 2048, CSA2_POOL_BLOCK = 8, CSA2_MAX_SWA = 128
};

/* Index-K page formats (the index_k_format field of the scoring calls). */
enum { CSA2_INDEX_FP8 = 0, CSA2_INDEX_FP4 = 1 };

/* Order of the reported top-k positions (the order field of the top-k and
 * Reindex calls).  The pages leave it open; the set is the same either way. */
enum {
  CSA2_ORDER_POSITION = 0, /* ascending position (groups a row's slot reads by page) */
  CSA2_ORDER_SCORE = 1     /* best first: score descending, ties to the lower position,
                              so the first k' < k entries are the row's top-k' */
};

/* Static description of a status code. */
CSA2_API const char* csa2_status_string(int status);
/* Human-readable detail of the last error returned on the calling thread
 * (thread-local; valid until the thread's next call). */
CSA2_API const char* csa2_last_error_detail(void);

/* Which query rows see which entries.  Row t belongs to sequence
 * row_seq[t] (row_seq NULL: sequence t, which needs T == B; an id outside
 * [0, B) makes the row see no entries).  The entries
 * visible to row t are E_t = n_visible[b] in decode (row_pos NULL), or
 * E_t = (row_pos[t] + 1) / ratio_m in prefill, clipped to n_visible[b] when
 * n_visible is given (CSA2 page, "候选池不减少存储": visible = (pos+1)//ratio).
 * At least one of n_visible, row_pos must be given. */
typedef struct {
  int32_t T;                  /* query rows, >= 1 */
  int32_t B;                  /* sequences, >= 1 */
  const int32_t* row_seq;     /* [T] in [0,B) or NULL */
  const int32_t* row_pos;     /* [T] token position or NULL */
  const int32_t* n_visible;   /* [B] visible entries or NULL */
  int32_t ratio_m;            /* 1 or 2 (only used with row_pos) */
} csa2_rows;

/* ---- 1. Lightning-Indexer score (Full layer) --------------------------------
 * scores[t][s] = k_scale[s] * sum_h (w[t,h] * q_scale[t,h]) * ReLU(q8[t,h] . k8[s])
 * which equals sum_h w[t,h] * ReLU(q[t,h] . k[s]) on the dequantised q and k
 * because q_scale, k_scale >= 0 (DSA page, "fp8 与 scale 的吸收").  No
 * 1/sqrt(H) or 1/sqrt(d) factor is applied.
 * Written: scores[t][s] for s < round_up(E_t, 128) clipped to ld_scores
 * (s >= E_t holds -inf); block_max[t][j] = max over the visible positions of
 * block j (8 positions) for j < ceil(E_t / 8), if block_max is not NULL.
 * Alignment: q_fp8, index_k 16 B (32 B for FP4 pages); ld_scores and
 * ld_block_max multiples of 4.
 * Prefill (row_pos given, B == 1, T >= 64, FP8 pages; T <= 16384) runs the
 * query-blocked tensor-core path (8 queries x 32 heads per MMA); everything
 * else the per-row scan (one query's 32 heads per MMA), which takes calls of
 * any T in launches of 2048 rows (hist: T <= 2048).  FP4 index-K pages are
 * scored on the per-row scan at every shape, prefill included (each query then
 * reads the keys anew, from L2 for a prefill chunk):
 * k = sum over its 4 blocks of 2^(u_b-127) * e2m1 codes. */
typedef struct {
  const uint8_t* q_fp8;       /* [T,32,128] e4m3 codes */
  const float* q_scale;       /* [T,32] >= 0 */
  const float* w;             /* [T,32] head weights */
  const uint8_t* index_k;     /* pages of 8448 B (FP8) or 4352 B (FP4) */
  int64_t index_k_pages;      /* number of pages in index_k */
  const int32_t* page_table;  /* [B, pt_stride] logical page -> physical page */
  int32_t pt_stride;
  csa2_rows rows;
  float* scores; int64_t ld_scores;           /* [T, ld_scores] */
  float* block_max; int64_t ld_block_max;     /* optional [T, ld_block_max] */
  /* optional [2, T, 2048] uint32, decode path only (else must be NULL): 2048-bin
   * histograms of the top 11 bits of the order-preserving key of every finite
   * visible score (rows 0..T-1) and of every finite block maximum (rows
   * T..2T-1, the newest block counted as +inf; untouched when block_max is
   * NULL).  The call ADDS into the buffer, which must hold zeros on entry:
   * zero it once when it is allocated; csa2_topk_with_candidates (or its
   * no-allocation variant) given the same buffer reads it and sets it back to
   * zero, so a step that pairs every scan with its top-k call needs no memset
   * between layers.  Passing it on saves the top-k call a pass over the
   * scores. */
  uint32_t* hist;
  int32_t index_k_format;     /* CSA2_INDEX_FP8 (0) or CSA2_INDEX_FP4 */
} csa2_index_score_args;
CSA2_API int csa2_index_score(const csa2_index_score_args* args, void* workspace, size_t ws_bytes, void* stream);

/* ---- 2. top-k with slot translation and the candidate pool ------------------
 * Per row: the k (<= 2048) positions s < E_t with the largest finite scores
 * (ties go to the lower position), in the order given by `order` (ascending
 * position by default), -1 filled when fewer than k are finite (DSA page,
 * "Top-k：选的是 token，不是 block").  topk_slot[t][i] = slot of topk_pos[t][i] (-1 kept).
 * Pool (pool_blocks not NULL; CSA2 page, "Hierarchical Sparse Indexer",
 * "attention 计算的落点" select_candidate_blocks): block scores are
 * block_max[t][0..ceil(E_t/8)); the newest block ceil(E_t/8)-1 is always kept
 * and counts toward pool_n; the other places go to the highest block maxima
 * (ties: lower block id); output ascending block ids, -1 padded; with at most
 * pool_n blocks every block is kept.
 * Workspace: csa2_workspace_size(CSA2_CALL_TOPK, args, &bytes). */
typedef struct {
  const float* scores; int64_t ld_scores;     /* [T, ld_scores] */
  const float* block_max; int64_t ld_block_max; /* [T, ld_block_max], needed for the pool */
  const int32_t* page_table; int32_t pt_stride; /* slot translation; NULL: no slots */
  csa2_rows rows;
  int32_t k;                                   /* 1..2048 */
  int32_t* topk_pos;                           /* [T, ld_topk] */
  int32_t* topk_slot;                          /* [T, ld_topk] or NULL */
  int64_t ld_topk;                             /* >= k */
  int32_t* pool_blocks;                        /* [T, pool_n] or NULL */
  int32_t pool_n;                              /* 1..2048 when pool_blocks is set */
  uint32_t* hist;                              /* optional: the histograms csa2_index_score wrote
                                                  for these scores and block maxima; read, then set
                                                  back to zero (both halves, also without a pool) */
  int32_t order;                               /* CSA2_ORDER_POSITION (0) or CSA2_ORDER_SCORE (1) */
} csa2_topk_args;
CSA2_API int csa2_topk_with_candidates(const csa2_topk_args* args, void* workspace, size_t ws_bytes, void* stream);

/* ---- top-k without workspace or allocation ------------------------------------
 * The pages have no counterpart of this call: it is a deployment convenience.
 * Same arguments, semantics and results as csa2_topk_with_candidates, but no
 * workspace: for callers that cannot provide or allocate device scratch (an
 * operator interface that passes only inputs and outputs, an engine whose
 * allocator cannot serve extra buffers, a path that must not call cudaMalloc).
 * The scratch is a static device array of CSA2_TOPK_NOALLOC_SCRATCH_BYTES that
 * every GPU loading the library holds until exit.  A call needs exactly what
 * csa2_workspace_size(CSA2_CALL_TOPK, args, ...) reports: nothing when
 * L <= 16384, else
 *     V * H + R + round_up(V * c * 4, 256) + V * c * 8192 bytes,
 * with L = ld_scores (the larger of ld_scores and ld_block_max when
 * pool_blocks is set), c = ceil(L / 4096), V = T (2T with a pool: the block
 * maxima are a second row per query), H = 8192 and R = round_up(V * 8, 256)
 * (H = R = 0 when hist is given).
 * That is about 2 B per element of L per row: a 1M-entry row needs 2.1 MB,
 * 4.2 MB with its pool, so the 8 MiB array takes three 1M rows, or one with
 * its pool, or seven 262,144-entry rows with their pools.  Calls needing more
 * return CSA2_ERR_WORKSPACE.  The library allocates nothing during the call.
 * The first call on each device looks up the array's device address, so make
 * it before any stream capture; the address is kept for the life of the
 * process, so do not use this call on a device after cudaDeviceReset.
 * All calls share the array: calls that overlap on the GPU race. */
#define CSA2_TOPK_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
CSA2_API int csa2_topk_with_candidates_noalloc(const csa2_topk_args* args, void* stream);

/* ---- 3. Reindex: pool-only rescoring and top-k ------------------------------
 * Candidate i of row t is position p = 8 * pool_blocks[t][i / 8] + i % 8; it
 * is scored like csa2_index_score when the block id is >= 0 and p < E_t, and
 * is -inf otherwise (CSA2 page, "Hierarchical Sparse Indexer" item 2: a
 * Reindex layer scores only the pool).  Then the top-k of those scores, as in
 * csa2_topk_with_candidates, reported as positions and slots.
 * pool_scores (optional, [T, 8*pool_n]) receives the candidate scores.
 * Workspace: csa2_workspace_size(CSA2_CALL_REINDEX, args, &bytes): the
 * candidate scores, unless pool_scores is given (then none). */
typedef struct {
  const uint8_t* q_fp8; const float* q_scale; const float* w;  /* as in index_score */
  const uint8_t* index_k; int64_t index_k_pages;
  const int32_t* page_table; int32_t pt_stride;
  csa2_rows rows;
  const int32_t* pool_blocks; int32_t pool_n;  /* [T, pool_n], pool_n <= 2048 */
  int32_t k;                                   /* 1..2048 */
  int32_t* topk_pos; int32_t* topk_slot; int64_t ld_topk;
  float* pool_scores;                          /* optional [T, 8*pool_n] */
  int32_t index_k_format;                      /* CSA2_INDEX_FP8 (0) or CSA2_INDEX_FP4 */
  int32_t order;                               /* CSA2_ORDER_POSITION (0) or CSA2_ORDER_SCORE (1) */
} csa2_reindex_args;
CSA2_API int csa2_reindex(const csa2_reindex_args* args, void* workspace, size_t ws_bytes, void* stream);

/* ---- 4. MQA sparse attention with SWA keys and an attention sink -----------
 * For row t and head i (CSA2 page, attention equation):
 *   logit_j = (q[t,i] . kv_j) * softmax_scale,  j over the valid SWA slots
 *             swa_slot[t][0..n_swa) and main slots topk_slot[t][0..k) (-1 skipped)
 *   out[t,i] = sum_j e^(logit_j - M) kv_j / (sum_j e^(logit_j - M) + e^(sink[i] - M))
 * kv_j is the dequantised 512-vector (K = V); the sink is not scaled.
 * lse[t,i] = M + ln(denominator) (natural log, sink included).
 * softmax_scale == 0 selects 1/sqrt(512).  Alignment: q, main_kv, swa_kv, out 16 B.
 * Two kernels: while rows x ceil((n_swa + k) / 80) is at most the SM count
 * (decode layers), each row's keys are split over a cluster of CTAs and merged
 * through L2 in the workspace (csa2_workspace_size); beyond, split-K CTAs walk
 * a row's keys with an online softmax and merge on chip (no workspace). */
typedef struct {
  const uint16_t* q;                           /* [T,64,512] bf16 */
  const uint8_t* main_kv; int64_t main_kv_slots;   /* 288-B records */
  const int32_t* topk_slot; int32_t k; int64_t ld_topk;  /* [T, ld_topk]; k <= 2048 */
  const uint8_t* swa_kv; int64_t swa_slots;        /* 528-B records */
  const int32_t* swa_slot; int32_t n_swa; int64_t ld_swa;  /* [T, ld_swa]; n_swa <= 128 */
  const float* sink;                           /* [64] */
  float softmax_scale;
  int32_t T;
  int32_t out_bf16;                            /* 0: fp32 out, 1: bf16 out */
  void* out;                                   /* [T,64,512] */
  float* lse;                                  /* optional [T,64] */
  /* 1: topk_slot, swa_slot, main_kv and swa_kv were written at least two
   * launches before this call on the stream (a Reuse layer's slots and caches,
   * written by its Full or Reindex layer), so the keys may be gathered before
   * the previous launch completes; q and sink are still read after it.  The two
   * launches before the call must be ordinary launches or kernels that signal
   * their dependents only after their own dependency wait (as every kernel of
   * this library does).  0: everything is read after the previous launch. */
  int32_t kv_ready;
  /* Optional (zero / NULL leaves each off):
   * q_pos [T]: position of each query row in its sequence.
   * out_inv_rope = 1: the output is rotated back by its query's RoPE before it
   *   is stored (CSA2 page, attention section: the output is un-RoPE'd before
   *   the grouped output projection): pair (448+2p, 449+2p) of out[t,i] turns
   *   by -q_pos[t] * rope_theta^(-2p/64), p < 32, the inverse of the rotation
   *   the keys carry.  rope_theta == 0 selects 10000.  lse is not affected.
   * swa_seg_start [T]: SWA bounded replay (CSA2 page, "Decoder SWA Bounded
   *   Replay"): swa_slot[t][j] holds the key at position
   *   q_pos[t] - n_swa + 1 + j, and a key at a position below
   *   swa_seg_start[t] is skipped, so the row at position i attends to the
   *   SWA keys of [max(s, i - n_swa + 1), i] only.
   * Both need q_pos.  q_pos and swa_seg_start are read together with the slots
   * (under kv_ready = 1 they too must be written two launches before). */
  const int32_t* q_pos;
  int32_t out_inv_rope;
  float rope_theta;
  const int32_t* swa_seg_start;
} csa2_sparse_attn_args;
CSA2_API int csa2_sparse_attn(const csa2_sparse_attn_args* args, void* workspace, size_t ws_bytes, void* stream);

/* ---- 5. main-KV entry build (m = 2, or m = 1) -------------------------------
 * Entry e (0 <= e < n_tokens / m) is built from tokens e*m .. e*m+m-1 of C, Z:
 *   m=2: x[c] = sum_j softmax_j(Z[2e+j][c]) * C[2e+j][c]  (per channel, no APE)
 *   m=1: x = C[e]                                         (weight identically 1)
 *   y = x / sqrt(mean(x^2) + eps) * gamma                 (RMSNorm)
 *   RoPE on dims 448..511 when apply_rope: pairs (448+2i, 449+2i) rotated by
 *   pos * rope_theta^(-2i/64), pos = entry_pos[e] if given, else (first_entry + e) * m
 *   FP4: per 32 elements u = k + 127 with k the smallest integer such that
 *   6 * 2^k >= amax (u = 127 for amax 0, clamped to [0,254]); codes = e2m1
 *   round-to-nearest-even of y / 2^k, saturating at 6; sign bit for y < 0.
 * The 288-B record goes to slot entry_slot[e] if given, else to
 * page_table[(first_entry + e) / 64] * 64 + (first_entry + e) % 64.
 * (CSA2 page item 3 and V4.1 Q&A page; V4.1-Flash report reading, section 六:
 * FP4 after RoPE, no global scale.)  latent_out (optional, fp32 [n_entries,512])
 * receives y after RoPE, before quantisation.  Alignment: C, Z 16 B.
 * Index keys (optional, w_ik not NULL; CSA2 page item 3, V4.1 Q&A page "the
 * indexer K is projected from the main KV"): from y before RoPE,
 *   k = RMSNorm(y W^IK) * k_gamma   (W^IK: 512 x 128, the same eps),
 *   RoPE on k's dims 64..127 (pairs (64+2i, 65+2i), the angles of the main
 *   latent's pair i), then quantised into the index-K page of the entry's slot
 *   (page slot/64, row slot%64): FP8: scale = amax/448 (fp32), codes = e4m3
 *   round-to-nearest-even of k/scale; FP4: e2m1 + ue8m0 per 32 dims as above.
 * index_latent_out (optional, fp32 [n_entries,128]) receives k before
 * quantisation. */
typedef struct {
  const uint16_t* C; const uint16_t* Z;        /* [n_tokens,512] bf16; Z unused for m=1 */
  int64_t n_tokens; int32_t ratio_m;
  const float* gamma; float eps;               /* [512], 16-B aligned */
  int32_t apply_rope; float rope_theta;
  int64_t first_entry;
  const int32_t* entry_pos;                    /* optional [n_entries] */
  uint8_t* main_kv; int64_t main_kv_slots;     /* 288-B records */
  const int32_t* page_table; int64_t pt_len;   /* [pt_len] of the one sequence, or NULL */
  const int32_t* entry_slot;                   /* optional [n_entries] direct slots */
  float* latent_out;                           /* optional [n_entries,512] */
  const uint16_t* w_ik;                        /* optional [512,128] bf16 W^IK (row = latent dim) */
  const float* k_gamma;                        /* [128] k_norm weight (with w_ik), 16-B aligned */
  uint8_t* index_k; int64_t index_k_pages;     /* index-K pages (with w_ik) */
  int32_t index_k_format;                      /* CSA2_INDEX_FP8 or CSA2_INDEX_FP4 */
  float* index_latent_out;                     /* optional [n_entries,128] */
} csa2_compress_args;
CSA2_API int csa2_compress_m2(const csa2_compress_args* args, void* stream);

/* ---- hidden-state projection of the entry build's inputs ---------------------
 * out[t] = hidden[t] W (fp32 accumulation, rounded to bf16) for t < T: the
 * per-token 512-vector the entry build takes as C (and, for m = 2, as Z).
 * CSA2 page item 3: with m = 1 the main-KV entry is one linear projection of
 * the token; CED (CSA2 page, report reading): the decoder layers' global KV
 * comes from the encoder output, C = H_{L/2} W^KV, the encoder layers' C and
 * Z from their own hidden states.  Sized for decode batches (T <= 64 rows;
 * the cost is the weight read, hidden_dim x 1 KB); a prefill chunk's
 * projection is a dense GEMM outside this call.  No workspace.  w is read
 * before the previous launch on the stream completes (weights are not
 * written by the step): it must not be written by the launch just before
 * this call.  Alignment: hidden, w, out 16 B. */
typedef struct {
  const uint16_t* hidden;      /* [T, hidden_dim] bf16 */
  const uint16_t* w;           /* [hidden_dim, 512] bf16 (row = input dim) */
  int32_t T;                   /* 1..64 */
  int32_t hidden_dim;          /* 512..16384, multiple of 512 */
  uint16_t* out;               /* [T, 512] bf16 */
} csa2_kv_project_args;
CSA2_API int csa2_kv_project(const csa2_kv_project_args* args, void* stream);

/* ---- workspace, device errors ------------------------------------------------ */
enum { CSA2_CALL_INDEX_SCORE = 1, CSA2_CALL_TOPK = 2, CSA2_CALL_REINDEX = 3, CSA2_CALL_SPARSE_ATTN = 4 };
/* Bytes of workspace the call needs with these arguments (0 if none). */
CSA2_API int csa2_workspace_size(int which_call, const void* args, size_t* bytes);
/* Synchronises the stream, then returns CSA2_ERR_DEVICE_BOUNDS or
 * CSA2_ERR_DEVICE_TIMEOUT if a kernel on this device recorded one since the
 * last check (and clears the record), else CSA2_OK.  The record is one word
 * per device for the whole process: every stream and every call of the
 * library on that device reports into it, so a check made after work on
 * stream A also reports an error that a kernel on stream B recorded, and
 * clears it for B's check.  Only the given stream is synchronised; the word
 * is read with a blocking copy. */
CSA2_API int csa2_check_device_error(void* stream);
/* Diagnostic (no counterpart in the pages): one CTA waits, with the bounded
 * wait every kernel of the library uses, on an mbarrier that nothing arrives
 * at and no copy completes; after `polls` polls (1..2^20; each poll may
 * suspend the thread for a short, hardware-defined time) it gives up and
 * records a timeout, so the next csa2_check_device_error returns
 * CSA2_ERR_DEVICE_TIMEOUT.  It exercises the failure path of the bounded
 * waits without a fault: nothing is left in flight and the context stays
 * usable.  In the kernels a wait gives up after 2^26 polls or 1 s of the
 * global timer without progress. */
CSA2_API int csa2_debug_bounded_wait(uint32_t polls, void* stream);
/* Library version string. */
CSA2_API const char* csa2_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H_ */
