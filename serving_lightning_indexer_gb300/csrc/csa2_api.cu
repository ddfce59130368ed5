// Host side of the CSA2 C ABI: argument validation, dispatch, workspace sizes,
// status strings and the device-side error word.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <string>

#include "csa2_device.cuh"
#include "csa2_internal.h"

namespace {

thread_local std::string g_detail;

// Device-side error word: kernels OR in kErrBounds / kErrTimeout.
__device__ uint32_t g_device_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_detail = buf;
  return code;
}

}  // namespace

namespace csa2 {
// Records the detail string of an error returned on this thread.
int set_error_detail(int code, const char* detail) {
  g_detail = detail;
  return code;
}
}  // namespace csa2

namespace {

int cuda_fail(cudaError_t e, const char* what) {
  return fail(CSA2_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxDevices = 64;
std::mutex g_ctx_mu;
csa2::DeviceCtx g_ctx[kMaxDevices];
bool g_ctx_ok[kMaxDevices];

int rows_check(const csa2_rows& r, const char* who) {
  if (r.T < 1 || r.B < 1) return fail(CSA2_ERR_SHAPE, "%s: T=%d and B=%d must be >= 1", who, r.T, r.B);
  if (!r.n_visible && !r.row_pos) return fail(CSA2_ERR_NULL, "%s: one of n_visible, row_pos is required", who);
  if (!r.row_seq && r.T != r.B) return fail(CSA2_ERR_SHAPE, "%s: row_seq NULL needs T == B (T=%d, B=%d)", who, r.T, r.B);
  if (r.row_pos && r.ratio_m != 1 && r.ratio_m != 2)
    return fail(CSA2_ERR_UNSUPPORTED, "%s: ratio_m=%d must be 1 or 2", who, r.ratio_m);
  return CSA2_OK;
}

csa2::RowsHost rows_host(const csa2_rows& r) {
  return csa2::RowsHost{r.T, r.B, r.row_seq, r.row_pos, r.n_visible, r.row_pos ? r.ratio_m : 1};
}

}  // namespace

namespace csa2 {

cudaError_t device_ctx(DeviceCtx* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_ctx_mu);
  if (!g_ctx_ok[dev]) {
    DeviceCtx c;
    c.device = dev;
    e = cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&c.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&c.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) return e;
    c.err = static_cast<uint32_t*>(p);
    g_ctx[dev] = c;
    g_ctx_ok[dev] = true;
  }
  *out = g_ctx[dev];
  return cudaSuccess;
}

static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

CUresult encode_tmap_2d_fp4(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tmap_encoder();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[2] = {128, rows};   // 4-bit elements per row, rows
  const cuuint64_t strides[1] = {64};       // bytes
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t rows,
                           uint64_t row_stride, uint32_t box_inner, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tmap_encoder();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[2] = {inner_bytes, rows};
  const cuuint64_t strides[1] = {row_stride};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace csa2

using csa2::DeviceCtx;

extern "C" {

const char* csa2_version(void) { return "csa2-gb300 0.1 (sm_103a)"; }

const char* csa2_status_string(int s) {
  switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_NULL: return "null pointer";
    case CSA2_ERR_SHAPE: return "bad shape or size";
    case CSA2_ERR_ALIGN: return "misaligned pointer or stride";
    case CSA2_ERR_UNSUPPORTED: return "unsupported argument combination";
    case CSA2_ERR_CUDA: return "CUDA error";
    case CSA2_ERR_DEVICE_BOUNDS: return "out-of-range page id or slot met on the device";
    case CSA2_ERR_WORKSPACE: return "workspace missing or too small";
    case CSA2_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
    default: return "unknown status";
  }
}

const char* csa2_last_error_detail(void) { return g_detail.c_str(); }

static int check_index_common(const uint8_t* q_fp8, const float* q_scale, const float* w, const uint8_t* index_k,
                              int64_t pages, const int32_t* pt, int32_t pt_stride, const csa2_rows& rows,
                              int32_t format, const char* who) {
  if (!q_fp8 || !q_scale || !w || !index_k || !pt) return fail(CSA2_ERR_NULL, "%s: null input pointer", who);
  if (format != CSA2_INDEX_FP8 && format != CSA2_INDEX_FP4)
    return fail(CSA2_ERR_UNSUPPORTED, "%s: index_k_format=%d is neither FP8 (0) nor FP4 (1)", who, format);
  if (!aligned16(q_fp8) || !aligned16(index_k)) return fail(CSA2_ERR_ALIGN, "%s: q_fp8 and index_k must be 16-B aligned", who);
  if (format == CSA2_INDEX_FP4 && (reinterpret_cast<uintptr_t>(index_k) & 31))
    return fail(CSA2_ERR_ALIGN, "%s: FP4 index_k pages must be 32-B aligned", who);
  if (pages < 1 || pages * 68 > 0x7FFFFFFFLL) return fail(CSA2_ERR_SHAPE, "%s: index_k_pages=%lld out of range", who, (long long)pages);
  if (pt_stride < 1) return fail(CSA2_ERR_SHAPE, "%s: pt_stride must be >= 1", who);
  return rows_check(rows, who);
}

int csa2_index_score(const csa2_index_score_args* a, void* ws, size_t ws_bytes, void* stream) {
  (void)ws;
  (void)ws_bytes;
  if (!a) return fail(CSA2_ERR_NULL, "csa2_index_score: args is NULL");
  int rc = check_index_common(a->q_fp8, a->q_scale, a->w, a->index_k, a->index_k_pages, a->page_table, a->pt_stride,
                              a->rows, a->index_k_format, "csa2_index_score");
  if (rc) return rc;
  if (!a->scores) return fail(CSA2_ERR_NULL, "csa2_index_score: scores is NULL");
  if (a->ld_scores < 1) return fail(CSA2_ERR_SHAPE, "csa2_index_score: ld_scores must be >= 1");
  if (!aligned16(a->scores) || (a->ld_scores & 3))
    return fail(CSA2_ERR_ALIGN, "csa2_index_score: scores must be 16-B aligned with ld_scores a multiple of 4");
  if (a->block_max && (!aligned16(a->block_max) || (a->ld_block_max & 3) || a->ld_block_max < 1))
    return fail(CSA2_ERR_ALIGN, "csa2_index_score: block_max must be 16-B aligned with ld a positive multiple of 4");
  // FP4 pages take the per-row scan at every shape (prefill included)
  const bool fp4 = a->index_k_format == CSA2_INDEX_FP4;
  const bool prefill = a->rows.row_pos && a->rows.B == 1 && a->rows.T >= 64 && !fp4;
  const int nq = prefill ? 8 : 1;
  if (prefill && a->rows.T > csa2::kIndexQueryBlocksPerLaunch * 8)
    return fail(CSA2_ERR_SHAPE, "csa2_index_score: at most %d rows per call on the prefill path",
                csa2::kIndexQueryBlocksPerLaunch * 8);
  if (a->hist && prefill)
    return fail(CSA2_ERR_UNSUPPORTED, "csa2_index_score: hist is produced on the per-row scan only (pass NULL)");
  if (a->hist && a->rows.T > csa2::kIndexQueryBlocksPerLaunch)
    return fail(CSA2_ERR_SHAPE, "csa2_index_score: hist needs at most %d rows per call", csa2::kIndexQueryBlocksPerLaunch);
  if (a->hist && !aligned16(a->hist)) return fail(CSA2_ERR_ALIGN, "csa2_index_score: hist must be 16-B aligned");
  DeviceCtx ctx;
  cudaError_t e = csa2::device_ctx(&ctx);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_index_score: device");
  // The per-row scan takes at most kIndexQueryBlocksPerLaunch rows a launch: rows
  // [t0, t0 + n) go with q, w, the outputs and the row arrays offset by t0.
  // Without row_seq the row is its own sequence, so the page table rows and
  // n_visible move along, and rows past the last sequence see nothing (no
  // launch).
  const int step = prefill ? a->rows.T : csa2::kIndexQueryBlocksPerLaunch;
  for (int t0 = 0; t0 < a->rows.T; t0 += step) {
    const int n = (a->rows.T - t0) < step ? (a->rows.T - t0) : step;
    csa2::IndexLaunch L{};
    L.q_fp8 = a->q_fp8 + static_cast<size_t>(t0) * 32 * 128;
    L.q_scale = a->q_scale + static_cast<size_t>(t0) * 32;
    L.w = a->w + static_cast<size_t>(t0) * 32;
    L.index_k = a->index_k;
    L.n_pages = a->index_k_pages;
    L.fp4 = fp4;
    L.page_table = a->page_table;
    L.pt_stride = a->pt_stride;
    L.rows = rows_host(a->rows);
    L.rows.T = n;
    if (a->rows.row_pos) L.rows.row_pos = a->rows.row_pos + t0;
    if (a->rows.row_seq) {
      L.rows.row_seq = a->rows.row_seq + t0;
    } else if (t0 > 0) {
      const int b_left = a->rows.B - t0;
      if (b_left <= 0) break;
      L.rows.B = b_left < n ? b_left : n;
      L.page_table = a->page_table + static_cast<size_t>(t0) * a->pt_stride;
      if (a->rows.n_visible) L.rows.n_visible = a->rows.n_visible + t0;
    }
    L.out = a->scores + static_cast<size_t>(t0) * a->ld_scores;
    L.ld_out = a->ld_scores;
    L.block_max = a->block_max ? a->block_max + static_cast<size_t>(t0) * a->ld_block_max : nullptr;
    L.ld_bm = a->ld_block_max;
    L.hist = a->hist;
    const char* why = "launch";
    e = csa2::launch_index_tiles(L, 0, nq, ctx, static_cast<cudaStream_t>(stream), &why);
    if (e != cudaSuccess) return cuda_fail(e, why);
  }
  return CSA2_OK;
}

}  // extern "C"

// Validates top-k arguments and fills the internal launch description; shared
// by every top-k entry point (`who` names the entry point in error details).
int csa2::topk_prepare(const csa2_topk_args* a, csa2::SelectLaunch* S, const char* who) {
  if (!a) return fail(CSA2_ERR_NULL, "%s: args is NULL", who);
  int rc = rows_check(a->rows, who);
  if (rc) return rc;
  if (!a->scores || !a->topk_pos) return fail(CSA2_ERR_NULL, "%s: scores/topk_pos is NULL", who);
  if (a->k < 1 || a->k > CSA2_MAX_TOPK) return fail(CSA2_ERR_SHAPE, "%s: k=%d not in 1..2048", who, a->k);
  if (a->ld_topk < a->k) return fail(CSA2_ERR_SHAPE, "%s: ld_topk < k", who);
  if (!aligned16(a->scores) || (a->ld_scores & 3) || a->ld_scores < 1)
    return fail(CSA2_ERR_ALIGN, "%s: scores must be 16-B aligned, ld a positive multiple of 4", who);
  if (a->topk_slot && !a->page_table) return fail(CSA2_ERR_NULL, "%s: topk_slot needs page_table", who);
  if (a->pool_blocks) {
    if (!a->block_max) return fail(CSA2_ERR_NULL, "%s: the pool needs block_max", who);
    if (a->pool_n < 1 || a->pool_n > CSA2_MAX_TOPK)
      return fail(CSA2_ERR_SHAPE, "%s: pool_n=%d not in 1..2048", who, a->pool_n);
    if (!aligned16(a->block_max) || (a->ld_block_max & 3) || a->ld_block_max < 1)
      return fail(CSA2_ERR_ALIGN, "%s: block_max must be 16-B aligned, ld a positive multiple of 4", who);
  }
  *S = csa2::SelectLaunch{};
  S->kind = 0;
  S->scores = a->scores;
  S->ld_scores = a->ld_scores;
  S->block_max = a->block_max;
  S->ld_bm = a->ld_block_max;
  S->page_table = a->page_table;
  S->pt_stride = a->pt_stride;
  S->rows = rows_host(a->rows);
  S->k = a->k;
  S->topk_pos = a->topk_pos;
  S->topk_slot = a->topk_slot;
  S->ld_topk = a->ld_topk;
  S->pool_out = a->pool_blocks;
  S->pool_n = a->pool_blocks ? a->pool_n : 0;
  if (a->hist && !aligned16(a->hist)) return fail(CSA2_ERR_ALIGN, "%s: hist must be 16-B aligned", who);
  S->hist = const_cast<uint32_t*>(a->hist);
  if (a->order != CSA2_ORDER_POSITION && a->order != CSA2_ORDER_SCORE)
    return fail(CSA2_ERR_SHAPE, "%s: order=%d must be 0 (positions) or 1 (best first)", who, a->order);
  S->order = a->order;
  return CSA2_OK;
}

extern "C" {

int csa2_topk_with_candidates(const csa2_topk_args* a, void* ws, size_t ws_bytes, void* stream) {
  csa2::SelectLaunch S;
  int rc = csa2::topk_prepare(a, &S, "csa2_topk_with_candidates");
  if (rc) return rc;
  const size_t need = csa2::select_workspace_bytes(S);
  if (need && (!ws || ws_bytes < need))
    return fail(CSA2_ERR_WORKSPACE, "csa2_topk_with_candidates: workspace of %zu bytes needed", need);
  if (need && !aligned16(ws)) return fail(CSA2_ERR_ALIGN, "csa2_topk_with_candidates: workspace must be 16-B aligned");
  DeviceCtx ctx;
  cudaError_t e = csa2::device_ctx(&ctx);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_topk_with_candidates: device");
  e = csa2::launch_select(S, ws, ws_bytes, ctx, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "csa2_topk_with_candidates: launch");
  return CSA2_OK;
}

// Reindex workspace: the candidate scores, unless pool_scores is given (the
// selection builds their histogram itself).
static size_t reindex_ws(const csa2_reindex_args* a) {
  return a->pool_scores ? 0 : ((static_cast<size_t>(a->rows.T) * a->pool_n * 8 * 4 + 255) & ~size_t(255));
}

int csa2_reindex(const csa2_reindex_args* a, void* ws, size_t ws_bytes, void* stream) {
  if (!a) return fail(CSA2_ERR_NULL, "csa2_reindex: args is NULL");
  int rc = check_index_common(a->q_fp8, a->q_scale, a->w, a->index_k, a->index_k_pages, a->page_table, a->pt_stride,
                              a->rows, a->index_k_format, "csa2_reindex");
  if (rc) return rc;
  if (a->rows.T > csa2::kIndexQueryBlocksPerLaunch)
    return fail(CSA2_ERR_SHAPE, "csa2_reindex: at most %d rows per call", csa2::kIndexQueryBlocksPerLaunch);
  if (!a->pool_blocks || !a->topk_pos) return fail(CSA2_ERR_NULL, "csa2_reindex: pool_blocks/topk_pos is NULL");
  if (a->pool_n < 1 || a->pool_n > CSA2_MAX_TOPK) return fail(CSA2_ERR_SHAPE, "csa2_reindex: pool_n=%d not in 1..2048", a->pool_n);
  if (a->k < 1 || a->k > CSA2_MAX_TOPK) return fail(CSA2_ERR_SHAPE, "csa2_reindex: k=%d not in 1..2048", a->k);
  if (a->ld_topk < a->k) return fail(CSA2_ERR_SHAPE, "csa2_reindex: ld_topk < k");
  if (a->pool_scores && !aligned16(a->pool_scores)) return fail(CSA2_ERR_ALIGN, "csa2_reindex: pool_scores must be 16-B aligned");
  if (a->order != CSA2_ORDER_POSITION && a->order != CSA2_ORDER_SCORE)
    return fail(CSA2_ERR_SHAPE, "csa2_reindex: order=%d must be 0 (positions) or 1 (best first)", a->order);
  const size_t need = reindex_ws(a);
  if (need && (!ws || ws_bytes < need)) return fail(CSA2_ERR_WORKSPACE, "csa2_reindex: workspace of %zu bytes needed", need);
  if (need && !aligned16(ws)) return fail(CSA2_ERR_ALIGN, "csa2_reindex: workspace must be 16-B aligned");
  DeviceCtx ctx;
  cudaError_t e = csa2::device_ctx(&ctx);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_reindex: device");
  float* ps = a->pool_scores ? a->pool_scores : static_cast<float*>(ws);
  csa2::IndexLaunch L{};
  L.q_fp8 = a->q_fp8;
  L.q_scale = a->q_scale;
  L.w = a->w;
  L.index_k = a->index_k;
  L.n_pages = a->index_k_pages;
  L.fp4 = a->index_k_format == CSA2_INDEX_FP4;
  L.page_table = a->page_table;
  L.pt_stride = a->pt_stride;
  L.rows = rows_host(a->rows);
  L.out = ps;
  L.ld_out = static_cast<long long>(a->pool_n) * 8;
  L.pool_blocks = a->pool_blocks;
  L.pool_n = a->pool_n;
  const char* why = "launch";
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  e = csa2::launch_index_tiles(L, 1, 1, ctx, st, &why);
  if (e != cudaSuccess) return cuda_fail(e, why);
  csa2::SelectLaunch S{};
  S.kind = 2;
  S.scores = ps;
  S.ld_scores = static_cast<long long>(a->pool_n) * 8;
  S.page_table = a->page_table;
  S.pt_stride = a->pt_stride;
  S.rows = rows_host(a->rows);
  S.k = a->k;
  S.topk_pos = a->topk_pos;
  S.topk_slot = a->topk_slot;
  S.ld_topk = a->ld_topk;
  S.pool_in = a->pool_blocks;
  S.pool_in_n = a->pool_n;
  S.order = a->order;
  e = csa2::launch_select(S, nullptr, 0, ctx, st);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_reindex: select launch");
  return CSA2_OK;
}

static int attn_check(const csa2_sparse_attn_args* a) {
  if (!a) return fail(CSA2_ERR_NULL, "csa2_sparse_attn: args is NULL");
  if (!a->q || !a->sink || !a->out) return fail(CSA2_ERR_NULL, "csa2_sparse_attn: q/sink/out is NULL");
  if (a->T < 1) return fail(CSA2_ERR_SHAPE, "csa2_sparse_attn: T must be >= 1");
  if (a->k < 0 || a->k > CSA2_MAX_TOPK) return fail(CSA2_ERR_SHAPE, "csa2_sparse_attn: k=%d not in 0..2048", a->k);
  if (a->n_swa < 0 || a->n_swa > CSA2_MAX_SWA) return fail(CSA2_ERR_SHAPE, "csa2_sparse_attn: n_swa=%d not in 0..128", a->n_swa);
  if (a->k > 0 && (!a->topk_slot || !a->main_kv)) return fail(CSA2_ERR_NULL, "csa2_sparse_attn: topk_slot/main_kv is NULL");
  if (a->n_swa > 0 && (!a->swa_slot || !a->swa_kv)) return fail(CSA2_ERR_NULL, "csa2_sparse_attn: swa_slot/swa_kv is NULL");
  if (a->k > 0 && a->ld_topk < a->k) return fail(CSA2_ERR_SHAPE, "csa2_sparse_attn: ld_topk < k");
  if (a->n_swa > 0 && a->ld_swa < a->n_swa) return fail(CSA2_ERR_SHAPE, "csa2_sparse_attn: ld_swa < n_swa");
  if (!aligned16(a->q) || !aligned16(a->out) || (a->main_kv && !aligned16(a->main_kv)) ||
      (a->swa_kv && !aligned16(a->swa_kv)))
    return fail(CSA2_ERR_ALIGN, "csa2_sparse_attn: q, out, main_kv, swa_kv must be 16-B aligned");
  if (!(a->softmax_scale >= 0.f) || !isfinite(a->softmax_scale))
    return fail(CSA2_ERR_SHAPE, "csa2_sparse_attn: softmax_scale must be finite and >= 0");
  if (a->out_inv_rope != 0 && a->out_inv_rope != 1)
    return fail(CSA2_ERR_SHAPE, "csa2_sparse_attn: out_inv_rope=%d must be 0 or 1", a->out_inv_rope);
  if ((a->out_inv_rope || a->swa_seg_start) && !a->q_pos)
    return fail(CSA2_ERR_NULL, "csa2_sparse_attn: out_inv_rope and swa_seg_start need q_pos");
  if (!(a->rope_theta >= 0.f) || !isfinite(a->rope_theta))
    return fail(CSA2_ERR_SHAPE, "csa2_sparse_attn: rope_theta must be finite and >= 0");
  return CSA2_OK;
}

int csa2_sparse_attn(const csa2_sparse_attn_args* a, void* ws, size_t ws_bytes, void* stream) {
  int rc = attn_check(a);
  if (rc) return rc;
  DeviceCtx ctx;
  cudaError_t e = csa2::device_ctx(&ctx);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_sparse_attn: device");
  const size_t need = csa2::attn_workspace_bytes(a->T, a->n_swa + a->k, ctx.num_sms);
  if (need && (!ws || ws_bytes < need)) return fail(CSA2_ERR_WORKSPACE, "csa2_sparse_attn: workspace of %zu bytes needed", need);
  if (need && !aligned16(ws)) return fail(CSA2_ERR_ALIGN, "csa2_sparse_attn: workspace must be 16-B aligned");
  csa2::AttnLaunch L{};
  L.q = a->q;
  L.main_kv = a->main_kv;
  L.main_slots = a->main_kv_slots;
  L.topk_slot = a->topk_slot;
  L.k = a->k;
  L.ld_topk = a->ld_topk;
  L.swa_kv = a->swa_kv;
  L.swa_slots = a->swa_slots;
  L.swa_slot = a->swa_slot;
  L.n_swa = a->n_swa;
  L.ld_swa = a->ld_swa;
  L.sink = a->sink;
  L.scale = a->softmax_scale > 0.f ? a->softmax_scale : 1.0f / sqrtf(512.0f);
  L.T = a->T;
  L.out_bf16 = a->out_bf16;
  L.out = a->out;
  L.lse = a->lse;
  L.kv_ready = a->kv_ready != 0;
  L.q_pos = a->q_pos;
  L.inv_rope = a->out_inv_rope;
  L.rope_theta = a->rope_theta > 0.f ? a->rope_theta : 10000.0f;
  L.swa_seg_start = a->swa_seg_start;
  e = csa2::launch_sparse_attn(L, ws, ws_bytes, ctx, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "csa2_sparse_attn: launch");
  return CSA2_OK;
}

int csa2_compress_m2(const csa2_compress_args* a, void* stream) {
  if (!a) return fail(CSA2_ERR_NULL, "csa2_compress_m2: args is NULL");
  if (!a->C || !a->gamma || !a->main_kv) return fail(CSA2_ERR_NULL, "csa2_compress_m2: C/gamma/main_kv is NULL");
  if (a->ratio_m != 1 && a->ratio_m != 2) return fail(CSA2_ERR_UNSUPPORTED, "csa2_compress_m2: ratio_m=%d must be 1 or 2", a->ratio_m);
  if (a->ratio_m == 2 && !a->Z) return fail(CSA2_ERR_NULL, "csa2_compress_m2: Z is NULL with ratio_m=2");
  if (a->n_tokens < 0) return fail(CSA2_ERR_SHAPE, "csa2_compress_m2: n_tokens < 0");
  if (!a->entry_slot && !a->page_table) return fail(CSA2_ERR_NULL, "csa2_compress_m2: entry_slot or page_table is required");
  if (!aligned16(a->C) || (a->Z && !aligned16(a->Z)) || !aligned16(a->main_kv) || !aligned16(a->gamma) ||
      (a->latent_out && !aligned16(a->latent_out)))
    return fail(CSA2_ERR_ALIGN, "csa2_compress_m2: C, Z, gamma, main_kv, latent_out must be 16-B aligned");
  if (!(a->eps >= 0.f)) return fail(CSA2_ERR_SHAPE, "csa2_compress_m2: eps must be >= 0");
  if (a->apply_rope && !(a->rope_theta > 0.f)) return fail(CSA2_ERR_SHAPE, "csa2_compress_m2: rope_theta must be > 0");
  if (a->first_entry < 0) return fail(CSA2_ERR_SHAPE, "csa2_compress_m2: first_entry < 0");
  if (a->w_ik) {
    if (!a->k_gamma || !a->index_k) return fail(CSA2_ERR_NULL, "csa2_compress_m2: w_ik needs k_gamma and index_k");
    if (a->index_k_format != CSA2_INDEX_FP8 && a->index_k_format != CSA2_INDEX_FP4)
      return fail(CSA2_ERR_UNSUPPORTED, "csa2_compress_m2: index_k_format=%d is neither FP8 (0) nor FP4 (1)",
                  a->index_k_format);
    if (!aligned16(a->w_ik) || !aligned16(a->k_gamma) || !aligned16(a->index_k) ||
        (a->index_latent_out && !aligned16(a->index_latent_out)))
      return fail(CSA2_ERR_ALIGN, "csa2_compress_m2: w_ik, k_gamma, index_k, index_latent_out must be 16-B aligned");
    if (a->index_k_pages < 1) return fail(CSA2_ERR_SHAPE, "csa2_compress_m2: index_k_pages must be >= 1");
  }
  DeviceCtx ctx;
  cudaError_t e = csa2::device_ctx(&ctx);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_compress_m2: device");
  csa2::CompressLaunch L{};
  L.C = a->C;
  L.Z = a->Z;
  L.n_entries = a->n_tokens / a->ratio_m;
  L.ratio_m = a->ratio_m;
  L.gamma = a->gamma;
  L.eps = a->eps;
  L.apply_rope = a->apply_rope;
  L.rope_theta = a->rope_theta;
  L.first_entry = a->first_entry;
  L.entry_pos = a->entry_pos;
  L.main_kv = a->main_kv;
  L.main_slots = a->main_kv_slots;
  L.page_table = a->page_table;
  L.pt_len = a->pt_len;
  L.entry_slot = a->entry_slot;
  L.latent_out = a->latent_out;
  L.w_ik = a->w_ik;
  L.k_gamma = a->k_gamma;
  L.index_k = a->index_k;
  L.index_k_pages = a->index_k_pages;
  L.index_k_fp4 = a->index_k_format == CSA2_INDEX_FP4;
  L.index_latent_out = a->index_latent_out;
  e = csa2::launch_compress(L, ctx, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "csa2_compress_m2: launch");
  return CSA2_OK;
}

int csa2_kv_project(const csa2_kv_project_args* a, void* stream) {
  if (!a) return fail(CSA2_ERR_NULL, "csa2_kv_project: args is NULL");
  if (!a->hidden || !a->w || !a->out) return fail(CSA2_ERR_NULL, "csa2_kv_project: hidden/w/out is NULL");
  if (a->T < 1 || a->T > 64) return fail(CSA2_ERR_SHAPE, "csa2_kv_project: T=%d not in 1..64", a->T);
  if (a->hidden_dim < 512 || a->hidden_dim > 16384 || (a->hidden_dim & 511))
    return fail(CSA2_ERR_SHAPE, "csa2_kv_project: hidden_dim=%d must be a multiple of 512 in 512..16384",
                a->hidden_dim);
  if (!aligned16(a->hidden) || !aligned16(a->w) || !aligned16(a->out))
    return fail(CSA2_ERR_ALIGN, "csa2_kv_project: hidden, w, out must be 16-B aligned");
  cudaError_t e = csa2::launch_kv_project(a->hidden, a->w, a->T, a->hidden_dim, a->out,
                                          static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "csa2_kv_project: launch");
  return CSA2_OK;
}

int csa2_workspace_size(int which, const void* args, size_t* bytes) {
  if (!args || !bytes) return fail(CSA2_ERR_NULL, "csa2_workspace_size: null argument");
  *bytes = 0;
  switch (which) {
    case CSA2_CALL_INDEX_SCORE:
      return CSA2_OK;
    case CSA2_CALL_TOPK: {
      csa2::SelectLaunch S;
      int rc = csa2::topk_prepare(static_cast<const csa2_topk_args*>(args), &S, "csa2_workspace_size");
      if (rc) return rc;
      *bytes = csa2::select_workspace_bytes(S);
      return CSA2_OK;
    }
    case CSA2_CALL_REINDEX:
      *bytes = reindex_ws(static_cast<const csa2_reindex_args*>(args));
      return CSA2_OK;
    case CSA2_CALL_SPARSE_ATTN: {
      const csa2_sparse_attn_args* a = static_cast<const csa2_sparse_attn_args*>(args);
      int rc = attn_check(a);
      if (rc) return rc;
      DeviceCtx ctx;
      cudaError_t e = csa2::device_ctx(&ctx);
      if (e != cudaSuccess) return cuda_fail(e, "csa2_workspace_size: device");
      *bytes = csa2::attn_workspace_bytes(a->T, a->n_swa + a->k, ctx.num_sms);
      return CSA2_OK;
    }
    default:
      return fail(CSA2_ERR_UNSUPPORTED, "csa2_workspace_size: unknown call %d", which);
  }
}

}  // extern "C"

namespace {
// One CTA waits, with the library's bounded wait, on an mbarrier that nothing
// arrives at and no copy completes; the wait gives up and records a timeout
// in the device error word exactly as the kernels of the library do.
__global__ void bounded_wait_probe_kernel(uint32_t polls, uint32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    csa2::mbar_init(&bar, 1);
    csa2::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !csa2::mbar_wait_polls(&bar, 0u, nullptr, polls)) csa2::set_error(err, csa2::kErrTimeout);
}
}  // namespace

extern "C" {

int csa2_debug_bounded_wait(uint32_t polls, void* stream) {
  if (polls < 1 || polls > (1u << 20)) return fail(CSA2_ERR_SHAPE, "csa2_debug_bounded_wait: polls=%u not in 1..2^20", polls);
  DeviceCtx ctx;
  cudaError_t e = csa2::device_ctx(&ctx);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_debug_bounded_wait: device");
  bounded_wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(polls, ctx.err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "csa2_debug_bounded_wait: launch");
  return CSA2_OK;
}

int csa2_check_device_error(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "csa2_check_device_error: stream");
  uint32_t v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "csa2_check_device_error: read");
  if (v) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "csa2_check_device_error: clear");
  }
  if (v & csa2::kErrTimeoutBit) return fail(CSA2_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait");
  if (v & csa2::kErrBoundsBit) return fail(CSA2_ERR_DEVICE_BOUNDS, "a kernel met an out-of-range page id or slot");
  return CSA2_OK;
}

}  // extern "C"
