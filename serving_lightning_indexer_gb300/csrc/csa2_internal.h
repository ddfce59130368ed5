// Internal declarations shared by the host side of the CSA2 library.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/csa2.h"

namespace csa2 {

// Bits of the device-side error word (the kernels use the same values).
constexpr uint32_t kErrBoundsBit = 1u;
constexpr uint32_t kErrTimeoutBit = 2u;

// Query blocks one indexer launch takes (the kernel keeps a table of them in
// shared memory): rows on the per-row scan and Reindex, blocks of 8 rows on
// the prefill path.
constexpr int kIndexQueryBlocksPerLaunch = 2048;

struct RowsHost {
  int T, B;
  const int* row_seq;
  const int* row_pos;
  const int* n_visible;
  int ratio_m;
};

// Per-device state: SM count and the device address of the error word.
struct DeviceCtx {
  int device;
  int num_sms;
  int smem_per_sm;        // shared memory per SM (bytes)
  int smem_reserved;      // shared memory the runtime reserves per CTA (bytes)
  uint32_t* err;
};
// CTAs of `smem_bytes` dynamic shared memory that fit on one SM (shared memory only).
inline int ctas_per_sm_by_smem(const DeviceCtx& c, size_t smem_bytes) {
  const long long per = static_cast<long long>(smem_bytes) + c.smem_reserved;
  const long long n = per > 0 ? c.smem_per_sm / per : 1;
  return n < 1 ? 1 : static_cast<int>(n);
}
// Prefer the largest shared-memory carveout for a kernel, so that consecutive
// kernels of the library never reconfigure the L1 / shared-memory split.
template <typename K>
inline cudaError_t prefer_max_smem(K kern, size_t dyn_smem) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       static_cast<int>(cudaSharedmemCarveoutMaxShared));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dyn_smem));
}
cudaError_t device_ctx(DeviceCtx* out);

// Lightning-Indexer tiles.  mode 0: scan (scores over consecutive entries),
// mode 1: gather (candidate blocks of a pool).  nq = queries per MMA tile (1 or 8).
struct IndexLaunch {
  const uint8_t* q_fp8;
  const float* q_scale;
  const float* w;
  const uint8_t* index_k;
  long long n_pages;
  const int* page_table;
  int pt_stride;
  RowsHost rows;
  float* out;
  long long ld_out;
  float* block_max;
  long long ld_bm;
  uint32_t* hist;
  const int* pool_blocks;
  int pool_n;
  int fp4;  // index-K pages: 0 FP8 (8448 B), 1 FP4 (4352 B)
};
cudaError_t launch_index_tiles(const IndexLaunch& a, int mode, int nq, const DeviceCtx& ctx, cudaStream_t st,
                               const char** why);

// Exact top-k selection (positions / pool blocks / Reindex candidates).
struct SelectLaunch {
  // kind 0: top-k over scores[t][0..E_t); kind 2: top-k over pool candidate scores
  int kind;
  const float* scores;
  long long ld_scores;
  const float* block_max;
  long long ld_bm;
  const int* page_table;
  int pt_stride;
  RowsHost rows;
  int k;
  int* topk_pos;
  int* topk_slot;
  long long ld_topk;
  int* pool_out;          // kind 0 only: candidate pool output [T, pool_n]
  int pool_n;
  const int* pool_in;     // kind 2: the pool the candidates come from [T, pool_in_n]
  int pool_in_n;
  uint32_t* hist;         // optional precomputed key histograms [V][2048] (returned to zero)
  int order;              // 0: ascending positions, 1: best first
};
size_t select_workspace_bytes(const SelectLaunch& a);
cudaError_t launch_select(const SelectLaunch& a, void* ws, size_t ws_bytes, const DeviceCtx& ctx, cudaStream_t st);

// Sparse attention.
struct AttnLaunch {
  const uint16_t* q;
  const uint8_t* main_kv;
  long long main_slots;
  const int* topk_slot;
  int k;
  long long ld_topk;
  const uint8_t* swa_kv;
  long long swa_slots;
  const int* swa_slot;
  int n_swa;
  long long ld_swa;
  const float* sink;
  float scale;
  int T;
  int out_bf16;
  void* out;
  float* lse;
  int kv_ready;  // slots and caches written at least two launches before: gather before the dependency wait
  const int* q_pos;          // [T] query positions (inverse RoPE, bounded replay)
  int inv_rope;              // rotate the output's last 64 dims back by the query's RoPE
  float rope_theta;
  const int* swa_seg_start;  // [T] bounded-replay segment starts, or null
};
int attn_num_splits(int T, int n_keys, int num_sms);
size_t attn_workspace_bytes(int T, int n_keys, int num_sms);
cudaError_t launch_sparse_attn(const AttnLaunch& a, void* ws, size_t ws_bytes, const DeviceCtx& ctx,
                               cudaStream_t st);

// Main-KV entry build.
struct CompressLaunch {
  const uint16_t* C;
  const uint16_t* Z;
  long long n_entries;
  int ratio_m;
  const float* gamma;
  float eps;
  int apply_rope;
  float rope_theta;
  long long first_entry;
  const int* entry_pos;
  uint8_t* main_kv;
  long long main_slots;
  const int* page_table;
  long long pt_len;
  const int* entry_slot;
  float* latent_out;
  const uint16_t* w_ik;  // optional index-key build
  const float* k_gamma;
  uint8_t* index_k;
  long long index_k_pages;
  int index_k_fp4;
  float* index_latent_out;
};
cudaError_t launch_compress(const CompressLaunch& a, const DeviceCtx& ctx, cudaStream_t st);
// C = H W (bf16 in and out, fp32 accumulation) for T hidden rows of width `hidden`.
cudaError_t launch_kv_project(const uint16_t* H, const uint16_t* W, int T, int hidden, uint16_t* out,
                              cudaStream_t st);

// Shared by the top-k entry points: argument checks + launch description;
// `who` names the entry point in the error detail.
int topk_prepare(const csa2_topk_args* a, SelectLaunch* S, const char* who);
// Records the per-thread detail string returned by csa2_last_error_detail().
int set_error_detail(int code, const char* detail);

// Launch with programmatic stream serialisation (see pdl_trigger / pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Tensor-map encoder from the driver (fetched once through the runtime).
// 2-D tensor map over rows of 128 packed e2m1 codes (64 B, row stride 64 B),
// unpacked to 16-byte chunks in shared memory, 128-byte swizzle, boxes of
// box_rows rows; base must be 32-byte aligned.
CUresult encode_tmap_2d_fp4(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows);
CUresult encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t rows,
                           uint64_t row_stride, uint32_t box_inner, uint32_t box_rows);

}  // namespace csa2
