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
  uint32_t* err;
};
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
  const int* pool_blocks;
  int pool_n;
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
};
int attn_num_splits(int T, int n_keys, int num_sms);
size_t attn_workspace_bytes(int T, int nsplit);
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
};
cudaError_t launch_compress(const CompressLaunch& a, const DeviceCtx& ctx, cudaStream_t st);

// Tensor-map encoder from the driver (fetched once through the runtime).
CUresult encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t rows,
                           uint64_t row_stride, uint32_t box_inner, uint32_t box_rows);

}  // namespace csa2
