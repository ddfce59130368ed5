// csa2_topk_with_candidates_noalloc: the top-k / candidate-pool call without a
// caller-provided workspace and without any device allocation.
//
// Some callers cannot give the library scratch memory: a plugin or operator
// interface that hands over only input and output pointers, an engine whose
// device memory is owned by its own allocator with no way to request extra
// buffers, or a latency-critical path that must not call cudaMalloc (which can
// synchronise the device).  For them the scratch (histograms, candidate
// counters and candidate lists) lives in one fixed array in device memory owned
// by this file.  Every GPU that loads the library holds
// CSA2_TOPK_NOALLOC_SCRATCH_BYTES of it until the process exits.
//
// All calls share that array and it keeps the last call's contents; each call
// clears the histogram and counter words it needs before using them.  Two
// calls whose executions overlap on the GPU (different streams, or concurrent
// host threads) race on the array: serialise them.
#include <stdio.h>

#include <mutex>

#include "csa2_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_topk_scratch[CSA2_TOPK_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_topk_scratch, per device

// In host code the array's name is only a host-side handle, not a device
// address: the address is looked up once per device, with that device current.
cudaError_t scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int csa2_topk_with_candidates_noalloc(const csa2_topk_args* a, void* stream) {
  csa2::SelectLaunch S;
  int rc = csa2::topk_prepare(a, &S, "csa2_topk_with_candidates_noalloc");
  if (rc) return rc;
  const size_t need = csa2::select_workspace_bytes(S);
  if (need > CSA2_TOPK_NOALLOC_SCRATCH_BYTES) {
    char buf[256];
    snprintf(buf, sizeof(buf),
             "csa2_topk_with_candidates_noalloc: these rows need %zu bytes of scratch but the static scratch holds "
             "%zu; use csa2_topk_with_candidates with a workspace, or fewer rows per call",
             need, static_cast<size_t>(CSA2_TOPK_NOALLOC_SCRATCH_BYTES));
    return csa2::set_error_detail(CSA2_ERR_WORKSPACE, buf);
  }
  csa2::DeviceCtx ctx;
  cudaError_t e = csa2::device_ctx(&ctx);
  if (e != cudaSuccess) return csa2::set_error_detail(CSA2_ERR_CUDA, cudaGetErrorString(e));
  void* ws = nullptr;
  e = scratch_address(ctx.device, &ws);
  if (e != cudaSuccess) return csa2::set_error_detail(CSA2_ERR_CUDA, cudaGetErrorString(e));
  e = csa2::launch_select(S, ws, CSA2_TOPK_NOALLOC_SCRATCH_BYTES, ctx, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return csa2::set_error_detail(CSA2_ERR_CUDA, cudaGetErrorString(e));
  return CSA2_OK;
}
