// Exact top-k selection with slot translation, and the block-max candidate pool.
//
// Semantics (DSA page, "Top-k：选的是 token，不是 block"; CSA2 page,
// "Hierarchical Sparse Indexer", "池里的 16384 个位置是哪些", "attention 计算的
// 落点"): per row keep the k largest finite scores, ties to the lower index;
// positions become physical slots page_table[p / 64] * 64 + p % 64, -1 filled;
// the pool keeps the newest block plus the blocks with the highest block
// maxima, reported in ascending block order.
//
// Every candidate carries a unique 64-bit key (ord(score) << 32 | ~index): the
// k largest keys are exactly the k best (score desc, index asc).  A "virtual
// row" is either a score row (k = top-k) or a block-maximum row (k = pool
// size, newest block forced to +inf).  Rows longer than kDirect go through:
//   hist   : 2048-bin histogram of the top 11 key bits (skipped when the
//            indexer scan already produced it)
//   filter : many CTAs per row append every element whose bin is at or above
//            the threshold bin to a per-row candidate list (at most kCap)
// and a final CTA per row runs an exact radix select over the 64-bit keys in
// shared memory, sorts the survivors and writes positions, slots or pools.
// Rows of at most kDirect elements are selected by the final CTA directly; a
// row whose candidate list overflowed (massive ties near the threshold) is
// selected by the final CTA streaming the row from global memory, still exact.
#include <math.h>

#include "csa2_device.cuh"
#include "csa2_internal.h"

namespace csa2 {

namespace {

constexpr int kBins = 2048;
constexpr int kCap = 16384;      // candidate list per row
constexpr int kDirect = 16384;   // rows up to this length are selected in shared memory directly
constexpr int kChunk = 16384;    // elements per CTA in the streaming passes
constexpr int kMaxK = 2048;
constexpr int kStreamThreads = 256;
constexpr int kFinalThreads = 1024;

struct SelParams {
  int kind;  // 0: positions (+ pool rows), 2: Reindex candidates
  const float* scores;
  long long ld_scores;
  const float* block_max;
  long long ld_bm;
  const int* page_table;
  int pt_stride;
  RowsDev rows;
  int k;
  int* topk_pos;
  int* topk_slot;
  long long ld_topk;
  int* pool_out;
  int pool_n;
  const int* pool_in;
  int pool_in_n;
  const uint32_t* hist;  // [V][kBins]: given, or built by the hist pass in `hist_ws`
  uint32_t* hist_ws;
  uint32_t* cnt;         // [V]
  uint32_t* cord;        // [V][kCap]
  uint32_t* cidx;        // [V][kCap]
  uint32_t* err;
};

struct VRow {
  const float* src;
  int n;
  int k;
  bool pool;  // block-maximum row: output ascending ids, newest block forced
  int t;
};

__device__ __forceinline__ VRow vrow_of(const SelParams& P, int v) {
  VRow r;
  const int T = P.rows.T;
  r.t = v % T;
  r.pool = (P.kind == 0 && v >= T);
  const int b = row_seq_of(P.rows, r.t);
  if (P.kind == 2) {
    r.src = P.scores + static_cast<long long>(r.t) * P.pool_in_n * 8;
    r.n = P.pool_in_n * 8;
    r.k = P.k;
  } else if (!r.pool) {
    const int e = visible_of(P.rows, r.t, b);
    r.src = P.scores + static_cast<long long>(r.t) * P.ld_scores;
    r.n = static_cast<int>(min(static_cast<long long>(e), P.ld_scores));
    r.k = P.k;
  } else {
    const int e = visible_of(P.rows, r.t, b);
    r.src = P.block_max + static_cast<long long>(r.t) * P.ld_bm;
    r.n = static_cast<int>(min(static_cast<long long>((e + 7) / 8), P.ld_bm));
    r.k = P.pool_n;
  }
  return r;
}

// Key of element i, or 0 when it is not selectable (-inf / NaN).  Valid keys
// are >= 0x00800000, so 0 never collides with one.
__device__ __forceinline__ uint32_t elem_key(const VRow& r, float val, int i) {
  if (r.pool && i == r.n - 1) return 0xFFFFFFFFu;
  return selectable(val) ? ord_key(val) : 0u;
}

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += v;
  }
  return x;
}

// Block-wide search of a 2048-bin histogram in shared memory, walked from the
// top bin: res[0] = bin b with count(bins > b) < need <= count(bins >= b) (or
// -1 when the histogram holds fewer than need), res[1] = count above b,
// res[2] = total.  Threads 0..255 each own 8 consecutive bins (two 16-B loads);
// every thread of the block must call it.
__device__ void block_find_bin(const uint32_t* h, uint32_t need, int* res, uint32_t* wsum) {
  const int t = threadIdx.x;
  const int lane = t & 31, w = t >> 5;
  uint32_t c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  uint32_t sum = 0, incl = 0;
  if (t < 256) {
    const uint4* p4 = reinterpret_cast<const uint4*>(h + (kBins - 8 - 8 * t));
    const uint4 a = p4[0], b = p4[1];
    c[0] = b.w; c[1] = b.z; c[2] = b.y; c[3] = b.x;  // bins 2047-8t, 2046-8t, ...
    c[4] = a.w; c[5] = a.z; c[6] = a.y; c[7] = a.x;
#pragma unroll
    for (int j = 0; j < 8; ++j) sum += c[j];
    incl = warp_incl_scan(sum);
    if (lane == 31) wsum[w] = incl;
  }
  __syncthreads();
  if (t < 256) {
    uint32_t off = 0, total = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t x = wsum[j];
      if (j < w) off += x;
      total += x;
    }
    incl += off;
    const uint32_t excl = incl - sum;
    if (t == 0) {
      res[2] = static_cast<int>(total);
      if (total < need) {
        res[0] = -1;
        res[1] = static_cast<int>(total);
      }
    }
    if (total >= need && excl < need && incl >= need) {
      uint32_t run = excl;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (run + c[j] >= need) {
          res[0] = kBins - 1 - 8 * t - j;
          res[1] = static_cast<int>(run);
          break;
        }
        run += c[j];
      }
    }
  }
  __syncthreads();
}

__device__ __forceinline__ void stage_hist(uint32_t* dst, const uint32_t* src) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (int i = threadIdx.x; i < kBins / 4; i += blockDim.x) d4[i] = s4[i];
}

// ---------------------------------------------------------------- streaming passes
__global__ void __launch_bounds__(kStreamThreads) sel_hist_kernel(const __grid_constant__ SelParams P) {
  pdl_trigger();
  pdl_wait();
  const int v = blockIdx.y;
  const VRow r = vrow_of(P, v);
  if (r.n <= kDirect) return;
  const int i0 = blockIdx.x * kChunk;
  if (i0 >= r.n) return;
  __shared__ uint32_t h[kBins];
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int i1 = min(i0 + kChunk, r.n);
  for (int i = i0 + threadIdx.x * 4; i < i1; i += blockDim.x * 4) {
    float4 v4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (i + 3 < i1) {
      v4 = __ldg(reinterpret_cast<const float4*>(r.src + i));
    } else {
      v4.x = r.src[i];
      if (i + 1 < i1) v4.y = r.src[i + 1];
      if (i + 2 < i1) v4.z = r.src[i + 2];
    }
    const float vals[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t key = (i + j < i1) ? elem_key(r, vals[j], i + j) : 0u;
      if (key) atomicAdd(&h[key >> 21], 1u);
    }
  }
  __syncthreads();
  uint32_t* gh = P.hist_ws + static_cast<long long>(v) * kBins;
  for (int i = threadIdx.x; i < kBins; i += blockDim.x)
    if (h[i]) atomicAdd(gh + i, h[i]);
}

__global__ void __launch_bounds__(kStreamThreads) sel_filter_kernel(const __grid_constant__ SelParams P) {
  pdl_trigger();
  pdl_wait();
  const int v = blockIdx.y;
  const VRow r = vrow_of(P, v);
  if (r.n <= kDirect) return;
  const int i0 = blockIdx.x * kChunk;
  if (i0 >= r.n) return;
  __shared__ __align__(16) uint32_t h[kBins];
  __shared__ int res[4];
  __shared__ uint32_t wsum[8];
  stage_hist(h, P.hist + static_cast<long long>(v) * kBins);
  if (threadIdx.x == 0) res[0] = -1;
  __syncthreads();
  block_find_bin(h, static_cast<uint32_t>(r.k), res, wsum);
  const int b1 = res[0];
  const uint32_t thr = b1 < 0 ? 0u : static_cast<uint32_t>(b1);
  const int lane = threadIdx.x & 31;
  uint32_t* cord = P.cord + static_cast<long long>(v) * kCap;
  uint32_t* cidx = P.cidx + static_cast<long long>(v) * kCap;
  const int i1 = min(i0 + kChunk, r.n);
  // loop bounds are uniform across the block so that every lane takes part in the warp scans
  for (int base = i0; base < i1; base += blockDim.x * 4) {
    const int i = base + threadIdx.x * 4;
    float4 v4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (i + 3 < i1) {
      v4 = __ldg(reinterpret_cast<const float4*>(r.src + i));
    } else if (i < i1) {
      v4.x = r.src[i];
      if (i + 1 < i1) v4.y = r.src[i + 1];
      if (i + 2 < i1) v4.z = r.src[i + 2];
    }
    const float vals[4] = {v4.x, v4.y, v4.z, v4.w};
    uint32_t keys[4];
    uint32_t mine = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t key = (i + j < i1) ? elem_key(r, vals[j], i + j) : 0u;
      keys[j] = (key && (key >> 21) >= thr) ? key : 0u;
      mine += keys[j] ? 1u : 0u;
    }
    const uint32_t incl = warp_incl_scan(mine);
    const uint32_t wtot = __shfl_sync(0xffffffffu, incl, 31);
    if (wtot == 0) continue;
    uint32_t wbase = 0;
    if (lane == 31) wbase = atomicAdd(P.cnt + v, wtot);
    wbase = __shfl_sync(0xffffffffu, wbase, 31);
    uint32_t slot = wbase + incl - mine;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (!keys[j]) continue;
      if (slot < static_cast<uint32_t>(kCap)) {
        cord[slot] = keys[j];
        cidx[slot] = static_cast<uint32_t>(i + j);
      }
      ++slot;
    }
  }
}

// ---------------------------------------------------------------- final select
struct FinalSmem {
  uint32_t* ord;   // [kDirect]
  uint32_t* idx;   // [kDirect]
  uint64_t* sel;   // [kMaxK]
  uint32_t* hist;  // [256]
  int* res;        // [8]
  uint32_t* wsum;  // [32]
};

__device__ __forceinline__ uint64_t key64(uint32_t ord, uint32_t idx) {
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint64_t>(~idx);
}

// Exact radix select of the `need` largest 64-bit keys, 8 bits per pass, ending
// as soon as the remaining need equals a whole digit bin.  GLOBAL: elements are
// streamed from the row each pass; else they are the n entries of sm.ord/idx.
template <bool GLOBAL>
__device__ void radix_select(const VRow& r, const FinalSmem& sm, int n, int need, uint64_t* prefix_out,
                             int* pbits_out) {
  uint64_t prefix = 0;
  int pbits = 0;
  const int lane = threadIdx.x & 31;
  const int nloop = GLOBAL ? r.n : n;
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) sm.hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < nloop; i += blockDim.x) {
      uint64_t kk;
      bool valid;
      if (GLOBAL) {
        const uint32_t o = elem_key(r, r.src[i], i);
        valid = o != 0u;
        kk = key64(o, static_cast<uint32_t>(i));
      } else {
        valid = true;
        kk = key64(sm.ord[i], sm.idx[i]);
      }
      if (valid && (pbits == 0 || (kk >> (64 - pbits)) == prefix))
        atomicAdd(&sm.hist[static_cast<uint32_t>((kk >> shift) & 0xFFu)], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l owns digits 255-8l .. 248-8l
      const uint4* p4 = reinterpret_cast<const uint4*>(sm.hist + (248 - 8 * lane));
      const uint4 a = p4[0], b = p4[1];
      const uint32_t c[8] = {b.w, b.z, b.y, b.x, a.w, a.z, a.y, a.x};
      uint32_t sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) sum += c[j];
      const uint32_t incl = warp_incl_scan(sum);
      const uint32_t excl = incl - sum;
      if (excl < static_cast<uint32_t>(need) && incl >= static_cast<uint32_t>(need)) {
        uint32_t run = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run + c[j] >= static_cast<uint32_t>(need)) {
            sm.res[0] = 255 - 8 * lane - j;
            sm.res[1] = static_cast<int>(run);
            sm.res[2] = static_cast<int>(c[j]);
            break;
          }
          run += c[j];
        }
      }
    }
    __syncthreads();
    const uint32_t d = static_cast<uint32_t>(sm.res[0]);
    const int above = sm.res[1];
    const int cnt = sm.res[2];
    need -= above;
    prefix = (prefix << 8) | d;
    pbits += 8;
    __syncthreads();
    if (cnt == need) break;
  }
  *prefix_out = prefix;
  *pbits_out = pbits;
}

__device__ __forceinline__ void bitonic_sort(uint64_t* a, int P, bool descending) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < P / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool up = ((lo & size) == 0) != descending;
        const uint64_t x = a[lo], y = a[hi];
        if ((x > y) == up) {
          a[lo] = y;
          a[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

// Block-wide compaction helper: this thread's slot for `take`, the block's
// takes counted in *counter (a shared word).  Every lane of the warp must call.
__device__ __forceinline__ uint32_t block_append(bool take, uint32_t* counter) {
  const int lane = threadIdx.x & 31;
  const unsigned m = __ballot_sync(0xffffffffu, take);
  uint32_t b0 = 0;
  if (m && lane == __ffs(m) - 1) b0 = atomicAdd(counter, __popc(m));
  b0 = __shfl_sync(0xffffffffu, b0, m ? __ffs(m) - 1 : 0);
  return b0 + __popc(m & ((1u << lane) - 1u));
}

__global__ void __launch_bounds__(kFinalThreads, 1) sel_final_kernel(const __grid_constant__ SelParams P) {
  extern __shared__ __align__(16) uint8_t fsm_raw[];
  FinalSmem sm;
  sm.ord = reinterpret_cast<uint32_t*>(fsm_raw);
  sm.idx = sm.ord + kDirect;
  sm.sel = reinterpret_cast<uint64_t*>(sm.idx + kDirect);
  sm.hist = reinterpret_cast<uint32_t*>(sm.sel + kMaxK);
  sm.res = reinterpret_cast<int*>(sm.hist + 256);
  sm.wsum = reinterpret_cast<uint32_t*>(sm.res + 8);
  uint32_t* counters = sm.wsum + 32;  // [0]: gathered, [1]: selected
  pdl_trigger();
  pdl_wait();
  const int v = blockIdx.x;
  const VRow r = vrow_of(P, v);
  if (threadIdx.x < 2) counters[threadIdx.x] = 0;
  __syncthreads();

  // 1. gather the candidates into shared memory, or decide to stream the row
  int mode = 0;  // 0: shared memory, 1: stream the row from global memory
  int n = 0;
  if (r.n <= kDirect) {
    const int nr = (r.n + blockDim.x - 1) / blockDim.x * blockDim.x;
    for (int i = threadIdx.x; i < nr; i += blockDim.x) {
      const uint32_t key = (i < r.n) ? elem_key(r, r.src[i], i) : 0u;
      const uint32_t slot = block_append(key != 0u, &counters[0]);
      if (key) {
        sm.ord[slot] = key;
        sm.idx[slot] = static_cast<uint32_t>(i);
      }
    }
    __syncthreads();
    n = static_cast<int>(counters[0]);
  } else {
    const uint32_t c = P.cnt[v];
    if (c <= static_cast<uint32_t>(kCap)) {
      const uint32_t* cord = P.cord + static_cast<long long>(v) * kCap;
      const uint32_t* cidx = P.cidx + static_cast<long long>(v) * kCap;
      for (int i = threadIdx.x; i < static_cast<int>(c); i += blockDim.x) {
        sm.ord[i] = cord[i];
        sm.idx[i] = cidx[i];
      }
      n = static_cast<int>(c);
    } else {  // overflow: count the selectable elements from the histogram
      stage_hist(sm.ord, P.hist + static_cast<long long>(v) * kBins);
      __syncthreads();
      block_find_bin(sm.ord, 1u, sm.res, sm.wsum);
      n = sm.res[2];
      mode = 1;
    }
    __syncthreads();
  }
  const int need = min(r.k, n);

  // 2. exact threshold over 64-bit keys, 3. collect exactly `need` survivors
  uint64_t prefix = 0;
  int pbits = 0;
  const bool take_all = (need == n);
  if (!take_all) {
    if (mode == 0) radix_select<false>(r, sm, n, need, &prefix, &pbits);
    else radix_select<true>(r, sm, n, need, &prefix, &pbits);
  }
  const int nloop = (mode == 0) ? n : r.n;
  const int nr = (nloop + blockDim.x - 1) / blockDim.x * blockDim.x;
  for (int i = threadIdx.x; i < nr; i += blockDim.x) {
    uint64_t kk = 0;
    bool valid = false;
    if (i < nloop) {
      if (mode == 0) {
        valid = true;
        kk = key64(sm.ord[i], sm.idx[i]);
      } else {
        const uint32_t o = elem_key(r, r.src[i], i);
        valid = o != 0u;
        kk = key64(o, static_cast<uint32_t>(i));
      }
    }
    const bool take = valid && (take_all || (kk >> (64 - pbits)) >= prefix);
    const uint32_t slot = block_append(take, &counters[1]);
    // pools sort by block id ascending, positions by key descending
    if (take && slot < static_cast<uint32_t>(kMaxK)) sm.sel[slot] = r.pool ? static_cast<uint64_t>(~kk & 0xFFFFFFFFull) : kk;
  }
  __syncthreads();
  const int got = min(static_cast<int>(counters[1]), kMaxK);

  // 4. sort the survivors
  int Pw = 1;
  while (Pw < got) Pw <<= 1;
  for (int i = got + threadIdx.x; i < Pw; i += blockDim.x) sm.sel[i] = r.pool ? ~0ull : 0ull;
  __syncthreads();
  bitonic_sort(sm.sel, Pw, !r.pool);

  // 5. outputs
  const int t = r.t;
  const int b = row_seq_of(P.rows, t);
  if (r.pool) {
    int* out = P.pool_out + static_cast<long long>(t) * P.pool_n;
    for (int i = threadIdx.x; i < P.pool_n; i += blockDim.x) out[i] = (i < got) ? static_cast<int>(sm.sel[i]) : -1;
    return;
  }
  int* opos = P.topk_pos + static_cast<long long>(t) * P.ld_topk;
  int* oslot = P.topk_slot ? P.topk_slot + static_cast<long long>(t) * P.ld_topk : nullptr;
  for (int i = threadIdx.x; i < r.k; i += blockDim.x) {
    int pos = -1;
    if (i < got) {
      const uint32_t idx = ~static_cast<uint32_t>(sm.sel[i] & 0xFFFFFFFFull);
      if (P.kind == 2) {
        const int blk = P.pool_in[static_cast<long long>(t) * P.pool_in_n + (idx >> 3)];
        pos = blk * 8 + static_cast<int>(idx & 7);
      } else {
        pos = static_cast<int>(idx);
      }
    }
    opos[i] = pos;
    if (oslot) {
      int slot = -1;
      if (pos >= 0 && P.page_table) {
        const int lp = pos >> 6;
        const int phys = (lp < P.pt_stride) ? P.page_table[static_cast<long long>(b) * P.pt_stride + lp] : -1;
        if (phys >= 0) slot = phys * 64 + (pos & 63);
        else set_error(P.err, kErrBounds);
      }
      oslot[i] = slot;
    }
  }
}

size_t final_smem_bytes() {
  return static_cast<size_t>(kDirect) * 8 + kMaxK * 8 + 256 * 4 + 8 * 4 + 64 * 4;
}

}  // namespace

size_t select_workspace_bytes(const SelectLaunch& a) {
  if (a.kind != 0) return 0;  // Reindex rows are short enough for the direct path
  const long long V = static_cast<long long>(a.rows.T) * (a.pool_out ? 2 : 1);
  const size_t hist = a.hist ? 0 : static_cast<size_t>(V) * kBins * 4;
  return hist + ((static_cast<size_t>(V) * 4 + 255) & ~size_t(255)) + static_cast<size_t>(V) * kCap * 8 + 256;
}

cudaError_t launch_select(const SelectLaunch& a, void* ws, size_t ws_bytes, const DeviceCtx& ctx, cudaStream_t st) {
  (void)ws_bytes;
  SelParams P;
  P.kind = a.kind;
  P.scores = a.scores;
  P.ld_scores = a.ld_scores;
  P.block_max = a.block_max;
  P.ld_bm = a.ld_bm;
  P.page_table = a.page_table;
  P.pt_stride = a.pt_stride;
  P.rows = RowsDev{a.rows.T, a.rows.B, a.rows.row_seq, a.rows.row_pos, a.rows.n_visible, a.rows.ratio_m};
  P.k = a.k;
  P.topk_pos = a.topk_pos;
  P.topk_slot = a.topk_slot;
  P.ld_topk = a.ld_topk;
  P.pool_out = a.pool_out;
  P.pool_n = a.pool_n;
  P.pool_in = a.pool_in;
  P.pool_in_n = a.pool_in_n;
  P.err = ctx.err;
  const int V = a.rows.T * ((a.kind == 0 && a.pool_out) ? 2 : 1);
  P.hist = a.hist;
  P.hist_ws = nullptr;
  P.cnt = nullptr;
  P.cord = P.cidx = nullptr;
  cudaError_t e;
  long long maxn = 0;
  if (a.kind == 0) {
    maxn = a.ld_scores;
    if (a.pool_out) maxn = maxn > a.ld_bm ? maxn : a.ld_bm;
  }
  if (maxn > kDirect) {
    uint8_t* w = static_cast<uint8_t*>(ws);
    if (!a.hist) {
      P.hist_ws = reinterpret_cast<uint32_t*>(w);
      P.hist = P.hist_ws;
      w += static_cast<size_t>(V) * kBins * 4;
    }
    P.cnt = reinterpret_cast<uint32_t*>(w);
    const size_t cnt_bytes = (static_cast<size_t>(V) * 4 + 255) & ~size_t(255);
    P.cord = reinterpret_cast<uint32_t*>(w + cnt_bytes);
    P.cidx = P.cord + static_cast<size_t>(V) * kCap;
    // zero the histogram being built (if any) and the candidate counters: one contiguous range
    const size_t zero_bytes = (a.hist ? 0 : static_cast<size_t>(V) * kBins * 4) + cnt_bytes;
    e = cudaMemsetAsync(a.hist ? static_cast<void*>(P.cnt) : ws, 0, zero_bytes, st);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>((maxn + kChunk - 1) / kChunk), static_cast<unsigned>(V));
    if ((e = prefer_max_smem(sel_hist_kernel, 0)) != cudaSuccess) return e;
    if ((e = prefer_max_smem(sel_filter_kernel, 0)) != cudaSuccess) return e;
    if (!a.hist && (e = launch_pdl(sel_hist_kernel, grid, dim3(kStreamThreads), 0, st, P)) != cudaSuccess) return e;
    if ((e = launch_pdl(sel_filter_kernel, grid, dim3(kStreamThreads), 0, st, P)) != cudaSuccess) return e;
  }
  const size_t smem = final_smem_bytes();
  e = prefer_max_smem(sel_final_kernel, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(sel_final_kernel, dim3(V), dim3(kFinalThreads), smem, st, P);
}

}  // namespace csa2
