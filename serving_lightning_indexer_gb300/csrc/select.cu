// Exact top-k selection with slot translation, and the block-max candidate pool.
//
// Semantics (DSA page, "Top-k：选的是 token，不是 block"; CSA2 page,
// "Hierarchical Sparse Indexer", "池里的 16384 个位置是哪些", "attention 计算的
// 落点"): per row keep the k largest finite scores, ties to the lower index,
// reported in ascending position order;
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
//   filter : CTAs of 4096 elements each store every element whose bin is at
//            or above the threshold bin in their own region (at most kRegion,
//            with the true count), so nothing shared needs zeroing
// and a final CTA per row runs an exact radix select over the 64-bit keys in
// shared memory and writes the survivors' positions, slots or pool blocks in
// ascending order (the compactions keep element order, so no sort is needed).
// Rows of at most kDirect elements are selected by the final CTA directly; a
// row whose candidate list overflowed (massive ties near the threshold) is
// selected by the final CTA streaming the row from global memory, still exact.
#include <math.h>

#include "csa2_device.cuh"
#include "csa2_internal.h"

namespace csa2 {

namespace {

constexpr int kBins = 2048;
constexpr int kCap = 16384;      // candidates of a row the final CTA holds in shared memory
// Candidates stored per filter CTA of 4096 elements (a larger count flags an
// overflow and sends the row to the streaming path).  A quarter of the chunk:
// block-maximum rows are narrow, and with 512 the pool rows of 32,768 blocks in
// the 38-layer decode step overflowed (623 candidates in one chunk).
constexpr int kRegion = 1024;
constexpr int kDirect = 16384;   // rows up to this length are selected in shared memory directly
constexpr int kChunk = 16384;    // elements per hist CTA (4x that when the rows make many waves of CTAs)
constexpr int kMaxK = 2048;
constexpr int kStreamThreads = 256;
constexpr int kFilterPer = 16;                             // elements per thread in the filter pass
constexpr int kFilterChunk = kStreamThreads * kFilterPer;  // elements per filter CTA
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
  uint32_t* hist;        // [V][kBins]: given, or built by the hist pass in `hist_ws`
  int order;             // 0: ascending positions, 1: best first (score desc, index asc)
  int hist_full;         // hist covers every row (given by the caller), not only the long ones;
                         // the final pass returns the caller's rows to zero after reading them
  uint32_t* hist_ws;
  uint32_t* hist_done;   // [V]: hist CTAs finished per row (zeroed with hist_ws), or null
  int* thr;              // [V]: threshold bin of each row found by its last hist CTA (-1: take all), or null
  uint32_t* cnt;         // [V][nchunks]: candidates found by each filter CTA (may exceed kRegion)
  uint2* cand;           // [V][nchunks][kRegion]: (key, index) of each filter CTA's candidates
  int nchunks;           // filter chunks of 4096 elements per row
  int filter_cpc;        // chunks per filter CTA
  int hist_chunk;        // elements per hist CTA
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
// As stage_hist, and sets the global histogram back to zero (the caller's
// histogram, read by nothing after the final pass).
__device__ __forceinline__ void stage_hist_clear(uint32_t* dst, uint32_t* src) {
  uint4* s4 = reinterpret_cast<uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (int i = threadIdx.x; i < kBins / 4; i += blockDim.x) {
    d4[i] = s4[i];
    s4[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Exclusive block-wide prefix sum of x (every thread calls); *total gets the sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t x, uint32_t* wsum, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const uint32_t incl = warp_incl_scan(x);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = (lane < nwarps) ? wsum[lane] : 0u;
    const uint32_t ws = warp_incl_scan(w);
    __syncwarp();
    wsum[lane] = ws;
  }
  __syncthreads();
  const uint32_t base = warp ? wsum[warp - 1] : 0u;
  *total = wsum[nwarps - 1];
  __syncthreads();  // wsum is reused by the next scan
  return base + incl - x;
}

// ---------------------------------------------------------------- streaming passes
__global__ void __launch_bounds__(kStreamThreads) sel_hist_kernel(const __grid_constant__ SelParams P) {
  pdl_wait();
  pdl_trigger();
  const int v = blockIdx.y;
  const VRow r = vrow_of(P, v);
  if (r.n <= kDirect) return;
  const int chunk = P.hist_chunk;
  const int i0 = blockIdx.x * chunk;
  if (i0 >= r.n) return;
  __shared__ uint32_t h[kBins];
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int i1 = min(i0 + chunk, r.n);
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
  // The row's last CTA to finish searches the complete histogram once for the
  // threshold bin, so that the filter CTAs read one word instead of each
  // searching the 8-KB histogram (the usual last-block pattern: each CTA's
  // additions are fenced before it counts itself done).
  __shared__ int last;
  __shared__ int res[4];
  __shared__ uint32_t wsum[32];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned nblk = static_cast<unsigned>((r.n + chunk - 1) / chunk);
    last = atomicAdd(P.hist_done + v, 1u) == nblk - 1;
    res[0] = -1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = __ldcg(gh + i);
  __syncthreads();
  block_find_bin(h, static_cast<uint32_t>(r.k), res, wsum);
  if (threadIdx.x == 0) P.thr[v] = res[0];
}

__global__ void __launch_bounds__(kStreamThreads) sel_filter_kernel(const __grid_constant__ SelParams P) {
  pdl_wait();
  pdl_trigger();
  const int v = blockIdx.y;
  const VRow r = vrow_of(P, v);
  if (r.n <= kDirect) return;
  // chunks filter_cpc * blockIdx.x .. of 4096 elements, one after the other
  // (several per CTA only when the rows x chunks make many waves of CTAs)
  const int ch0 = blockIdx.x * P.filter_cpc;
  if (ch0 * kFilterChunk >= r.n) return;
  const int ch1 = min(ch0 + P.filter_cpc, (r.n + kFilterChunk - 1) / kFilterChunk);
  __shared__ __align__(16) uint32_t h[kBins];
  __shared__ int res[4];
  __shared__ uint32_t wsum[32];
  // this thread's kFilterPer consecutive elements of chunk ch
  float vals[kFilterPer];
  auto load_chunk = [&](int ch) {
    const int i = ch * kFilterChunk + threadIdx.x * kFilterPer;
    const int i1 = min(ch * kFilterChunk + kFilterChunk, r.n);
#pragma unroll
    for (int q = 0; q < kFilterPer / 4; ++q) {
      const int e = i + 4 * q;
      float4 v4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      if (e + 3 < i1) {
        v4 = *reinterpret_cast<const float4*>(r.src + e);
      } else if (e < i1) {
        v4.x = r.src[e];
        if (e + 1 < i1) v4.y = r.src[e + 1];
        if (e + 2 < i1) v4.z = r.src[e + 2];
      }
      vals[4 * q] = v4.x;
      vals[4 * q + 1] = v4.y;
      vals[4 * q + 2] = v4.z;
      vals[4 * q + 3] = v4.w;
    }
  };
  // the first chunk's elements are requested before the threshold, so that
  // the two latencies overlap
  load_chunk(ch0);
  int b1;
  if (P.thr) {  // found once per row by the hist pass
    b1 = __ldcg(P.thr + v);
  } else {
    stage_hist(h, P.hist + static_cast<long long>(v) * kBins);
    if (threadIdx.x == 0) res[0] = -1;
    __syncthreads();
    block_find_bin(h, static_cast<uint32_t>(r.k), res, wsum);
    b1 = res[0];
  }
  const uint32_t thr = b1 < 0 ? 0u : static_cast<uint32_t>(b1);
  for (int ch = ch0; ch < ch1; ++ch) {
    const int i = ch * kFilterChunk + threadIdx.x * kFilterPer;
    const int i1 = min(ch * kFilterChunk + kFilterChunk, r.n);
    uint32_t keys[kFilterPer];
    uint32_t mine = 0;
#pragma unroll
    for (int j = 0; j < kFilterPer; ++j) {
      const uint32_t key = (i + j < i1) ? elem_key(r, vals[j], i + j) : 0u;
      keys[j] = (key && (key >> 21) >= thr) ? key : 0u;
      mine += keys[j] ? 1u : 0u;
    }
    if (ch + 1 < ch1) load_chunk(ch + 1);  // in flight during this chunk's compaction
    // the chunk's own region, in element order (each thread holds consecutive
    // elements; a block prefix sum places them), and its true count: no
    // counter shared across CTAs, nothing to zero
    uint32_t total;
    uint32_t slot = block_excl_scan(mine, wsum, &total);
    uint2* cand = P.cand + (static_cast<long long>(v) * P.nchunks + ch) * kRegion;
#pragma unroll
    for (int j = 0; j < kFilterPer; ++j) {
      if (!keys[j]) continue;
      if (slot < static_cast<uint32_t>(kRegion)) cand[slot] = make_uint2(keys[j], static_cast<uint32_t>(i + j));
      ++slot;
    }
    if (threadIdx.x == 0) P.cnt[static_cast<long long>(v) * P.nchunks + ch] = total;
  }
}

// ---------------------------------------------------------------- final select
constexpr int kPerThread = kDirect / kFinalThreads;  // direct-row values held in registers per thread
constexpr int kMaxChunks = kMaxK;                    // filter CTAs per row the final CTA can gather (counts + offsets in sel)

struct FinalSmem {
  uint32_t* ord;      // [kDirect] candidate keys (score part)
  uint32_t* idx;      // [kDirect] candidate element indices
  uint64_t* sel;      // [kMaxK] survivors
  uint64_t* xchg;     // [kMaxK] second buffer of the merge sort
  uint32_t* hist;     // [kBins]
  int* res;           // [8]
  uint32_t* wsum;     // [32]
  uint32_t* counters; // [4]: [0] candidates, [1] survivors
};

__device__ __forceinline__ FinalSmem final_smem(uint8_t* base) {
  FinalSmem sm;
  sm.ord = reinterpret_cast<uint32_t*>(base);
  sm.idx = sm.ord + kDirect;
  sm.sel = reinterpret_cast<uint64_t*>(sm.idx + kDirect);
  sm.xchg = sm.sel + kMaxK;
  sm.hist = reinterpret_cast<uint32_t*>(sm.xchg + kMaxK);
  sm.res = reinterpret_cast<int*>(sm.hist + kBins);
  sm.wsum = reinterpret_cast<uint32_t*>(sm.res + 8);
  sm.counters = sm.wsum + 32;
  return sm;
}

__device__ __forceinline__ uint64_t key64(uint32_t ord, uint32_t idx) {
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint64_t>(~idx);
}

__device__ __forceinline__ void hist_add(uint32_t* h, bool on, uint32_t bin) {
  if (on) atomicAdd(h + bin, 1u);
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

// Radix refinement below a known prefix: the candidates sm.ord/idx[0..n) whose
// key starts with *prefix (of *pbits bits) are narrowed digit by digit (11, 10,
// 11, 11, 10 bits: the rest of the score, then ~index) until the threshold
// digit's bin is needed whole.  On return the keys whose top *pbits bits are
// >= *prefix are exactly the `need` best plus those above the entry prefix.
__device__ void radix_refine(const FinalSmem& sm, int n, int need, uint64_t* prefix_io, int* pbits_io) {
  uint64_t prefix = *prefix_io;
  int pbits = *pbits_io;
  const int nr = (n + blockDim.x - 1) / blockDim.x * blockDim.x;
  while (pbits < 64) {
    const int width = (pbits == 22 || pbits == 54) ? 10 : 11;
    const int shift = 64 - pbits - width;
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) sm.hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < nr; i += blockDim.x) {
      bool on = false;
      uint32_t bin = 0;
      if (i < n) {
        const uint64_t kk = key64(sm.ord[i], sm.idx[i]);
        on = (kk >> (64 - pbits)) == prefix;
        bin = static_cast<uint32_t>(kk >> shift) & ((1u << width) - 1u);
      }
      hist_add(sm.hist, on, bin);
    }
    __syncthreads();
    block_find_bin(sm.hist, static_cast<uint32_t>(need), sm.res, sm.wsum);
    const int d = sm.res[0];
    const int above = sm.res[1];
    const int cnt = static_cast<int>(sm.hist[d]);
    __syncthreads();  // res and hist are rewritten by the next digit
    need -= above;
    prefix = (prefix << width) | static_cast<uint32_t>(d);
    pbits += width;
    if (cnt == need) break;
  }
  *prefix_io = prefix;
  *pbits_io = pbits;
}

// Exact radix select streaming the row from global memory each pass (rows
// whose candidate list overflowed), 8-bit digits of the 64-bit keys.
__device__ void radix_select_stream(const VRow& r, const FinalSmem& sm, int need, uint64_t* prefix_out,
                                    int* pbits_out) {
  uint64_t prefix = 0;
  int pbits = 0;
  const int lane = threadIdx.x & 31;
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) sm.hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < r.n; i += blockDim.x) {
      const uint32_t o = elem_key(r, r.src[i], i);
      const uint64_t kk = key64(o, static_cast<uint32_t>(i));
      if (o != 0u && (pbits == 0 || (kk >> (64 - pbits)) == prefix))
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

// Descending sort of sel[0..got), got <= kMaxK: warps sort runs of 32 keys with
// shuffles, then runs are merged pairwise, each key placed by a binary search in
// the partner run (ties keep the left run first, so equal padding keys stay a
// permutation).  The result is back in sel.
__device__ void sort_desc(const FinalSmem& sm, int got) {
  int P2 = 32, lgP = 5;
  while (P2 < got) {
    P2 <<= 1;
    ++lgP;
  }
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  uint64_t* A = sm.sel;
  uint64_t* B = sm.xchg;
  for (int run = warp; run < (P2 >> 5); run += nwarps) {
    const int e = (run << 5) + lane;
    uint64_t x = e < got ? A[e] : 0ull;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const uint64_t y = __shfl_xor_sync(0xffffffffu, x, stride);
        const bool lower = (lane & stride) == 0;
        const bool asc = (lane & size) != 0;
        x = (lower == asc) ? (x < y ? x : y) : (x > y ? x : y);
      }
    }
    A[e] = x;
  }
  __syncthreads();
  for (int lg = 5; lg < lgP; ++lg) {
    const int L = 1 << lg;
    for (int i = tid; i < P2; i += blockDim.x) {
      const uint64_t key = A[i];
      const int run = i >> lg, off = i & (L - 1);
      const bool left = (run & 1) == 0;
      const uint64_t* pr = A + ((run ^ 1) << lg);
      // number of partner keys placed before this one: a prefix of the run
      int pos = 0;
      for (int step = L >> 1; step > 0; step >>= 1) {
        const uint64_t m = pr[pos + step - 1];
        if (left ? (m > key) : (m >= key)) pos += step;
      }
      {
        const uint64_t m = pr[pos];
        if (left ? (m > key) : (m >= key)) ++pos;
      }
      B[((run & ~1) << lg) + off + pos] = key;
    }
    __syncthreads();
    uint64_t* t = A;
    A = B;
    B = t;
  }
  if (A != sm.sel) {
    for (int i = tid; i < got; i += blockDim.x) sm.sel[i] = A[i];
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kFinalThreads, 1) sel_final_kernel(const __grid_constant__ SelParams P) {
  extern __shared__ __align__(16) uint8_t fsm_raw[];
  const FinalSmem sm = final_smem(fsm_raw);
  pdl_wait();
  pdl_trigger();
  const int v = blockIdx.x;
  const VRow r = vrow_of(P, v);
  const int tid = threadIdx.x;
  if (tid < 4) sm.counters[tid] = 0;
  if (P.hist_full && P.kind == 0 && P.pool_out == nullptr) {
    // the scan's block-maximum histogram of this row has no pool row to read it
    uint4* hb = reinterpret_cast<uint4*>(P.hist + (static_cast<long long>(P.rows.T) + v) * kBins);
    for (int i = tid; i < kBins / 4; i += blockDim.x) hb[i] = make_uint4(0u, 0u, 0u, 0u);
  }

  // 1. the 2048-bin histogram of the top 11 key bits: the caller's (the
  //    scan's) or the hist pass's, else built here from the values of a short
  //    row (kept in registers)
  int mode;  // 0: short row, 1: candidate list, 2: overflowed candidate list (stream the row)
  uint32_t ord[kPerThread];  // direct rows: elements e0 .. e0 + kPerThread - 1 of this thread
  const int e0 = tid * kPerThread;
  if (r.n <= kDirect) {
    mode = 0;
    float val[kPerThread];
#pragma unroll
    for (int q = 0; q < kPerThread / 4; ++q) {
      const int e = e0 + 4 * q;
      float4 v4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      if (e + 3 < r.n) {
        v4 = *reinterpret_cast<const float4*>(r.src + e);
      } else if (e < r.n) {
        v4.x = r.src[e];
        if (e + 1 < r.n) v4.y = r.src[e + 1];
        if (e + 2 < r.n) v4.z = r.src[e + 2];
      }
      val[4 * q] = v4.x;
      val[4 * q + 1] = v4.y;
      val[4 * q + 2] = v4.z;
      val[4 * q + 3] = v4.w;
    }
    if (P.hist_full) {
      stage_hist_clear(sm.hist, P.hist + static_cast<long long>(v) * kBins);
    } else {
      for (int i = tid; i < kBins; i += blockDim.x) sm.hist[i] = 0;
    }
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) ord[j] = (e0 + j < r.n) ? elem_key(r, val[j], e0 + j) : 0u;
    if (!P.hist_full) {
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kPerThread; ++j) hist_add(sm.hist, ord[j] != 0u, ord[j] >> 21);
    }
  } else {
    // the per-CTA candidate counts of the filter pass (over the sel area, free until the collect)
    const int nch = (r.n + kFilterChunk - 1) / kFilterChunk;
    uint32_t* scnt = reinterpret_cast<uint32_t*>(sm.sel);  // [kMaxChunks] counts, then offsets
    mode = (nch <= kMaxChunks) ? 1 : 2;
    if (mode == 1)
      for (int i = tid; i < nch; i += blockDim.x) scnt[i] = P.cnt[static_cast<long long>(v) * P.nchunks + i];
    if (P.hist_full) stage_hist_clear(sm.hist, P.hist + static_cast<long long>(v) * kBins);
    else stage_hist(sm.hist, P.hist + static_cast<long long>(v) * kBins);
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) ord[j] = 0u;
  }
  __syncthreads();
  block_find_bin(sm.hist, static_cast<uint32_t>(r.k), sm.res, sm.wsum);
  const int b1 = sm.res[0];
  const int above1 = sm.res[1];
  const int total = sm.res[2];
  const int cnt1 = b1 >= 0 ? static_cast<int>(sm.hist[b1]) : 0;
  const uint32_t thr = b1 >= 0 ? static_cast<uint32_t>(b1) : 0u;
  const bool take_all = total <= r.k;
  __syncthreads();

  // 2. the candidates in shared memory: keys whose top 11 bits reach the threshold bin
  int n = 0;
  if (mode == 0) {
    uint32_t tmask = 0, mine = 0;
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      if (ord[j] != 0u && (ord[j] >> 21) >= thr) {
        tmask |= 1u << j;
        ++mine;
      }
    }
    uint32_t total_c;
    uint32_t slot = block_excl_scan(mine, sm.wsum, &total_c);  // candidates stay in element order
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      if ((tmask >> j) & 1u) {
        sm.ord[slot] = ord[j];
        sm.idx[slot] = static_cast<uint32_t>(e0 + j);
        ++slot;
      }
    }
    n = static_cast<int>(total_c);
    __syncthreads();
  } else if (mode == 1) {
    // concatenate the filter CTAs' regions: offsets by a block prefix sum (two
    // chunks per thread); an overflowed region or list falls back to streaming
    const int nch = (r.n + kFilterChunk - 1) / kFilterChunk;
    uint32_t* scnt = reinterpret_cast<uint32_t*>(sm.sel);
    uint32_t* soff = scnt + kMaxChunks;
    const int c0 = 2 * tid;
    const uint32_t x0 = (c0 < nch) ? scnt[c0] : 0u, x1 = (c0 + 1 < nch) ? scnt[c0 + 1] : 0u;
    const bool over = x0 > static_cast<uint32_t>(kRegion) || x1 > static_cast<uint32_t>(kRegion);
    uint32_t total_c;
    const uint32_t off = block_excl_scan(x0 + x1, sm.wsum, &total_c);
    if (c0 < nch) soff[c0] = off;
    if (c0 + 1 < nch) soff[c0 + 1] = off + x0;
    const bool any_over = __syncthreads_or(over) != 0;
    if (any_over || total_c > static_cast<uint32_t>(kCap)) {
      mode = 2;
    } else {
      const int lane = tid & 31, warp = tid >> 5;
      for (int ch = warp; ch < nch; ch += blockDim.x >> 5) {
        const int nc = static_cast<int>(scnt[ch]);
        const int o0 = static_cast<int>(soff[ch]);
        const uint2* src = P.cand + (static_cast<long long>(v) * P.nchunks + ch) * kRegion;
        for (int i = lane; i < nc; i += 32) {
          const uint2 e = src[i];
          sm.ord[o0 + i] = e.x;
          sm.idx[o0 + i] = e.y;
        }
      }
      n = static_cast<int>(total_c);
    }
    __syncthreads();
  }

  // 3. the exact threshold over the 64-bit keys
  uint64_t prefix = thr;
  int pbits = 11;
  if (!take_all) {
    if (mode == 2) {
      radix_select_stream(r, sm, r.k, &prefix, &pbits);
    } else if (cnt1 != r.k - above1) {
      radix_refine(sm, n, r.k - above1, &prefix, &pbits);
    }
  }

  // 4. collect the survivors (exactly min(k, selectable) of them) in element
  //    order.  Candidates i = j * blockDim + tid form rounds j; a survivor's
  //    place is the count of survivors in earlier rounds plus earlier warps of
  //    its round (one prefix over [round][warp]) plus earlier lanes (ballot).
  if (mode != 2) {
    const int nper = (n + blockDim.x - 1) / blockDim.x;  // <= kPerThread
    const int lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    uint32_t* wcnt = sm.hist;  // [kPerThread][32] survivors per round and warp, then their prefix
    uint32_t tmask = 0;
    for (int j = 0; j < nper; ++j) {
      const int i = j * blockDim.x + tid;
      const bool take = i < n && (take_all || (key64(sm.ord[i], sm.idx[i]) >> (64 - pbits)) >= prefix);
      const unsigned m = __ballot_sync(0xffffffffu, take);
      if (take) tmask |= 1u << j;
      if (lane == 0) wcnt[j * 32 + warp] = __popc(m);
    }
    __syncthreads();
    if (warp == 0) {  // exclusive prefix over the nper x nwarps counts, 16 per lane
      const int cells = nper * 32;
      const int per = (cells + 31) / 32;
      uint32_t loc[16];
      uint32_t sum = 0;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int cidx = lane * per + u;
        loc[u] = (u < per && cidx < cells && (cidx & 31) < nwarps) ? wcnt[cidx] : 0u;
        sum += loc[u];
      }
      const uint32_t incl = warp_incl_scan(sum);
      uint32_t run = incl - sum;
      __syncwarp();
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int cidx = lane * per + u;
        if (u < per && cidx < cells) wcnt[cidx] = run;
        run += loc[u];
      }
      if (lane == 31) sm.counters[1] = incl;
    }
    __syncthreads();
    for (int j = 0; j < nper; ++j) {
      const bool take = (tmask >> j) & 1u;
      const unsigned m = __ballot_sync(0xffffffffu, take);
      if (take) {
        const uint32_t place = wcnt[j * 32 + warp] + __popc(m & ((1u << lane) - 1u));
        if (place < static_cast<uint32_t>(kMaxK)) sm.sel[place] = sm.idx[j * blockDim.x + tid];
      }
    }
  } else {
    const int nr = (r.n + blockDim.x - 1) / blockDim.x * blockDim.x;
    for (int i = tid; i < nr; i += blockDim.x) {
      uint64_t kk = 0;
      bool valid = false;
      if (i < r.n) {
        const uint32_t o = elem_key(r, r.src[i], i);
        valid = o != 0u;
        kk = key64(o, static_cast<uint32_t>(i));
      }
      const bool take = valid && (take_all || (kk >> (64 - pbits)) >= prefix);
      const uint32_t slot = block_append(take, &sm.counters[1]);
      // ~index: the descending sort below then leaves ascending indices
      if (take && slot < static_cast<uint32_t>(kMaxK)) sm.sel[slot] = static_cast<uint64_t>(~static_cast<uint32_t>(i));
    }
  }
  __syncthreads();
  const int got = min(static_cast<int>(sm.counters[1]), kMaxK);
  if (mode == 2) {  // streamed survivors arrive in no particular order
    sort_desc(sm, got);
    for (int i = tid; i < got; i += blockDim.x) sm.sel[i] = ~static_cast<uint32_t>(sm.sel[i]);
    __syncthreads();
  }

  // best first: the survivors' 64-bit keys sorted descending (ties of the
  // score go to the lower index through ~index in the low word)
  if (P.order == 1 && !r.pool) {
    for (int i = tid; i < got; i += blockDim.x) {
      const uint32_t id = static_cast<uint32_t>(sm.sel[i]);
      sm.sel[i] = key64(elem_key(r, r.src[id], static_cast<int>(id)), id);
    }
    __syncthreads();
    sort_desc(sm, got);
    for (int i = tid; i < got; i += blockDim.x) sm.sel[i] = ~static_cast<uint32_t>(sm.sel[i]);
    __syncthreads();
  }

  // 5. write: sel holds the survivors' element indices in ascending order (or best first)
  const int t = r.t;
  const int b = row_seq_of(P.rows, t);
  if (r.pool) {
    int* out = P.pool_out + static_cast<long long>(t) * P.pool_n;
    for (int i = tid; i < P.pool_n; i += blockDim.x) out[i] = (i < got) ? static_cast<int>(sm.sel[i]) : -1;
    return;
  }
  int* opos = P.topk_pos + static_cast<long long>(t) * P.ld_topk;
  int* oslot = P.topk_slot ? P.topk_slot + static_cast<long long>(t) * P.ld_topk : nullptr;
  for (int i = tid; i < r.k; i += blockDim.x) {
    int pos = -1;
    if (i < got) {
      const uint32_t id = static_cast<uint32_t>(sm.sel[i]);
      if (P.kind == 2) {
        const int blk = P.pool_in[static_cast<long long>(t) * P.pool_in_n + (id >> 3)];
        pos = blk * 8 + static_cast<int>(id & 7);
      } else {
        pos = static_cast<int>(id);
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
  return static_cast<size_t>(2 * kDirect) * 4 + 2 * kMaxK * 8 + kBins * 4 + 8 * 4 + 32 * 4 + 4 * 4;
}

}  // namespace

// Workspace of rows longer than kDirect: [histograms, unless given][per-CTA
// candidate counts][per-CTA candidate regions]
static long long select_maxn(const SelectLaunch& a) {
  if (a.kind != 0) return 0;  // Reindex rows are short enough for the direct path
  long long maxn = a.ld_scores;
  if (a.pool_out) maxn = maxn > a.ld_bm ? maxn : a.ld_bm;
  return maxn;
}
static size_t select_cnt_bytes(long long V, long long nch) {
  return (static_cast<size_t>(V) * nch * 4 + 255) & ~size_t(255);
}
// the hist pass's per-row words: a done count and the threshold bin
static size_t select_row_words_bytes(long long V) { return (static_cast<size_t>(V) * 8 + 255) & ~size_t(255); }

size_t select_workspace_bytes(const SelectLaunch& a) {
  const long long maxn = select_maxn(a);
  if (maxn <= kDirect) return 0;
  const long long V = static_cast<long long>(a.rows.T) * (a.pool_out ? 2 : 1);
  const long long nch = (maxn + kFilterChunk - 1) / kFilterChunk;
  const size_t hist = a.hist ? 0 : static_cast<size_t>(V) * kBins * 4 + select_row_words_bytes(V);
  return hist + select_cnt_bytes(V, nch) + static_cast<size_t>(V) * nch * kRegion * 8;
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
  P.order = a.order;
  P.err = ctx.err;
  const int V = a.rows.T * ((a.kind == 0 && a.pool_out) ? 2 : 1);
  P.hist = a.hist;
  P.hist_full = a.hist != nullptr;
  P.hist_ws = nullptr;
  P.hist_done = nullptr;
  P.thr = nullptr;
  P.cnt = nullptr;
  P.cand = nullptr;
  P.nchunks = 0;
  P.filter_cpc = 1;
  P.hist_chunk = kChunk;
  cudaError_t e;
  const long long maxn = select_maxn(a);
  if (maxn > kDirect) {
    const long long nch = (maxn + kFilterChunk - 1) / kFilterChunk;
    uint8_t* w = static_cast<uint8_t*>(ws);
    if (!a.hist) {
      P.hist_ws = reinterpret_cast<uint32_t*>(w);
      P.hist = P.hist_ws;
      w += static_cast<size_t>(V) * kBins * 4;
      P.hist_done = reinterpret_cast<uint32_t*>(w);
      P.thr = reinterpret_cast<int*>(w + static_cast<size_t>(V) * 4);
      w += select_row_words_bytes(V);
      // the histogram pass accumulates and counts its CTAs: zero both (the
      // only memset; given histograms need none)
      e = cudaMemsetAsync(P.hist_ws, 0, static_cast<size_t>(V) * kBins * 4 + select_row_words_bytes(V), st);
      if (e != cudaSuccess) return e;
    }
    P.cnt = reinterpret_cast<uint32_t*>(w);
    P.cand = reinterpret_cast<uint2*>(w + select_cnt_bytes(V, nch));
    P.nchunks = static_cast<int>(nch);
    // one filter chunk per CTA while the rows' chunks make at most 8 waves of
    // CTAs (decode), else up to 8 chunks per CTA, which spreads the CTA's
    // setup (row, threshold) and overlaps a chunk's loads with the previous
    // chunk's compaction (prefill: thousands of rows)
    const long long wave = static_cast<long long>(ctx.num_sms) * 4;  // 256-thread CTAs at 64 registers: 4 an SM
    const long long fct = static_cast<long long>(V) * nch;
    long long cpc = fct > 8 * wave ? (fct + 4 * wave - 1) / (4 * wave) : 1;
    cpc = cpc < 1 ? 1 : (cpc > 8 ? 8 : cpc);
    P.filter_cpc = static_cast<int>(cpc);
    // hist CTAs: 4x the elements each when the rows make more than 8 waves of
    // them (fewer CTAs to zero and add in a histogram; measured 1.41 -> 1.37 ms
    // for the 4,096-row prefill top-k)
    if (static_cast<long long>(V) * ((maxn + kChunk - 1) / kChunk) > 8 * wave) P.hist_chunk = 4 * kChunk;
    const dim3 grid(static_cast<unsigned>((maxn + P.hist_chunk - 1) / P.hist_chunk), static_cast<unsigned>(V));
    const dim3 fgrid(static_cast<unsigned>((nch + cpc - 1) / cpc), static_cast<unsigned>(V));
    if ((e = prefer_max_smem(sel_hist_kernel, 0)) != cudaSuccess) return e;
    if ((e = prefer_max_smem(sel_filter_kernel, 0)) != cudaSuccess) return e;
    if (!a.hist && (e = launch_pdl(sel_hist_kernel, grid, dim3(kStreamThreads), 0, st, P)) != cudaSuccess) return e;
    if ((e = launch_pdl(sel_filter_kernel, fgrid, dim3(kStreamThreads), 0, st, P)) != cudaSuccess) return e;
  }
  const size_t smem = final_smem_bytes();
  e = prefer_max_smem(sel_final_kernel, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(sel_final_kernel, dim3(V), dim3(kFinalThreads), smem, st, P);
}

}  // namespace csa2
