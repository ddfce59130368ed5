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
// k largest keys are exactly the k best (score desc, index asc).  Long rows go
// through three streaming passes over L2-resident scores, many CTAs per row:
//   hist   : 2048-bin histogram of the top 11 key bits
//   refine : (only if the threshold bin is crowded) histogram of the next 11
//            bits inside that bin
//   filter : append every element at or above the threshold prefix to a
//            per-row candidate list (at most kCap)
// and a final per-row CTA runs an exact radix select over 64-bit keys in shared
// memory, sorts the survivors and writes positions, slots or pool blocks.
// Rows of at most kDirect elements skip the streaming passes; a row whose
// candidate list overflowed (massive ties) is selected by the final CTA
// streaming the row from global memory, which stays exact.
#include <math.h>

#include "csa2_device.cuh"
#include "csa2_internal.h"

namespace csa2 {

namespace {

constexpr int kBins = 2048;
constexpr int kCap = 4096;       // candidate list per row
constexpr int kDirect = 16384;   // rows up to this length are selected in shared memory directly
constexpr int kChunk = 8192;     // elements per CTA in the streaming passes
constexpr int kMaxK = 2048;

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
  int n_vrows;
  uint32_t* hist1;   // [V][kBins]
  uint32_t* hist2;   // [V][kBins]
  uint32_t* cnt;     // [V]
  uint32_t* cord;    // [V][kCap]
  uint32_t* cidx;    // [V][kCap]
  uint32_t* err;
};

struct VRow {
  const float* src;
  int n;
  int k;
  bool force_last;  // pool rows: the newest block is always kept
  bool pool;        // output is a pool (ascending ids)
  int t;
};

__device__ __forceinline__ VRow vrow_of(const SelParams& P, int v) {
  VRow r;
  const int T = P.rows.T;
  r.t = v % T;
  r.pool = (P.kind == 0 && v >= T);
  r.force_last = r.pool;
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
  if (r.force_last && i == r.n - 1) return 0xFFFFFFFFu;
  return selectable(val) ? ord_key(val) : 0u;
}

// Find the bin b such that count(bins > b) < need <= count(bins >= b), by one
// warp over a 2048-bin histogram in global memory.  Returns b (or -1 when the
// histogram holds fewer than need elements) and the count above b; *total gets
// the histogram total.
__device__ int find_bin_warp(const uint32_t* h, int need, uint32_t* above_out, uint32_t* total_out) {
  const int lane = threadIdx.x & 31;
  // lane l covers bins [2047 - 64 l - 63, 2047 - 64 l], walked from the top
  uint32_t sum = 0;
  for (int j = 0; j < 64; ++j) sum += h[kBins - 1 - (lane * 64 + j)];
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
  *total_out = total;
  if (total < static_cast<uint32_t>(need)) {
    *above_out = total;
    return -1;
  }
  const uint32_t excl = incl - sum;
  const unsigned hit = __ballot_sync(0xffffffffu, excl < static_cast<uint32_t>(need) && incl >= static_cast<uint32_t>(need));
  const int src = __ffs(hit) - 1;
  int bin = -1;
  uint32_t above = 0;
  if (lane == src) {
    uint32_t run = excl;
    for (int j = 0; j < 64; ++j) {
      const int bb = kBins - 1 - (lane * 64 + j);
      const uint32_t c = h[bb];
      if (run + c >= static_cast<uint32_t>(need)) {
        bin = bb;
        above = run;
        break;
      }
      run += c;
    }
  }
  bin = __shfl_sync(0xffffffffu, bin, src);
  above = __shfl_sync(0xffffffffu, above, src);
  *above_out = above;
  return bin;
}

// Threshold of a row computed from its histograms: an element is a candidate
// iff (key >> shift) >= thr.  shift == 32 means "every selectable element".
struct Thresh {
  int shift;
  uint32_t thr;
};

__device__ Thresh row_threshold(const SelParams& P, int v, int k, bool* need_refine) {
  uint32_t above1, total;
  const uint32_t* h1 = P.hist1 + static_cast<long long>(v) * kBins;
  const int b1 = find_bin_warp(h1, k, &above1, &total);
  Thresh th{32, 0};
  *need_refine = false;
  if (b1 < 0) return th;
  const uint32_t c1 = h1[b1];
  if (above1 + c1 <= static_cast<uint32_t>(kCap)) {
    th.shift = 21;
    th.thr = static_cast<uint32_t>(b1);
    return th;
  }
  *need_refine = true;
  th.shift = 21;
  th.thr = static_cast<uint32_t>(b1);
  return th;
}

__global__ void __launch_bounds__(256) sel_hist1_kernel(const __grid_constant__ SelParams P) {
  const int v = blockIdx.y;
  const VRow r = vrow_of(P, v);
  if (r.n <= kDirect) return;
  const int i0 = blockIdx.x * kChunk;
  if (i0 >= r.n) return;
  __shared__ uint32_t h[kBins];
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int i1 = min(i0 + kChunk, r.n);
  for (int base = i0; base < i1; base += blockDim.x * 4) {
    const int i = base + threadIdx.x * 4;
    float4 v4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (i + 3 < i1) {
      v4 = __ldg(reinterpret_cast<const float4*>(r.src + i));
    } else {
      if (i < i1) v4.x = r.src[i];
      if (i + 1 < i1) v4.y = r.src[i + 1];
      if (i + 2 < i1) v4.z = r.src[i + 2];
    }
    const float vals[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t key = (i + j < i1) ? elem_key(r, vals[j], i + j) : 0u;
      const uint32_t bin = key ? (key >> 21) : 0xFFFFFFFFu;
      const unsigned grp = __match_any_sync(0xffffffffu, bin);
      if (key && (threadIdx.x & 31) == __ffs(grp) - 1) atomicAdd(&h[bin], __popc(grp));
    }
  }
  __syncthreads();
  uint32_t* gh = P.hist1 + static_cast<long long>(v) * kBins;
  for (int i = threadIdx.x; i < kBins; i += blockDim.x)
    if (h[i]) atomicAdd(gh + i, h[i]);
}

__global__ void __launch_bounds__(256) sel_refine_kernel(const __grid_constant__ SelParams P) {
  const int v = blockIdx.y;
  const VRow r = vrow_of(P, v);
  if (r.n <= kDirect) return;
  const int i0 = blockIdx.x * kChunk;
  if (i0 >= r.n) return;
  __shared__ uint32_t h[kBins];
  __shared__ int s_b1;
  __shared__ int s_refine;
  if (threadIdx.x < 32) {
    bool refine;
    const Thresh th = row_threshold(P, v, r.k, &refine);
    if (threadIdx.x == 0) {
      s_b1 = static_cast<int>(th.thr);
      s_refine = refine ? 1 : 0;
    }
  }
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
  __syncthreads();
  if (!s_refine) return;
  const uint32_t b1 = static_cast<uint32_t>(s_b1);
  const int i1 = min(i0 + kChunk, r.n);
  for (int base = i0; base < i1; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const uint32_t key = (i < i1) ? elem_key(r, r.src[i], i) : 0u;
    const bool in = key && (key >> 21) == b1;
    const uint32_t bin = in ? ((key >> 10) & (kBins - 1)) : 0xFFFFFFFFu;
    const unsigned grp = __match_any_sync(0xffffffffu, bin);
    if (in && (threadIdx.x & 31) == __ffs(grp) - 1) atomicAdd(&h[bin], __popc(grp));
  }
  __syncthreads();
  uint32_t* gh = P.hist2 + static_cast<long long>(v) * kBins;
  for (int i = threadIdx.x; i < kBins; i += blockDim.x)
    if (h[i]) atomicAdd(gh + i, h[i]);
}

__global__ void __launch_bounds__(256) sel_filter_kernel(const __grid_constant__ SelParams P) {
  const int v = blockIdx.y;
  const VRow r = vrow_of(P, v);
  if (r.n <= kDirect) return;
  const int i0 = blockIdx.x * kChunk;
  if (i0 >= r.n) return;
  __shared__ int s_shift;
  __shared__ uint32_t s_thr;
  if (threadIdx.x < 32) {
    bool refine;
    Thresh th = row_threshold(P, v, r.k, &refine);
    if (refine) {
      const uint32_t* h1 = P.hist1 + static_cast<long long>(v) * kBins;
      uint32_t above1, total1;
      const int b1 = find_bin_warp(h1, r.k, &above1, &total1);
      uint32_t above2, total2;
      const int b2 = find_bin_warp(P.hist2 + static_cast<long long>(v) * kBins, r.k - static_cast<int>(above1),
                                   &above2, &total2);
      th.shift = 10;
      th.thr = (static_cast<uint32_t>(b1) << 11) | static_cast<uint32_t>(max(b2, 0));
    }
    if (threadIdx.x == 0) {
      s_shift = th.shift;
      s_thr = th.thr;
    }
  }
  __syncthreads();
  const int shift = s_shift;
  const uint32_t thr = s_thr;
  const int lane = threadIdx.x & 31;
  uint32_t* cord = P.cord + static_cast<long long>(v) * kCap;
  uint32_t* cidx = P.cidx + static_cast<long long>(v) * kCap;
  const int i1 = min(i0 + kChunk, r.n);
  for (int base = i0; base < i1; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const uint32_t key = (i < i1) ? elem_key(r, r.src[i], i) : 0u;
    const bool take = key && (shift >= 32 || (key >> shift) >= thr);
    const unsigned m = __ballot_sync(0xffffffffu, take);
    if (m == 0) continue;
    uint32_t basepos = 0;
    if (lane == __ffs(m) - 1) basepos = atomicAdd(P.cnt + v, __popc(m));
    basepos = __shfl_sync(0xffffffffu, basepos, __ffs(m) - 1);
    if (take) {
      const uint32_t slot = basepos + __popc(m & ((1u << lane) - 1u));
      if (slot < static_cast<uint32_t>(kCap)) {
        cord[slot] = key;
        cidx[slot] = static_cast<uint32_t>(i);
      }
    }
  }
}

// ---------------------------------------------------------------- final select
struct FinalSmem {
  uint32_t* ord;       // [kDirect]
  uint32_t* idx;       // [kDirect]
  uint64_t* sel;       // [kMaxK]
  uint32_t* hist;      // [256]
  uint32_t* misc;      // [8]
};

__device__ __forceinline__ uint64_t key64(uint32_t ord, uint32_t idx) {
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint64_t>(~idx);
}

// Exact radix select of the `need` largest 64-bit keys.  GLOBAL: elements are
// streamed from the row each pass; else they are the n entries of sm.ord/idx.
template <bool GLOBAL>
__device__ void radix_select(const VRow& r, const FinalSmem& sm, int n, int need, uint64_t* prefix_out,
                             int* pbits_out) {
  uint64_t prefix = 0;
  int pbits = 0;
  const int lane = threadIdx.x & 31;
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) sm.hist[i] = 0;
    __syncthreads();
    const int nloop = GLOBAL ? r.n : n;
    for (int base = 0; base < nloop; base += blockDim.x) {
      const int i = base + threadIdx.x;
      uint64_t kk = 0;
      bool valid = false;
      if (i < nloop) {
        if (GLOBAL) {
          const uint32_t o = elem_key(r, r.src[i], i);
          valid = o != 0u;
          kk = key64(o, static_cast<uint32_t>(i));
        } else {
          valid = true;
          kk = key64(sm.ord[i], sm.idx[i]);
        }
      }
      const bool in = valid && (pbits == 0 || (kk >> (64 - pbits)) == prefix);
      const uint32_t bin = in ? static_cast<uint32_t>((kk >> shift) & 0xFFu) : 0xFFFFFFFFu;
      const unsigned grp = __match_any_sync(0xffffffffu, bin);
      if (in && lane == __ffs(grp) - 1) atomicAdd(&sm.hist[bin], __popc(grp));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l covers digits [255 - 8 l - 7, 255 - 8 l]
      uint32_t sum = 0;
      for (int j = 0; j < 8; ++j) sum += sm.hist[255 - (lane * 8 + j)];
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t excl = incl - sum;
      const unsigned hit =
          __ballot_sync(0xffffffffu, excl < static_cast<uint32_t>(need) && incl >= static_cast<uint32_t>(need));
      const int src = __ffs(hit) - 1;
      if (lane == src) {
        uint32_t run = excl;
        for (int j = 0; j < 8; ++j) {
          const int d = 255 - (lane * 8 + j);
          const uint32_t c = sm.hist[d];
          if (run + c >= static_cast<uint32_t>(need)) {
            sm.misc[0] = static_cast<uint32_t>(d);
            sm.misc[1] = run;
            sm.misc[2] = c;
            break;
          }
          run += c;
        }
      }
    }
    __syncthreads();
    const uint32_t d = sm.misc[0];
    const uint32_t above = sm.misc[1];
    const uint32_t cnt = sm.misc[2];
    need -= static_cast<int>(above);
    prefix = (prefix << 8) | d;
    pbits += 8;
    __syncthreads();
    if (cnt == static_cast<uint32_t>(need)) break;
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

__global__ void __launch_bounds__(1024, 1) sel_final_kernel(const __grid_constant__ SelParams P) {
  extern __shared__ uint8_t fsm_raw[];
  FinalSmem sm;
  sm.ord = reinterpret_cast<uint32_t*>(fsm_raw);
  sm.idx = sm.ord + kDirect;
  sm.sel = reinterpret_cast<uint64_t*>(sm.idx + kDirect);
  sm.hist = reinterpret_cast<uint32_t*>(sm.sel + kMaxK);
  sm.misc = sm.hist + 256;
  const int v = blockIdx.x;
  const VRow r = vrow_of(P, v);
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) sm.misc[4] = 0;
  __syncthreads();

  // 1. gather the candidates (or decide to stream the row)
  int mode;  // 0: smem direct/candidates, 1: global stream
  int n = 0;
  if (r.n <= kDirect) {
    for (int base = 0; base < r.n; base += blockDim.x) {
      const int i = base + threadIdx.x;
      const uint32_t key = (i < r.n) ? elem_key(r, r.src[i], i) : 0u;
      const unsigned m = __ballot_sync(0xffffffffu, key != 0u);
      uint32_t b0 = 0;
      if (m && lane == __ffs(m) - 1) b0 = atomicAdd(&sm.misc[4], __popc(m));
      b0 = __shfl_sync(0xffffffffu, b0, m ? __ffs(m) - 1 : 0);
      if (key) {
        const uint32_t slot = b0 + __popc(m & ((1u << lane) - 1u));
        sm.ord[slot] = key;
        sm.idx[slot] = static_cast<uint32_t>(i);
      }
    }
    __syncthreads();
    n = static_cast<int>(sm.misc[4]);
    mode = 0;
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
      mode = 0;
    } else {
      // overflow (massive ties): count the selectable elements from the histogram
      if (threadIdx.x < 32) {
        uint32_t above, total;
        find_bin_warp(P.hist1 + static_cast<long long>(v) * kBins, 1, &above, &total);
        if (threadIdx.x == 0) sm.misc[4] = total;
      }
      __syncthreads();
      n = static_cast<int>(sm.misc[4]);
      mode = 1;
    }
    __syncthreads();
  }
  const int need = min(r.k, n);

  // 2. exact threshold over 64-bit keys, 3. collect exactly `need` survivors
  if (threadIdx.x == 0) sm.misc[5] = 0;
  __syncthreads();
  uint64_t prefix = 0;
  int pbits = 0;
  const bool take_all = (need == n);
  if (!take_all) {
    if (mode == 0) radix_select<false>(r, sm, n, need, &prefix, &pbits);
    else radix_select<true>(r, sm, n, need, &prefix, &pbits);
  }
  const int nloop = (mode == 0) ? n : r.n;
  for (int base = 0; base < nloop; base += blockDim.x) {
    const int i = base + threadIdx.x;
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
    const unsigned m = __ballot_sync(0xffffffffu, take);
    uint32_t b0 = 0;
    if (m && lane == __ffs(m) - 1) b0 = atomicAdd(&sm.misc[5], __popc(m));
    b0 = __shfl_sync(0xffffffffu, b0, m ? __ffs(m) - 1 : 0);
    if (take) {
      const uint32_t slot = b0 + __popc(m & ((1u << lane) - 1u));
      if (slot < static_cast<uint32_t>(kMaxK)) {
        // pools sort by block id ascending, positions by key descending
        sm.sel[slot] = r.pool ? static_cast<uint64_t>(~kk & 0xFFFFFFFFull) : kk;
      }
    }
  }
  __syncthreads();
  const int got = min(static_cast<int>(sm.misc[5]), kMaxK);

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
    for (int i = threadIdx.x; i < P.pool_n; i += blockDim.x)
      out[i] = (i < got) ? static_cast<int>(sm.sel[i]) : -1;
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

}  // namespace

size_t select_workspace_bytes(const SelectLaunch& a) {
  const long long V = static_cast<long long>(a.rows.T) * ((a.kind == 0 && a.pool_out) ? 2 : 1);
  // hist1 + hist2 + cnt (one memset), candidate lists
  return static_cast<size_t>(V) * (2 * kBins + 1) * 4 + static_cast<size_t>(V) * kCap * 8 + 256;
}

cudaError_t launch_select(const SelectLaunch& a, void* ws, size_t ws_bytes, const DeviceCtx& ctx, cudaStream_t st) {
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
  P.n_vrows = V;
  uint8_t* w = static_cast<uint8_t*>(ws);
  P.hist1 = reinterpret_cast<uint32_t*>(w);
  P.hist2 = P.hist1 + static_cast<size_t>(V) * kBins;
  P.cnt = P.hist2 + static_cast<size_t>(V) * kBins;
  uint8_t* cand = w + ((static_cast<size_t>(V) * (2 * kBins + 1) * 4 + 255) & ~size_t(255));
  P.cord = reinterpret_cast<uint32_t*>(cand);
  P.cidx = P.cord + static_cast<size_t>(V) * kCap;

  // longest row that may need the streaming passes
  long long maxn = 0;
  if (a.kind == 0) {
    maxn = a.ld_scores;
    if (a.pool_out) maxn = maxn > a.ld_bm ? maxn : a.ld_bm;
  }
  cudaError_t e;
  if (maxn > kDirect) {
    e = cudaMemsetAsync(ws, 0, static_cast<size_t>(V) * (2 * kBins + 1) * 4, st);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>((maxn + kChunk - 1) / kChunk), static_cast<unsigned>(V));
    sel_hist1_kernel<<<grid, 256, 0, st>>>(P);
    sel_refine_kernel<<<grid, 256, 0, st>>>(P);
    sel_filter_kernel<<<grid, 256, 0, st>>>(P);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const size_t smem = static_cast<size_t>(kDirect) * 8 + kMaxK * 8 + 256 * 4 + 64;
  e = cudaFuncSetAttribute(sel_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  sel_final_kernel<<<V, 1024, smem, st>>>(P);
  return cudaGetLastError();
}

}  // namespace csa2
