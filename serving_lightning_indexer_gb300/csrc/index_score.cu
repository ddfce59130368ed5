// Lightning-Indexer scoring on the 5th-generation tensor cores.
//
// Score (CSA2 page, "一层 CSA2 的 attention 具体怎么算" item 4; DSA page,
// "打分公式" and "fp8 与 scale 的吸收"):
//     I[t,s] = k_scale[s] * sum_h w'[t,h] * ReLU(q8[t,h] . k8[s]),  w' = w * q_scale
//
// One persistent, warp-specialised kernel serves three tilings:
//   * scan,   NQ=1: decode.  A tile is 128 consecutive entries (two 64-entry
//                   pages) of one row's sequence x the row's 32 heads.
//   * scan,   NQ=8: prefill of one sequence.  A tile is 128 entries x 8
//                   consecutive query rows (256 = 8 x 32 head columns).
//   * gather, NQ=1: Reindex.  A tile is 16 candidate blocks of 8 entries
//                   (CSA2 page, "Hierarchical Sparse Indexer": a Reindex
//                   layer scores only the pool) x the row's 32 heads.
// The contraction D[key, (query, head)] = K8 . Q8^T (K = 128) runs as
// tcgen05.mma kind::f8f6f4 with keys on M = 128 and (query, head) on N,
// both operands TMA-staged in the 128-byte swizzle layout, the fp32
// accumulator in TMEM (a ring of 4 in decode, 2 in prefill).  The epilogue
// applies ReLU, the head weights, the per-key scale and the visibility mask,
// and emits the 8-entry block maxima used by the candidate pool:
//   * decode / Reindex: one key row per thread (tcgen05.ld 32x32b), head
//     weights broadcast from shared memory, score and block-max histograms
//     for the selection kernels;
//   * prefill: q is staged head-major (row 8 h + j = head h of query j), so a
//     16x256b load gives each thread two queries of a key pair and all 64 of
//     its head weights stay in registers (packed fp32x2 FMA, ReLU split
//     between the ALU and FMA pipes).
//
// Roles (320 threads): warp 0 = TMA producer (the whole warp walks the stage
// loop), warp 1 = TMEM owner + MMA issuer, warps 2..9 = two epilogue groups
// (warp w reads TMEM lanes 32*(w%4)...).  In decode the groups take alternate
// tiles; in prefill both read every accumulator (group g the 16-lane half g
// of each lane quadrant) and release it before the key scales, stores and
// block maxima, so the next MMA starts as early as possible.
#include <math.h>

#include "csa2_device.cuh"
#include "csa2_internal.h"

namespace csa2 {

namespace {

constexpr int kModeScan = 0;
constexpr int kModeGather = 1;
constexpr int kTileKeys = 128;
constexpr int kRowBytes = 128;                       // one FP8 key / one head of q
constexpr int kMaxQB = 2048;                         // query blocks per launch

struct IdxParams {
  const float* q_scale;
  const float* w;
  const uint8_t* index_k;
  long long n_pages;
  const int* page_table;
  int pt_stride;
  RowsDev rows;
  float* out;
  long long ld_out;
  float* block_max;
  long long ld_bm;
  uint32_t* hist;  // optional [2][T][2048]: key histograms of the scores and of the block maxima
  const int* pool_blocks;
  int pool_n;
  uint32_t* err;
};

constexpr int kHistBins = 2048;  // top 11 bits of the order-preserving key

constexpr int kEpiGroups = 2;                        // epilogue groups of 4 warps, alternating tiles
constexpr int kThreads = 64 + kEpiGroups * 128;

// Index-K page formats: FP8 (8448 B = 64 x 128 e4m3 codes + 64 fp32 scales,
// seen as 66 rows of 128 B) and FP4 (4352 B = 64 x 64 B of e2m1 codes + 64 x
// 4 ue8m0 scales, one per 32 dims, seen as 68 rows of 64 B).
template <bool F4>
struct PageFmt {
  static constexpr int kBytes = F4 ? 4352 : 8448;
  static constexpr int kRows = F4 ? 68 : 66;        // rows of the 2-D tensor view per page
  static constexpr int kScaleOff = F4 ? 4096 : 8192;
};

template <int NQ, bool F4 = false>
struct IdxCfg {
  // decode: the two epilogue groups take alternate tiles; prefill: both groups
  // read every accumulator.  Each epilogue warp of a tile releases its stage
  // once it has read the key scales.
  static constexpr int kEpiWarpsPerTile = (NQ == 1) ? 4 : 8;
  // decode runs two CTAs per SM (two producers per SM measured ~1.5x the HBM
  // throughput of one CTA with deeper staging); prefill one CTA with 8 stages
  static constexpr int kStages = (NQ == 1) ? 4 : 8;
  static constexpr int kCtasPerSm = (NQ == 1) ? 2 : 1;
  // TMEM accumulator ring.  FP4 keys: one 32-column accumulator per 32-dim
  // block of the key (the MMA has no per-block scale here; the epilogue
  // applies the ue8m0 block scales), 128 columns a tile.
  static constexpr int kNumAcc = F4 ? 2 : ((NQ == 1) ? 4 : 2);
  static constexpr int kQBytes = NQ * 32 * kRowBytes;
  static constexpr int kAccCols = F4 ? 4 * NQ * 32 : NQ * 32;
  static constexpr int kTmemCols = kNumAcc * kAccCols;
  static constexpr int kKeyBytes = kTileKeys * kRowBytes;
  static constexpr int kOffKeys = 0;
  static constexpr int kOffQ = kOffKeys + kStages * kKeyBytes;
  static constexpr int kOffScales = kOffQ + 2 * kQBytes;
  static constexpr int kOffW = kOffScales + kStages * kTileKeys * 4;
  static constexpr int kOffBars = kOffW + kEpiGroups * NQ * 32 * 4;
  static constexpr int kNumBars = 2 * kStages + 4 + 2 * kNumAcc;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kOffLookup = kOffMisc + 16;         // 32 resolved copy sources of the producer warp
  // per epilogue group: score and block-max key histograms of the current row (decode only)
  static constexpr int kHistWords = (NQ == 1) ? 2 * kHistBins : 0;
  static constexpr int kOffHist = kOffLookup + 32 * 4;
  static constexpr int kOffPrefix = kOffHist + kEpiGroups * kHistWords * 4;
  // prefix [nqb+1], then the sequence and the visible entries of every query block [nqb] each
  static size_t smem_bytes(int nqb) { return 1024 + kOffPrefix + static_cast<size_t>(3 * nqb + 1) * 4; }
};
static_assert(128 == IdxCfg<1>::kTmemCols, "decode accumulators: 4 x 32 columns");
static_assert(512 == IdxCfg<8>::kTmemCols, "prefill accumulators: 2 x 256 columns");
static_assert(256 == IdxCfg<1, true>::kTmemCols, "FP4 decode accumulators: 2 x 128 columns");
static_assert(kEpiGroups == 2 && IdxCfg<1>::kNumAcc % kEpiGroups == 0 && IdxCfg<8>::kNumAcc % kEpiGroups == 0,
              "each epilogue group owns the accumulators of its tiles");

// Sequence, entries visible to the rows of a query block, and its tile count.
template <int NQ, int MODE>
__device__ __forceinline__ int qb_tiles(const IdxParams& p, int qb, int* seq, int* emax_out) {
  const int t0 = (MODE == kModeScan) ? qb * NQ : qb;
  const int b = row_seq_of(p.rows, t0);
  int emax = 0;
#pragma unroll
  for (int j = 0; j < (MODE == kModeScan ? NQ : 1); ++j)
    if (t0 + j < p.rows.T) emax = max(emax, visible_of(p.rows, t0 + j, b));
  *seq = b;
  *emax_out = emax;
  if (MODE == kModeGather) return (p.pool_n * 8 + kTileKeys - 1) / kTileKeys;
  return (emax + kTileKeys - 1) / kTileKeys;
}

// ReLU on two pipes (prefill epilogue).  A dot product of two FP8 e4m3 vectors
// of 128 elements is below 128 * 448^2 < 2^25 in magnitude, so a saturating
// multiply by 2^-25 (clamp to [0, 1], on the FMA pipe) returns ReLU(x) * 2^-25
// exactly; the head weight of such a head is stored times 2^25, so the product
// w' * ReLU(x) and every rounding step are those of the max-based form (on
// the ALU pipe).  One head in four takes the multiply, which balances the two
// pipes.
constexpr float kSatUp = 33554432.f;  // 2^25
__host__ __device__ constexpr bool kSatHead(int h) { return (h & 3) == 3; }
__device__ __forceinline__ float relu_mixed(uint32_t bits, bool sat) {
  const float x = __uint_as_float(bits);
  if (!sat) return fmaxf(x, 0.f);
  float y;
  asm("mul.rn.sat.f32 %0, %1, 0f33000000;" : "=f"(y) : "f"(x));  // x * 2^-25 clamped to [0, 1]
  return y;
}

// Value 2^(u-127) of a ue8m0 scale byte (u = 0: 2^-127; u = 255: NaN).
__device__ __forceinline__ float ue8m0_to_float(uint32_t u) {
  return u == 0u ? __uint_as_float(0x00400000u) : (u == 255u ? __uint_as_float(0x7FC00000u) : __uint_as_float(u << 23));
}

__device__ __forceinline__ int find_qb(const int* prefix, int nqb, long long g) {
  int lo = 0, hi = nqb - 1;  // largest qb with prefix[qb] <= g
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int NQ, int MODE, bool F4>
__global__ void __launch_bounds__(kThreads, IdxCfg<NQ, F4>::kCtasPerSm)
    index_tiles_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_kv,
                       const __grid_constant__ IdxParams p) {
  using Cfg = IdxCfg<NQ, F4>;
  using Fmt = PageFmt<F4>;
  static_assert(!F4 || NQ == 1, "FP4 index keys on the decode scan and the Reindex gather");
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_keys = smem + Cfg::kOffKeys;
  uint8_t* s_q = smem + Cfg::kOffQ;
  float* s_scales = reinterpret_cast<float*>(smem + Cfg::kOffScales);
  float* s_w = reinterpret_cast<float*>(smem + Cfg::kOffW);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBars);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* qfull = bars + 2 * S;
  uint64_t* qempty = qfull + 2;
  uint64_t* tfull = qempty + 2;
  uint64_t* tempty = tfull + Cfg::kNumAcc;
  constexpr int NA = Cfg::kNumAcc;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  int* s_lookup = reinterpret_cast<int*>(smem + Cfg::kOffLookup);
  int* s_prefix = reinterpret_cast<int*>(smem + Cfg::kOffPrefix);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = p.rows.T;
  const int nqb = (MODE == kModeScan) ? (T + NQ - 1) / NQ : T;

  int* s_seq = s_prefix + nqb + 1;
  int* s_emax = s_seq + nqb;
  // barriers and TMEM are set up while the previous kernel may still run; the
  // next kernel may start only once this CTA holds its TMEM (so that it can
  // never take the TMEM this CTA waits for)
  if (threadIdx.x == 0) {
    s_prefix[0] = 0;
    *s_abort = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1 + Cfg::kEpiWarpsPerTile);  // MMA commit + one arrival per epilogue warp of the tile
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 1);
    }
    for (int i = 0; i < NA; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], Cfg::kEpiWarpsPerTile);  // the epilogue warps reading this accumulator
    }
    fence_mbar_init();
    prefetch_tmap(&map_q);
    prefetch_tmap(&map_kv);
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, Cfg::kTmemCols);
    tmem_relinquish();
  }
  pdl_wait();  // global memory is touched only after the previous kernel completed
  pdl_trigger();
  for (int i = threadIdx.x; i < nqb; i += blockDim.x) s_prefix[i + 1] = qb_tiles<NQ, MODE>(p, i, &s_seq[i], &s_emax[i]);
  __syncthreads();
  if (warp == 0) {  // inclusive scan of the tile counts by one warp
    const int per = (nqb + 31) / 32;
    const int lo = 1 + lane * per;
    const int hi = min(lo + per, nqb + 1);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += s_prefix[i];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int i = lo; i < hi; ++i) {
      run += s_prefix[i];
      s_prefix[i] = run;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const long long total = s_prefix[nqb];
  const long long g_begin = total * blockIdx.x / gridDim.x;
  const long long g_end = total * (blockIdx.x + 1) / gridDim.x;

  if (g_begin < g_end) {
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      // The warp resolves the copy sources of a group of tiles in parallel (one
      // page or candidate block per lane), then lane 0 waits for free stages
      // and issues the TMA / bulk copies.
      constexpr int SLOTS = (MODE == kModeScan) ? 2 : 16;  // copies per tile
      constexpr int GT = 32 / SLOTS;                       // tiles per group
      const uint64_t pol_keys = (MODE == kModeScan && NQ > 1) ? l2_policy_evict_last() : l2_policy_evict_first();
      const uint64_t pol_q = l2_policy_evict_last();
      int cur_qb = -1, qcount = 0;
      long long it = 0;
      bool ok = true;
      for (long long g0 = g_begin; g0 < g_end; g0 += GT) {
        {
          const long long gl = g0 + lane / SLOTS;
          const int sl = lane % SLOTS;
          int rid = -1;  // row of the 66-row page view to copy from
          if (gl < g_end) {
            const int qbl = find_qb(s_prefix, nqb, gl);
            const int kb = static_cast<int>(gl - s_prefix[qbl]);
            const int b = s_seq[qbl], emax = s_emax[qbl];
            const int* ptab = p.page_table + static_cast<long long>(b) * p.pt_stride;
            if (MODE == kModeScan) {
              const int lp = kb * 2 + sl;
              if (lp * 64 < emax) {
                const int phys = (lp < p.pt_stride) ? __ldg(ptab + lp) : -1;
                if (phys >= 0 && phys < p.n_pages) rid = phys * Fmt::kRows;
                else set_error(p.err, kErrBounds);
              }
            } else {
              const int cb = kb * 16 + sl;
              const int blk = (cb < p.pool_n) ? __ldg(p.pool_blocks + static_cast<long long>(qbl) * p.pool_n + cb) : -1;
              if (blk >= 0 && blk * 8 < emax) {
                const int phys = ((blk >> 3) < p.pt_stride) ? __ldg(ptab + (blk >> 3)) : -1;
                if (phys >= 0 && phys < p.n_pages) rid = phys * Fmt::kRows + (blk & 7) * 8;
                else set_error(p.err, kErrBounds);
              }
            }
          }
          s_lookup[lane] = rid;
        }
        __syncwarp();
        // The whole warp walks the group's tiles in step (a warp whose lanes
        // wait at different points measurably slows the epilogue warps sharing
        // its scheduler): it switches q when the row changes, reserves a stage
        // per tile and lane 0 announces its bytes.  The copies are issued by
        // lane 0 (scan: 2 pages per tile; q: one lane per head box in prefill)
        // or, after the walk, by one lane per copy source (gather: 16
        // candidate blocks per tile, whose serial issue would dominate).
        const long long it0 = it;  // tile j of the group uses stage (it0 + j) % S
        int ntile = 0;
        {
          int qb = find_qb(s_prefix, nqb, g0);
          for (int j = 0; j < GT && g0 + j < g_end; ++j, ++it) {
            const long long g = g0 + j;
            while (g >= s_prefix[qb + 1]) ++qb;
            if (qb != cur_qb) {
              cur_qb = qb;
              const int slot = qcount & 1;
              if (!(ok = mbar_wait(&qempty[slot], ((qcount >> 1) & 1) ^ 1, s_abort))) break;
              const int t0 = (MODE == kModeScan) ? qb * NQ : qb;
              if (lane == 0) mbar_arrive_expect_tx(&qfull[slot], Cfg::kQBytes);
              __syncwarp();
              if (NQ == 1) {
                if (lane == 0) tma_load_2d(s_q + slot * Cfg::kQBytes, &map_q, 0, t0 * 32, &qfull[slot], pol_q);
              } else {
                // head-major tile: rows h * NQ + j hold head h of query t0 + j
                tma_load_2d(s_q + slot * Cfg::kQBytes + lane * NQ * kRowBytes, &map_q, lane * kRowBytes, t0,
                            &qfull[slot], pol_q);
              }
              ++qcount;
            }
            const int s = static_cast<int>(it % S);
            if (!(ok = mbar_wait(&empty[s], static_cast<uint32_t>((it / S) & 1) ^ 1u, s_abort))) break;
            constexpr int kRows = (MODE == kModeScan) ? 64 : 8;  // key rows per copy
            // bytes a key row adds to the stage's transaction count: the 128 B
            // of an FP8 key; the 64 B of packed codes of an FP4 key (unpacked
            // into 128 B of shared memory by the copy)
            constexpr uint32_t kKeyTxBytes = F4 ? 64 : kRowBytes;
            ntile = j + 1;
            if (lane == 0) {
              uint32_t bytes = 0;
#pragma unroll
              for (int c = 0; c < SLOTS; ++c)
                if (s_lookup[j * SLOTS + c] >= 0) bytes += kRows * (kKeyTxBytes + 4);
              mbar_arrive_expect_tx(&full[s], bytes);
              if (MODE == kModeScan) {
                uint8_t* kdst = s_keys + s * Cfg::kKeyBytes;
                float* sdst = s_scales + s * kTileKeys;
#pragma unroll
                for (int c = 0; c < SLOTS; ++c) {
                  const int rid = s_lookup[j * SLOTS + c];
                  if (rid < 0) continue;
                  const int phys = rid / Fmt::kRows;
                  const int r = rid - phys * Fmt::kRows;
                  tma_load_2d(kdst + c * kRows * kRowBytes, &map_kv, 0, rid, &full[s], pol_keys);
                  bulk_load(sdst + c * kRows, p.index_k + static_cast<long long>(phys) * Fmt::kBytes + Fmt::kScaleOff + r * 4,
                            kRows * 4, &full[s], pol_keys);
                }
              }
            }
            __syncwarp();
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (MODE == kModeGather) {
          const int j = lane / SLOTS, c = lane % SLOTS;
          const int rid = s_lookup[lane];
          if (j < ntile && rid >= 0) {
            constexpr int kRows = 8;
            const int s = static_cast<int>((it0 + j) % S);
            const int phys = rid / Fmt::kRows;
            const int r = rid - phys * Fmt::kRows;
            tma_load_2d(s_keys + s * Cfg::kKeyBytes + c * kRows * kRowBytes, &map_kv, 0, rid, &full[s], pol_keys);
            bulk_load(s_scales + s * kTileKeys + c * kRows,
                      p.index_k + static_cast<long long>(phys) * Fmt::kBytes + Fmt::kScaleOff + r * 4, kRows * 4, &full[s],
                      pol_keys);
          }
        }
        if (!ok) break;
        __syncwarp();
      }
      if (lane == 0) {
        if (!ok) {
          *s_abort = 1;
          set_error(p.err, kErrTimeout);
        }
        // the copies of the last stages must land before the CTA may exit
        for (long long i = (it > S ? it - S : 0); i < it; ++i)
          mbar_wait(&full[i % S], static_cast<uint32_t>((i / S) & 1), nullptr);
      }
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      // FP4 keys: A is e2m1 (format 5 of kind::f8f6f4), in the 16-byte chunks
      // the tensor copy unpacks them to (8 bytes of codes, 8 bytes of gap)
      constexpr uint32_t idesc = idesc_e4m3_f32(128, NQ * 32) | (F4 ? (5u << 7) : 0u);
      int qb = find_qb(s_prefix, nqb, g_begin);
      int cur_qb = -1, qcount = 0, slot = 0;
      long long it = 0;
      bool ok = true;
      for (long long g = g_begin; g < g_end; ++g, ++it) {
        while (g >= s_prefix[qb + 1]) ++qb;
        if (qb != cur_qb) {
          if (cur_qb >= 0) mma_commit(&qempty[slot]);
          cur_qb = qb;
          slot = qcount & 1;
          if (!(ok = mbar_wait(&qfull[slot], (qcount >> 1) & 1, s_abort))) break;
          ++qcount;
        }
        const int s = static_cast<int>(it % S);
        if (!(ok = mbar_wait(&full[s], static_cast<uint32_t>((it / S) & 1), s_abort))) break;
        const int a = static_cast<int>(it % NA);
        if (!(ok = mbar_wait(&tempty[a], static_cast<uint32_t>((it / NA) & 1) ^ 1u, s_abort))) break;
        tc_fence_after();
        const uint64_t adesc = smem_desc_sw128(s_keys + s * Cfg::kKeyBytes);
        const uint64_t bdesc = smem_desc_sw128(s_q + slot * Cfg::kQBytes);
        const uint32_t d = tmem_base + a * Cfg::kAccCols;
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // K = 128 = 4 steps of 32 elements (32 B of the swizzled rows)
          if (F4)  // one accumulator per 32-dim block: the block scales differ
            mma_e4m3(d + k * NQ * 32, adesc + 2 * k, bdesc + 2 * k, idesc, 0u);
          else
            mma_e4m3(d, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
        }
        mma_commit(&tfull[a]);
        mma_commit(&empty[s]);
      }
      if (!ok) {
        *s_abort = 1;
        set_error(p.err, kErrTimeout);
      }
    } else if (warp >= 2 && NQ == 8) {
      // ------------------------------------------------------------ prefill epilogue
      // The accumulator's columns are head-major (column 8 h + j: head h of
      // query t0 + j).  Both groups read every accumulator: group g reads the
      // 16-lane half g of its warp's lane quadrant, as eight 16x256b.x4 loads
      // of 32 columns (heads 4c .. 4c+3), each issued before the previous one
      // is consumed.  Lane l gets rows ra = 16 g + l/4 and ra + 8 of the
      // quadrant for queries qa = t0 + 2 (l % 4) and qa + 1, so its 64 head
      // weights stay in registers and a key's head sum needs no exchange
      // between threads.  The accumulator is released as soon as it has been
      // read; the key scales, the stores and the block maxima follow.
      const int grp = (warp - 2) >> 2;
      const int quad = warp & 3;
      const int pc = lane & 3, prr = lane >> 2;
      const int ra = quad * 32 + grp * 16 + prr;
      const uint32_t lane_addr = static_cast<uint32_t>(quad * 32 + grp * 16) << 16;
      uint64_t wq[32];  // wq[h] = (w'[qa][h], w'[qa + 1][h])
      int Ea = 0, Eb = 0, ta = 0;
      int qb = find_qb(s_prefix, nqb, g_begin);
      int cur_qb = -1;
      uint32_t a = 0, aph = 0;  // accumulator ring position and phase
      uint32_t st = 0, sph = 0;  // key stage and its phase
      bool ok = true;
      for (long long g = g_begin; g < g_end; ++g) {
        while (g >= s_prefix[qb + 1]) ++qb;
        const int kb = static_cast<int>(g - s_prefix[qb]);
        if (qb != cur_qb) {
          cur_qb = qb;
          const int t0 = qb * NQ;
          const int b = s_seq[qb];
          ta = t0 + 2 * pc;
          const int tb = ta + 1;
          const float* wa = p.w + static_cast<long long>(ta) * 32;
          const float* sa = p.q_scale + static_cast<long long>(ta) * 32;
#pragma unroll
          for (int h = 0; h < 32; ++h) {
            const float k = kSatHead(h) ? kSatUp : 1.f;
            wq[h] = pack_f32x2(ta < T ? __ldg(wa + h) * __ldg(sa + h) * k : 0.f,
                               tb < T ? __ldg(wa + 32 + h) * __ldg(sa + 32 + h) * k : 0.f);
          }
          Ea = (ta < T) ? visible_of(p.rows, ta, b) : 0;
          Eb = (tb < T) ? visible_of(p.rows, tb, b) : 0;
        }
        const uint32_t ca = a, cph = aph, cs = st, csph = sph;
        if (++a == static_cast<uint32_t>(NA)) {
          a = 0;
          aph ^= 1u;
        }
        if (++st == static_cast<uint32_t>(S)) {
          st = 0;
          sph ^= 1u;
        }
        // on a timeout the warp keeps walking the tiles without waiting
        if (ok) ok = mbar_wait(&tfull[ca], cph, s_abort);
        if (!ok) continue;
        tc_fence_after();
        const uint32_t tbase = tmem_base + ca * Cfg::kAccCols + lane_addr;
        uint64_t accA0 = 0, accA1 = 0, accB0 = 0, accB1 = 0;  // (qa, qa + 1) of rows ra / ra + 8
        uint32_t v0[16], v1[16];
        tmem_ld16x256_x4(tbase, v0);
        tmem_wait_ld16(v0);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t(&cur)[16] = (c & 1) ? v1 : v0;
          uint32_t(&nxt)[16] = (c & 1) ? v0 : v1;
          if (c + 1 < 8) tmem_ld16x256_x4(tbase + (c + 1) * 32, nxt);
#pragma unroll
          for (int n = 0; n < 4; ++n) {
            const bool sat = kSatHead(4 * c + n);
            const uint64_t xa = pack_f32x2(relu_mixed(cur[4 * n + 0], sat), relu_mixed(cur[4 * n + 1], sat));
            const uint64_t xb = pack_f32x2(relu_mixed(cur[4 * n + 2], sat), relu_mixed(cur[4 * n + 3], sat));
            if (n & 1) {
              accA1 = fma_f32x2(xa, wq[4 * c + n], accA1);
              accB1 = fma_f32x2(xb, wq[4 * c + n], accB1);
            } else {
              accA0 = fma_f32x2(xa, wq[4 * c + n], accA0);
              accB0 = fma_f32x2(xb, wq[4 * c + n], accB0);
            }
          }
          if (c + 1 < 8) tmem_wait_ld16(nxt);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[ca]);
        // The accumulator is free again.  The stage's key scales are read only
        // now, off the path from one MMA to the next; the stage is released
        // after that read.
        if (ok) ok = mbar_wait(&full[cs], csph, s_abort);
        if (!ok) continue;
        const float ksA = s_scales[cs * kTileKeys + ra], ksB = s_scales[cs * kTileKeys + ra + 8];
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[cs]);
        const float2 a0 = unpack_f32x2(accA0), a1 = unpack_f32x2(accA1);
        const float2 b0 = unpack_f32x2(accB0), b1 = unpack_f32x2(accB1);
        const int posA = kb * kTileKeys + ra, posB = posA + 8;
        const int tb = ta + 1;
        // scores (row, query): [0] (ra, qa), [1] (ra, qa+1), [2] (ra+8, qa), [3] (ra+8, qa+1)
        float sc[4];
        sc[0] = posA < Ea ? (a0.x + a1.x) * ksA : -INFINITY;
        sc[1] = posA < Eb ? (a0.y + a1.y) * ksA : -INFINITY;
        sc[2] = posB < Ea ? (b0.x + b1.x) * ksB : -INFINITY;
        sc[3] = posB < Eb ? (b0.y + b1.y) * ksB : -INFINITY;
        if (ta < T) {
          if (posA < p.ld_out) p.out[static_cast<long long>(ta) * p.ld_out + posA] = sc[0];
          if (posB < p.ld_out) p.out[static_cast<long long>(ta) * p.ld_out + posB] = sc[2];
        }
        if (tb < T) {
          if (posA < p.ld_out) p.out[static_cast<long long>(tb) * p.ld_out + posA] = sc[1];
          if (posB < p.ld_out) p.out[static_cast<long long>(tb) * p.ld_out + posB] = sc[3];
        }
        if (p.block_max != nullptr) {
          // rows ra of the 8 lanes sharing lane % 4 are one block of 8 entries
          // (posA is a multiple of 8 on lane / 4 == 0), rows ra + 8 the next
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            sc[e] = fmaxf(sc[e], __shfl_xor_sync(0xffffffffu, sc[e], 4));
            sc[e] = fmaxf(sc[e], __shfl_xor_sync(0xffffffffu, sc[e], 8));
            sc[e] = fmaxf(sc[e], __shfl_xor_sync(0xffffffffu, sc[e], 16));
          }
          if (prr == 0) {
            const int blk = posA >> 3;
            const int na = (Ea + 7) / 8, nb = (Eb + 7) / 8;
            float* bma = p.block_max + static_cast<long long>(ta) * p.ld_bm;
            float* bmb = p.block_max + static_cast<long long>(tb) * p.ld_bm;
            if (ta < T && blk < na && blk < p.ld_bm) bma[blk] = sc[0];
            if (tb < T && blk < nb && blk < p.ld_bm) bmb[blk] = sc[1];
            if (ta < T && blk + 1 < na && blk + 1 < p.ld_bm) bma[blk + 1] = sc[2];
            if (tb < T && blk + 1 < nb && blk + 1 < p.ld_bm) bmb[blk + 1] = sc[3];
          }
        }
      }
      if (!ok) {
        *s_abort = 1;
        set_error(p.err, kErrTimeout);
      }
    } else if (warp >= 2) {
      // ------------------------------------------------------------ epilogue
      // Two groups of four warps take alternate tiles; inside a group warp w
      // reads TMEM lane quadrant w % 4.
      const int grp = (warp - 2) >> 2;
      const int gtid = threadIdx.x - 64 - grp * 128;
      const int quad = warp & 3;
      const int r = quad * 32 + lane;  // key row of this thread within the tile
      float* s_wg = s_w + grp * NQ * 32;
      constexpr bool kHist = (NQ == 1);  // decode scan and Reindex gather
      const bool hist_on = kHist && p.hist != nullptr;
      uint32_t* hs = reinterpret_cast<uint32_t*>(smem + Cfg::kOffHist) + grp * Cfg::kHistWords;
      uint32_t* hb = hs + kHistBins;
      if (hist_on)
        for (int i = gtid; i < 2 * kHistBins; i += 128) hs[i] = 0u;
      // adds the group's histograms of row t to the global ones and clears them
      auto flush_hist = [&](int t) {
        uint32_t* gs = p.hist + static_cast<long long>(t) * kHistBins;
        uint32_t* gb = p.hist + (static_cast<long long>(T) + t) * kHistBins;
        for (int i = gtid; i < kHistBins; i += 128) {
          const uint32_t a = hs[i];
          if (a) atomicAdd(gs + i, a);
          hs[i] = 0u;
          if (MODE == kModeScan) {
            const uint32_t c = hb[i];
            if (c) atomicAdd(gb + i, c);
            hb[i] = 0u;
          }
        }
      };
      int qb = find_qb(s_prefix, nqb, g_begin);
      int cur_qb = -1, t0 = 0;
      int E[NQ];
      long long it = 0;
      bool ok = true;
      for (long long g = g_begin; g < g_end; ++g, ++it) {
        while (g >= s_prefix[qb + 1]) ++qb;
        if ((it & (kEpiGroups - 1)) != grp) continue;
        const int kb = static_cast<int>(g - s_prefix[qb]);
        if (qb != cur_qb) {
          named_bar_sync(1 + grp, 128);
          if (hist_on && cur_qb >= 0) {
            flush_hist(t0);
            named_bar_sync(1 + grp, 128);
          }
          cur_qb = qb;
          t0 = (MODE == kModeScan) ? qb * NQ : qb;
          const int b = row_seq_of(p.rows, t0);
          for (int i = gtid; i < NQ * 32; i += 128) {
            const int t = t0 + i / 32;
            s_wg[i] = (t < T) ? __ldg(p.w + static_cast<long long>(t) * 32 + (i & 31)) *
                                   __ldg(p.q_scale + static_cast<long long>(t) * 32 + (i & 31))
                             : 0.f;
          }
#pragma unroll
          for (int j = 0; j < NQ; ++j) E[j] = (t0 + j < T) ? visible_of(p.rows, t0 + j, b) : 0;
          named_bar_sync(1 + grp, 128);
        }
        const int a = static_cast<int>(it % NA);
        const int s = static_cast<int>(it % S);
        int pos;
        long long ci = 0;
        if (MODE == kModeScan) {
          pos = kb * kTileKeys + r;
        } else {  // the candidate's block id is loaded before the wait to hide its latency
          ci = static_cast<long long>(kb) * kTileKeys + r;
          const int cb = static_cast<int>(ci >> 3);
          const int blk = (cb < p.pool_n) ? __ldg(p.pool_blocks + static_cast<long long>(t0) * p.pool_n + cb) : -1;
          pos = blk >= 0 ? blk * 8 + static_cast<int>(ci & 7) : -1;
        }
        // On a timeout this warp keeps walking the tiles without waiting, so the
        // other warps of its group never stall on the named barrier above.
        if (ok) ok = mbar_wait(&tfull[a], static_cast<uint32_t>((it / NA) & 1), s_abort);
        if (ok) ok = mbar_wait(&full[s], static_cast<uint32_t>((it / S) & 1), s_abort);  // acquire the scales
        if (!ok) continue;
        tc_fence_after();
        // the key scale is read first, so the stage goes back to the producer
        // while the accumulator is still being read
        // FP8 keys: one fp32 scale per key; FP4 keys: four ue8m0 block scales
        const float ks = F4 ? 1.f : s_scales[s * kTileKeys + r];
        const uint32_t ub = F4 ? reinterpret_cast<const uint32_t*>(s_scales)[s * kTileKeys + r] : 0u;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll 1
        for (int j = 0; j < NQ; ++j) {
          const uint32_t tq = tmem_base + a * Cfg::kAccCols + (static_cast<uint32_t>(quad * 32) << 16);
          const float4* w4 = reinterpret_cast<const float4*>(s_wg + j * 32);
          float acc0 = 0.f, acc1 = 0.f;
          if constexpr (F4) {
            // q . k = sum over the 4 blocks of 2^(u_b - 127) * (q . e2m1 codes of
            // block b); 16 heads at a time, two heads per packed fp32x2 FMA (each
            // element rounded as by fmaf: the same values as one head at a time)
            uint64_t sb[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const float f = ue8m0_to_float((ub >> (8 * b)) & 0xFFu);
              sb[b] = pack_f32x2(f, f);
            }
            const uint64_t nz = pack_f32x2(-0.f, -0.f);  // x * y + (-0) == x * y, zeros' signs included
            uint64_t acc = pack_f32x2(0.f, 0.f);        // heads 2i (low) and 2i + 1 (high)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              // the four blocks' loads are issued together, then one wait
              uint32_t d[4][16];
#pragma unroll
              for (int b = 0; b < 4; ++b) tmem_ld32x16_async(tq + b * 32 + hh * 16, d[b]);
#pragma unroll
              for (int b = 0; b < 4; ++b) tmem_wait_ld16(d[b]);
#pragma unroll
              for (int i = 0; i < 16; i += 2) {
                uint64_t x = fma_f32x2(pack_f32x2(__uint_as_float(d[0][i]), __uint_as_float(d[0][i + 1])), sb[0], nz);
                x = fma_f32x2(pack_f32x2(__uint_as_float(d[1][i]), __uint_as_float(d[1][i + 1])), sb[1], x);
                x = fma_f32x2(pack_f32x2(__uint_as_float(d[2][i]), __uint_as_float(d[2][i + 1])), sb[2], x);
                x = fma_f32x2(pack_f32x2(__uint_as_float(d[3][i]), __uint_as_float(d[3][i + 1])), sb[3], x);
                const float2 v = unpack_f32x2(x);
                const float2 ww = reinterpret_cast<const float2*>(w4)[8 * hh + i / 2];
                acc = fma_f32x2(pack_f32x2(fmaxf(v.x, 0.f), fmaxf(v.y, 0.f)), pack_f32x2(ww.x, ww.y), acc);
              }
            }
            const float2 a2 = unpack_f32x2(acc);
            acc0 = a2.x;
            acc1 = a2.y;
          } else {
            float v[32];
            tmem_ld32(tq + j * 32, v);
#pragma unroll
            for (int h4 = 0; h4 < 8; ++h4) {
              const float4 ww = w4[h4];
              acc0 = fmaf(ww.x, fmaxf(v[4 * h4 + 0], 0.f), acc0);
              acc1 = fmaf(ww.y, fmaxf(v[4 * h4 + 1], 0.f), acc1);
              acc0 = fmaf(ww.z, fmaxf(v[4 * h4 + 2], 0.f), acc0);
              acc1 = fmaf(ww.w, fmaxf(v[4 * h4 + 3], 0.f), acc1);
            }
          }
          const int t = t0 + j;
          const bool valid = pos >= 0 && pos < E[j];
          const float sc = valid ? (acc0 + acc1) * ks : -INFINITY;
          if (MODE == kModeScan) {
            if (t < T && pos < p.ld_out) p.out[static_cast<long long>(t) * p.ld_out + pos] = sc;
            if (hist_on && valid && selectable(sc)) atomicAdd(&hs[ord_key(sc) >> 21], 1u);
            if (p.block_max != nullptr) {
              float m = sc;
              m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
              m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
              m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
              const int blk = pos >> 3;
              const int nblk = (E[j] + 7) / 8;
              if ((lane & 7) == 0 && t < T && blk < nblk && blk < p.ld_bm) {
                p.block_max[static_cast<long long>(t) * p.ld_bm + blk] = m;
                // the newest block is always kept by the pool: it counts as +inf
                if (hist_on && (blk == nblk - 1 || selectable(m)))
                  atomicAdd(&hb[(blk == nblk - 1 ? 0xFFFFFFFFu : ord_key(m)) >> 21], 1u);
              }
            }
          } else {
            if (ci < static_cast<long long>(p.pool_n) * 8) p.out[static_cast<long long>(t) * p.pool_n * 8 + ci] = sc;
            if (hist_on && valid && selectable(sc)) atomicAdd(&hs[ord_key(sc) >> 21], 1u);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[a]);
      }
      if (hist_on && cur_qb >= 0) {
        named_bar_sync(1 + grp, 128);
        flush_hist(t0);
      }
      if (!ok) {
        *s_abort = 1;
        set_error(p.err, kErrTimeout);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

template <int NQ, int MODE, bool F4>
cudaError_t launch_variant(const IndexLaunch& a, const DeviceCtx& ctx, cudaStream_t st, const char** why) {
  using Cfg = IdxCfg<NQ, F4>;
  using Fmt = PageFmt<F4>;
  const int nqb = (MODE == kModeScan) ? (a.rows.T + NQ - 1) / NQ : a.rows.T;
  if (nqb > kMaxQB) {
    *why = "too many query rows for one launch";
    return cudaErrorInvalidValue;
  }
  CUtensorMap map_q, map_kv;
  // decode: q as [T * 32 rows of 128 B], one 32-row box per query; prefill: q
  // as [T rows of 32 * 128 B], boxes of one head (128 B) x NQ queries
  const CUresult qe = (NQ == 1) ? encode_tmap_2d_u8(&map_q, a.q_fp8, kRowBytes, static_cast<uint64_t>(a.rows.T) * 32,
                                                    kRowBytes, kRowBytes, 32)
                                : encode_tmap_2d_u8(&map_q, a.q_fp8, 32 * kRowBytes, static_cast<uint64_t>(a.rows.T),
                                                    32 * kRowBytes, kRowBytes, NQ);
  if (qe != CUDA_SUCCESS) {
    *why = "tensor map of q could not be encoded";
    return cudaErrorInvalidValue;
  }
  // FP8 pages as rows of 128 B; FP4 pages as rows of 128 e2m1 codes (64 B),
  // unpacked by the tensor copy into 16-byte chunks of 8 code bytes + 8 gap
  // bytes (128 B of shared memory per key, the layout of a 4-bit MMA operand)
  const uint64_t kv_rows = static_cast<uint64_t>(a.n_pages) * Fmt::kRows;
  const CUresult ke = F4 ? encode_tmap_2d_fp4(&map_kv, a.index_k, kv_rows, MODE == kModeScan ? 64 : 8)
                         : encode_tmap_2d_u8(&map_kv, a.index_k, kRowBytes, kv_rows, kRowBytes, kRowBytes,
                                             MODE == kModeScan ? 64 : 8);
  if (ke != CUDA_SUCCESS) {
    *why = "tensor map of the index-K cache could not be encoded";
    return cudaErrorInvalidValue;
  }
  IdxParams p;
  p.q_scale = a.q_scale;
  p.w = a.w;
  p.index_k = a.index_k;
  p.n_pages = a.n_pages;
  p.page_table = a.page_table;
  p.pt_stride = a.pt_stride;
  p.rows = RowsDev{a.rows.T, a.rows.B, a.rows.row_seq, a.rows.row_pos, a.rows.n_visible, a.rows.ratio_m};
  p.out = a.out;
  p.ld_out = a.ld_out;
  p.block_max = a.block_max;
  p.ld_bm = a.ld_bm;
  p.hist = a.hist;
  p.pool_blocks = a.pool_blocks;
  p.pool_n = a.pool_n;
  p.err = ctx.err;
  if (a.hist && NQ != 1) {
    *why = "score histograms are produced on the decode and Reindex paths only";
    return cudaErrorInvalidValue;
  }
  // the histograms accumulate into the caller's zeroed buffer: [2][T][2048]
  // (scores, block maxima); the top-k call that reads them zeroes them again
  const size_t smem = Cfg::smem_bytes(nqb);
  auto kern = index_tiles_kernel<NQ, MODE, F4>;
  cudaError_t e = prefer_max_smem(kern, smem);
  if (e != cudaSuccess) return e;
  // CTAs per SM: bounded by shared memory, the register budget of the launch
  // bounds and the TMEM columns (kTmemCols per CTA, 512 per SM)
  int occ = ctas_per_sm_by_smem(ctx, smem);
  occ = occ > Cfg::kCtasPerSm ? Cfg::kCtasPerSm : occ;
  static_assert(IdxCfg<1>::kTmemCols * IdxCfg<1>::kCtasPerSm <= 512 &&
                    IdxCfg<1, true>::kTmemCols * IdxCfg<1, true>::kCtasPerSm <= 512,
                "TMEM of the CTAs sharing an SM");
  return launch_pdl(kern, dim3(ctx.num_sms * occ), dim3(kThreads), smem, st, map_q, map_kv, p);
}

}  // namespace

cudaError_t launch_index_tiles(const IndexLaunch& a, int mode, int nq, const DeviceCtx& ctx, cudaStream_t st,
                               const char** why) {
  if (a.fp4) {
    if (mode == kModeScan && nq == 1) return launch_variant<1, kModeScan, true>(a, ctx, st, why);
    if (mode == kModeGather && nq == 1) return launch_variant<1, kModeGather, true>(a, ctx, st, why);
    *why = "FP4 index keys are scored on the decode scan and the Reindex gather only";
    return cudaErrorInvalidValue;
  }
  if (mode == kModeScan && nq == 1) return launch_variant<1, kModeScan, false>(a, ctx, st, why);
  if (mode == kModeScan && nq == 8) return launch_variant<8, kModeScan, false>(a, ctx, st, why);
  if (mode == kModeGather && nq == 1) return launch_variant<1, kModeGather, false>(a, ctx, st, why);
  *why = "unsupported index tiling";
  return cudaErrorInvalidValue;
}

}  // namespace csa2
