// MQA sparse attention over SWA keys + selected main-KV entries + attention sink.
//
// CSA2 page, "一层 CSA2 的 attention 具体怎么算" (attention equation): per
// query row t and head i, one joint softmax over the layer's SWA keys and the
// <= k main-KV entries of the row's top-k, with the per-head sink s_i only in
// the denominator; K = V is one shared 512-vector (MQA, 64 heads).
//
// The key list of a row is [SWA slots..., main slots...].  Rows of up to 16
// chunks of 80 keys (decode and prefill: 128 SWA + 512 main keys) take the
// tcgen05 kernel further below.  Longer rows take this split-K kernel: the
// list is cut into chunks of 64 keys, and a thread-block cluster of S CTAs
// works on one row, CTA r taking a contiguous range of chunks.  Per chunk a CTA
//   * gathers the records with bulk async copies (one per key, completing on an
//     mbarrier) into a staging area, the row's q arriving the same way,
//   * dequantises them to bf16 rows in shared memory (FP8 e4m3 x fp32 scale for
//     SWA, e2m1 x ue8m0 through byte-permute tables for main KV),
//   * computes S = q K^T on the tensor cores (mma.sync m16n8k16 bf16, fp32
//     accumulate; 16 warps, each 16 heads x 16 keys over all 512 dims), a
//     running max / sum per head, and O += P V (each warp 16 heads x 128 dims),
// gathering the next chunk's records meanwhile.  The partial results of a row
// are merged through distributed shared memory: the CTAs exchange their (max,
// sum) per head, scale their O by exp(max - M) / denominator, and each CTA sums
// a share of the heads over the cluster and writes it.  No global scratch.
#include <math.h>

#include "csa2_device.cuh"
#include "csa2_rope.cuh"
#include "csa2_internal.h"

namespace csa2 {

namespace {

constexpr int kH = 64;
constexpr int kD = 512;
constexpr int kCK = 64;              // keys per chunk
constexpr int kQStride = kD + 8;     // bf16 per shared row (1040 B: conflict-free ldmatrix)
constexpr int kSStride = kCK + 4;    // floats
constexpr int kPStride = kCK + 8;    // bf16
constexpr int kRawStride = 528;      // staging bytes per key (largest record)
constexpr int kMaxCluster = 16;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnParams {
  const __nv_bfloat16* q;
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
  float scale_log2;
  int T;
  int out_bf16;
  void* out;
  float* lse;
  int nsplit;             // CTAs per row = cluster size
  int chunks_per_split;
  const int* q_pos;          // [T] query positions (inverse RoPE, bounded replay)
  const int* swa_seg_start;  // [T] bounded-replay segment starts, or null
  int inv_rope;              // rotate the output's last 64 dims back by the query's RoPE
  uint64_t inv_freq[32];     // theta^(-2p/64) as a fixed-point turn rate (rope_turn_rate)
  uint32_t* err;
};

struct AttnSmem {
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kH * kQStride * 2;
  static constexpr int kOffRaw = kOffK + kCK * kQStride * 2;
  static constexpr int kOffS = kOffRaw + kCK * kRawStride;
  static constexpr int kOffP = kOffS + kH * kSStride * 4;
  static constexpr int kOffStats = kOffP + kH * kPStride * 2;  // m, l, alpha [64] each
  static constexpr int kOffKind = kOffStats + 3 * kH * 4;       // [64] 0 none, 1 SWA, 2 main
  static constexpr int kOffBars = kOffKind + kCK * 4;           // q, records, merge receive
  static constexpr int kBytes = kOffBars + 24;
  // merge: send rows [64][kQStride] bf16 over q, receive rows [ns][ceil(64/ns)][512] bf16 after them
  static constexpr int kRecvRowsMax = 75;                       // max over ns of ns * ceil(64 / ns)
  static constexpr int kOffSend = 0;
  static constexpr int kOffRecv = kOffSend + kH * kQStride * 2;
  static_assert(kOffRecv + kRecvRowsMax * kD * 2 <= kOffS, "the merge buffers fit over q, K and the staging");
};
// ns * recv_rows_per_rank(ns) peaks at 75 (ns = 15) for 1 <= ns <= 16.
__host__ __device__ constexpr int recv_rows_per_rank(int ns) { return (kH + ns - 1) / ns; }
static_assert(15 * ((kH + 14) / 15) == AttnSmem::kRecvRowsMax, "receive rows");

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- cluster helpers
// Bulk asynchronous copy from this CTA's shared memory into a cluster peer's,
// completing on the peer's mbarrier (dst and mbar in the cluster window).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
                   "r"(dst),
               "r"(smem_u32(src)), "r"(bytes), "r"(mbar)
               : "memory");
}

// ---------------------------------------------------------------- dequantisation
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Byte tables of the bf16 bit patterns of the 8 e2m1 magnitudes times 2^(u-127)
// (0, .5, 1, 1.5, 2, 3, 4, 6): L = low bytes, H = high bytes, entries 0-3 in
// the first word, 4-7 in the second.  Valid for 2 <= u <= 252 (the scaled
// magnitudes stay normal bf16 numbers).
struct E2m1Tables {
  uint32_t L0, L1, H0, H1;
};
__device__ __forceinline__ E2m1Tables e2m1_tables(uint32_t u) {
  const int k = static_cast<int>(u) - 127;
  constexpr uint32_t base[8] = {0u, 0x3F00u, 0x3F80u, 0x3FC0u, 0x4000u, 0x4040u, 0x4080u, 0x40C0u};
  uint32_t P[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) P[m] = m ? static_cast<uint32_t>(static_cast<int>(base[m]) + (k << 7)) : 0u;
  E2m1Tables t;
  t.L0 = (P[0] & 0xFFu) | ((P[1] & 0xFFu) << 8) | ((P[2] & 0xFFu) << 16) | ((P[3] & 0xFFu) << 24);
  t.L1 = (P[4] & 0xFFu) | ((P[5] & 0xFFu) << 8) | ((P[6] & 0xFFu) << 16) | ((P[7] & 0xFFu) << 24);
  t.H0 = (P[0] >> 8) | ((P[1] >> 8) << 8) | ((P[2] >> 8) << 16) | ((P[3] >> 8) << 24);
  t.H1 = (P[4] >> 8) | ((P[5] >> 8) << 8) | ((P[6] >> 8) << 16) | ((P[7] >> 8) << 24);
  return t;
}
// Four e2m1 codes (the 4 nibbles of c, element 0 lowest) -> two bf16x2 words.
__device__ __forceinline__ void e2m1x4_bf16(uint32_t c, const E2m1Tables& t, uint32_t& o0, uint32_t& o1) {
  const uint32_t mag = c & 0x7777u;              // 3-bit magnitude indices
  const uint32_t lo = prmt(t.L0, t.L1, mag);
  uint32_t hi = prmt(t.H0, t.H1, mag);
  // byte i of sm = 0xFF when element i is negative: replicate the bit that
  // holds the nibble's sign (c << 4 moves the even nibbles' sign to bit 7)
  const uint32_t sm = prmt(c << 4, c, 0xD9C8u);
  hi |= sm & 0x80808080u;
  o0 = prmt(lo, hi, 0x5140u);                    // (lo0,hi0,lo1,hi1): elements 0, 1
  o1 = prmt(lo, hi, 0x7362u);                    // elements 2, 3
}
// e2m1 code (4 bits) times a power-of-two scale (exact float path).
__device__ __forceinline__ float e2m1_scaled(uint32_t c, float scale) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  const float mag = e ? __uint_as_float(((e + 126u) << 23) | (m << 22)) : (m ? 0.5f : 0.f);
  const float v = mag * scale;
  return (c & 8u) ? -v : v;
}
__device__ __forceinline__ float ue8m0_value(uint32_t u) {
  return u ? __uint_as_float(u << 23) : __uint_as_float(0x00400000u);  // 2^(u-127)
}
// Two e4m3 codes (low byte first) -> two floats, exactly (e4m3 is a subset of f16).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(two)));
  __half2 hh = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(hh);
}
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 16-B chunk c (elements 8c .. 8c+7) of a staged record -> 8 bf16.
__device__ __forceinline__ uint4 dequant_chunk(const uint8_t* raw, int kind, int c) {
  if (kind == 2) {  // main KV: 512 e2m1 codes, ue8m0 per 32 elements
    const uint32_t w = *reinterpret_cast<const uint32_t*>(raw + 4 * c);
    const uint32_t u = raw[256 + (c >> 2)];
    uint4 o;
    if (u >= 2u && u <= 252u) {
      const E2m1Tables tb = e2m1_tables(u);
      e2m1x4_bf16(w & 0xFFFFu, tb, o.x, o.y);
      e2m1x4_bf16(w >> 16, tb, o.z, o.w);
    } else {
      const float sc = ue8m0_value(u);
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t byte = (w >> (8 * e)) & 0xFFu;
        pk[e] = pack_bf16(e2m1_scaled(byte & 0xFu, sc), e2m1_scaled(byte >> 4, sc));
      }
      o = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    return o;
  }
  if (kind == 1) {  // SWA: 512 e4m3 codes, fp32 scale per 128 channels
    const uint2 w = *reinterpret_cast<const uint2*>(raw + 8 * c);
    const float sc = *reinterpret_cast<const float*>(raw + 512 + (c >> 4) * 4);
    const float2 a = e4m3x2_to_float2(w.x & 0xFFFFu), b = e4m3x2_to_float2(w.x >> 16);
    const float2 d = e4m3x2_to_float2(w.y & 0xFFFFu), e = e4m3x2_to_float2(w.y >> 16);
    return make_uint4(pack_bf16(a.x * sc, a.y * sc), pack_bf16(b.x * sc, b.y * sc), pack_bf16(d.x * sc, d.y * sc),
                      pack_bf16(e.x * sc, e.y * sc));
  }
  return make_uint4(0u, 0u, 0u, 0u);
}

// Slot and kind of key j of row t (kind 0: empty or out of range).
__device__ __forceinline__ int key_slot(const AttnParams& p, int t, int j, int* kind) {
  int slot = -1;
  *kind = 0;
  if (j < p.n_swa) {
    slot = __ldg(p.swa_slot + static_cast<long long>(t) * p.ld_swa + j);
    // bounded replay: slot j holds position q_pos - n_swa + 1 + j; keys before
    // the segment start are not attended to
    if (p.swa_seg_start &&
        static_cast<long long>(__ldg(p.q_pos + t)) - p.n_swa + 1 + j < __ldg(p.swa_seg_start + t))
      slot = -1;
    if (slot >= p.swa_slots) {
      set_error(p.err, kErrBounds);
      slot = -1;
    }
    if (slot >= 0) *kind = 1;
  } else if (j < p.n_swa + p.k) {
    slot = __ldg(p.topk_slot + static_cast<long long>(t) * p.ld_topk + (j - p.n_swa));
    if (slot >= p.main_slots) {
      set_error(p.err, kErrBounds);
      slot = -1;
    }
    if (slot >= 0) *kind = 2;
  }
  return slot;
}

__global__ void __launch_bounds__(512, 1) sparse_attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(128) uint8_t sm[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(sm + AttnSmem::kOffQ);
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(sm + AttnSmem::kOffK);
  uint8_t* sRaw = sm + AttnSmem::kOffRaw;
  float* sS = reinterpret_cast<float*>(sm + AttnSmem::kOffS);
  __nv_bfloat16* sP = reinterpret_cast<__nv_bfloat16*>(sm + AttnSmem::kOffP);
  float* sM = reinterpret_cast<float*>(sm + AttnSmem::kOffStats);
  float* sL = sM + kH;
  float* sA = sL + kH;
  int* sKind = reinterpret_cast<int*>(sm + AttnSmem::kOffKind);
  uint64_t* bar_q = reinterpret_cast<uint64_t*>(sm + AttnSmem::kOffBars);
  uint64_t* bar_raw = bar_q + 1;
  uint64_t* bar_recv = bar_q + 2;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.y;
  const uint32_t rank = (p.nsplit > 1) ? cluster_rank() : 0u;
  const int L = p.n_swa + p.k;
  const int nchunks = (L + kCK - 1) / kCK;
  const int c0 = static_cast<int>(rank) * p.chunks_per_split;
  const int c1 = min(c0 + p.chunks_per_split, nchunks);

  if (tid == 0) {
    mbar_init(bar_q, kH);     // one arrival per q row copy
    mbar_init(bar_raw, kCK);  // one arrival per key of a chunk
    mbar_init(bar_recv, 1);   // the merge: one local arrival + the bytes pushed by the cluster
    fence_mbar_init();
  }
  if (tid < kH) {
    sM[tid] = -INFINITY;
    sL[tid] = 0.f;
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  const uint64_t pol = l2_policy_evict_first();
  // q rows and the first chunk's records: bulk copies, one per thread of the first 64
  int next_slot = -1, next_kind = 0;
  if (tid < kCK) {
    mbar_arrive_expect_tx(bar_q, kD * 2);
    bulk_load(sQ + tid * kQStride, p.q + (static_cast<long long>(t) * kH + tid) * kD, kD * 2, bar_q,
              l2_policy_evict_last());
    if (c0 < c1) next_slot = key_slot(p, t, c0 * kCK + tid, &next_kind);
  }
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  const int hg = warp & 3;       // 16-head group
  const int xg = warp >> 2;      // S: 16-key group; PV: 128-dim group
  const int g = lane >> 2, cq = lane & 3;
  bool ok = true;

  // records of one chunk, key = tid (threads 0..63)
  auto issue_records = [&](int slot, int kind) {
    sKind[tid] = kind;
    if (kind == 0) {
      mbar_arrive(bar_raw);
    } else {
      const uint32_t bytes = kind == 1 ? 528u : 288u;
      const uint8_t* src = (kind == 1 ? p.swa_kv : p.main_kv) + static_cast<long long>(slot) * bytes;
      mbar_arrive_expect_tx(bar_raw, bytes);
      bulk_load(sRaw + tid * kRawStride, src, bytes, bar_raw, pol);
    }
  };
  if (tid < kCK && c0 < c1) issue_records(next_slot, next_kind);

  int it = 0;
  for (int ch = c0; ch < c1; ++ch, ++it) {
    // the next chunk's slots load now; its records are issued once this chunk is dequantised
    if (tid < kCK) {
      next_slot = -1;
      next_kind = 0;
      if (ch + 1 < c1) next_slot = key_slot(p, t, (ch + 1) * kCK + tid, &next_kind);
    }
    if (ok) ok = mbar_wait(bar_raw, static_cast<uint32_t>(it & 1), nullptr);
    if (!ok) set_error(p.err, kErrTimeout);
    // ---- dequantise: warp w owns keys 4w..4w+3, lane l the 16-B chunks l and l+32 of each
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int key = warp * 4 + kk;
      const int kind = ok ? sKind[key] : 0;
      const uint8_t* raw = sRaw + key * kRawStride;
      uint4* dst = reinterpret_cast<uint4*>(sK + key * kQStride);
      dst[lane] = dequant_chunk(raw, kind, lane);
      dst[lane + 32] = dequant_chunk(raw, kind, lane + 32);
    }
    const unsigned kmask_lo = __ballot_sync(0xffffffffu, ok && sKind[lane] != 0);
    const unsigned kmask_hi = __ballot_sync(0xffffffffu, ok && sKind[32 + lane] != 0);
    __syncthreads();  // sK ready; the staging area and sKind are free again
    if (tid < kCK && ch + 1 < c1) issue_records(next_slot, next_kind);
    if (it == 0) {
      if (ok) ok = mbar_wait(bar_q, 0u, nullptr);
      if (!ok) set_error(p.err, kErrTimeout);
    }

    // ---- S tile: heads 16hg.., keys 16xg.., all 512 dims
    {
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const uint32_t aBase = smem_u32(sQ + (16 * hg + (lane & 15)) * kQStride + (lane >> 4) * 8);
      const uint32_t bBase =
          smem_u32(sK + (16 * xg + (lane & 7) + ((lane >> 4) << 3)) * kQStride + ((lane >> 3) & 1) * 8);
#pragma unroll 8
      for (int ks = 0; ks < kD / 16; ++ks) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(aBase + ks * 32, a0, a1, a2, a3);
        ldsm_x4(bBase + ks * 32, b0, b1, b2, b3);
        mma_bf16(acc[0], a0, a1, a2, a3, b0, b1);
        mma_bf16(acc[1], a0, a1, a2, a3, b2, b3);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int col = 16 * xg + nt * 8 + 2 * cq;
        sS[(16 * hg + g) * kSStride + col] = acc[nt][0];
        sS[(16 * hg + g) * kSStride + col + 1] = acc[nt][1];
        sS[(16 * hg + g + 8) * kSStride + col] = acc[nt][2];
        sS[(16 * hg + g + 8) * kSStride + col + 1] = acc[nt][3];
      }
    }
    __syncthreads();

    // ---- online softmax: thread -> (head tid/8, keys 8*(tid%8)..)
    {
      const int h = tid >> 3, sub = tid & 7;
      float x[8];
      float cmax = -INFINITY;
      const unsigned km = (sub < 4) ? kmask_lo : kmask_hi;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int key = sub * 8 + i;
        x[i] = ((km >> (key & 31)) & 1u) ? sS[h * kSStride + key] * p.scale_log2 : -INFINITY;
        cmax = fmaxf(cmax, x[i]);
      }
      cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 1));
      cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 2));
      cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 4));
      const float m_old = sM[h];
      const float m_new = fmaxf(m_old, cmax);
      float sum = 0.f;
      uint32_t packed[4];
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        const float e0 = (m_new == -INFINITY) ? 0.f : exp2f(x[i] - m_new);
        const float e1 = (m_new == -INFINITY) ? 0.f : exp2f(x[i + 1] - m_new);
        sum += e0 + e1;
        packed[i / 2] = pack_bf16(e0, e1);
      }
      *reinterpret_cast<uint4*>(sP + h * kPStride + sub * 8) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      sum += __shfl_xor_sync(0xffffffffu, sum, 4);
      __syncwarp();
      if (sub == 0) {
        const float alpha = (m_old == -INFINITY) ? 0.f : exp2f(m_old - m_new);
        sA[h] = alpha;
        sL[h] = sL[h] * alpha + sum;
        sM[h] = m_new;
      }
    }
    __syncthreads();

    // ---- O += P V: heads 16hg.., dims 128xg..
    {
      const float al0 = sA[16 * hg + g], al1 = sA[16 * hg + g + 8];
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        o[nt][0] *= al0;
        o[nt][1] *= al0;
        o[nt][2] *= al1;
        o[nt][3] *= al1;
      }
      const uint32_t aBase = smem_u32(sP + (16 * hg + (lane & 15)) * kPStride + (lane >> 4) * 8);
      const int mi = lane >> 3, rr = lane & 7;
      const uint32_t vBase = smem_u32(sK + (rr + (mi & 1) * 8) * kQStride + 128 * xg + (mi >> 1) * 8);
#pragma unroll
      for (int ks = 0; ks < kCK / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(aBase + ks * 32, a0, a1, a2, a3);
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vBase + (ks * 16 * kQStride + np * 16) * 2, b0, b1, b2, b3);
          mma_bf16(o[2 * np], a0, a1, a2, a3, b0, b1);
          mma_bf16(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();
  }
  if (c0 >= c1 && ok) {  // a CTA without chunks still owns the copies of q
    ok = mbar_wait(bar_q, 0u, nullptr);
    if (!ok) set_error(p.err, kErrTimeout);
  }

  const int h0 = 16 * hg + g, h1 = h0 + 8;
  const long long obase = static_cast<long long>(t) * kH * kD;
  if (p.nsplit == 1) {
    const float s0 = __ldg(p.sink + h0) * kLog2e, s1 = __ldg(p.sink + h1) * kLog2e;
    const float m0 = sM[h0], m1 = sM[h1];
    const float M0 = fmaxf(m0, s0), M1 = fmaxf(m1, s1);
    const float w0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - M0);
    const float w1 = (m1 == -INFINITY) ? 0.f : exp2f(m1 - M1);
    const float d0 = sL[h0] * w0 + exp2f(s0 - M0);
    const float d1 = sL[h1] * w1 + exp2f(s1 - M1);
    const float f0 = w0 / d0, f1 = w1 / d1;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int d = 128 * xg + nt * 8 + 2 * cq;
      float a0 = o[nt][0] * f0, b0 = o[nt][1] * f0, a1 = o[nt][2] * f1, b1 = o[nt][3] * f1;
      if (p.inv_rope && d >= kD - 64) {  // (d, d + 1) is RoPE pair (d - 448) / 2
        const long long pos = __ldg(p.q_pos + t);
        const uint64_t fr = p.inv_freq[(d - (kD - 64)) >> 1];
        inv_rope_pair(a0, b0, pos, fr);
        inv_rope_pair(a1, b1, pos, fr);
      }
      if (p.out_bf16) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + obase;
        *reinterpret_cast<__nv_bfloat162*>(out + h0 * kD + d) = __floats2bfloat162_rn(a0, b0);
        *reinterpret_cast<__nv_bfloat162*>(out + h1 * kD + d) = __floats2bfloat162_rn(a1, b1);
      } else {
        float* out = static_cast<float*>(p.out) + obase;
        *reinterpret_cast<float2*>(out + h0 * kD + d) = make_float2(a0, b0);
        *reinterpret_cast<float2*>(out + h1 * kD + d) = make_float2(a1, b1);
      }
    }
    if (p.lse && xg == 0 && cq == 0) {
      p.lse[static_cast<long long>(t) * kH + h0] = (M0 + log2f(d0)) * kLn2;
      p.lse[static_cast<long long>(t) * kH + h1] = (M1 + log2f(d1)) * kLn2;
    }
    return;
  }

  // ---- merge over the cluster.  Head h belongs to CTA h % ns.  The CTAs
  // exchange their (max, sum) per head, each scales its O rows by its weight
  // exp2(max_r - M) / denominator and stores them as bf16, bulk copies push each
  // 1-KB head row to the owner, and the owner sums its heads' rows.
  const int ns = p.nsplit;
  const int rows_pr = recv_rows_per_rank(ns);                 // receive rows per source rank
  const int my_heads = (kH - static_cast<int>(rank) + ns - 1) / ns;
  __nv_bfloat16* sendO = reinterpret_cast<__nv_bfloat16*>(sm + AttnSmem::kOffSend);  // [64][kQStride]
  __nv_bfloat16* recvO = reinterpret_cast<__nv_bfloat16*>(sm + AttnSmem::kOffRecv);  // [ns][rows_pr][512]
  cluster_sync();  // (max, sum) of every CTA final; q, K and the staging area no longer read
  float* sF = sA;  // this CTA's weight per head
  if (tid < kH) {
    const int h = tid;
    float mr[kMaxCluster], lr[kMaxCluster];
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) {
      mr[r] = -INFINITY;
      lr[r] = 0.f;
      if (r < ns) {
        mr[r] = ld_cluster_f32(map_rank(smem_u32(&sM[h]), r));
        lr[r] = ld_cluster_f32(map_rank(smem_u32(&sL[h]), r));
      }
    }
    const float sk = __ldg(p.sink + h) * kLog2e;
    float M = sk;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) M = fmaxf(M, mr[r]);
    float dsum = exp2f(sk - M);
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      if (mr[r] != -INFINITY) dsum += exp2f(mr[r] - M) * lr[r];
    const float mine = sM[h];
    sF[h] = (mine == -INFINITY) ? 0.f : exp2f(mine - M) / dsum;
    if (p.lse && static_cast<uint32_t>(h % ns) == rank)
      p.lse[static_cast<long long>(t) * kH + h] = (M + log2f(dsum)) * kLn2;
  }
  if (tid == 0) mbar_arrive_expect_tx(bar_recv, static_cast<uint32_t>(ns * my_heads * kD * 2));
  __syncthreads();
  {
    const float f0 = sF[h0], f1 = sF[h1];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int d = 128 * xg + nt * 8 + 2 * cq;
      *reinterpret_cast<__nv_bfloat162*>(sendO + h0 * kQStride + d) = __floats2bfloat162_rn(o[nt][0] * f0, o[nt][1] * f0);
      *reinterpret_cast<__nv_bfloat162*>(sendO + h1 * kQStride + d) = __floats2bfloat162_rn(o[nt][2] * f1, o[nt][3] * f1);
    }
  }
  fence_proxy_async_smem();  // the rows are read next by the bulk-copy engine
  cluster_sync();            // every send row written, every receive barrier armed
  if (tid < kH) {
    const int h = tid;
    const uint32_t owner = static_cast<uint32_t>(h % ns);
    const uint32_t dst = map_rank(smem_u32(recvO + (static_cast<int>(rank) * rows_pr + h / ns) * kD), owner);
    bulk_copy_to_peer(dst, sendO + h * kQStride, kD * 2, map_rank(smem_u32(bar_recv), owner));
  }
  if (!mbar_wait(bar_recv, 0u, nullptr)) set_error(p.err, kErrTimeout);
  {
    constexpr int kPerHead = kD / 8;  // 8 bf16 per thread and step
    for (int i = tid; i < my_heads * kPerHead; i += blockDim.x) {
      const int li = i / kPerHead;
      const int h = static_cast<int>(rank) + li * ns;
      const int d = (i % kPerHead) * 8;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int r = 0; r < ns; ++r) {
        const uint4 v = *reinterpret_cast<const uint4*>(recvO + (r * rows_pr + li) * kD + d);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[j]));
          acc[2 * j] += f2.x;
          acc[2 * j + 1] += f2.y;
        }
      }
      if (p.inv_rope && d >= kD - 64) {
        const long long pos = __ldg(p.q_pos + t);
#pragma unroll
        for (int j = 0; j < 4; ++j) inv_rope_pair(acc[2 * j], acc[2 * j + 1], pos, p.inv_freq[(d - (kD - 64)) / 2 + j]);
      }
      const long long oo = obase + static_cast<long long>(h) * kD + d;
      if (p.out_bf16) {
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + oo) =
            make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]), pack_bf16(acc[4], acc[5]),
                       pack_bf16(acc[6], acc[7]));
      } else {
        float4* out = reinterpret_cast<float4*>(static_cast<float*>(p.out) + oo);
        out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      }
    }
  }
  cluster_sync();  // no CTA leaves while its rows may still be copied out of its shared memory
}


// ================================================================ tensor-core path
// One CTA per 80-key chunk of a row; the row's CTAs form a cluster.  Per CTA:
//   * the row's q (64 heads x 512, bf16) and the chunk's records are staged in
//     shared memory; the records are dequantised to bf16 key rows.  Both tiles
//     use the 128-byte swizzled layout of the tensor cores: 8 atoms of 64
//     dims, each [64 rows x 128 B], rows of an atom 1024 B per group of 8.
//   * S = q K^T on tcgen05 (M = 64 heads, N = 80 keys, K = 512) into TMEM;
//     an M = 64 accumulator puts head h in lane 32 (h / 16) + h % 16.
//   * four lanes per head (4 warps, one per TMEM lane quadrant) read its S
//     row, mask absent keys, and form P = exp2(S*scale - max) (bf16, swizzled)
//     with its max and sum, combined across the four lanes by shuffles.
//   * O = P V on tcgen05 (M = 64 heads, N = 256 dims twice, K = 80 keys; V
//     is the key tile read MN-major) into TMEM.
//   * O / sum is stored as bf16 straight from the accumulator into a per-row
//     scratch in global memory, with (max, sum) per head; after a cluster
//     barrier the CTA of rank r loads its range of heads of every chunk from
//     L2 and combines them with the sink.
// Scratch of one chunk: O / sum as bf16 in [64 blocks of 8 dims][64 heads][16 B]
// (a readout warp's 16 heads of one block are 256 contiguous bytes), plus
// (max, sum) per head in a separate array [rows][chunks][64] of float2.
constexpr int kPartBlocks = kD / 8;                     // blocks of 8 dims
constexpr int kPartBlockBytes = kH * 16;                // one block: 64 heads x 8 bf16
constexpr int kPartChunkBytes = kPartBlocks * kPartBlockBytes;
constexpr int kTcKeys = 80;  // keys per CTA: 640 keys of a decode row in 8 CTAs, so two clusters share a GPC
struct TcSmem {
  static constexpr int kQAtom = 8192;                           // 64 rows x 128 B (q, P)
  static constexpr int kKAtom = kTcKeys * 128;                  // 80 key rows x 128 B
  static constexpr int kOffQ = 0;                               // 8 q atoms
  static constexpr int kOffK = kOffQ + 8 * kQAtom;              // 8 key atoms
  static constexpr int kOffP = kOffK + 8 * kKAtom;              // 2 P atoms: keys 0-63, keys 64-79
  static constexpr int kOffRaw = kOffP + 2 * kQAtom;            // [kTcKeys][kRawStride]
  static constexpr int kOffKind = kOffRaw + kTcKeys * kRawStride;  // int[kTcKeys]
  static constexpr int kOffStat = kOffKind + kTcKeys * 4;       // float m[64], l[64], sink[64]
  static constexpr int kOffBar = kOffStat + 3 * kH * 4;             // raw, S done, O halves done, q halves
  static constexpr int kOffTmem = kOffBar + 6 * 8;
  static constexpr int kBytes = kOffTmem + 8;
  static constexpr int kAlloc = kBytes + 1024;                  // the base is rounded up to 1024 B
  static_assert(kKAtom % 1024 == 0 && kOffK % 1024 == 0 && kOffP % 1024 == 0, "swizzle atoms are 1024-B aligned");
  static_assert(kAlloc <= 227 * 1024, "one CTA per SM");
};
constexpr int kTcWorkers = 640;              // dequantisation (80 keys x 8 blocks per wave), softmax, readout, combine
constexpr int kTcThreads = kTcWorkers;       // 20 warps: 5 per SM sub-partition, up to 96 registers a thread
constexpr int kTcMmaThread = 19 * 32;         // issues the copies and MMAs; its warp takes no part in softmax or readout
constexpr uint32_t kTmemCols = 512;  // O: 2 x 256 columns; S (64 columns) shares the second half

struct TcParams {
  const __nv_bfloat16* q;
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
  float scale_log2;
  int T;          // rows of this launch
  int t_base;     // first row
  int out_bf16;
  void* out;
  float* lse;
  int kv_ready;   // gather the keys before the dependency wait
  int nsplit;     // CTAs (80-key chunks) per row = cluster size
  uint8_t* part;     // [T][nsplit][64 blocks][64 heads][16 B]: O / sum of each chunk (bf16)
  float2* part_ml;   // [T][nsplit][64]: (max, sum) of each chunk and head, log2 units
  uint32_t* err;
  const int* q_pos;          // [T] query positions (inverse RoPE, bounded replay)
  const int* swa_seg_start;  // [T] bounded-replay segment starts, or null
  int inv_rope;              // rotate the output's last 64 dims back by the query's RoPE
  uint64_t inv_freq[32];     // theta^(-2p/64) as a fixed-point turn rate (rope_turn_rate)
};

__device__ __forceinline__ int key_slot_tc(const TcParams& p, int t, int j, int* kind) {
  int slot = -1;
  *kind = 0;
  if (j < p.n_swa) {
    slot = __ldg(p.swa_slot + static_cast<long long>(t) * p.ld_swa + j);
    // bounded replay: slot j holds position q_pos - n_swa + 1 + j; keys before
    // the segment start are not attended to
    if (p.swa_seg_start &&
        static_cast<long long>(__ldg(p.q_pos + t)) - p.n_swa + 1 + j < __ldg(p.swa_seg_start + t))
      slot = -1;
    if (slot >= p.swa_slots) {
      set_error(p.err, kErrBounds);
      slot = -1;
    }
    if (slot >= 0) *kind = 1;
  } else if (j < p.n_swa + p.k) {
    slot = __ldg(p.topk_slot + static_cast<long long>(t) * p.ld_topk + (j - p.n_swa));
    if (slot >= p.main_slots) {
      set_error(p.err, kErrBounds);
      slot = -1;
    }
    if (slot >= 0) *kind = 2;
  }
  return slot;
}

// 32 dims (block b) of one staged record -> 32 bf16 in o[0..3] (8 each).
__device__ __forceinline__ void dequant_block32(const uint8_t* raw, int kind, int b, uint4 (&o)[4]) {
  if (kind == 2) {  // main KV: e2m1 codes, one ue8m0 scale per 32 dims
    const uint4 w = *reinterpret_cast<const uint4*>(raw + 16 * b);
    const uint32_t u = raw[256 + b];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    if (u >= 2u && u <= 252u) {
      const E2m1Tables tb = e2m1_tables(u);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        e2m1x4_bf16(ws[j] & 0xFFFFu, tb, o[j].x, o[j].y);
        e2m1x4_bf16(ws[j] >> 16, tb, o[j].z, o[j].w);
      }
    } else {
      const float sc = ue8m0_value(u);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t byte = (ws[j] >> (8 * e)) & 0xFFu;
          pk[e] = pack_bf16(e2m1_scaled(byte & 0xFu, sc), e2m1_scaled(byte >> 4, sc));
        }
        o[j] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
  } else if (kind == 1) {  // SWA: e4m3 codes, one fp32 scale per 128 dims
    const uint4 w0 = *reinterpret_cast<const uint4*>(raw + 32 * b);
    const uint4 w1 = *reinterpret_cast<const uint4*>(raw + 32 * b + 16);
    const float sc = *reinterpret_cast<const float*>(raw + 512 + (b >> 2) * 4);
    const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 a = e4m3x2_to_float2(ws[j] & 0xFFFFu), c = e4m3x2_to_float2(ws[j] >> 16);
      pk[2 * j] = pack_bf16(a.x * sc, a.y * sc);
      pk[2 * j + 1] = pack_bf16(c.x * sc, c.y * sc);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = make_uint4(0u, 0u, 0u, 0u);
  }
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


// One dequantisation wave of the chunk: thread -> key tid % 80, 32-dim block
// tid / 80 + 8 wave, written as bf16 into the swizzled key atoms; ends in a CTA
// barrier.  Out of line, so the kernel's four call sites share one copy of the
// code: with the copies inlined, Full and Reindex layers (whose waves run after
// the dependency wait) measured 12.4 us a launch against 11.1 us (instruction
// fetches on the critical path), the decode step 0.8564 against 0.8518 ms.
__device__ __noinline__ void tc_dequant_wave(const uint8_t* sRaw, uint8_t* sK, const int* sKind, bool ok, int wave) {
  const int tid = threadIdx.x;
  if (tid < kTcWorkers) {
    const int key = tid % kTcKeys;
    const int b = tid / kTcKeys + 8 * wave;
    uint4 o[4];
    dequant_block32(sRaw + key * kRawStride, ok ? sKind[key] : 0, b, o);
    uint8_t* row = sK + (b >> 1) * TcSmem::kKAtom + key * 128;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = ((b & 1) << 2) + j;
      *reinterpret_cast<uint4*>(row + ((c ^ (key & 7)) << 4)) = o[j];
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
}

// NS: the cluster size when fixed at compile time (8: the 640-key decode row,
// whose instantiation has the combine's per-chunk loops at 8 instead of 16,
// less code on the critical path), or 0 (p.nsplit, up to 16 chunks).
template <int NS>
__global__ void __launch_bounds__(kTcThreads, 1)
    sparse_attn_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ TcParams p) {
  constexpr int kMaxNs = NS > 0 ? NS : kMaxCluster;
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + TcSmem::kOffQ;
  uint8_t* sK = sm + TcSmem::kOffK;
  uint8_t* sP = sm + TcSmem::kOffP;
  uint8_t* sRaw = sm + TcSmem::kOffRaw;
  int* sKind = reinterpret_cast<int*>(sm + TcSmem::kOffKind);
  float* sM = reinterpret_cast<float*>(sm + TcSmem::kOffStat);
  float* sL = sM + kH;
  float* sSink = sL + kH;
  uint64_t* bar_raw = reinterpret_cast<uint64_t*>(sm + TcSmem::kOffBar);
  uint64_t* bar_s = bar_raw + 1;
  uint64_t* bar_o = bar_raw + 2;  // [2]
  uint64_t* bar_q = bar_raw + 4;  // the row's q tile: dims 0-255 on bar_q[0], 256-511 on bar_q[1]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + TcSmem::kOffTmem);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int rank = blockIdx.x;  // the cluster spans gridDim.x
  const int ns = NS > 0 ? NS : p.nsplit;
  const int tl = blockIdx.y;    // row within this launch
  const int t = p.t_base + tl;

  if (tid == 0) {
    mbar_init(bar_raw, kTcKeys);
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init(bar_o + 1, 1);
    mbar_init(bar_q, 1);
    mbar_init(bar_q + 1, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  // ---- records of this chunk (one bulk copy per key): before the dependency
  // wait when the caller marks the slots and caches as written two or more
  // launches earlier (every launch before the previous one has completed when
  // this CTA starts), else after it; then the row's q and the sink
  auto issue_records = [&]() {
    if (tid < kTcKeys) {
      int kind;
      const int slot = key_slot_tc(p, t, rank * kTcKeys + tid, &kind);
      sKind[tid] = kind;
      if (kind == 0) {
        mbar_arrive(bar_raw);
      } else {
        const uint32_t bytes = kind == 1 ? 528u : 288u;
        const uint8_t* src = (kind == 1 ? p.swa_kv : p.main_kv) + static_cast<long long>(slot) * bytes;
        mbar_arrive_expect_tx(bar_raw, bytes);
        bulk_load(sRaw + tid * kRawStride, src, bytes, bar_raw, l2_policy_evict_first());
      }
    }
  };
  // ---- dequantisation: two waves of 4 atoms (256 dims); thread -> key tid % 80,
  // 32-dim block tid / 80 of the wave.  S = q K^T -> TMEM columns 256..335.
  bool ok = true;
  unsigned kmask[3] = {0u, 0u, 0u};  // keys 0-31, 32-63, 64-79 present
  auto wait_records = [&]() {
    ok = mbar_wait(bar_raw, 0u, nullptr);
    if (!ok) set_error(p.err, kErrTimeout);
    kmask[0] = __ballot_sync(0xffffffffu, ok && sKind[lane] != 0);
    kmask[1] = __ballot_sync(0xffffffffu, ok && sKind[32 + lane] != 0);
    kmask[2] = __ballot_sync(0xffffffffu, ok && lane < kTcKeys - 64 && sKind[64 + lane] != 0);
  };
  auto dequant_wave = [&](int wave) {  // every thread calls (it ends in a barrier)
    tc_dequant_wave(sRaw, sK, sKind, ok, wave);
  };
  auto issue_s = [&](int wave) {  // the MMA thread, once q and the wave's keys are in place
    tc_fence_after();
    constexpr uint32_t idesc = idesc_bf16_f32(64, kTcKeys, 0, 0);
#pragma unroll
    for (int a = 4 * wave; a < 4 * wave + 4; ++a) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        umma_bf16(tmem + 256, smem_desc_sw128(sQ + a * TcSmem::kQAtom + kk * 32),
                  smem_desc_sw128(sK + a * TcSmem::kKAtom + kk * 32), idesc, (a | kk) != 0 ? 1u : 0u);
      }
    }
    if (wave == 1) mma_commit(bar_s);
  };
  auto wait_q = [&](int half) {  // the S MMAs of a wave need that half of q only
    if (!mbar_wait(bar_q + half, 0u, nullptr)) set_error(p.err, kErrTimeout);
  };

  // Records and S waves each have one call site (a loop that is not
  // unrolled), so every launch runs the same copy of their code whether the
  // keys are gathered before the dependency wait (kv_ready, pass 0) or after
  // it (pass 1): instruction fetches of code a previous launch has run are
  // cheaper on the critical path.
  const int rec_pass = p.kv_ready ? 0 : 1;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    if (pass == 1) {
      pdl_wait();
      pdl_trigger();
      // the row's q: eight 64-head x 64-dim atoms, swizzled by the tensor copy,
      // in two halves so that the first wave's S MMAs start on the first half
      if (tid == kTcMmaThread) {
        mbar_arrive_expect_tx(bar_q, kH * kD);
        mbar_arrive_expect_tx(bar_q + 1, kH * kD);
#pragma unroll
        for (int a = 0; a < 8; ++a)
          tma_load_2d(sQ + a * TcSmem::kQAtom, &map_q, a * 128, t * kH, bar_q + (a >> 2), l2_policy_evict_first());
      }
      if (tid < kH) sSink[tid] = __ldg(p.sink + tid) * kLog2e;
    }
    if (pass == rec_pass) {
      issue_records();
      wait_records();
      if (pass == 0) {  // kv_ready: both waves before the wait
        dequant_wave(0);
        dequant_wave(1);
      }
    }
  }
  // the S MMAs: after the wait, the first wave's MMAs run while the second
  // wave is dequantised (keys gathered after the wait)
#pragma unroll 1
  for (int w = 0; w < 2; ++w) {
    if (!p.kv_ready) dequant_wave(w);
    if (tid == kTcMmaThread) {
      wait_q(w);
      issue_s(w);
    }
  }

  // ---- softmax of the chunk: warps 0-3, one per TMEM lane quadrant q (an
  // M = 64 accumulator holds heads 16q .. 16q+15 in lanes 0-15 of quadrant q).
  // Three 16x256b loads give lane l heads hA = 16q + l/4 and hB = hA + 8, keys
  // 8g + 2(l%4) and the next of every 8-key group g (keys 80-95 are masked);
  // the four lanes of a head combine max and sum by shuffles.
  if (warp < 4) {
    const int q = warp;
    const int hA = 16 * q + (lane >> 2), hB = hA + 8;
    const int kc = 2 * (lane & 3);  // this lane's first key of each 8-key group
    bool oks = mbar_wait(bar_s, 0u, nullptr);
    if (!oks) set_error(p.err, kErrTimeout);
    tc_fence_after();
    uint32_t r0[16], r1[16], r2[16];
    const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) + 256;
    tmem_ld16x256_x4(ta, r0);
    tmem_ld16x256_x4(ta + 32, r1);
    tmem_ld16x256_x4(ta + 64, r2);
    tmem_wait_ld16(r0);
    tmem_wait_ld16(r1);
    tmem_wait_ld16(r2);
    constexpr int kG = kTcKeys / 8;  // 8-key groups of the chunk
    float xA[2 * kG], xB[2 * kG];
    float mA = -INFINITY, mB = -INFINITY;
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      const uint32_t* rr = (g < 4) ? r0 : (g < 8) ? r1 : r2;
      const int gi = g & 3;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int k = 8 * g + kc + u;
        const bool valid = oks && ((kmask[k >> 5] >> (k & 31)) & 1u);
        xA[2 * g + u] = valid ? __uint_as_float(rr[4 * gi + u]) * p.scale_log2 : -INFINITY;
        xB[2 * g + u] = valid ? __uint_as_float(rr[4 * gi + 2 + u]) * p.scale_log2 : -INFINITY;
        mA = fmaxf(mA, xA[2 * g + u]);
        mB = fmaxf(mB, xB[2 * g + u]);
      }
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, o));
      mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, o));
    }
    float sA = 0.f, sB = 0.f;
    uint8_t* prA = sP + hA * 128;
    uint8_t* prB = sP + hB * 128;
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      const float a0 = (mA == -INFINITY) ? 0.f : ex2_approx(xA[2 * g] - mA);
      const float a1 = (mA == -INFINITY) ? 0.f : ex2_approx(xA[2 * g + 1] - mA);
      const float b0 = (mB == -INFINITY) ? 0.f : ex2_approx(xB[2 * g] - mB);
      const float b1 = (mB == -INFINITY) ? 0.f : ex2_approx(xB[2 * g + 1] - mB);
      sA += a0 + a1;
      sB += b0 + b1;
      // P rows: keys 0-63 in atom 0 (16-B chunks 0-7), keys 64-79 in chunks
      // 0-1 of atom 1; this lane's key pair is bytes 2 kc .. 2 kc + 3 of chunk g % 8
      const int off = (g >> 3) * TcSmem::kQAtom + 2 * kc;
      *reinterpret_cast<uint32_t*>(prA + off + (((g & 7) ^ (hA & 7)) << 4)) = pack_bf16(a0, a1);
      *reinterpret_cast<uint32_t*>(prB + off + (((g & 7) ^ (hB & 7)) << 4)) = pack_bf16(b0, b1);
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      sA += __shfl_xor_sync(0xffffffffu, sA, o);
      sB += __shfl_xor_sync(0xffffffffu, sB, o);
    }
    if ((lane & 3) == 0) {
      sM[hA] = mA;
      sL[hA] = sA;
      sM[hB] = mB;
      sL[hB] = sB;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();

  // ---- O = P V  (dims 0-255 -> columns 0..255, committed to bar_o[0]; dims
  // 256-511 -> columns 256..511, bar_o[1])
  if (tid == kTcMmaThread) {
    tc_fence_after();
    constexpr uint32_t idesc = idesc_bf16_f32(64, 256, 0, 1);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
      for (int kk = 0; kk < kTcKeys / 16; ++kk) {  // 16 keys per step: P atom kk / 4, V rows 16 kk ..
        umma_bf16(tmem + 256 * hh, smem_desc_sw128(sP + (kk >> 2) * TcSmem::kQAtom + (kk & 3) * 32),
                  smem_desc_sw128_mn(sK + 4 * hh * TcSmem::kKAtom + kk * 2048, TcSmem::kKAtom, 1024), idesc,
                  kk != 0 ? 1u : 0u);
      }
      mma_commit(bar_o + hh);  // dims 0-255 done: bar_o[0]; dims 256-511: bar_o[1]
    }
  }

  // ---- partial results: O / sum (bf16) and (max, sum) per head, stored from
  // the accumulator straight into the scratch.  Warps 0-15: lane quadrant
  // warp % 4 (heads 16 q .. 16 q + 15 in its lanes 0-15), column group warp / 4
  // of 128 dims; each 16-B store of a warp covers one 8-dim block of its 16
  // heads (256 contiguous bytes).
  const long long rowbase = static_cast<long long>(tl) * ns;
  if (warp < 16) {
    const int qd = warp & 3, g = warp >> 2;
    const int h = qd * 16 + (lane & 15);
    const bool act = lane < 16;
    bool oko = mbar_wait(bar_o + (g >> 1), 0u, nullptr);  // column groups 0-1: dims 0-255
    if (!oko) set_error(p.err, kErrTimeout);
    tc_fence_after();
    const float l = sL[h];
    const float inv = (l > 0.f && oko) ? 1.f / l : 0.f;
    uint8_t* dst = p.part + (rowbase + rank) * kPartChunkBytes + h * 16;
    // eight 16-column loads, each issued before the previous one is consumed
    const uint32_t tcol = tmem + (static_cast<uint32_t>(qd * 32) << 16) + 128 * g;
    uint32_t ra[16], rb[16];
    tmem_ld32x16_async(tcol, ra);
    tmem_wait_ld16(ra);
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      uint32_t(&cur)[16] = (cc & 1) ? rb : ra;
      uint32_t(&nxt)[16] = (cc & 1) ? ra : rb;
      if (cc + 1 < 8) tmem_ld32x16_async(tcol + 16 * (cc + 1), nxt);
#pragma unroll
      for (int j = 0; j < 2; ++j) {  // block 16 g + 2 cc + j
        const uint32_t* w = cur + 8 * j;
        if (act)
          *reinterpret_cast<uint4*>(dst + (16 * g + 2 * cc + j) * kPartBlockBytes) = make_uint4(
              pack_bf16(__uint_as_float(w[0]) * inv, __uint_as_float(w[1]) * inv),
              pack_bf16(__uint_as_float(w[2]) * inv, __uint_as_float(w[3]) * inv),
              pack_bf16(__uint_as_float(w[4]) * inv, __uint_as_float(w[5]) * inv),
              pack_bf16(__uint_as_float(w[6]) * inv, __uint_as_float(w[7]) * inv));
      }
      if (cc + 1 < 8) tmem_wait_ld16(nxt);
    }
    if (act && g == 0) p.part_ml[(rowbase + rank) * kH + h] = make_float2(oko ? sM[h] : -INFINITY, oko ? l : 0.f);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();  // every chunk's partial of this row is in the scratch
  float* sRope = sM;  // (cos, sin) of the 32 RoPE pairs at the query's position; sM is no longer read
  if (p.inv_rope && tid < 32) {
    float sn, cs;
    rope_angle(__ldg(p.q_pos + t), p.inv_freq[tid], &sn, &cs);
    sRope[2 * tid] = cs;
    sRope[2 * tid + 1] = sn;
  }

  // ---- combine: this CTA owns heads [hb, hb + nh).  The cluster barrier
  // above orders the chunks' stores before these loads (L2, generic proxy
  // on both sides).  A thread takes one head and 8-dim block: the chunk
  // weights exp2(max_r - M) sum_r / D (the sink in D) from the (max, sum)
  // pairs, then the weighted sum of the chunks' O / sum.
  const int hb = (kH * rank) / ns;
  const int nh = (kH * (rank + 1)) / ns - hb;
  if (p.inv_rope) __syncthreads();  // sRope written
  for (int task = tid; task < nh * kPartBlocks; task += kTcThreads) {
    // consecutive threads: consecutive heads, then blocks (64-B runs of nh
    // heads per load and store of a warp)
    const int li = task % nh, c = task / nh;
    const int h = hb + li;
    const uint8_t* src = p.part + (rowbase * kPartBlocks + c) * kPartBlockBytes + h * 16;
    auto load_batch = [&](int r0, uint4 (&pv)[8]) {
#pragma unroll
      for (int r = 0; r < 8; ++r)
        pv[r] = (r0 + r < ns) ? __ldcg(reinterpret_cast<const uint4*>(src + static_cast<long long>(r0 + r) * kPartChunkBytes))
                              : make_uint4(0u, 0u, 0u, 0u);
    };
    // the first 8 chunks' rows are requested before the (max, sum) pairs, so
    // both arrive in one round trip to L2
    uint4 pv[8];
    load_batch(0, pv);
    float wr[kMaxNs], ml_l[kMaxNs];
    float M = sSink[h];
#pragma unroll
    for (int r = 0; r < kMaxNs; ++r) {
      float2 ml = make_float2(-INFINITY, 0.f);
      if (r < ns) ml = __ldcg(p.part_ml + (rowbase + r) * kH + h);
      wr[r] = ml.x;
      M = fmaxf(M, ml.x);
      ml_l[r] = ml.y;
    }
    float D = ex2_approx(sSink[h] - M);
#pragma unroll
    for (int r = 0; r < kMaxNs; ++r) {
      wr[r] = (wr[r] == -INFINITY) ? 0.f : ex2_approx(wr[r] - M) * ml_l[r];
      D += wr[r];
    }
    const float invD = 1.f / D;
    if (c == 0 && p.lse) p.lse[static_cast<long long>(t) * kH + h] = (M + log2f(D)) * kLn2;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r0 = 0; r0 < kMaxNs; r0 += 8) {  // 8 chunks' loads in flight at a time
      if (r0 > 0) {
        if (r0 >= ns) break;
        load_batch(r0, pv);
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float w = wr[r0 + r] * invD;
        const uint32_t wv[4] = {pv[r].x, pv[r].y, pv[r].z, pv[r].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[j]));
          acc[2 * j] = fmaf(w, f2.x, acc[2 * j]);
          acc[2 * j + 1] = fmaf(w, f2.y, acc[2 * j + 1]);
        }
      }
    }
    if (p.inv_rope && c >= (kD - 64) / 8) {  // dims 8c .. 8c+7 are RoPE pairs 4(c - 56) .. +3
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int pp = 4 * (c - (kD - 64) / 8) + j;
        const float cs = sRope[2 * pp], sn = sRope[2 * pp + 1];
        const float x = acc[2 * j], y = acc[2 * j + 1];
        acc[2 * j] = x * cs + y * sn;
        acc[2 * j + 1] = y * cs - x * sn;
      }
    }
    const long long oo = (static_cast<long long>(t) * kH + h) * kD + 8 * c;
    if (p.out_bf16) {
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + oo) =
          make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]), pack_bf16(acc[4], acc[5]),
                     pack_bf16(acc[6], acc[7]));
    } else {
      float4* out = reinterpret_cast<float4*>(static_cast<float*>(p.out) + oo);
      out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
  }
}

}  // namespace

// CTAs per row: one per 64-key chunk while the rows of the launch still fit the
// SMs with one CTA each, at most 16 (the cluster limit); the chunks are then
// spread evenly over that many CTAs.
int attn_num_splits(int T, int n_keys, int num_sms) {
  const int nchunks = (n_keys + kCK - 1) / kCK;
  if (nchunks <= 1) return 1;
  int s = num_sms / (T > 0 ? T : 1);
  if (s < 1) s = 1;
  if (s > nchunks) s = nchunks;
  if (s > kMaxCluster) s = kMaxCluster;
  const int cps = (nchunks + s - 1) / s;
  return (nchunks + cps - 1) / cps;
}

// The tensor-core path takes rows of 1..16 chunks (up to 1280 keys), one CTA
// per chunk, in launches of at most kTcRowsPerLaunch rows sharing one scratch.
// It is a latency design (a row's chunks in parallel on a cluster, merged
// through L2): it is taken while all rows' CTAs fit one wave (rows x chunks
// <= SMs, e.g. 8-row decode layers).  Beyond that the split-K kernel, fewer
// CTAs a row each walking its chunks with an online softmax, measured faster
// (640 keys a row: 28 against 31 us at 32 rows, 477 against 785 us at 1,024
// rows, 1.84 against 3.14 ms for a 4,096-query prefill chunk; 16 against
// 10.6 us at 8 rows).
constexpr int kTcRowsPerLaunch = 256;
static bool use_tc_path(int T, int n_keys, int num_sms) {
  const int nchunks = (n_keys + kTcKeys - 1) / kTcKeys;
  return nchunks >= 1 && nchunks <= kMaxCluster && static_cast<long long>(T) * nchunks <= num_sms;
}
static size_t tc_part_bytes(int rows, int nchunks) {
  return static_cast<size_t>(rows) * nchunks * (kPartChunkBytes + kH * sizeof(float2));
}

size_t attn_workspace_bytes(int T, int n_keys, int num_sms) {
  if (!use_tc_path(T, n_keys, num_sms)) return 0;  // the split-K kernel merges on chip
  const int nchunks = (n_keys + kTcKeys - 1) / kTcKeys;
  const int rows = T < kTcRowsPerLaunch ? T : kTcRowsPerLaunch;
  return tc_part_bytes(rows, nchunks);
}

static cudaError_t launch_sparse_attn_tc(const AttnLaunch& a, void* ws, const DeviceCtx& ctx, cudaStream_t st) {
  const int L = a.n_swa + a.k;
  const int nchunks = (L + kTcKeys - 1) / kTcKeys;
  TcParams p;
  p.q = reinterpret_cast<const __nv_bfloat16*>(a.q);
  p.main_kv = a.main_kv;
  p.main_slots = a.main_slots;
  p.topk_slot = a.topk_slot;
  p.k = a.k;
  p.ld_topk = a.ld_topk;
  p.swa_kv = a.swa_kv;
  p.swa_slots = a.swa_slots;
  p.swa_slot = a.swa_slot;
  p.n_swa = a.n_swa;
  p.ld_swa = a.ld_swa;
  p.sink = a.sink;
  p.scale_log2 = a.scale * kLog2e;
  p.out_bf16 = a.out_bf16;
  p.out = a.out;
  p.lse = a.lse;
  p.kv_ready = a.kv_ready;
  p.nsplit = nchunks;
  p.err = ctx.err;
  // scratch: O / sum of [rows][chunks] as 2-D rows of 64 heads x 16 B (one row
  // per 8-dim block), then (max, sum) [rows][chunks][64]
  const int rows_max = a.T < kTcRowsPerLaunch ? a.T : kTcRowsPerLaunch;
  p.part = static_cast<uint8_t*>(ws);
  p.part_ml = reinterpret_cast<float2*>(p.part + static_cast<size_t>(rows_max) * nchunks * kPartChunkBytes);
  p.q_pos = a.q_pos;
  p.swa_seg_start = a.swa_seg_start;
  p.inv_rope = a.inv_rope;
  for (int i = 0; i < 32; ++i) p.inv_freq[i] = rope_turn_rate(static_cast<double>(a.rope_theta), i);
  // q viewed as [T*64 rows of 1024 B]; a 128-B x 64-row box is one swizzled atom
  CUtensorMap map_q;
  if (encode_tmap_2d_u8(&map_q, a.q, static_cast<uint64_t>(kD) * 2, static_cast<uint64_t>(a.T) * kH,
                        static_cast<uint64_t>(kD) * 2, 128, kH) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // rows of 8 chunks (640 keys: 128 SWA + 512) take the instantiation with the
  // cluster size fixed at 8
  auto kern = nchunks == 8 ? sparse_attn_tc_kernel<8> : sparse_attn_tc_kernel<0>;
  cudaError_t e = prefer_max_smem(kern, TcSmem::kAlloc);
  if (e != cudaSuccess) return e;
  if (nchunks > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  for (int t0 = 0; t0 < a.T; t0 += kTcRowsPerLaunch) {
    p.t_base = t0;
    p.T = (a.T - t0) < kTcRowsPerLaunch ? (a.T - t0) : kTcRowsPerLaunch;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nchunks, p.T);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = TcSmem::kAlloc;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = nchunks;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, map_q, p);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_sparse_attn(const AttnLaunch& a, void* ws, size_t ws_bytes, const DeviceCtx& ctx,
                               cudaStream_t st) {
  (void)ws_bytes;
  if (use_tc_path(a.T, a.n_swa + a.k, ctx.num_sms)) return launch_sparse_attn_tc(a, ws, ctx, st);
  AttnParams p;
  p.q = reinterpret_cast<const __nv_bfloat16*>(a.q);
  p.main_kv = a.main_kv;
  p.main_slots = a.main_slots;
  p.topk_slot = a.topk_slot;
  p.k = a.k;
  p.ld_topk = a.ld_topk;
  p.swa_kv = a.swa_kv;
  p.swa_slots = a.swa_slots;
  p.swa_slot = a.swa_slot;
  p.n_swa = a.n_swa;
  p.ld_swa = a.ld_swa;
  p.sink = a.sink;
  p.scale_log2 = a.scale * kLog2e;
  p.T = a.T;
  p.out_bf16 = a.out_bf16;
  p.out = a.out;
  p.lse = a.lse;
  p.err = ctx.err;
  p.q_pos = a.q_pos;
  p.swa_seg_start = a.swa_seg_start;
  p.inv_rope = a.inv_rope;
  for (int i = 0; i < 32; ++i) p.inv_freq[i] = rope_turn_rate(static_cast<double>(a.rope_theta), i);
  const int L = a.n_swa + a.k;
  const int nchunks = (L + kCK - 1) / kCK;
  const int nsplit = attn_num_splits(a.T, L, ctx.num_sms);
  cudaError_t e = prefer_max_smem(sparse_attn_kernel, AttnSmem::kBytes);
  if (e != cudaSuccess) return e;
  if (nsplit > 8) {
    e = cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  p.nsplit = nsplit;
  p.chunks_per_split = nsplit > 1 ? (nchunks + nsplit - 1) / nsplit : (nchunks > 0 ? nchunks : 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nsplit, a.T);
  cfg.blockDim = dim3(512);
  cfg.dynamicSmemBytes = AttnSmem::kBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = nsplit;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, sparse_attn_kernel, p);
}

}  // namespace csa2
