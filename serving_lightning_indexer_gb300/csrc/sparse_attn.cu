// MQA sparse attention over SWA keys + selected main-KV entries + attention sink.
//
// CSA2 page, "一层 CSA2 的 attention 具体怎么算" (attention equation): per
// query row t and head i, one joint softmax over the layer's SWA keys and the
// <= k main-KV entries of the row's top-k, with the per-head sink s_i only in
// the denominator; K = V is one shared 512-vector (MQA, 64 heads).
//
// A CTA takes one query row and a contiguous range of 64-key chunks of the
// row's key list [SWA slots..., main slots...].  Per chunk it gathers the
// records (FP8 SWA, FP4 main KV), dequantises them to bf16 in shared memory,
// computes S = q K^T on the tensor cores (mma.sync m16n8k16 bf16, fp32
// accumulation; 16 warps, each a 16-head x 16-key tile over all 512 dims),
// updates a running max / sum per head, and accumulates O += P V (each warp a
// 16-head x 128-dim tile).  Small batches split the key list over several
// CTAs and merge the partial (max, sum, O) by log-sum-exp in a second kernel.
#include <math.h>

#include "csa2_device.cuh"
#include "csa2_internal.h"

namespace csa2 {

namespace {

constexpr int kH = 64;
constexpr int kD = 512;
constexpr int kCK = 64;              // keys per chunk
constexpr int kQStride = kD + 8;     // bf16 per shared row (1040 B: conflict-free ldmatrix)
constexpr int kSStride = kCK + 4;    // floats
constexpr int kPStride = kCK + 8;    // bf16
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
  int nsplit;
  int chunks_per_split;
  float* ws_o;    // [T][nsplit][64][512]
  float* ws_ml;   // [T][nsplit][64][2]
  uint32_t* err;
};

struct AttnSmem {
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kH * kQStride * 2;
  static constexpr int kOffS = kOffK + kCK * kQStride * 2;
  static constexpr int kOffP = kOffS + kH * kSStride * 4;
  static constexpr int kOffStats = kOffP + kH * kPStride * 2;  // m, l, alpha [64] each
  static constexpr int kOffValid = kOffStats + 3 * kH * 4;
  static constexpr int kBytes = kOffValid + kCK * 4;
};

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
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// e2m1 code (4 bits) times a power-of-two scale.
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
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
  __half2 hh = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(hh);
}

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

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(512, 1) sparse_attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(16) uint8_t sm[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(sm + AttnSmem::kOffQ);
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(sm + AttnSmem::kOffK);
  float* sS = reinterpret_cast<float*>(sm + AttnSmem::kOffS);
  __nv_bfloat16* sP = reinterpret_cast<__nv_bfloat16*>(sm + AttnSmem::kOffP);
  float* sM = reinterpret_cast<float*>(sm + AttnSmem::kOffStats);
  float* sL = sM + kH;
  float* sA = sL + kH;
  int* sValid = reinterpret_cast<int*>(sm + AttnSmem::kOffValid);

  const int split = blockIdx.x;
  const int t = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  pdl_trigger();
  pdl_wait();
  const int L = p.n_swa + p.k;
  const int nchunks = (L + kCK - 1) / kCK;
  const int c0 = split * p.chunks_per_split;
  const int c1 = min(c0 + p.chunks_per_split, nchunks);

  // q -> shared (async), stats init
  {
    const __nv_bfloat16* gq = p.q + static_cast<long long>(t) * kH * kD;
    for (int i = tid; i < kH * (kD / 8); i += blockDim.x) {
      const int h = i / (kD / 8), c = i % (kD / 8);
      cp_async16(sQ + h * kQStride + c * 8, gq + h * kD + c * 8);
    }
  }
  if (tid < kH) {
    sM[tid] = -INFINITY;
    sL[tid] = 0.f;
  }
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  const int hg = warp & 3;       // 16-head group
  const int xg = warp >> 2;      // S: 16-key group; PV: 128-dim group
  const int g = lane >> 2, cq = lane & 3;

  for (int ch = c0; ch < c1; ++ch) {
    // ---- gather + dequantise 64 keys: thread -> (key kk, 64-dim part)
    {
      const int kk = tid >> 3, part = tid & 7;
      const int j = ch * kCK + kk;
      int slot = -1;
      bool swa = false;
      if (j < p.n_swa) {
        slot = __ldg(p.swa_slot + static_cast<long long>(t) * p.ld_swa + j);
        swa = true;
        if (slot >= p.swa_slots) {
          set_error(p.err, kErrBounds);
          slot = -1;
        }
      } else if (j < L) {
        slot = __ldg(p.topk_slot + static_cast<long long>(t) * p.ld_topk + (j - p.n_swa));
        if (slot >= p.main_slots) {
          set_error(p.err, kErrBounds);
          slot = -1;
        }
      }
      uint4* dst = reinterpret_cast<uint4*>(sK + kk * kQStride + part * 64);
      if (slot < 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
      } else if (swa) {
        const uint8_t* rec = p.swa_kv + static_cast<long long>(slot) * 528;
        const float sc = __ldg(reinterpret_cast<const float*>(rec + 512) + (part >> 1));
        const uint4* src = reinterpret_cast<const uint4*>(rec + part * 64);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 raw = __ldg(src + i);  // 16 codes
          const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t packed[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 lo = e4m3x2_to_float2(static_cast<uint16_t>(w4[q] & 0xFFFFu));
            const float2 hi = e4m3x2_to_float2(static_cast<uint16_t>(w4[q] >> 16));
            packed[2 * q] = pack_bf16(lo.x * sc, lo.y * sc);
            packed[2 * q + 1] = pack_bf16(hi.x * sc, hi.y * sc);
          }
          dst[2 * i] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          dst[2 * i + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        }
      } else {
        const uint8_t* rec = p.main_kv + static_cast<long long>(slot) * 288;
        const uint4* src = reinterpret_cast<const uint4*>(rec + part * 32);
        const uint32_t sbytes = __ldg(reinterpret_cast<const unsigned short*>(rec + 256) + part);
        const uint4 raw0 = __ldg(src), raw1 = __ldg(src + 1);
#pragma unroll
        for (int i = 0; i < 2; ++i) {  // 32 elements per 16-B load, one scale each
          const uint4 raw = i ? raw1 : raw0;
          const uint32_t u = i ? (sbytes >> 8) : (sbytes & 0xFFu);
          const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
          if (u >= 2u && u <= 252u) {
            const E2m1Tables tb = e2m1_tables(u);
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // 8 codes per word
              uint32_t o0, o1, o2, o3;
              e2m1x4_bf16(w4[q] & 0xFFFFu, tb, o0, o1);
              e2m1x4_bf16(w4[q] >> 16, tb, o2, o3);
              dst[4 * i + q] = make_uint4(o0, o1, o2, o3);
            }
          } else {  // scales at the ends of the ue8m0 range: exact float path
            const float sc = ue8m0_value(u);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t packed[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const uint32_t byte = (w4[q] >> (8 * e)) & 0xFFu;
                packed[e] = pack_bf16(e2m1_scaled(byte & 0xFu, sc), e2m1_scaled(byte >> 4, sc));
              }
              dst[4 * i + q] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            }
          }
        }
      }
      if (part == 0) sValid[kk] = slot >= 0 ? 1 : 0;
    }
    cp_async_wait_all();
    __syncthreads();

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
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int key = sub * 8 + i;
        x[i] = sValid[key] ? sS[h * kSStride + key] * p.scale_log2 : -INFINITY;
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

  cp_async_wait_all();  // a CTA without chunks still owns in-flight copies of q
  // ---- epilogue
  const int h0 = 16 * hg + g, h1 = h0 + 8;
  if (p.nsplit == 1) {
    const float s0 = __ldg(p.sink + h0) * kLog2e, s1 = __ldg(p.sink + h1) * kLog2e;
    const float m0 = sM[h0], m1 = sM[h1];
    const float M0 = fmaxf(m0, s0), M1 = fmaxf(m1, s1);
    const float w0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - M0);
    const float w1 = (m1 == -INFINITY) ? 0.f : exp2f(m1 - M1);
    const float d0 = sL[h0] * w0 + exp2f(s0 - M0);
    const float d1 = sL[h1] * w1 + exp2f(s1 - M1);
    const float f0 = w0 / d0, f1 = w1 / d1;
    const long long base = static_cast<long long>(t) * kH * kD;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int d = 128 * xg + nt * 8 + 2 * cq;
      if (p.out_bf16) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + base;
        *reinterpret_cast<__nv_bfloat162*>(out + h0 * kD + d) = __floats2bfloat162_rn(o[nt][0] * f0, o[nt][1] * f0);
        *reinterpret_cast<__nv_bfloat162*>(out + h1 * kD + d) = __floats2bfloat162_rn(o[nt][2] * f1, o[nt][3] * f1);
      } else {
        float* out = static_cast<float*>(p.out) + base;
        *reinterpret_cast<float2*>(out + h0 * kD + d) = make_float2(o[nt][0] * f0, o[nt][1] * f0);
        *reinterpret_cast<float2*>(out + h1 * kD + d) = make_float2(o[nt][2] * f1, o[nt][3] * f1);
      }
    }
    if (p.lse && xg == 0 && cq == 0) {
      p.lse[static_cast<long long>(t) * kH + h0] = (M0 + log2f(d0)) * kLn2;
      p.lse[static_cast<long long>(t) * kH + h1] = (M1 + log2f(d1)) * kLn2;
    }
  } else {
    const long long ps = static_cast<long long>(t) * p.nsplit + split;
    float* wo = p.ws_o + ps * kH * kD;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int d = 128 * xg + nt * 8 + 2 * cq;
      *reinterpret_cast<float2*>(wo + h0 * kD + d) = make_float2(o[nt][0], o[nt][1]);
      *reinterpret_cast<float2*>(wo + h1 * kD + d) = make_float2(o[nt][2], o[nt][3]);
    }
    if (tid < kH) {
      p.ws_ml[(ps * kH + tid) * 2] = sM[tid];
      p.ws_ml[(ps * kH + tid) * 2 + 1] = sL[tid];
    }
  }
}

// Merge of the per-split (max, sum, O) of one (row, head): one warp turns the
// split statistics into normalised weights, then every thread sums its four
// dims over the splits with independent loads.
constexpr int kMaxSplits = 32;

__global__ void __launch_bounds__(128) attn_combine_kernel(const __grid_constant__ AttnParams p) {
  const int t = blockIdx.x, h = blockIdx.y;
  __shared__ float s_wt[kMaxSplits];
  pdl_trigger();
  pdl_wait();
  const int ns = p.nsplit;
  const long long base = static_cast<long long>(t) * ns;
  if (threadIdx.x < 32) {
    const int s = threadIdx.x;
    float m = -INFINITY, l = 0.f;
    if (s < ns) {
      m = p.ws_ml[((base + s) * kH + h) * 2];
      l = p.ws_ml[((base + s) * kH + h) * 2 + 1];
    }
    const float sk = __ldg(p.sink + h) * kLog2e;
    float M = fmaxf(m, sk);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = (s < ns && m != -INFINITY) ? exp2f(m - M) : 0.f;
    float den = w * l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    den += exp2f(sk - M);
    s_wt[s] = w / den;
    if (s == 0 && p.lse) p.lse[static_cast<long long>(t) * kH + h] = (M + log2f(den)) * kLn2;
  }
  __syncthreads();
  const int d = threadIdx.x * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
  for (int s = 0; s < ns; ++s) {
    const float w = s_wt[s];
    const float4 v = *reinterpret_cast<const float4*>(p.ws_o + ((base + s) * kH + h) * kD + d);
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  const long long o = (static_cast<long long>(t) * kH + h) * kD + d;
  if (p.out_bf16) {
    __nv_bfloat162* out = reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.out) + o);
    out[0] = __floats2bfloat162_rn(acc.x, acc.y);
    out[1] = __floats2bfloat162_rn(acc.z, acc.w);
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(p.out) + o) = acc;
  }
}

}  // namespace

int attn_num_splits(int T, int n_keys, int num_sms) {
  const int nchunks = (n_keys + kCK - 1) / kCK;
  if (nchunks <= 1) return 1;
  int s = (2 * num_sms + T - 1) / T;
  if (s < 1) s = 1;
  if (s > nchunks) s = nchunks;
  if (s > kMaxSplits) s = kMaxSplits;
  // equalise the chunk count per split
  const int cps = (nchunks + s - 1) / s;
  return (nchunks + cps - 1) / cps;
}

size_t attn_workspace_bytes(int T, int nsplit) {
  if (nsplit <= 1) return 0;
  return static_cast<size_t>(T) * nsplit * kH * (kD + 2) * sizeof(float) + 256;
}

cudaError_t launch_sparse_attn(const AttnLaunch& a, void* ws, size_t ws_bytes, const DeviceCtx& ctx,
                               cudaStream_t st) {
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
  const int L = a.n_swa + a.k;
  const int nchunks = (L + kCK - 1) / kCK;
  const int nsplit = attn_num_splits(a.T, L, ctx.num_sms);
  p.nsplit = nsplit;
  p.chunks_per_split = nsplit > 1 ? (nchunks + nsplit - 1) / nsplit : (nchunks > 0 ? nchunks : 1);
  p.ws_o = nullptr;
  p.ws_ml = nullptr;
  if (nsplit > 1) {
    p.ws_o = static_cast<float*>(ws);
    p.ws_ml = p.ws_o + static_cast<size_t>(a.T) * nsplit * kH * kD;
  }
  cudaError_t e = prefer_max_smem(sparse_attn_kernel, AttnSmem::kBytes);
  if (e != cudaSuccess) return e;
  if ((e = prefer_max_smem(attn_combine_kernel, 0)) != cudaSuccess) return e;
  e = launch_pdl(sparse_attn_kernel, dim3(nsplit, a.T), dim3(512), AttnSmem::kBytes, st, p);
  if (e != cudaSuccess) return e;
  if (nsplit > 1) e = launch_pdl(attn_combine_kernel, dim3(a.T, kH), dim3(128), 0, st, p);
  return e;
}

}  // namespace csa2
