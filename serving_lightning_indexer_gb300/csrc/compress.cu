// Main-KV entry build of a Full layer.
//
// CSA2 page, "一层 CSA2 的 attention 具体怎么算" item 3, and the V4.1 Q&A page
// (compression operator): with m = 2 an entry is the per-channel
// softmax-weighted sum of two adjacent, non-overlapping tokens (no APE); with
// m = 1 the weight is identically 1.  The result goes through RMSNorm, RoPE on
// the last 64 dims, and FP4 quantisation after RoPE (V4.1-Flash report
// reading, section 六), into a 288-B record (e2m1 codes + ue8m0 scale per 32).
//
// One warp per entry, lane l owning channels 16l .. 16l+15 (two e2m1 scale
// groups span a lane pair).  HBM-bound: 2 KB (m=2: 4 KB) read, 288 B written.
//
// With W^IK the kernel also writes each entry's index key (V4.1 Q&A page:
// k = RMSNorm(y W^IK) from the latent before RoPE, RoPE on its last 64 dims;
// CSA2 page item 3: wk -> k_norm -> RoPE -> quantisation).  The CTA's 8
// latents go to shared memory and the 8 warps split the 512 x 128 projection
// by input rows (each warp's 64 rows of W^IK are loaded before the dependency
// wait), so W^IK is read once per CTA.
#include <cuda_fp8.h>
#include <math.h>

#include "csa2_device.cuh"
#include "csa2_rope.cuh"
#include "csa2_internal.h"

namespace csa2 {

namespace {

struct CompressParams {
  const __nv_bfloat16* C;
  const __nv_bfloat16* Z;
  long long n_entries;
  int ratio_m;
  const float* gamma;
  float eps;
  int apply_rope;
  uint64_t inv_freq[32];   // theta^(-2i/64) as a fixed-point turn rate (rope_turn_rate)
  long long first_entry;
  const int* entry_pos;
  uint8_t* main_kv;
  long long main_slots;
  const int* page_table;
  long long pt_len;
  const int* entry_slot;
  float* latent_out;
  const __nv_bfloat16* w_ik;  // optional index-key build: [512][128] W^IK
  const float* k_gamma;
  uint8_t* index_k;
  long long index_k_pages;
  int index_k_fp4;
  float* index_latent_out;
  uint32_t* err;
};

__device__ __forceinline__ void load16_bf16(const __nv_bfloat16* src, float (&v)[16]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 r = __ldg(s + i);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[j]);
      const float2 f = __bfloat1622float2(b);
      v[8 * i + 2 * j] = f.x;
      v[8 * i + 2 * j + 1] = f.y;
    }
  }
}

// e2m1 code of a value already divided by its group scale: nearest magnitude
// among 0, .5, 1, 1.5, 2, 3, 4, 6 with ties to the even code, saturating.
// The FP4 block exponent: the smallest k with 6 * 2^k >= a, for a finite a > 0
// (a = f * 2^ex with f in [0.5, 1): k = ex - 3 when f <= 0.75, else ex - 2),
// read from the bits of a; frexpf for a subnormal a.
__device__ __forceinline__ int fp4_block_exp(float a) {
  const uint32_t b = __float_as_uint(a);
  const int e = static_cast<int>(b >> 23);
  if (e == 0) {
    int ex;
    const float f = frexpf(a, &ex);
    return (f <= 0.75f) ? ex - 3 : ex - 2;
  }
  return ((b & 0x7FFFFFu) <= 0x400000u) ? e - 129 : e - 128;  // ex = e - 126; f <= 0.75 iff mantissa <= 2^22
}
// 2^(127 - u) for a scale byte u in 0..254, exact (2^-127 is subnormal):
// multiplying by it equals ldexpf(v, 127 - u), rounding included.
__device__ __forceinline__ float fp4_unscale(int u) {
  const int e = 254 - u;
  return e >= 1 ? __uint_as_float(static_cast<uint32_t>(e) << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ uint32_t e2m1_code(float v) {
  const float a = fabsf(v);
  uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
  return c | (v < 0.f ? 8u : 0u);
}

// Shared memory of the index-key phase: the CTA's 8 latents before RoPE,
// [512 channels][8 entries], then the partial projections [8 warps][8 entries][128].
template <int EPC>
constexpr int ik_smem_floats() { return 512 * EPC + 8 * EPC * 128; }

// IK: also the index keys (W^IK given); EPC: entries per CTA (8, or 1 so that
// few entries spread over more SMs: the other warps then only help project)
template <bool IK, int EPC>
__global__ void __launch_bounds__(256, IK ? 1 : 4) compress_kernel(const __grid_constant__ CompressParams p) {
  extern __shared__ float s_ik[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // W^IK is a weight (no earlier kernel writes it): this warp's 64 rows, lane
  // l's 4 columns 4l .. 4l+3, are loaded before the dependency wait
  uint2 wr[IK ? 64 : 1];
  float4 kg = make_float4(1.f, 1.f, 1.f, 1.f);  // k_norm weights of outputs 4l .. 4l+3
  if constexpr (IK) {
#pragma unroll
    for (int r = 0; r < 64; ++r)
      wr[r] = __ldg(reinterpret_cast<const uint2*>(p.w_ik + (64 * warp + r) * 128 + 4 * lane));
    kg = __ldg(reinterpret_cast<const float4*>(p.k_gamma) + lane);
  }
  // the RMSNorm weights of this lane's 16 channels, likewise
  const int c0 = lane * 16;
  float gam[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 g4 = __ldg(reinterpret_cast<const float4*>(p.gamma + c0) + i);
    gam[4 * i] = g4.x;
    gam[4 * i + 1] = g4.y;
    gam[4 * i + 2] = g4.z;
    gam[4 * i + 3] = g4.w;
  }
  pdl_wait();
  pdl_trigger();
  const long long e_raw = static_cast<long long>(blockIdx.x) * EPC + warp;
  const bool active = warp < EPC && e_raw < p.n_entries;  // other warps help the index-key phase only
  const long long e = active ? e_raw : p.n_entries - 1;
  long long pos = 0, slot = -1;
  bool slot_ok = false;
  float rope_sn = 0.f, rope_cs = 1.f;  // RoPE pair `lane` of the entry (below)
  if (warp < EPC) {
  // the entry's position and destination slot are requested with its tokens
  pos = p.entry_pos ? static_cast<long long>(__ldg(p.entry_pos + e)) : (p.first_entry + e) * p.ratio_m;
  if (p.entry_slot) {
    slot = __ldg(p.entry_slot + e);
  } else {
    const long long ent = p.first_entry + e;
    const long long lp = ent >> 6;
    slot = (lp < p.pt_len) ? static_cast<long long>(__ldg(p.page_table + lp)) * 64 + (ent & 63) : -1;
  }
  // RoPE pair `lane` of the entry (the latent's dims 448 + 2 lane, +1, and the
  // index key's 64 + 2 lane, +1 turn by the same angle): one angle a lane,
  // handed to the lanes that rotate the pair by shuffles
  if (p.apply_rope) rope_angle(pos, p.inv_freq[lane], &rope_sn, &rope_cs);
  float x[16];
  if (p.ratio_m == 1) {
    load16_bf16(p.C + e * 512 + c0, x);
  } else {
    // the two tokens' 16 channels of C and Z, kept packed (bf16) until used
    const long long r0 = e * 2;
    uint4 pk[4][2];  // C token 0, C token 1, Z token 0, Z token 1; 8 channels each
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      pk[0][h] = __ldg(reinterpret_cast<const uint4*>(p.C + r0 * 512 + c0) + h);
      pk[1][h] = __ldg(reinterpret_cast<const uint4*>(p.C + (r0 + 1) * 512 + c0) + h);
      pk[2][h] = __ldg(reinterpret_cast<const uint4*>(p.Z + r0 * 512 + c0) + h);
      pk[3][h] = __ldg(reinterpret_cast<const uint4*>(p.Z + (r0 + 1) * 512 + c0) + h);
    }
    auto chan = [&](int s_, int i) {  // channel c0 + i of stream s_ as fp32 (exact)
      const uint4& q = pk[s_][i >> 3];
      const int w = (i >> 1) & 3;
      const uint32_t word = w == 0 ? q.x : (w == 1 ? q.y : (w == 2 ? q.z : q.w));
      return __uint_as_float((i & 1) ? (word & 0xFFFF0000u) : (word << 16));
    };
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float za = chan(2, i), zb = chan(3, i);
      const float zm = fmaxf(za, zb);
      const float ea = expf(za - zm), eb = expf(zb - zm);
      x[i] = (ea * chan(0, i) + eb * chan(1, i)) / (ea + eb);
    }
  }
  // RMSNorm over the 512 channels
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = 1.0f / sqrtf(ss / 512.0f + p.eps);
  float y[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) y[i] = x[i] * inv * gam[i];
  if constexpr (IK) {  // the latent before RoPE feeds the index key
#pragma unroll
    for (int i = 0; i < 16; ++i) s_ik[(c0 + i) * EPC + warp] = y[i];
  }
  // RoPE on dims 448..511: interleaved pairs, angle pos * theta^(-2i/64)
  if (p.apply_rope) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = lane >= 28 ? (c0 - 448) / 2 + j : j;  // pair i (every lane takes part in the shuffle)
      const float sn = __shfl_sync(0xffffffffu, rope_sn, i), cs = __shfl_sync(0xffffffffu, rope_cs, i);
      if (lane >= 28) {
        const float a = y[2 * j], b = y[2 * j + 1];
        y[2 * j] = a * cs - b * sn;
        y[2 * j + 1] = a * sn + b * cs;
      }
    }
  }
  if (p.latent_out && active) {
    float4* lo = reinterpret_cast<float4*>(p.latent_out + e * 512 + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i) lo[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
  }
  // FP4: group of 32 = lanes (2g, 2g+1)
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(y[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  int u = 127;
  if (amax > 0.f) u = min(max(fp4_block_exp(amax) + 127, 0), 254);  // smallest k with 6 * 2^k >= amax
  const float unscale = fp4_unscale(u);
  uint32_t packed[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t code = e2m1_code(y[i] * unscale);
    packed[i >> 3] |= code << (4 * (i & 7));
  }
  slot_ok = slot >= 0 && slot < p.main_slots;
  if (active && !slot_ok && lane == 0) set_error(p.err, kErrBounds);
  if (active && slot_ok) {
    uint8_t* rec = p.main_kv + slot * 288;
    *reinterpret_cast<uint2*>(rec + lane * 8) = make_uint2(packed[0], packed[1]);
    if ((lane & 1) == 0) rec[256 + (lane >> 1)] = static_cast<uint8_t>(u);
    if (lane < 4) *reinterpret_cast<uint32_t*>(rec + 272 + lane * 4) = 0u;
  }
  }  // warp < EPC
  if constexpr (!IK) return;

  // ---- index keys of the CTA's entries (V4.1 Q&A page): k = RMSNorm(y W^IK) *
  // k_gamma from the latents before RoPE, RoPE on dims 64..127, then the FP8 or
  // FP4 entry.  Warp w multiplies channels 64w .. 64w+63 of all 8 latents by
  // its rows of W^IK (lane l: outputs 4l .. 4l+3); the 8 partial sums of each
  // entry are then added by the entry's own warp.
  __syncthreads();
  float acc[EPC][4];
#pragma unroll
  for (int q = 0; q < EPC; ++q)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[q][j] = 0.f;
#pragma unroll
  for (int r = 0; r < 64; ++r) {
    float yv[EPC];
    if constexpr (EPC == 8) {
      const float4 ya = *reinterpret_cast<const float4*>(s_ik + (64 * warp + r) * 8);
      const float4 yb = *reinterpret_cast<const float4*>(s_ik + (64 * warp + r) * 8 + 4);
      yv[0] = ya.x; yv[1] = ya.y; yv[2] = ya.z; yv[3] = ya.w;
      yv[4] = yb.x; yv[5] = yb.y; yv[6] = yb.z; yv[7] = yb.w;
    } else {
#pragma unroll
      for (int q = 0; q < EPC; ++q) yv[q] = s_ik[(64 * warp + r) * EPC + q];
    }
    const float2 w01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wr[r].x));
    const float2 w23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wr[r].y));
#pragma unroll
    for (int q = 0; q < EPC; ++q) {
      acc[q][0] = fmaf(yv[q], w01.x, acc[q][0]);
      acc[q][1] = fmaf(yv[q], w01.y, acc[q][1]);
      acc[q][2] = fmaf(yv[q], w23.x, acc[q][2]);
      acc[q][3] = fmaf(yv[q], w23.y, acc[q][3]);
    }
  }
  float* s_part = s_ik + 512 * EPC;  // [warp][entry][128]
#pragma unroll
  for (int q = 0; q < EPC; ++q)
    *reinterpret_cast<float4*>(s_part + (warp * EPC + q) * 128 + 4 * lane) =
        make_float4(acc[q][0], acc[q][1], acc[q][2], acc[q][3]);
  __syncthreads();
  if (warp >= EPC) return;
  float kk[4] = {0.f, 0.f, 0.f, 0.f};  // k[4 lane + j] of this warp's entry
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const float4 v = *reinterpret_cast<const float4*>(s_part + (w * EPC + warp) * 128 + 4 * lane);
    kk[0] += v.x;
    kk[1] += v.y;
    kk[2] += v.z;
    kk[3] += v.w;
  }
  float s2 = (kk[0] * kk[0] + kk[1] * kk[1]) + (kk[2] * kk[2] + kk[3] * kk[3]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
  const float inv2 = 1.0f / sqrtf(s2 / 128.0f + p.eps);
  kk[0] *= inv2 * kg.x;
  kk[1] *= inv2 * kg.y;
  kk[2] *= inv2 * kg.z;
  kk[3] *= inv2 * kg.w;
  if (p.apply_rope) {  // dims 64..127: pairs (4l, 4l+1), (4l+2, 4l+3) = pair 2l-32, 2l-31
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = lane >= 16 ? 2 * lane - 32 + h : h;
      const float sn = __shfl_sync(0xffffffffu, rope_sn, i), cs = __shfl_sync(0xffffffffu, rope_cs, i);
      if (lane >= 16) {
        const float a = kk[2 * h], b = kk[2 * h + 1];
        kk[2 * h] = a * cs - b * sn;
        kk[2 * h + 1] = a * sn + b * cs;
      }
    }
  }
  if (!active) return;
  if (p.index_latent_out)
    *reinterpret_cast<float4*>(p.index_latent_out + e * 128 + 4 * lane) = make_float4(kk[0], kk[1], kk[2], kk[3]);
  if (!slot_ok) return;
  const long long page = slot >> 6;
  const int row = static_cast<int>(slot & 63);
  if (page >= p.index_k_pages) {
    if (lane == 0) set_error(p.err, kErrBounds);
    return;
  }
  if (!p.index_k_fp4) {  // FP8: one fp32 scale amax / 448, e4m3 codes round-to-nearest-even
    float am = fmaxf(fmaxf(fabsf(kk[0]), fabsf(kk[1])), fmaxf(fabsf(kk[2]), fabsf(kk[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    const float sc = am > 0.f ? am / 448.0f : 1.0f;
    uint8_t* pg = p.index_k + page * 8448;
    uint32_t word = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      word |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(kk[j] / sc, __NV_SATFINITE, __NV_E4M3)) << (8 * j);
    *reinterpret_cast<uint32_t*>(pg + row * 128 + 4 * lane) = word;
    if (lane == 0) *reinterpret_cast<float*>(pg + 8192 + row * 4) = sc;
  } else {  // FP4: e2m1 + one ue8m0 scale per 32 dims (lanes 8b .. 8b+7)
    float am = fmaxf(fmaxf(fabsf(kk[0]), fabsf(kk[1])), fmaxf(fabsf(kk[2]), fabsf(kk[3])));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    int ue = 127;
    if (am > 0.f) ue = min(max(fp4_block_exp(am) + 127, 0), 254);
    const float unscale = fp4_unscale(ue);
    uint32_t half = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) half |= e2m1_code(kk[j] * unscale) << (4 * j);
    uint8_t* pg = p.index_k + page * 4352;
    *reinterpret_cast<uint16_t*>(pg + row * 64 + 2 * lane) = static_cast<uint16_t>(half);
    if ((lane & 7) == 0) pg[4096 + row * 4 + (lane >> 3)] = static_cast<uint8_t>(ue);
  }
}


// ---------------------------------------------------------------- hidden-state projection
// C = H W for the per-token inputs of the entry build (CSA2 page item 3: with
// m = 1 the main-KV entry is one linear projection of the token; CED: the
// decoder layers' C = H_{L/2} W^KV, the encoder layers' C and Z from their
// own hidden state).  Decode-sized row counts (T <= 64): the weight read
// (hidden x 1 KB) is the cost, so every SM streams a share of it at once.
// Grid: 16 column blocks of 32 x 8 slices of the hidden dimension; the 8 CTAs
// of a column block form a cluster and add their partial sums through
// distributed shared memory.  A thread owns 8 columns (one 16-B weight load)
// of one row in each round of 64 rows; a batch of up to 16 rounds of weights
// is loaded into registers at once (the first batch before the dependency
// wait: weights are not produced by the step), the batch's hidden-state
// columns are staged in shared memory, and 4 rows of H at a time are
// accumulated with packed fp32x2 FMAs.  The 64 threads of a column chunk are
// reduced by a shuffle reduce-scatter (xor 16, 8, 4) and through shared memory.
constexpr int kPjD = 512;           // width of the projected token vector
constexpr int kPjCols = 32;         // output columns per CTA
constexpr int kPjSplit = 8;         // CTAs (slices of the hidden dimension) per column block
constexpr int kPjThreads = 256;     // 64 rows x 4 column chunks of 8
constexpr int kPjRounds = 16;       // rounds of 64 rows per batch
constexpr int kPjBatch = 64 * kPjRounds;

size_t kv_project_smem(int T, int hidden) {
  const int batch = min(hidden / kPjSplit, kPjBatch);
  return static_cast<size_t>(T) * batch * 2 + 8 * 4 * 32 * 4 + static_cast<size_t>(T) * kPjCols * 4;
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__global__ void __launch_bounds__(kPjThreads, 1) kv_project_kernel(const __nv_bfloat16* __restrict__ H,
                                                                   const __nv_bfloat16* __restrict__ W, int T,
                                                                   int hidden, __nv_bfloat16* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t pj_smem[];
  const int hs = hidden / kPjSplit;       // rows of this CTA's slice (a multiple of 64)
  const int batch = min(hs, kPjBatch);
  __nv_bfloat16* h_s = reinterpret_cast<__nv_bfloat16*>(pj_smem);            // [T][batch]
  float* red = reinterpret_cast<float*>(pj_smem + static_cast<size_t>(T) * batch * 2);  // [8 warps][4 chunks][32]
  float* part = red + 8 * 4 * 32;                                              // [T][32]
  const uint32_t rank = cluster_rank();
  const int col0 = blockIdx.x * kPjCols;
  const int tid = threadIdx.x, cc = tid & 3, rsub = tid >> 2;
  const int lane = tid & 31, warp = tid >> 5;
  const int k_begin = static_cast<int>(rank) * hs;
  for (int i = tid; i < T * kPjCols; i += kPjThreads) part[i] = 0.f;
  bool waited = false;
  for (int kb = k_begin; kb < k_begin + hs; kb += batch) {
    const int nb = min(batch, k_begin + hs - kb);  // a multiple of 64
    uint4 wv[kPjRounds];
#pragma unroll
    for (int i = 0; i < kPjRounds; ++i) {
      wv[i] = make_uint4(0u, 0u, 0u, 0u);
      if (i * 64 < nb)
        wv[i] = __ldg(reinterpret_cast<const uint4*>(W + static_cast<long long>(kb + i * 64 + rsub) * kPjD + col0 +
                                                     cc * 8));
    }
    if (!waited) {
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
    __syncthreads();  // the previous batch's h_s is no longer read
    const int per_row = nb / 8;
    for (int i = tid; i < T * per_row; i += kPjThreads) {
      const int t = i / per_row, u = i - t * per_row;
      *reinterpret_cast<uint4*>(h_s + t * batch + u * 8) =
          __ldg(reinterpret_cast<const uint4*>(H + static_cast<long long>(t) * hidden + kb + u * 8));
    }
    __syncthreads();
    for (int t0 = 0; t0 < T; t0 += 4) {
      uint64_t acc[4][4];
#pragma unroll
      for (int tt = 0; tt < 4; ++tt)
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) acc[tt][jp] = 0ull;
#pragma unroll
      for (int i = 0; i < kPjRounds; ++i) {
        if (i * 64 < nb) {
          const int kl = i * 64 + rsub;
          const uint32_t w32[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
          uint64_t wp[4];
#pragma unroll
          for (int jp = 0; jp < 4; ++jp) wp[jp] = pack_f32x2(bf16_lo(w32[jp]), bf16_hi(w32[jp]));
#pragma unroll
          for (int tt = 0; tt < 4; ++tt) {
            const float h = (t0 + tt < T) ? __bfloat162float(h_s[(t0 + tt) * batch + kl]) : 0.f;
            const uint64_t hh = pack_f32x2(h, h);
#pragma unroll
            for (int jp = 0; jp < 4; ++jp) acc[tt][jp] = fma_f32x2(hh, wp[jp], acc[tt][jp]);
          }
        }
      }
      // value q = 8 tt + j of this thread (row t0 + tt, column cc * 8 + j)
      float v[32];
#pragma unroll
      for (int tt = 0; tt < 4; ++tt)
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {
          const float2 f = unpack_f32x2(acc[tt][jp]);
          v[tt * 8 + 2 * jp] = f.x;
          v[tt * 8 + 2 * jp + 1] = f.y;
        }
      // reduce-scatter over the 8 lanes of the warp that hold chunk cc: after
      // the xor-16, -8 and -4 steps lane l holds values (l >> 2) * 4 + i, i < 4
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const bool hi = lane & 16;
        const float keep = hi ? v[16 + i] : v[i], send = hi ? v[i] : v[16 + i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const bool hi = lane & 8;
        const float keep = hi ? v[8 + i] : v[i], send = hi ? v[i] : v[8 + i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool hi = lane & 4;
        const float keep = hi ? v[4 + i] : v[i], send = hi ? v[i] : v[4 + i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
      }
      *reinterpret_cast<float4*>(red + (warp * 4 + cc) * 32 + (lane >> 2) * 4) = make_float4(v[0], v[1], v[2], v[3]);
      __syncthreads();
      if (tid < 128) {
        const int c2 = tid >> 5, q = tid & 31;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) sum += red[(w * 4 + c2) * 32 + q];
        const int tt = q >> 3, j = q & 7;
        if (t0 + tt < T) part[(t0 + tt) * kPjCols + c2 * 8 + j] += sum;
      }
      __syncthreads();  // red is rewritten by the next rows
    }
  }
  cluster_sync();  // every slice's partial sums are final
  // the column block's T x 32 outputs, split over the cluster's CTAs
  for (int o = static_cast<int>(rank) * kPjThreads + tid; o < T * kPjCols; o += kPjSplit * kPjThreads) {
    const uint32_t a = smem_u32(part + o);
    float sum = 0.f;
#pragma unroll
    for (int r = 0; r < kPjSplit; ++r) sum += ld_cluster_f32(map_rank(a, static_cast<uint32_t>(r)));
    out[static_cast<long long>(o / kPjCols) * kPjD + col0 + (o % kPjCols)] = __float2bfloat16_rn(sum);
  }
  cluster_sync();  // no CTA leaves while its partial sums may still be read
}

}  // namespace

cudaError_t launch_compress(const CompressLaunch& a, const DeviceCtx& ctx, cudaStream_t st) {
  CompressParams p;
  p.C = reinterpret_cast<const __nv_bfloat16*>(a.C);
  p.Z = reinterpret_cast<const __nv_bfloat16*>(a.Z);
  p.n_entries = a.n_entries;
  p.ratio_m = a.ratio_m;
  p.gamma = a.gamma;
  p.eps = a.eps;
  p.apply_rope = a.apply_rope;
  for (int i = 0; i < 32; ++i) p.inv_freq[i] = rope_turn_rate(static_cast<double>(a.rope_theta), i);
  p.first_entry = a.first_entry;
  p.entry_pos = a.entry_pos;
  p.main_kv = a.main_kv;
  p.main_slots = a.main_slots;
  p.page_table = a.page_table;
  p.pt_len = a.pt_len;
  p.entry_slot = a.entry_slot;
  p.latent_out = a.latent_out;
  p.w_ik = reinterpret_cast<const __nv_bfloat16*>(a.w_ik);
  p.k_gamma = a.k_gamma;
  p.index_k = a.index_k;
  p.index_k_pages = a.index_k_pages;
  p.index_k_fp4 = a.index_k_fp4;
  p.index_latent_out = a.index_latent_out;
  p.err = ctx.err;
  if (a.n_entries == 0) return cudaSuccess;
  if (!a.w_ik) {
    const long long blocks = (a.n_entries + 7) / 8;
    cudaError_t e = prefer_max_smem(compress_kernel<false, 8>, 0);
    if (e != cudaSuccess) return e;
    return launch_pdl(compress_kernel<false, 8>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, p);
  }
  // with index keys: up to one entry per SM, one entry per CTA (the projection
  // of an entry spread over 8 warps); beyond, 8 entries per CTA (W^IK read
  // once per 8 entries)
  if (a.n_entries <= ctx.num_sms) {
    constexpr size_t smem = ik_smem_floats<1>() * sizeof(float);
    cudaError_t e = prefer_max_smem(compress_kernel<true, 1>, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(compress_kernel<true, 1>, dim3(static_cast<unsigned>(a.n_entries)), dim3(256), smem, st, p);
  }
  const long long blocks = (a.n_entries + 7) / 8;
  constexpr size_t smem = ik_smem_floats<8>() * sizeof(float);
  cudaError_t e = prefer_max_smem(compress_kernel<true, 8>, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(compress_kernel<true, 8>, dim3(static_cast<unsigned>(blocks)), dim3(256), smem, st, p);
}

cudaError_t launch_kv_project(const uint16_t* H, const uint16_t* W, int T, int hidden, uint16_t* out,
                              cudaStream_t st) {
  const size_t smem = kv_project_smem(T, hidden);
  cudaError_t e = prefer_max_smem(kv_project_kernel, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kPjD / kPjCols, kPjSplit);
  cfg.blockDim = dim3(kPjThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = kPjSplit;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kv_project_kernel, reinterpret_cast<const __nv_bfloat16*>(H),
                            reinterpret_cast<const __nv_bfloat16*>(W), T, hidden, reinterpret_cast<__nv_bfloat16*>(out));
}

}  // namespace csa2
