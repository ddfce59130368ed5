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
#include <cuda_fp8.h>
#include <math.h>

#include "csa2_device.cuh"
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
  double inv_freq[32];     // theta^(-2i/64), computed on the host in double
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

// Sum over the warp of 32 values per lane, scattered: lane l returns the total
// of element l (five butterfly halvings, 31 shuffles).
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int j = 0; j < s; ++j) {
      const float send = up ? v[j] : v[j + s];
      const float keep = up ? v[j + s] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return v[0];
}

// sin and cos of pos * inv_freq: the angle reaches ~1e6 rad, so it is formed
// and reduced modulo 2 pi in double (2 pi split in two parts), then sin/cos
// run in fp32 on the reduced angle.
__device__ __forceinline__ void rope_angle(long long pos, double inv_freq, float* sn, float* cs) {
  constexpr double kTwoPiHi = 6.283185307179586;
  constexpr double kTwoPiLo = 2.4492935982947064e-16;
  constexpr double kInvTwoPi = 0.15915494309189535;
  const double ang = static_cast<double>(pos) * inv_freq;
  const double kq = rint(ang * kInvTwoPi);
  const double red = fma(-kq, kTwoPiLo, fma(-kq, kTwoPiHi, ang));
  sincosf(static_cast<float>(red), sn, cs);
}

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
__device__ __forceinline__ uint32_t e2m1_code(float v) {
  const float a = fabsf(v);
  uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
  return c | (v < 0.f ? 8u : 0u);
}

__global__ void __launch_bounds__(256) compress_kernel(const __grid_constant__ CompressParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  const long long e = static_cast<long long>(blockIdx.x) * 8 + warp;
  if (e >= p.n_entries) return;
  const int c0 = lane * 16;
  float x[16];
  if (p.ratio_m == 1) {
    load16_bf16(p.C + e * 512 + c0, x);
  } else {
    float ca[16], cb[16], za[16], zb[16];
    const long long r0 = e * 2;
    load16_bf16(p.C + r0 * 512 + c0, ca);
    load16_bf16(p.C + (r0 + 1) * 512 + c0, cb);
    load16_bf16(p.Z + r0 * 512 + c0, za);
    load16_bf16(p.Z + (r0 + 1) * 512 + c0, zb);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float zm = fmaxf(za[i], zb[i]);
      const float ea = expf(za[i] - zm), eb = expf(zb[i] - zm);
      x[i] = (ea * ca[i] + eb * cb[i]) / (ea + eb);
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
  for (int i = 0; i < 16; ++i) y[i] = x[i] * inv * __ldg(p.gamma + c0 + i);
  const long long pos = p.entry_pos ? static_cast<long long>(__ldg(p.entry_pos + e)) : (p.first_entry + e) * p.ratio_m;
  // index key (V4.1 Q&A page): k = RMSNorm(y W^IK) * k_gamma from the latent
  // before RoPE, then RoPE on dims 64..127; lane l holds k[32 b + l], b < 4
  float kk[4] = {0.f, 0.f, 0.f, 0.f};
  if (p.w_ik) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float part[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) part[j] = 0.f;
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const uint4* wr = reinterpret_cast<const uint4*>(p.w_ik + (c0 + i) * 128 + 32 * b);
        const float yi = y[i];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 r = __ldg(wr + q);
          const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
          for (int t2 = 0; t2 < 4; ++t2) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[t2]));
            part[8 * q + 2 * t2] = fmaf(yi, f.x, part[8 * q + 2 * t2]);
            part[8 * q + 2 * t2 + 1] = fmaf(yi, f.y, part[8 * q + 2 * t2 + 1]);
          }
        }
      }
      kk[b] = reduce_scatter32(part, lane);
    }
    float s2 = (kk[0] * kk[0] + kk[1] * kk[1]) + (kk[2] * kk[2] + kk[3] * kk[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    const float inv2 = 1.0f / sqrtf(s2 / 128.0f + p.eps);
#pragma unroll
    for (int b = 0; b < 4; ++b) kk[b] = kk[b] * inv2 * __ldg(p.k_gamma + 32 * b + lane);
    if (p.apply_rope) {
#pragma unroll
      for (int b = 2; b < 4; ++b) {  // dims 64..127: pair i = (dim - 64) / 2 of lanes (2j, 2j+1)
        float sn, cs;
        rope_angle(pos, p.inv_freq[16 * (b - 2) + (lane >> 1)], &sn, &cs);
        const float other = __shfl_xor_sync(0xffffffffu, kk[b], 1);
        kk[b] = (lane & 1) ? fmaf(other, sn, kk[b] * cs) : fmaf(-other, sn, kk[b] * cs);
      }
    }
  }
  // RoPE on dims 448..511: interleaved pairs, angle pos * theta^(-2i/64)
  if (p.apply_rope && lane >= 28) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = (c0 - 448) / 2 + j;
      float sn, cs;
      rope_angle(pos, p.inv_freq[i], &sn, &cs);
      const float a = y[2 * j], b = y[2 * j + 1];
      y[2 * j] = a * cs - b * sn;
      y[2 * j + 1] = a * sn + b * cs;
    }
  }
  if (p.latent_out) {
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
  if (amax > 0.f) {
    int ex;
    const float f = frexpf(amax, &ex);           // amax = f * 2^ex, f in [0.5, 1)
    const int k = (f <= 0.75f) ? ex - 3 : ex - 2;  // smallest k with 6 * 2^k >= amax
    u = min(max(k + 127, 0), 254);
  }
  uint32_t packed[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t code = e2m1_code(ldexpf(y[i], 127 - u));
    packed[i >> 3] |= code << (4 * (i & 7));
  }
  // destination slot
  long long slot;
  if (p.entry_slot) {
    slot = __ldg(p.entry_slot + e);
  } else {
    const long long ent = p.first_entry + e;
    const long long lp = ent >> 6;
    slot = (lp < p.pt_len) ? static_cast<long long>(__ldg(p.page_table + lp)) * 64 + (ent & 63) : -1;
  }
  if (slot < 0 || slot >= p.main_slots) {
    if (lane == 0) set_error(p.err, kErrBounds);
    return;
  }
  uint8_t* rec = p.main_kv + slot * 288;
  *reinterpret_cast<uint2*>(rec + lane * 8) = make_uint2(packed[0], packed[1]);
  if ((lane & 1) == 0) rec[256 + (lane >> 1)] = static_cast<uint8_t>(u);
  if (lane < 4) *reinterpret_cast<uint32_t*>(rec + 272 + lane * 4) = 0u;
  if (p.w_ik) {
    if (p.index_latent_out) {
#pragma unroll
      for (int b = 0; b < 4; ++b) p.index_latent_out[e * 128 + 32 * b + lane] = kk[b];
    }
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
#pragma unroll
      for (int b = 0; b < 4; ++b)
        pg[row * 128 + 32 * b + lane] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(kk[b] / sc, __NV_SATFINITE, __NV_E4M3));
      if (lane == 0) *reinterpret_cast<float*>(pg + 8192 + row * 4) = sc;
    } else {  // FP4: e2m1 + one ue8m0 scale per 32 dims (a block = one register across the warp)
      uint8_t* pg = p.index_k + page * 4352;
      uint32_t ub = 0u;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float am = fabsf(kk[b]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        int ue = 127;
        if (am > 0.f) {
          int ex;
          const float f = frexpf(am, &ex);
          const int k = (f <= 0.75f) ? ex - 3 : ex - 2;
          ue = min(max(k + 127, 0), 254);
        }
        const uint32_t code = e2m1_code(ldexpf(kk[b], 127 - ue));
        const uint32_t hi = __shfl_xor_sync(0xffffffffu, code, 1);
        if ((lane & 1) == 0) pg[row * 64 + 16 * b + (lane >> 1)] = static_cast<uint8_t>(code | (hi << 4));
        ub |= static_cast<uint32_t>(ue) << (8 * b);
      }
      if (lane == 0) *reinterpret_cast<uint32_t*>(pg + 4096 + row * 4) = ub;
    }
  }
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
  for (int i = 0; i < 32; ++i) p.inv_freq[i] = pow(static_cast<double>(a.rope_theta), -2.0 * i / 64.0);
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
  const long long blocks = (a.n_entries + 7) / 8;
  cudaError_t e = prefer_max_smem(compress_kernel, 0);
  if (e != cudaSuccess) return e;
  return launch_pdl(compress_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, p);
}

}  // namespace csa2
