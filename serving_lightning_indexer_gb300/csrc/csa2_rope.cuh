// RoPE angle helpers shared by the entry build (RoPE of new entries) and the
// attention output (inverse RoPE at the query position).  RoPE acts on the
// last 64 of the 512 dims in interleaved pairs, pair p turning by
// pos * theta^(-2p/64) (CSA2 page, attention section: RoPE only on the last 64
// dims).
#pragma once
#include <cuda_runtime.h>
#include <math.h>

namespace csa2 {

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

// Inverse RoPE of one interleaved pair (a, b): rotation by -pos * inv_freq.
__device__ __forceinline__ void inv_rope_pair(float& a, float& b, long long pos, double inv_freq) {
  float sn, cs;
  rope_angle(pos, inv_freq, &sn, &cs);
  const float x = a, y = b;
  a = x * cs + y * sn;
  b = y * cs - x * sn;
}

}  // namespace csa2
