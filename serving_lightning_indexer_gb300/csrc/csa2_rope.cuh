// RoPE angle helpers shared by the entry build (RoPE of new entries) and the
// attention output (inverse RoPE at the query position).  RoPE acts on the
// last 64 of the 512 dims in interleaved pairs, pair p turning by
// pos * theta^(-2p/64) (CSA2 page, attention section: RoPE only on the last 64
// dims).
#pragma once
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

namespace csa2 {

// A pair's rate in turns per position, as a 64-bit fixed-point fraction of a
// turn: 2^64 * frac(theta^(-2p/64) / (2 pi)), computed on the host in double
// (53 significant bits: pos * rate is then off by under 1e-8 rad for
// pos < 2^31; whole turns are dropped, as the angle is taken modulo 2 pi).
inline uint64_t rope_turn_rate(double theta, int p) {
  const double turns = pow(theta, -2.0 * p / 64.0) / 6.283185307179586;
  const double fr = turns - floor(turns);  // in [0, 1)
  return static_cast<uint64_t>(ldexp(fr, 64));
}

// sin and cos of pos * theta^(-2p/64): the angle reaches ~1e6 rad.  pos times
// the fixed-point rate, modulo 2^64 (the integer product's low word), is the
// angle's fraction of a turn, exactly reduced; its top 32 bits as a signed
// fraction of [-pi, pi) go to fp32 sin/cos (the fp32 angle carries the same
// 2^-24 relative rounding as any fp32 argument).
__device__ __forceinline__ void rope_angle(long long pos, uint64_t turn_rate, float* sn, float* cs) {
  const uint64_t frac = static_cast<uint64_t>(pos) * turn_rate;
  const int32_t t = static_cast<int32_t>(static_cast<uint32_t>(frac >> 32));
  sincosf(static_cast<float>(t) * 1.4629180792671596e-09f, sn, cs);  // 2 pi / 2^32
}

// Inverse RoPE of one interleaved pair (a, b): rotation by -pos * rate.
__device__ __forceinline__ void inv_rope_pair(float& a, float& b, long long pos, uint64_t inv_freq) {
  float sn, cs;
  rope_angle(pos, inv_freq, &sn, &cs);
  const float x = a, y = b;
  a = x * cs + y * sn;
  b = y * cs - x * sn;
}

}  // namespace csa2
