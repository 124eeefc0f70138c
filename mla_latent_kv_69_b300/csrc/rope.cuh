// RoPE of the 64-wide decoupled query/key ("DeepSeek-V2 机制拆解" (discosf.com), §解耦
// RoPE 与 YaRN: a separate 64-wide query and a shared key carry the position). Pairs
// (i, i + 32) turn by theta_i = pos * base^(-2i/64) (rotate-half pairing).
//
// Positions reach 131071 and beyond, where an fp32 product pos * freq would be off by
// ~1e-2 rad, so the angle is reduced exactly: f_i = base^(-2i/64) / (2 pi) is held as a
// 64-bit fixed-point fraction of a turn (computed on the host in double), the turn
// count's fraction is the wrapping 64-bit product pos * f_i, and only the reduced angle
// goes through fp32 sincos.
#pragma once
#include <cmath>
#include <cstdint>
#include <mutex>

#include "common.cuh"

namespace mla {

struct RopeTurns {
  unsigned long long f[kRope / 2];   // base^(-2i/64) / (2 pi) as an unsigned 0.64 fixed-point fraction
};

// The turn table of `rope_base`, computed once per base (host).
inline RopeTurns rope_turns(float rope_base) {
  static std::mutex mu;
  static float last_base = 0.f;
  static RopeTurns last;
  std::lock_guard<std::mutex> lock(mu);
  if (rope_base != last_base) {
    for (int i = 0; i < kRope / 2; ++i) {
      const double f = std::pow((double)rope_base, -2.0 * i / (double)kRope) / (2.0 * M_PI);   // < 1/(2 pi)
      last.f[i] = (unsigned long long)std::ldexp(f, 64);
    }
    last_base = rope_base;
  }
  return last;
}

// sin and cos of pair i's angle at position `pos` (>= 0).
__device__ __forceinline__ void rope_sincos(int pos, unsigned long long f, float* sn, float* cs) {
  const unsigned long long frac = (unsigned long long)(long long)pos * f;
  const float ang = (float)(frac >> 40) * (6.283185307179586f / 16777216.f);
  sincosf(ang, sn, cs);
}

}  // namespace mla
