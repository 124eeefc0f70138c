// RoPE of the 64-wide decoupled query/key ("DeepSeek-V2 机制拆解" (discosf.com), §解耦
// RoPE 与 YaRN: a separate 64-wide query and a shared key carry the position). Pairs
// (i, i + 32) turn by pos * theta_i (rotate-half pairing), theta_i from rope_freq.
//
// Positions reach 131071 and beyond, where an fp32 product pos * freq would be off by
// ~1e-2 rad, so the angle is reduced exactly: f_i = theta_i / (2 pi) is held as a
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
  unsigned long long f[kRope / 2];   // theta_i / (2 pi) as an unsigned 0.64 fixed-point fraction
};

// Angular frequency of pair i: base^(-2i/64), or, extended by YaRN, that frequency where
// the pair turns more than beta times over the original context (r_i = L_0 theta_i / 2 pi),
// theta_i / scale where it turns less than alpha times, and the linear blend in r between
// ("DeepSeek-V2 机制拆解", §解耦 RoPE 与 YaRN: YaRN with scale 40, alpha 1, beta 32 on the
// decoupled key; the pages give no formula, this is the published YaRN frequency rule).
inline double rope_freq(const RopeSpec& r, int i) {
  const double theta = std::pow(r.base, -2.0 * i / (double)kRope);
  if (r.yarn_scale == 1.0) return theta;
  const double turns = r.original_max_pos * theta / (2.0 * M_PI);
  double g = (turns - r.yarn_alpha) / (r.yarn_beta - r.yarn_alpha);
  g = g < 0.0 ? 0.0 : (g > 1.0 ? 1.0 : g);
  return (1.0 - g) * theta / r.yarn_scale + g * theta;
}

// The turn table of `r`, computed once per distinct spec (host).
inline RopeTurns rope_turns(const RopeSpec& r) {
  static std::mutex mu;
  static RopeSpec last_spec = {0.0, 0.0, 0.0, 0.0, 0};
  static RopeTurns last;
  std::lock_guard<std::mutex> lock(mu);
  if (r.base != last_spec.base || r.yarn_scale != last_spec.yarn_scale || r.yarn_alpha != last_spec.yarn_alpha ||
      r.yarn_beta != last_spec.yarn_beta || r.original_max_pos != last_spec.original_max_pos) {
    for (int i = 0; i < kRope / 2; ++i) {
      const double f = rope_freq(r, i) / (2.0 * M_PI);   // turns per position, < 1/(2 pi)
      last.f[i] = (unsigned long long)std::ldexp(f, 64);
    }
    last_spec = r;
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
