#include "decode_tc.cuh"

namespace mla {

bool decode_tc_supported(const DecodeParams&) { return false; }

cudaError_t launch_decode_tc(const DecodeParams&, int, cudaStream_t) { return cudaErrorNotSupported; }

int decode_tc_num_splits(int B, int tiles, int n_h, int sms) {
  (void)n_h;
  const int pairs = sms / 2 > 0 ? sms / 2 : 1;
  int best = 1;
  double best_t = 1e30;
  for (int S = 1; S <= MLA_MAX_SPLITS && S <= tiles; ++S) {
    const int per = ceil_div(tiles, S);
    const int waves = ceil_div(B * S, pairs);
    // time in tile units: waves of `per` tiles, plus ~3.6 tile-equivalents of
    // partial-result traffic per unit (256 KB fp32 written, read back by the merge)
    const double t = waves * (per + 3.6) + 3.6 * (double)B * S / pairs;
    if (t < best_t - 1e-9) {
      best_t = t;
      best = S;
    }
  }
  return best;
}

}  // namespace mla
