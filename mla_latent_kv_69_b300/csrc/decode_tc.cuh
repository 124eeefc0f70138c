// Tensor-core (tcgen05 + TMEM + TMA) split-KV decode: host-side entry points.
#pragma once
#include "common.cuh"

namespace mla {

// True when the tcgen05 kernel handles this configuration.
bool decode_tc_supported(const DecodeParams& p);
// Launch; max_seq_len sizes nothing on the device side but is kept for heuristics.
cudaError_t launch_decode_tc(const DecodeParams& p, int max_seq_len, cudaStream_t st);
// Split count for B sequences of up to `tiles` 64-token tiles.
int decode_tc_num_splits(int B, int tiles, int n_h, int sms);

}  // namespace mla
