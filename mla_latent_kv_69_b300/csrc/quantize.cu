// mla_quantize_fp8: one warp per 576-element row (quantize.cuh).
#include "quantize.cuh"

namespace mla {
namespace {

constexpr int kQuantWarps = 8;

__global__ void __launch_bounds__(kQuantWarps * 32)
quantize_fp8_kernel(const __nv_bfloat16* __restrict__ rows, int64_t n, uint8_t* __restrict__ codes,
                    float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
  if (r >= n) return;
  quantize_row_e4m3(rows + r * kRow, codes + r * kRow, scales + r, lane);
}

}  // namespace

cudaError_t launch_quantize_fp8(const __nv_bfloat16* rows, int64_t n, uint8_t* codes, float* scales,
                                cudaStream_t st) {
  const int64_t blocks = ceil_div64(n, kQuantWarps);
  quantize_fp8_kernel<<<(unsigned)blocks, kQuantWarps * 32, 0, st>>>(rows, n, codes, scales);
  return cudaGetLastError();
}

}  // namespace mla
