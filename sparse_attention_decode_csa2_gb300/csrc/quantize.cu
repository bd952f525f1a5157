// FP4 main-KV packer: fp32 latent rows -> E2M1 codes + one E4M3 scale per
// 16 channels (DeepSeek-V4.1-Flash paper walkthrough, 1.(5).4 "FP4 Main KV
// Cache"; release summary, "CSA2").  One warp per 512-channel row; the row
// arithmetic (and why it is bit-exact) is in quant_fp4.cuh.
#include "quant_fp4.cuh"

namespace csa2 {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
quantize_kv_fp4_kernel(const float* __restrict__ x, int64_t n_rows, uint8_t* __restrict__ out) {
  __shared__ __align__(16) uint8_t rowbuf[kWarps][kRowBytes];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint8_t* buf = rowbuf[warp];
  for (int64_t row = (int64_t)blockIdx.x * kWarps + warp; row < n_rows;
       row += (int64_t)gridDim.x * kWarps) {
    quantize_fp4_row_warp(x + row * kD, out + row * kRowBytes, buf, lane);
  }
}

}  // namespace

cudaError_t launch_quantize_kv_fp4(const float* x, int64_t n_rows, uint8_t* out,
                                   cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  int64_t blocks = (n_rows + kWarps - 1) / kWarps;
  int64_t cap = (int64_t)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  quantize_kv_fp4_kernel<<<(unsigned)blocks, kWarps * 32, 0, stream>>>(x, n_rows, out);
  return cudaGetLastError();
}

}  // namespace csa2
