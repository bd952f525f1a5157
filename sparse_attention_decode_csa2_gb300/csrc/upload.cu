// A decode step's host inputs in one host-to-device copy: the caller packs
// every input of the step (queries, positions, the entries the step's tokens
// append to the caches, as fp32 latent rows for the FP4 main-KV cache) into one
// pinned buffer behind a table of segments; csa2_upload copies the whole
// buffer to a device staging area and one kernel moves each segment to its
// place, packing the appended latent rows into FP4 cache rows on the way
// (the same row arithmetic as csa2_quantize_kv_fp4, quant_fp4.cuh).
#include "quant_fp4.cuh"

namespace csa2 {
namespace {

constexpr int kUpThreads = 256;
constexpr int kUpWarps = kUpThreads / 32;

__global__ void __launch_bounds__(kUpThreads)
upload_kernel(const uint8_t* __restrict__ stage, int n_segs) {
  __shared__ __align__(16) uint8_t rowbuf[kUpWarps][kRowBytes];
  const csa2_upload_seg* segs = reinterpret_cast<const csa2_upload_seg*>(stage);
  const int64_t nthreads = (int64_t)gridDim.x * kUpThreads;
  const int64_t gtid = (int64_t)blockIdx.x * kUpThreads + threadIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nwarps = (int64_t)gridDim.x * kUpWarps;
  const int64_t gwarp = (int64_t)blockIdx.x * kUpWarps + warp;
  for (int i = 0; i < n_segs; ++i) {
    const csa2_upload_seg sg = segs[i];
    uint8_t* dst = reinterpret_cast<uint8_t*>(sg.dst);
    const uint8_t* src = stage + sg.src_off;
    if (sg.kind == CSA2_UPLOAD_KV_FP4) {
      // one warp per latent row: 512 fp32 channels -> one 288-byte FP4 row
      for (int64_t r = gwarp; r < (int64_t)sg.rows; r += nwarps)
        quantize_fp4_row_warp(reinterpret_cast<const float*>(src + r * sg.row_bytes),
                              dst + r * sg.dst_stride, rowbuf[warp], lane);
    } else if (((sg.dst | sg.src_off | sg.row_bytes | sg.dst_stride) & 15u) == 0) {
      const int64_t per_row = (int64_t)(sg.row_bytes >> 4);  // 16-byte units
      const int64_t units = per_row * (int64_t)sg.rows;
      for (int64_t u = gtid; u < units; u += nthreads) {
        const int64_t r = u / per_row, c = u - r * per_row;
        *reinterpret_cast<uint4*>(dst + r * sg.dst_stride + 16 * c) =
            *reinterpret_cast<const uint4*>(src + r * sg.row_bytes + 16 * c);
      }
    } else {
      const int64_t per_row = (int64_t)sg.row_bytes;
      const int64_t units = per_row * (int64_t)sg.rows;
      for (int64_t u = gtid; u < units; u += nthreads) {
        const int64_t r = u / per_row, c = u - r * per_row;
        dst[r * sg.dst_stride + c] = src[r * sg.row_bytes + c];
      }
    }
  }
}

}  // namespace

cudaError_t launch_upload(const void* host_packed, size_t bytes, int n_segs, void* dev_stage,
                          int64_t work_units, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyAsync(dev_stage, host_packed, bytes, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess || n_segs == 0) return e;
  // about four 16-byte units (or one warp-row per warp) per thread, at most two
  // CTAs per SM
  int64_t blocks = (work_units + 4 * kUpThreads - 1) / (4 * kUpThreads);
  const int64_t cap = (int64_t)device_sm_count() * 2;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  upload_kernel<<<(unsigned)blocks, kUpThreads, 0, stream>>>(
      reinterpret_cast<const uint8_t*>(dev_stage), n_segs);
  return cudaGetLastError();
}

}  // namespace csa2
