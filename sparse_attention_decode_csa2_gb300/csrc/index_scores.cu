// Indexer scores restricted to a candidate pool (DeepSeek-V4.1-Flash paper
// walkthrough, 1.(4).2 "Hierarchical Sparse Indexer": later layers score only
// the pool positions chosen by the first Full layer), and the entry point of
// the full indexer scan, which runs on the tensor cores (index_tc.cu).
//
// Pool scoring gathers one 64-byte indexer-K row per pool slot, so it is a
// gather of small rows rather than a dense GEMM; it runs on CUDA cores with
// the head sum taken first: qsum[d] = sum_h qI[h][d] (E4M3 values are integer
// multiples of 2^-9 below 2^9, so for H_I <= 32 every qsum[d] is exact in
// fp32) and score = qsum . KI[j] in fp32 FMA (exact for integer inputs).
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 256;

// qsum[d] = sum_h e4m3(q[h][d]) for one query.  The H_I x D_I bytes are
// fetched with one 16-byte load per thread (a single memory latency), decoded
// into `qf` and summed over heads from shared memory.  Needs H_I * D_I <= 16 *
// blockDim.x; ends with a barrier.
__device__ __forceinline__ void load_qsum(const uint8_t* __restrict__ q, int H_I, int D_I,
                                          float* __restrict__ qf, float* __restrict__ qsum) {
  const int nchunks = H_I * D_I / 16;
  if ((int)threadIdx.x < nchunks) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(q) + threadIdx.x);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float* dst = qf + threadIdx.x * 16;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 lo = half2_bits_to_float2(e4m3x2_to_f16x2((uint16_t)(w[i] & 0xFFFFu)));
      const float2 hi = half2_bits_to_float2(e4m3x2_to_f16x2((uint16_t)(w[i] >> 16)));
      dst[4 * i + 0] = lo.x;
      dst[4 * i + 1] = lo.y;
      dst[4 * i + 2] = hi.x;
      dst[4 * i + 3] = hi.y;
    }
  }
  __syncthreads();
  for (int d = threadIdx.x; d < D_I; d += blockDim.x) {
    float s = 0.0f;
    for (int h = 0; h < H_I; ++h) s += qf[h * D_I + d];
    qsum[d] = s;
  }
  __syncthreads();
}

// 16 E4M3 bytes (a uint4) dotted with 16 fp32 weights.
__device__ __forceinline__ float dot16(uint4 v, const float* w) {
  uint32_t words[4] = {v.x, v.y, v.z, v.w};
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 lo = half2_bits_to_float2(e4m3x2_to_f16x2((uint16_t)(words[i] & 0xFFFFu)));
    float2 hi = half2_bits_to_float2(e4m3x2_to_f16x2((uint16_t)(words[i] >> 16)));
    acc = fmaf(lo.x, w[4 * i + 0], acc);
    acc = fmaf(lo.y, w[4 * i + 1], acc);
    acc = fmaf(hi.x, w[4 * i + 2], acc);
    acc = fmaf(hi.y, w[4 * i + 3], acc);
  }
  return acc;
}

// Pool scoring: one CTA scores 1024 pool slots of one query (gathered rows).
template <int D_I>
__global__ void __launch_bounds__(kThreads)
pool_scores_kernel(const uint8_t* __restrict__ q_fp8, const uint8_t* __restrict__ k_fp8, int H_I,
                   int64_t N, int64_t kv_seq_stride, int q_per_seq,
                   const int32_t* __restrict__ pool, int P, float* __restrict__ pool_scores,
                   int32_t* status) {
  constexpr int TPE = D_I / 16;
  constexpr int EPI = kThreads / TPE;
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(16) float qf[32 * 128];
  __shared__ float qsum[D_I];
  const int q = blockIdx.y;
  load_qsum(q_fp8 + (int64_t)q * H_I * D_I, H_I, D_I, qf, qsum);
  const int sub = threadIdx.x % TPE;
  float w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = qsum[sub * 16 + i];
  const uint8_t* kseq = k_fp8 + (int64_t)(q / q_per_seq) * kv_seq_stride * D_I;
  const int32_t* prow = pool + (int64_t)q * P;
  for (int it = 0; it < 1024 / EPI; ++it) {
    const int p = blockIdx.x * 1024 + it * EPI + threadIdx.x / TPE;
    int32_t j = -1;
    bool ok = false;
    if (p < P) {
      j = prow[p];
      ok = (j >= 0 && j < N);
      if (sub == 0) {
        bool bad = (j >= N) || (j < -1);
        if (p > 0) {
          int32_t prev = prow[p - 1];
          if (j >= 0 && (prev < 0 || prev >= j)) bad = true;  // not ascending / -1 not at tail
        }
        if (bad) set_status(status, kStatusBadIndex);
      }
    }
    uint4 v = ok ? __ldg(reinterpret_cast<const uint4*>(kseq + (int64_t)j * D_I) + sub)
                 : make_uint4(0, 0, 0, 0);
    float s = dot16(v, w);
#pragma unroll
    for (int o = TPE / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (sub == 0 && p < P) pool_scores[(int64_t)q * P + p] = ok ? s : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_index_scores(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I,
                                int D_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                const int32_t* q_pos, int ratio, float* scores, int32_t* status,
                                cudaStream_t stream) {
  if (B == 0 || N == 0) return cudaSuccess;
  return launch_index_scores_tc(q_fp8, k_fp8, B, H_I, D_I, N, kv_seq_stride, q_per_seq, q_pos,
                                ratio, scores, status, stream);
}

cudaError_t launch_pool_scores(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I,
                               int D_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                               const int32_t* pool, int P, float* pool_scores, int32_t* n_valid,
                               int32_t* status, cudaStream_t stream) {
  (void)n_valid;
  if (B == 0 || P == 0) return cudaSuccess;
  dim3 grid((unsigned)((P + 1023) / 1024), (unsigned)B);
  switch (D_I) {
    case 32:
      pool_scores_kernel<32><<<grid, kThreads, 0, stream>>>(q_fp8, k_fp8, H_I, N, kv_seq_stride,
                                                           q_per_seq, pool, P, pool_scores, status);
      break;
    case 64:
      pool_scores_kernel<64><<<grid, kThreads, 0, stream>>>(q_fp8, k_fp8, H_I, N, kv_seq_stride,
                                                           q_per_seq, pool, P, pool_scores, status);
      break;
    default:
      pool_scores_kernel<128><<<grid, kThreads, 0, stream>>>(
          q_fp8, k_fp8, H_I, N, kv_seq_stride, q_per_seq, pool, P, pool_scores, status);
  }
  return cudaGetLastError();
}

}  // namespace csa2
