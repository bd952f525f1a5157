// Indexer scores restricted to a candidate pool (DeepSeek-V4.1-Flash paper
// walkthrough, 1.(4).2 "Hierarchical Sparse Indexer": later layers score only
// the pool positions chosen by the first Full layer), and the entry point of
// the full indexer scan, which runs on the tensor cores (index_tc.cu).
//
// Pool scoring gathers one D_I-byte indexer-K row per pool slot, so it is a
// gather of small rows rather than a dense GEMM.  The head sum is taken first:
// qsum[d] = sum_h qI[h][d] (E4M3 values are integer multiples of 2^-9 below
// 2^9, so for H_I <= 32 every qsum[d] is exact in fp32), and score = qsum .
// KI[j].  The dot products run as warp-level m16n8k16 MMAs, 16 gathered
// entries per group: each E4M3 pair of a row converts straight into an f16x2
// A register (exact), B holds qsum as two f16 parts (its f16 rounding and the
// rounding of the remainder: 22 significant bits, exact for integer inputs)
// in columns 0 and 1, and the products accumulate in fp32.  Lane (g, t)
// decodes word 4s + t of entries g and g + 8 for k16 step s: in step s,
// k = 2t + {0,1} is element 16s + 4t + {0,1} and k = 2t + 8 + {0,1} is element
// 16s + 4t + 2 + {0,1}, and B follows the same order.
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

__device__ __forceinline__ void mma_16816_f16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// f16 part p of x (p = 0: rounding of x, p = 1: rounding of the remainder).
__device__ __forceinline__ uint16_t f16_part(float x, int p) {
  const __half h = __float2half_rn(x);
  return __half_as_ushort(p ? __float2half_rn(x - __half2float(h)) : h);
}

// Pool scoring: one CTA scores 1024 pool slots of one query (gathered rows),
// each warp 16 entries at a time.
template <int D_I>
__global__ void __launch_bounds__(kThreads)
pool_scores_kernel(const uint8_t* __restrict__ q_fp8, const uint8_t* __restrict__ k_fp8, int H_I,
                   int64_t N, int64_t kv_seq_stride, int q_per_seq,
                   const int32_t* __restrict__ pool, int P, float* __restrict__ pool_scores,
                   int32_t* status) {
  constexpr int kSteps = D_I / 16;  // k16 steps (one code word per entry per step)
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(16) float qf[32 * 128];
  __shared__ float qsum[D_I];
  const int q = blockIdx.y;
  load_qsum(q_fp8 + (int64_t)q * H_I * D_I, H_I, D_I, qf, qsum);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  // B registers of lane (g, t): column g = part g of qsum (g < 2), zero otherwise
  uint32_t bq[kSteps][2];
#pragma unroll
  for (int st = 0; st < kSteps; ++st)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = 16 * st + 4 * t + 2 * h;
      bq[st][h] = g < 2 ? ((uint32_t)f16_part(qsum[e], g) |
                           ((uint32_t)f16_part(qsum[e + 1], g) << 16))
                        : 0u;
    }
  const uint8_t* kseq = k_fp8 + (int64_t)(q / q_per_seq) * kv_seq_stride * D_I;
  const int32_t* prow = pool + (int64_t)q * P;
  constexpr int kGroups = 1024 / 16 / (kThreads / 32);  // per warp
  for (int it = 0; it < kGroups; ++it) {
    const int p0 = blockIdx.x * 1024 + (it * (kThreads / 32) + warp) * 16;
    const int pA = p0 + g, pB = pA + 8;
    int32_t jA = -1, jB = -1;
    if (pA < P) jA = __ldg(prow + pA);
    if (pB < P) jB = __ldg(prow + pB);
    // lanes t = 0 / 1 check slots g / g + 8: in range, ascending, -1 only at the tail
    if (t < 2) {
      const int p = t == 0 ? pA : pB;
      const int32_t j = t == 0 ? jA : jB;
      if (p < P) {
        bool bad = (j >= N) || (j < -1);
        if (p > 0) {
          const int32_t prev = __ldg(prow + p - 1);
          if (j >= 0 && (prev < 0 || prev >= j)) bad = true;
        }
        if (bad) set_status(status, kStatusBadIndex);
      }
    }
    const bool okA = jA >= 0 && jA < N, okB = jB >= 0 && jB < N;
    const uint32_t* rwA = reinterpret_cast<const uint32_t*>(kseq + (int64_t)(okA ? jA : 0) * D_I);
    const uint32_t* rwB = reinterpret_cast<const uint32_t*>(kseq + (int64_t)(okB ? jB : 0) * D_I);
    uint32_t wA[kSteps], wB[kSteps];
#pragma unroll
    for (int st = 0; st < kSteps; ++st) {
      wA[st] = okA ? __ldg(rwA + 4 * st + t) : 0u;
      wB[st] = okB ? __ldg(rwB + 4 * st + t) : 0u;
    }
    float c[4] = {0.f, 0.f, 0.f, 0.f}, d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int st = 0; st < kSteps; ++st) {
      const uint32_t a0 = e4m3x2_to_f16x2((uint16_t)(wA[st] & 0xFFFFu));
      const uint32_t a1 = e4m3x2_to_f16x2((uint16_t)(wB[st] & 0xFFFFu));
      const uint32_t a2 = e4m3x2_to_f16x2((uint16_t)(wA[st] >> 16));
      const uint32_t a3 = e4m3x2_to_f16x2((uint16_t)(wB[st] >> 16));
      if (st & 1)
        mma_16816_f16(d, a0, a1, a2, a3, bq[st][0], bq[st][1]);
      else
        mma_16816_f16(c, a0, a1, a2, a3, bq[st][0], bq[st][1]);
    }
    // lane (g, 0) holds columns 0, 1 (the two parts) of entries g and g + 8
    if (t == 0) {
      if (pA < P) pool_scores[(int64_t)q * P + pA] = okA ? (c[0] + d[0]) + (c[1] + d[1]) : -INFINITY;
      if (pB < P) pool_scores[(int64_t)q * P + pB] = okB ? (c[2] + d[2]) + (c[3] + d[3]) : -INFINITY;
    }
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
                               const int32_t* pool, int P, float* pool_scores, int32_t* status,
                               cudaStream_t stream) {
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
