// Lightweight indexer: scores main-KV entries with indexer q and indexer K
// (DeepSeek-V4.1-Flash paper walkthrough, 1.(4) "CSA2"; Reindex layers use
// their own q against the shared K, 1.(4).1; pool-restricted scoring,
// 1.(4).2).
//
// score[q][j] = sum_h sum_d qI[q][h][d] * KI[j][d].  Because every indexer
// head reads the same per-entry K vector, the head sum is taken first:
// qsum[d] = sum_h qI[h][d].  E4M3 values are integer multiples of 2^-9 below
// 2^9, so for H_I <= 32 every qsum[d] is an integer multiple of 2^-9 below
// 2^14: exact in fp32.  The 64-term dot product qsum . KI[j] then runs in
// fp32 FMA, exact whenever the partial sums are representable (integer
// inputs), and within a few fp32 ulps otherwise.
//
// Decode layout (few queries per context): one CTA scores 1024 entries of one
// query; D_I/16 threads share one 16-byte chunk of an entry row each, so a
// warp streams 8 (D_I = 64) whole rows per load instruction.
// Prefill layout (many queries share one context): one CTA scores a tile of
// 16 queries x 256 entries, each thread owns one entry row in registers.
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

template <int D_I>
__global__ void __launch_bounds__(kThreads)
index_scores_decode_kernel(const uint8_t* __restrict__ q_fp8, const uint8_t* __restrict__ k_fp8,
                           int H_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                           const int32_t* __restrict__ q_pos, int ratio,
                           float* __restrict__ scores) {
  constexpr int TPE = D_I / 16;               // threads per entry
  constexpr int EPI = kThreads / TPE;         // entries per iteration
  constexpr int ITERS = 1024 / EPI;
  constexpr int U = ITERS < 8 ? ITERS : 8;
  __shared__ __align__(16) float qf[32 * 128];
  __shared__ float qsum[D_I];
  const int q = blockIdx.y;
  const int sub = threadIdx.x % TPE;
  const int64_t nv = n_visible(q_pos, q, ratio, N);
  const uint8_t* kseq = k_fp8 + (int64_t)(q / q_per_seq) * kv_seq_stride * D_I;
  float* srow = scores + (int64_t)q * N;
  const int64_t base = (int64_t)blockIdx.x * 1024 + threadIdx.x / TPE;
  // first batch of K rows in flight before the q prologue
  uint4 v[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t e = base + (int64_t)u * EPI;
    v[u] = (e < nv) ? __ldg(reinterpret_cast<const uint4*>(kseq + e * D_I) + sub)
                    : make_uint4(0, 0, 0, 0);
  }
  load_qsum(q_fp8 + (int64_t)q * H_I * D_I, H_I, D_I, qf, qsum);
  float w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = qsum[sub * 16 + i];
#pragma unroll
  for (int it0 = 0; it0 < ITERS; it0 += U) {
    if (it0 > 0) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t e = base + (int64_t)(it0 + u) * EPI;
        v[u] = (e < nv) ? __ldg(reinterpret_cast<const uint4*>(kseq + e * D_I) + sub)
                        : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t e = base + (int64_t)(it0 + u) * EPI;
      float s = dot16(v[u], w);
#pragma unroll
      for (int o = TPE / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (sub == 0 && e < N) srow[e] = (e < nv) ? s : -INFINITY;
    }
  }
}

// Many queries per context: a CTA scores QT consecutive queries of one
// sequence against ET = 256 entries; thread t owns entry t of the tile.
template <int D_I>
__global__ void __launch_bounds__(kThreads)
index_scores_tiled_kernel(const uint8_t* __restrict__ q_fp8, const uint8_t* __restrict__ k_fp8,
                          int B, int H_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                          const int32_t* __restrict__ q_pos, int ratio,
                          float* __restrict__ scores) {
  constexpr int QT = 16;
  __shared__ __align__(16) float qsum[QT][D_I];
  __shared__ __align__(16) uint8_t qbytes[QT * 32 * 128];
  const int q0 = blockIdx.y * QT;
  const int nq = min(QT, B - q0);
  {
    // all queries' bytes with one 16-byte load per thread per round
    const int chunks = nq * H_I * D_I / 16;
    const uint4* src = reinterpret_cast<const uint4*>(q_fp8 + (int64_t)q0 * H_I * D_I);
    for (int c = threadIdx.x; c < chunks; c += kThreads)
      reinterpret_cast<uint4*>(qbytes)[c] = __ldg(src + c);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < QT * D_I; i += kThreads) {
    const int qq = i / D_I, d = i % D_I;
    float s = 0.0f;
    if (qq < nq)
      for (int h = 0; h < H_I; ++h)
        s += half2_bits_to_float2(e4m3x2_to_f16x2((uint16_t)qbytes[(qq * H_I + h) * D_I + d])).x;
    qsum[qq][d] = s;
  }
  __syncthreads();
  const int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  if (e >= N) return;
  const uint8_t* kseq = k_fp8 + (int64_t)(q0 / q_per_seq) * kv_seq_stride * D_I;
  float kv[D_I];
  {
    const uint4* src = reinterpret_cast<const uint4*>(kseq + e * D_I);
#pragma unroll
    for (int c = 0; c < D_I / 16; ++c) {
      uint4 v = __ldg(src + c);
      uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 lo = half2_bits_to_float2(e4m3x2_to_f16x2((uint16_t)(words[i] & 0xFFFFu)));
        float2 hi = half2_bits_to_float2(e4m3x2_to_f16x2((uint16_t)(words[i] >> 16)));
        kv[16 * c + 4 * i + 0] = lo.x;
        kv[16 * c + 4 * i + 1] = lo.y;
        kv[16 * c + 4 * i + 2] = hi.x;
        kv[16 * c + 4 * i + 3] = hi.y;
      }
    }
  }
#pragma unroll 1
  for (int qq = 0; qq < QT; ++qq) {
    const int q = q0 + qq;
    if (q >= B) break;
    const float4* qs = reinterpret_cast<const float4*>(qsum[qq]);
    float acc = 0.0f;
#pragma unroll
    for (int d4 = 0; d4 < D_I / 4; ++d4) {
      float4 w = qs[d4];
      acc = fmaf(kv[4 * d4 + 0], w.x, acc);
      acc = fmaf(kv[4 * d4 + 1], w.y, acc);
      acc = fmaf(kv[4 * d4 + 2], w.z, acc);
      acc = fmaf(kv[4 * d4 + 3], w.w, acc);
    }
    const int64_t nv = n_visible(q_pos, q, ratio, N);
    scores[(int64_t)q * N + e] = (e < nv) ? acc : -INFINITY;
  }
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

template <int D_I>
cudaError_t launch_scores_t(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I, int64_t N,
                            int64_t kv_seq_stride, int q_per_seq, const int32_t* q_pos, int ratio,
                            float* scores, cudaStream_t stream) {
  if (q_per_seq >= 16 && q_per_seq % 16 == 0) {
    dim3 grid((unsigned)((N + kThreads - 1) / kThreads), (unsigned)((B + 15) / 16));
    index_scores_tiled_kernel<D_I><<<grid, kThreads, 0, stream>>>(
        q_fp8, k_fp8, B, H_I, N, kv_seq_stride, q_per_seq, q_pos, ratio, scores);
  } else {
    dim3 grid((unsigned)((N + 1023) / 1024), (unsigned)B);
    index_scores_decode_kernel<D_I><<<grid, kThreads, 0, stream>>>(
        q_fp8, k_fp8, H_I, N, kv_seq_stride, q_per_seq, q_pos, ratio, scores);
  }
  return cudaGetLastError();
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
