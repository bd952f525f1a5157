// MXFP4 lightweight indexer (DeepSeek-V4.1-Flash paper walkthrough, 1.(5).4:
// the indexer query and key are FP4 in the OCP MXFP4 format; 1.(4) "CSA2" and
// 1.(4).2 for what the scores feed).
//
// Row format (OCP MX, MXFP4): D_I / 2 bytes of E2M1 codes (element 2j in the
// low nibble of byte j), then D_I / 32 E8M0 scale bytes (2^(byte - 127)), one
// per block of 32 elements.  At D_I = 128 a row is 68 bytes.
//
// Scoring.  The score is a sum over indexer heads of q_h . K_j, so the head
// sum is formed first (qsum = sum_h q_h, compensated fp32 summation of exact
// decoded values) and each entry costs one 128-long dot product: 68 bytes of
// HBM for 128 multiply-adds.  That is a matrix-vector product bounded by HBM
// bandwidth, so it runs on the CUDA cores, not the tensor cores:
//  * full scan: a persistent grid (a multiple of the SM count) walks
//    contiguous runs of 128-entry tiles (8704 bytes); one producer warp
//    streams the tiles into a 4-stage shared-memory ring with 1D bulk
//    copies (cp.async.bulk, mbarrier completion), four consumer warps score
//    them.  Four lanes share an entry, one 32-element block each, and add
//    their partial dot products with two shuffles.
//  * pool scan (Reindex layers): the same per-entry arithmetic on gathered
//    rows, one entry per four lanes.
// Products are fp32 FMAs of exact decoded values; the per-block partial is
// scaled by the entry's E8M0 scale.
#include "csa2_internal.cuh"
#include "tc_common.cuh"

namespace csa2 {
namespace {

constexpr int kMxDI = 128;
constexpr int kMxRow = kMxDI / 2 + kMxDI / 32;  // 68
constexpr int kMxCodes = kMxDI / 2;             // 64
constexpr int kTileRows = 128;
constexpr int kTileBytes = kTileRows * kMxRow;  // 8704, a multiple of 16
constexpr int kStages = 4;
constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kScanThreads = kConsumers + 32;  // + one producer warp
constexpr int kQChunk = 8;                     // queries whose qsum is staged at once

__device__ __forceinline__ float e8m0_to_float(uint32_t b) {
  return __uint_as_float(b ? (b << 23) : 0x00400000u);  // 2^(b-127); b = 0 is 2^-127
}

// E2M1 code of x for a power-of-two block scale X: the code whose value is
// nearest to the exact |x| / X, ties to the even code, saturating at 6.  The
// midpoints t * X are exact in fp32 (t has <= 3 significant bits, X a power of
// two >= 2^-127), so the comparisons are exact; strict / non-strict encode
// ties-to-even (0.25, 1.25, 2.5, 5 round down; 0.75, 1.75, 3.5 round up).
__device__ __forceinline__ uint32_t e2m1_code_pow2(float x, float X) {
  const uint32_t sign = __float_as_uint(x) >> 31;
  const float m = fabsf(x);
  const uint32_t c = (m > 0.25f * X) + (m >= 0.75f * X) + (m > 1.25f * X) + (m >= 1.75f * X) +
                     (m > 2.5f * X) + (m >= 3.5f * X) + (m > 5.0f * X);
  return (sign << 3) | c;
}

// One warp per 128 elements of a row: lane l takes elements 4l..4l+3, so a
// 32-element block sits in 8 consecutive lanes.  Shared exponent =
// floor(log2(absmax)) - 2 clamped to >= -127, i.e. scale byte =
// max(exponent field of absmax - 2, 0) (a zero or subnormal absmax gives 0).
__global__ void __launch_bounds__(256)
quantize_mxfp4_kernel(const float* __restrict__ x, int64_t n_rows, int d,
                      uint8_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int chunks = (d + 127) / 128;
  const int64_t rb = d / 2 + d / 32;
  const int64_t n_items = n_rows * chunks;
  for (int64_t it = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < n_items;
       it += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int64_t row = it / chunks;
    const int c0 = (int)(it % chunks) * 128;
    const bool active = c0 + 4 * lane < d;  // d % 32 == 0: whole 8-lane blocks
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active) v = __ldg(reinterpret_cast<const float4*>(x + row * d + c0) + lane);
    float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
    const int ef = (int)((__float_as_uint(a) >> 23) & 0xFFu);
    const uint32_t sbyte = (uint32_t)(ef > 2 ? ef - 2 : 0);
    const float X = e8m0_to_float(sbyte);
    if (active) {
      const uint32_t c0c = e2m1_code_pow2(v.x, X), c1c = e2m1_code_pow2(v.y, X);
      const uint32_t c2c = e2m1_code_pow2(v.z, X), c3c = e2m1_code_pow2(v.w, X);
      uint8_t* orow = out + row * rb;
      const int byte0 = (c0 + 4 * lane) / 2;
      orow[byte0] = (uint8_t)(c0c | (c1c << 4));
      orow[byte0 + 1] = (uint8_t)(c2c | (c3c << 4));
      if ((lane & 7) == 0) orow[d / 2 + (c0 + 4 * lane) / 32] = (uint8_t)sbyte;
    }
  }
}

// fp32 pair FMA (Blackwell packed FP32 pipe): acc += a * b, element-wise.
__device__ __forceinline__ void ffma2(float2& acc, float2 a, float2 b) {
  uint64_t d;
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%1, %2};\n\tmov.b64 rb, {%3, %4};\n\tmov.b64 rc, {%5, %6};\n\t"
      "fma.rn.f32x2 %0, ra, rb, rc;\n\t}"
      : "=l"(d)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(acc.x), "f"(acc.y));
  acc.x = __uint_as_float((uint32_t)d);
  acc.y = __uint_as_float((uint32_t)(d >> 32));
}

// Dot product of one 32-element block (16 code bytes in w[0..3]) with the
// matching 32 qsum values (in registers), unscaled.
__device__ __forceinline__ float block_dot(const uint32_t w[4], const float* qs) {
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = half2_bits_to_float2(e2m1x2_to_f16x2((w[c] >> (8 * j)) & 0xFFu));
      const float2 q = make_float2(qs[8 * c + 2 * j], qs[8 * c + 2 * j + 1]);
      if (j & 1) ffma2(acc1, f, q);
      else ffma2(acc0, f, q);
    }
  }
  return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

// qsum[d] = sum_h value(q[h][d]) for one query (MXFP4 rows of kMxDI), by
// compensated (Neumaier) fp32 summation of the exact decoded values; thread t
// of `nthreads` computes dims t, t + nthreads, ...
__device__ __forceinline__ float mx_qsum_dim(const uint8_t* __restrict__ q, int H_I, int d) {
  float s = 0.0f, comp = 0.0f;
  for (int h = 0; h < H_I; ++h) {
    const uint8_t* row = q + (int64_t)h * kMxRow;
    const uint32_t byte = __ldg(row + d / 2);
    const uint32_t code = (d & 1) ? (byte >> 4) : (byte & 15u);
    const float v =
        half2_bits_to_float2(e2m1x2_to_f16x2(code)).x * e8m0_to_float(__ldg(row + kMxCodes + d / 32));
    const float t = s + v;
    comp += (fabsf(s) >= fabsf(v)) ? ((s - t) + v) : ((v - t) + s);
    s = t;
  }
  return s + comp;
}

struct ScanSmem {
  uint8_t tiles[kStages][kTileBytes];
  float qsum[kQChunk][kMxDI];
  uint64_t full[kStages];
  uint64_t empty[kStages];
};

// Entries of the tile that must be read: those visible to some query of the
// sequence.  Both the producer and the consumers evaluate it.
__device__ __forceinline__ int tile_rows_loaded(int64_t vis_max, int64_t row0) {
  const int64_t r = vis_max - row0;
  return r <= 0 ? 0 : (r >= kTileRows ? kTileRows : (int)r);
}

__device__ __forceinline__ int64_t seq_vis_max(const int32_t* q_pos, int s, int q_per_seq, int B,
                                               int ratio, int64_t N) {
  int64_t m = 0;
  const int q_end = min(B, (s + 1) * q_per_seq);
  for (int q = s * q_per_seq; q < q_end; ++q) {
    const int64_t v = n_visible(q_pos, q, ratio, N);
    m = v > m ? v : m;
  }
  return m;
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Full scan.  Tiles are numbered (sequence, tile) row-major, T tiles of 128
// entries per sequence; CTA c takes the contiguous run [c*total/C, (c+1)*total/C),
// so it meets few sequence changes (each recomputes the staged qsum).
__global__ void __launch_bounds__(kScanThreads, 3)
mx_scores_kernel(const uint8_t* __restrict__ q_mx, const uint8_t* __restrict__ k_mx, int B,
                 int H_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                 const int32_t* __restrict__ q_pos, int ratio, float* __restrict__ scores,
                 int32_t* status) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  ScanSmem& sm = *reinterpret_cast<ScanSmem*>(smem_raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int S = (B + q_per_seq - 1) / q_per_seq;
  const int64_t T = (N + kTileRows - 1) / kTileRows;
  const int64_t total = (int64_t)S * T;
  const int64_t t_begin = total * blockIdx.x / gridDim.x;
  const int64_t t_end = total * (blockIdx.x + 1) / gridDim.x;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(tc::su32(&sm.full[i]), 1);
      tc::mbar_init(tc::su32(&sm.empty[i]), kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();

  if (warp == kConsumerWarps) {
    // ---------------- producer: one lane issues the tile copies ----------------
    if (lane != 0) return;
    int64_t n = 0;  // loads issued
    int cur_s = -1;
    int64_t vis = 0;
    for (int64_t tile = t_begin; tile < t_end; ++tile) {
      const int s = (int)(tile / T);
      const int64_t row0 = (tile - (int64_t)s * T) * kTileRows;
      if (s != cur_s) {
        cur_s = s;
        vis = seq_vis_max(q_pos, s, q_per_seq, B, ratio, N);
      }
      const int rows = tile_rows_loaded(vis, row0);
      if (rows == 0) continue;
      const int st = (int)(n % kStages);
      if (n >= kStages &&
          !tc::mbar_wait(tc::su32(&sm.empty[st]), (uint32_t)((n / kStages - 1) & 1), status))
        return;
      const uint8_t* src = k_mx + ((int64_t)s * kv_seq_stride + row0) * kMxRow;
      const uint32_t bytes = (uint32_t)rows * kMxRow;
      const uint32_t b16 = bytes & ~15u;
      // the tail of a ragged tile (< 16 bytes, whole words) by plain loads,
      // so that no copy reads past the last entry
      for (uint32_t o = b16; o < bytes; o += 4)
        *reinterpret_cast<uint32_t*>(&sm.tiles[st][o]) =
            __ldg(reinterpret_cast<const uint32_t*>(src + o));
      tc::proxy_fence();
      tc::mbar_expect_tx(tc::su32(&sm.full[st]), b16);
      bulk_copy(tc::su32(&sm.tiles[st][0]), src, b16, tc::su32(&sm.full[st]));
      ++n;
    }
    return;
  }

  // ---------------- consumers ----------------
  const int blk = lane & 3;                 // 32-element block of this lane
  const int rsub = tid >> 2;                // 0..31: rows rsub + 32 i
  int64_t n = 0;                            // loads consumed
  int cur_s = -1, cur_chunk = -1;
  int64_t vis = 0;
  for (int64_t tile = t_begin; tile < t_end; ++tile) {
    const int s = (int)(tile / T);
    const int64_t row0 = (tile - (int64_t)s * T) * kTileRows;
    if (s != cur_s) {
      cur_s = s;
      cur_chunk = -1;
      vis = seq_vis_max(q_pos, s, q_per_seq, B, ratio, N);
    }
    const int rows = tile_rows_loaded(vis, row0);
    const int rows_in_tile = (int)((N - row0) < kTileRows ? (N - row0) : kTileRows);
    const int st = (int)(n % kStages);
    if (rows > 0 &&
        !tc::mbar_wait(tc::su32(&sm.full[st]), (uint32_t)((n / kStages) & 1), status))
      return;
    const uint8_t* tileb = sm.tiles[st];
    const int q_first = s * q_per_seq;
    const int q_last = min(B, q_first + q_per_seq);
    for (int qc = q_first; qc < q_last; qc += kQChunk) {
      const int nq = min(kQChunk, q_last - qc);
      if (qc != cur_chunk) {
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
        for (int i = tid; i < nq * kMxDI; i += kConsumers)
          sm.qsum[i / kMxDI][i % kMxDI] =
              mx_qsum_dim(q_mx + (int64_t)(qc + i / kMxDI) * H_I * kMxRow, H_I, i % kMxDI);
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
        cur_chunk = qc;
      }
      for (int ql = 0; ql < nq; ++ql) {
        const int q = qc + ql;
        const int64_t nv = n_visible(q_pos, q, ratio, N);
        float qs[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 v4 = *reinterpret_cast<const float4*>(&sm.qsum[ql][32 * blk + 4 * i]);
          qs[4 * i] = v4.x;
          qs[4 * i + 1] = v4.y;
          qs[4 * i + 2] = v4.z;
          qs[4 * i + 3] = v4.w;
        }
        float* srow = scores + (int64_t)q * N + row0;
#pragma unroll
        for (int i = 0; i < kTileRows / 32; ++i) {
          const int r = rsub + 32 * i;
          float part = 0.0f;
          if (r < rows) {
            const uint32_t* rw = reinterpret_cast<const uint32_t*>(tileb + r * kMxRow);
            uint32_t w[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) w[c] = rw[4 * blk + c];
            const uint32_t sb = (rw[kMxCodes / 4] >> (8 * blk)) & 0xFFu;
            part = block_dot(w, qs) * e8m0_to_float(sb);
          }
          part += __shfl_xor_sync(0xffffffffu, part, 1);
          part += __shfl_xor_sync(0xffffffffu, part, 2);
          if (blk == 0 && r < rows_in_tile) srow[r] = (row0 + r < nv) ? part : -INFINITY;
        }
      }
    }
    if (rows > 0) {
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::su32(&sm.empty[st]));
      ++n;
    }
  }
}

// Pool scan: CTA (x, q) scores pool slots [1024 x, 1024 x + 1024) of query q.
constexpr int kPoolThreads = 256;
constexpr int kPoolSlots = 1024;

__global__ void __launch_bounds__(kPoolThreads)
mx_pool_scores_kernel(const uint8_t* __restrict__ q_mx, const uint8_t* __restrict__ k_mx, int H_I,
                      int64_t N, int64_t kv_seq_stride, int q_per_seq,
                      const int32_t* __restrict__ pool, int P, float* __restrict__ pool_scores,
                      int32_t* status) {
  __shared__ __align__(16) float qsum[kMxDI];
  pdl_trigger();
  pdl_wait();
  const int q = blockIdx.y;
  for (int d = threadIdx.x; d < kMxDI; d += kPoolThreads)
    qsum[d] = mx_qsum_dim(q_mx + (int64_t)q * H_I * kMxRow, H_I, d);
  __syncthreads();
  const int blk = threadIdx.x & 3;
  float qs[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) qs[i] = qsum[32 * blk + i];
  const uint8_t* kseq = k_mx + (int64_t)(q / q_per_seq) * kv_seq_stride * kMxRow;
  const int32_t* prow = pool + (int64_t)q * P;
  for (int it = 0; it < kPoolSlots / (kPoolThreads / 4); ++it) {
    const int p = blockIdx.x * kPoolSlots + it * (kPoolThreads / 4) + (threadIdx.x >> 2);
    int32_t j = -1;
    bool ok = false;
    if (p < P) {
      j = prow[p];
      ok = (j >= 0 && j < N);
      if (blk == 0) {
        bool bad = (j >= N) || (j < -1);
        if (p > 0) {
          const int32_t prev = prow[p - 1];
          if (j >= 0 && (prev < 0 || prev >= j)) bad = true;  // not ascending / -1 not at tail
        }
        if (bad) set_status(status, kStatusBadIndex);
      }
    }
    float part = 0.0f;
    if (ok) {
      const uint32_t* rw = reinterpret_cast<const uint32_t*>(kseq + (int64_t)j * kMxRow);
      uint32_t w[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) w[c] = __ldg(rw + 4 * blk + c);
      const uint32_t sb = (__ldg(rw + kMxCodes / 4) >> (8 * blk)) & 0xFFu;
      part = block_dot(w, qs) * e8m0_to_float(sb);
    }
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    part += __shfl_xor_sync(0xffffffffu, part, 2);
    if (blk == 0 && p < P) pool_scores[(int64_t)q * P + p] = ok ? part : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_quantize_mxfp4(const float* x, int64_t n_rows, int d, uint8_t* out,
                                  cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  const int64_t warps = n_rows * ((d + 127) / 128);
  int64_t blocks = (warps + 7) / 8;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  quantize_mxfp4_kernel<<<(unsigned)blocks, 256, 0, stream>>>(x, n_rows, d, out);
  return cudaGetLastError();
}

cudaError_t launch_index_scores_mxfp4(const uint8_t* q_mx, const uint8_t* k_mx, int B, int H_I,
                                      int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                      const int32_t* q_pos, int ratio, float* scores,
                                      int32_t* status, cudaStream_t stream) {
  if (B == 0 || N == 0) return cudaSuccess;
  const size_t smem = sizeof(ScanSmem);
  static bool attr_set = false;  // per process; the attribute is per kernel
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(mx_scores_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int S = (B + q_per_seq - 1) / q_per_seq;
  const int64_t total = (int64_t)S * ((N + kTileRows - 1) / kTileRows);
  int dev = 0, smem_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  int per_sm = smem_sm > 0 ? smem_sm / (int)(smem + 1024) : 1;
  per_sm = per_sm < 1 ? 1 : (per_sm > 3 ? 3 : per_sm);
  int64_t grid = (int64_t)per_sm * device_sm_count();
  if (grid > total) grid = total;
  return launch_kernel(mx_scores_kernel, dim3((unsigned)grid), dim3(kScanThreads), smem, stream,
                       false, q_mx, k_mx, B, H_I, N, kv_seq_stride, q_per_seq, q_pos, ratio,
                       scores, status);
}

cudaError_t launch_pool_scores_mxfp4(const uint8_t* q_mx, const uint8_t* k_mx, int B, int H_I,
                                     int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                     const int32_t* pool, int P, float* pool_scores,
                                     int32_t* status, cudaStream_t stream) {
  if (B == 0 || P == 0) return cudaSuccess;
  dim3 grid((unsigned)((P + kPoolSlots - 1) / kPoolSlots), (unsigned)B);
  return launch_kernel(mx_pool_scores_kernel, grid, dim3(kPoolThreads), 0, stream, false, q_mx,
                       k_mx, H_I, N, kv_seq_stride, q_per_seq, pool, P, pool_scores, status);
}

}  // namespace csa2
