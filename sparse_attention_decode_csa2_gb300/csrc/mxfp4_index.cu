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
// HBM for 128 multiply-adds, a matrix-vector product bounded by HBM bandwidth.
// What limits it on the SM is decoding: one E2M1 pair -> f16x2 conversion
// per code byte is the only per-element instruction left; the multiply-adds
// run as warp-level m16n8k16 MMAs (f16 operands, fp32 accumulation) that
// take the decoded registers directly, 16 entries per MMA group, with the
// head sum in B split into two f16 parts (22 significant bits).
//  * full scan: a persistent grid (a multiple of the SM count) walks
//    contiguous runs of 128-entry tiles (8704 bytes); one producer warp
//    streams the tiles into a 4-stage shared-memory ring with 1D bulk
//    copies (cp.async.bulk, mbarrier completion), four consumer warps score
//    them, 32 entries each.
//  * pool scan (Reindex layers): the same per-group arithmetic on gathered
//    rows loaded straight from global memory.
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

// ---------------------------------------------------------------------------
// Dot products of 16 entries with one query on the warp's tensor cores.
//
// mma.sync m16n8k16 (f16 in, fp32 accumulate) with A = 16 entries x 16
// elements and B = 16 elements x 8 columns.  Lane (g, t) (g = lane / 4,
// t = lane % 4) supplies entries g and g + 8 of the group; of each entry it
// decodes code word 4b + t of every 32-element block b: 8 elements, i.e. the
// four A registers of two k16 steps.  The k order inside a step is therefore
// a permutation of the elements, and B follows the same permutation: in step
// (b, cc), k = 2t + {0,1} is element 32b + 8t + 4cc + {0,1} and k = 2t + 8 +
// {0,1} is element 32b + 8t + 4cc + 2 + {0,1}.
// Column n = 2b + p of B holds part p (p = 0: f16 rounding, p = 1: f16
// rounding of the remainder) of the query's head sum, scaled by 2^-e_b, on
// the rows of block b and zero elsewhere.  After the 8 steps lane (g, t)
// holds the block-t partials of entries g and g + 8 in accumulator columns
// 2t (part 0) and 2t + 1 (part 1); it scales them by the entry's E8M0 scale
// and 2^e_t and four lanes add them.  Products of two f16 values are exact in
// fp32.
// ---------------------------------------------------------------------------

// code word (8 E2M1 elements) -> 4 f16x2 registers (byte j -> register j,
// low nibble in the low half).  The byte unpack costs no instruction.
__device__ __forceinline__ void e2m1_word_to_f16x2(uint32_t w, uint32_t h[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ void mma_16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// wA[b], wB[b]: code word 4b + t of entries g and g + 8; bq[b]: the lane's B
// registers of steps (b, 0) and (b, 1).  The two steps of a block go to
// separate accumulators (two independent MMA chains), added at the end.
__device__ __forceinline__ void mx16_dot(const uint32_t wA[4], const uint32_t wB[4],
                                         const uint4 bq[4], float c[4]) {
  float d[4] = {0.f, 0.f, 0.f, 0.f};
  c[0] = c[1] = c[2] = c[3] = 0.0f;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    uint32_t hA[4], hB[4];
    e2m1_word_to_f16x2(wA[b], hA);
    e2m1_word_to_f16x2(wB[b], hB);
    mma_16816(c, hA[0], hB[0], hA[1], hB[1], bq[b].x, bq[b].y);
    mma_16816(d, hA[2], hB[2], hA[3], hB[3], bq[b].z, bq[b].w);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] += d[i];
}

// Two groups of 16 entries (32 entries) at once: four independent MMA chains.
__device__ __forceinline__ void mx32_dot(const uint32_t w[2][2][4], const uint4 bq[4],
                                         float c[2][4]) {
  float d[2][4];
#pragma unroll
  for (int x = 0; x < 2; ++x)
#pragma unroll
    for (int i = 0; i < 4; ++i) c[x][i] = d[x][i] = 0.0f;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      uint32_t hA[4], hB[4];
      e2m1_word_to_f16x2(w[x][0][b], hA);
      e2m1_word_to_f16x2(w[x][1][b], hB);
      mma_16816(c[x], hA[0], hB[0], hA[1], hB[1], bq[b].x, bq[b].y);
      mma_16816(d[x], hA[2], hB[2], hA[3], hB[3], bq[b].z, bq[b].w);
    }
  }
#pragma unroll
  for (int x = 0; x < 2; ++x)
#pragma unroll
    for (int i = 0; i < 4; ++i) c[x][i] += d[x][i];
}

// qsum[d] = sum_h value(q[h][d]) of one query from its H_I rows staged in
// shared memory, by compensated (Neumaier) fp32 summation of the exact
// decoded values.
__device__ __forceinline__ float mx_qsum_dim(const uint8_t* q, int H_I, int d) {
  float s = 0.0f, comp = 0.0f;
  for (int h = 0; h < H_I; ++h) {
    const uint8_t* row = q + h * kMxRow;
    const uint32_t byte = row[d / 2];
    const uint32_t code = (d & 1) ? (byte >> 4) : (byte & 15u);
    const float v =
        half2_bits_to_float2(e2m1x2_to_f16x2(code)).x * e8m0_to_float(row[kMxCodes + d / 32]);
    const float t = s + v;
    comp += (fabsf(s) >= fabsf(v)) ? ((s - t) + v) : ((v - t) + s);
    s = t;
  }
  return s + comp;
}

constexpr int kMaxHI = 64;

// The B registers of up to kQChunk queries, built by kThreads threads (a
// multiple of 32, >= 64): qsum of each dim, a power-of-two scale 2^e_b per
// 32-dim block putting the block's largest |qsum| in [2^14, 2^15), then the
// f16 parts.  frag[ql][b][lane] holds lane's registers of steps (b, 0),
// (b, 1); qscale[ql][b] = 2^e_b.  Each query's H_I rows are first copied to
// shared memory with independent loads (one memory latency, not H_I).
struct QFrag {
  __align__(16) uint8_t qraw[kMaxHI * kMxRow];
  float qs[kQChunk][kMxDI];
  uint4 frag[kQChunk][4][32];
  float qscale[kQChunk][4];
};

__device__ __forceinline__ uint32_t f16_part_pair(float x0, float x1, int p) {
  __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
  if (p) {
    h0 = __float2half_rn(x0 - __half2float(h0));
    h1 = __float2half_rn(x1 - __half2float(h1));
  }
  return (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
}

template <int kThreads, int kBarId>
__device__ __forceinline__ void build_qfrag(QFrag& f, const uint8_t* __restrict__ q_mx, int H_I,
                                            int q0, int nq) {
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int nbytes = H_I * kMxRow;
  for (int ql = 0; ql < nq; ++ql) {
    const uint8_t* src = q_mx + (int64_t)(q0 + ql) * nbytes;
    if ((reinterpret_cast<uintptr_t>(src) & 3u) == 0) {  // rows are 68 bytes: words
      constexpr int kPer = (kMaxHI * kMxRow / 4 + kThreads - 1) / kThreads;
      const uint32_t* s4 = reinterpret_cast<const uint32_t*>(src);
      uint32_t* d4 = reinterpret_cast<uint32_t*>(f.qraw);
      uint32_t v[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int o = tid + i * kThreads;
        v[i] = o < nbytes / 4 ? __ldg(s4 + o) : 0u;
      }
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int o = tid + i * kThreads;
        if (o < nbytes / 4) d4[o] = v[i];
      }
    } else {
      for (int o = tid; o < nbytes; o += kThreads) f.qraw[o] = __ldg(src + o);
    }
    asm volatile("bar.sync %0, %1;" ::"n"(kBarId), "n"(kThreads) : "memory");
    for (int d = tid; d < kMxDI; d += kThreads) {  // whole warps: a warp's dims form one block
      const float x = mx_qsum_dim(f.qraw, H_I, d);
      float a = fabsf(x);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      int e = 0;
      if (a > 0.0f) {
        int ex;
        frexpf(a, &ex);  // a = m 2^ex, m in [0.5, 1): floor(log2 a) = ex - 1
        e = ex - 1 - 14;
      }
      f.qs[ql][d] = ldexpf(x, -e);
      if (lane == 0) f.qscale[ql][d / 32] = ldexpf(1.0f, e);
    }
    asm volatile("bar.sync %0, %1;" ::"n"(kBarId), "n"(kThreads) : "memory");
  }
  asm volatile("bar.sync %0, %1;" ::"n"(kBarId), "n"(kThreads) : "memory");
  uint32_t* words = reinterpret_cast<uint32_t*>(&f.frag[0][0][0]);
  for (int i = tid; i < nq * 4 * 32 * 4; i += kThreads) {
    const int ql = i / 512, b = (i / 128) % 4, ln = (i / 4) % 32, w = i % 4;
    const int g = ln >> 2, t = ln & 3, cc = w >> 1, h = w & 1;
    uint32_t val = 0;
    if ((g >> 1) == b) {
      const int e = 32 * b + 8 * t + 4 * cc + 2 * h;
      val = f16_part_pair(f.qs[ql][e], f.qs[ql][e + 1], g & 1);
    }
    words[i] = val;
  }
  asm volatile("bar.sync %0, %1;" ::"n"(kBarId), "n"(kThreads) : "memory");
}

struct ScanSmem {
  uint8_t tiles[kStages][kTileBytes];
  QFrag qf;
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
// so it meets few sequence changes (each rebuilds the staged query registers).
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
    int s = (int)(t_begin / T);
    int64_t tt = t_begin - (int64_t)s * T;
    for (int64_t tile = t_begin; tile < t_end; ++tile, ++tt) {
      if (tt == T) {
        tt = 0;
        ++s;
      }
      const int64_t row0 = tt * kTileRows;
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

  // ---------------- consumers: warp w scores entries 32w .. 32w + 31 of a tile ----------------
  // Entries past the loaded rows of a ragged tile read stale (or never
  // written) shared memory: any byte is a valid pair of E2M1 codes, so the
  // products stay finite, and their scale is taken as 0.
  const int g = lane >> 2, t = lane & 3;
  int64_t n = 0;  // loads consumed
  int cur_s = -1, cur_chunk = -1, reg_q = -1;
  int64_t vis = 0;
  uint4 bq[4];
  float qs_t = 0.0f;
  int s = (int)(t_begin / T);
  int64_t tt = t_begin - (int64_t)s * T;
  for (int64_t tile = t_begin; tile < t_end; ++tile, ++tt) {
    if (tt == T) {
      tt = 0;
      ++s;
    }
    const int64_t row0 = tt * kTileRows;
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
    const uint32_t* tw = reinterpret_cast<const uint32_t*>(tileb);
    const int q_first = s * q_per_seq;
    const int q_last = min(B, q_first + q_per_seq);
    const int r0 = warp * 32 + g;  // entries r0, r0 + 8, r0 + 16, r0 + 24
    for (int qc = q_first; qc < q_last; qc += kQChunk) {
      const int nq = min(kQChunk, q_last - qc);
      if (qc != cur_chunk) {
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
        build_qfrag<kConsumers, 1>(sm.qf, q_mx, H_I, qc, nq);
        cur_chunk = qc;
        reg_q = -1;
      }
      for (int ql = 0; ql < nq; ++ql) {
        const int q = qc + ql;
        if (q != reg_q) {
#pragma unroll
          for (int b = 0; b < 4; ++b) bq[b] = sm.qf.frag[ql][b][lane];
          qs_t = sm.qf.qscale[ql][t];
          reg_q = q;
        }
        const int64_t nv = n_visible(q_pos, q, ratio, N);
        float* srow = scores + (int64_t)q * N + row0;
        float p[4] = {0.f, 0.f, 0.f, 0.f};  // entries r0 + 8 i
        if (rows > 0) {  // tile-uniform
          uint32_t w[2][2][4];
#pragma unroll
          for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int y = 0; y < 2; ++y)
#pragma unroll
              for (int b = 0; b < 4; ++b)
                w[x][y][b] = tw[(r0 + 16 * x + 8 * y) * (kMxRow / 4) + 4 * b + t];
          float c[2][4];
          mx32_dot(w, bq, c);
#pragma unroll
          for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int y = 0; y < 2; ++y) {
              const int r = r0 + 16 * x + 8 * y;
              const float ks = r < rows ? e8m0_to_float(tileb[r * kMxRow + kMxCodes + t]) : 0.0f;
              p[2 * x + y] = (c[x][2 * y] + c[x][2 * y + 1]) * (ks * qs_t);
            }
#pragma unroll
          for (int i = 0; i < 4; ++i) p[i] += __shfl_xor_sync(0xffffffffu, p[i], 1);
#pragma unroll
          for (int i = 0; i < 4; ++i) p[i] += __shfl_xor_sync(0xffffffffu, p[i], 2);
        }
        // lane t of the quad stores entry r0 + 8 t
        const float v = t == 0 ? p[0] : (t == 1 ? p[1] : (t == 2 ? p[2] : p[3]));
        const int r = r0 + 8 * t;
        if (r < rows_in_tile) srow[r] = (row0 + r < nv) ? v : -INFINITY;
      }
    }
    if (rows > 0) {
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::su32(&sm.empty[st]));
      ++n;
    }
  }
}

// Pool scan: CTA (x, q) scores pool slots [1024 x, 1024 x + 1024) of query q,
// each warp 16 gathered entries at a time.
constexpr int kPoolThreads = 256;
constexpr int kPoolSlots = 1024;

struct PoolSmem {
  QFrag qf;
};

__global__ void __launch_bounds__(kPoolThreads)
mx_pool_scores_kernel(const uint8_t* __restrict__ q_mx, const uint8_t* __restrict__ k_mx, int H_I,
                      int64_t N, int64_t kv_seq_stride, int q_per_seq,
                      const int32_t* __restrict__ pool, int P, float* __restrict__ pool_scores,
                      int32_t* status) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  PoolSmem& sm = *reinterpret_cast<PoolSmem*>(smem_raw);
  pdl_trigger();
  pdl_wait();
  const int q = blockIdx.y;
  build_qfrag<kPoolThreads, 1>(sm.qf, q_mx, H_I, q, 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  uint4 bq[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) bq[b] = sm.qf.frag[0][b][lane];
  const float qs_t = sm.qf.qscale[0][t];
  const uint8_t* kseq = k_mx + (int64_t)(q / q_per_seq) * kv_seq_stride * kMxRow;
  const int32_t* prow = pool + (int64_t)q * P;
  constexpr int kGroups = kPoolSlots / 16 / (kPoolThreads / 32);  // per warp
  for (int it = 0; it < kGroups; ++it) {
    const int p0 = blockIdx.x * kPoolSlots + (it * (kPoolThreads / 32) + warp) * 16;
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
    const uint32_t* rwA = reinterpret_cast<const uint32_t*>(kseq + (int64_t)(okA ? jA : 0) * kMxRow);
    const uint32_t* rwB = reinterpret_cast<const uint32_t*>(kseq + (int64_t)(okB ? jB : 0) * kMxRow);
    uint32_t wA[4], wB[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      wA[b] = okA ? __ldg(rwA + 4 * b + t) : 0u;
      wB[b] = okB ? __ldg(rwB + 4 * b + t) : 0u;
    }
    const uint32_t sA = okA ? __ldg(reinterpret_cast<const uint8_t*>(rwA) + kMxCodes + t) : 0u;
    const uint32_t sB = okB ? __ldg(reinterpret_cast<const uint8_t*>(rwB) + kMxCodes + t) : 0u;
    float c[4];
    mx16_dot(wA, wB, bq, c);
    float vA = (c[0] + c[1]) * (e8m0_to_float(sA) * qs_t);
    float vB = (c[2] + c[3]) * (e8m0_to_float(sB) * qs_t);
    vA += __shfl_xor_sync(0xffffffffu, vA, 1);
    vB += __shfl_xor_sync(0xffffffffu, vB, 1);
    vA += __shfl_xor_sync(0xffffffffu, vA, 2);
    vB += __shfl_xor_sync(0xffffffffu, vB, 2);
    if (t == 0 && pA < P) pool_scores[(int64_t)q * P + pA] = okA ? vA : -INFINITY;
    if (t == 1 && pB < P) pool_scores[(int64_t)q * P + pB] = okB ? vB : -INFINITY;
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
  // set on every call: the attribute belongs to the current device's context
  cudaError_t e = cudaFuncSetAttribute(mx_scores_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int S = (B + q_per_seq - 1) / q_per_seq;
  const int64_t total = (int64_t)S * ((N + kTileRows - 1) / kTileRows);
  int dev = 0, smem_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  int per_sm = smem_sm > 0 ? smem_sm / (int)(smem + 1024) : 1;
  per_sm = per_sm < 1 ? 1 : (per_sm > 4 ? 4 : per_sm);
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
  const size_t smem = sizeof(PoolSmem);
  // set on every call: the attribute belongs to the current device's context
  cudaError_t e = cudaFuncSetAttribute(mx_pool_scores_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((P + kPoolSlots - 1) / kPoolSlots), (unsigned)B);
  return launch_kernel(mx_pool_scores_kernel, grid, dim3(kPoolThreads), smem, stream, false, q_mx,
                       k_mx, H_I, N, kv_seq_stride, q_per_seq, pool, P, pool_scores, status);
}

}  // namespace csa2
