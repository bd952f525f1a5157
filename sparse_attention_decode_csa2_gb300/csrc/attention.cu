// Sparse MQA attention over the selected FP4 entries (DeepSeek-V4.1-Flash
// paper walkthrough, 1.(4) "CSA2": each query attends its selected main-KV
// entries; 1.(5).4: the FP4 cache is dequantised before attention; 2.(2).1:
// 64 query heads of 512 dims).  K = V = the dequantised 512-channel latent,
// shared by every head.
//
// Work split: one CTA per (query, chunk of its selected slots); chunks are
// merged by log-sum-exp in a second kernel when a query has several.
// Per 64-entry tile:
//   gather  : 288-byte FP4 rows copied global -> shared with cp.async (16 B
//             granules, zero-fill for -1 / out-of-range slots), double-buffered
//   dequant : E2M1 x E4M3 -> fp16 (exact: <= 6 significant bits, range
//             2^-10 .. 2688), written to a padded [64][512] tile
//   S = Q V^T  (fp16 tensor-core MMA, fp32 accumulate), masked, online softmax
//             in fp32 with exp2 on pre-scaled logits
//   O += P V   (P rounded to fp16, fp32 accumulate in registers)
// Q is converted bf16 -> fp16 once per CTA (values below 2^-14 lose bits as
// fp16 subnormals; the effect on a logit is below 2^-25 per element).
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;                 // entries per tile
constexpr int kRowH = kD + 8;             // padded fp16 row (1040 B): conflict-free ldmatrix
constexpr int kPRowH = kTile + 8;         // padded P row (144 B)
constexpr int kChunks16 = kRowBytes / 16; // 18 granules per FP4 row

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int H>
struct AttnSmem {
  static constexpr size_t q_off = 0;
  static constexpr size_t v_off = q_off + (size_t)H * kRowH * 2;
  static constexpr size_t raw_off = v_off + (size_t)kTile * kRowH * 2;
  static constexpr size_t p_off = raw_off + 2 * (size_t)kTile * kRowBytes;
  static constexpr size_t valid_off = p_off + (size_t)H * kPRowH * 2;
  static constexpr size_t red_off = valid_off + 2 * kTile * 4;
  static constexpr size_t bytes = red_off + 8 * (size_t)H * 4;
};

// Issue the cp.async copies of one tile's FP4 rows into raw[stage].
__device__ __forceinline__ void issue_tile(const uint8_t* __restrict__ kvseq, int64_t N,
                                           const int32_t* __restrict__ slots, int s_begin,
                                           int s_end, uint8_t* raw, int32_t* valid,
                                           int32_t* status) {
  for (int c = threadIdx.x; c < kTile * kChunks16; c += kThreads) {
    const int r = c / kChunks16, part = c - r * kChunks16;
    const int s = s_begin + r;
    int32_t j = (s < s_end) ? slots[s] : -1;
    const bool ok = (j >= 0) && (j < N);
    if (part == 0) {
      valid[r] = ok ? 1 : 0;
      if (j >= N || j < -1) set_status(status, kStatusBadIndex);
    }
    const uint8_t* src = ok ? kvseq + (int64_t)j * kRowBytes + part * 16 : kvseq;
    cp_async16(smem_u32(raw + r * kRowBytes + part * 16), src, ok);
  }
  cp_async_commit();
}

template <int H>
__global__ void __launch_bounds__(kThreads, 1)
sparse_attn_kernel(const uint16_t* __restrict__ q_bf16, const uint8_t* __restrict__ kv_fp4,
                   int64_t N, int64_t kv_seq_stride, int q_per_seq,
                   const int32_t* __restrict__ idx, int k, int chunk, float scale_log2,
                   float* __restrict__ out, float* __restrict__ lse, float* __restrict__ part_o,
                   float* __restrict__ part_lse, int32_t* status) {
  constexpr int HG = H / 16;        // head groups of 16 rows
  constexpr int WP = 8 / HG;        // warps sharing a head group
  constexpr int EW = kTile / WP;    // entries per warp in S
  constexpr int NT = EW / 8;        // n-tiles per warp in S
  constexpr int CW = kD / WP;       // channels per warp in O
  constexpr int CNT = CW / 8;       // n-tiles per warp in O
  using L = AttnSmem<H>;
  extern __shared__ __align__(128) uint8_t smem[];
  __half* Qs = reinterpret_cast<__half*>(smem + L::q_off);
  __half* Vs = reinterpret_cast<__half*>(smem + L::v_off);
  uint8_t* raw = smem + L::raw_off;
  __half* Ps = reinterpret_cast<__half*>(smem + L::p_off);
  int32_t* valid = reinterpret_cast<int32_t*>(smem + L::valid_off);
  float* red = reinterpret_cast<float*>(smem + L::red_off);  // [WP][H]

  const int b = blockIdx.y;
  const int split = blockIdx.x;
  const int nsplit = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hg = warp % HG, part = warp / HG;
  const int g = lane >> 2, t4 = lane & 3;

  const int s0 = split * chunk;
  const int s1 = min(k, s0 + chunk);
  const int ntiles = s1 > s0 ? (s1 - s0 + kTile - 1) / kTile : 0;
  const int32_t* slots = idx + (int64_t)b * k;
  const uint8_t* kvseq = kv_fp4 + (int64_t)(b / q_per_seq) * kv_seq_stride * kRowBytes;

  if (ntiles > 0) issue_tile(kvseq, N, slots, s0, s1, raw, valid, status);

  // Q: bf16 -> fp16, [H][512] padded rows
  {
    const uint4* qsrc = reinterpret_cast<const uint4*>(q_bf16 + (int64_t)b * H * kD);
    for (int c = tid; c < H * kD / 8; c += kThreads) {
      uint4 v = __ldg(qsrc + c);
      const int h = c / (kD / 8), col = (c % (kD / 8)) * 8;
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o[i] = pack_half2(bf16_bits_to_float((uint16_t)(w[i] & 0xFFFF)),
                          bf16_bits_to_float((uint16_t)(w[i] >> 16)));
      *reinterpret_cast<uint4*>(Qs + h * kRowH + col) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }

  float o_acc[CNT][4];
#pragma unroll
  for (int i = 0; i < CNT; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};  // rows g and g+8, raw (unscaled) units
  float l_run[2] = {0.f, 0.f};              // this thread's share of the row sums

  const uint32_t q_base = smem_u32(Qs);
  const uint32_t v_base = smem_u32(Vs);
  const uint32_t p_base = smem_u32(Ps);

  for (int t = 0; t < ntiles; ++t) {
    const int stage = t & 1;
    if (t + 1 < ntiles) {
      issue_tile(kvseq, N, slots, s0 + (t + 1) * kTile, s1, raw + (stage ^ 1) * kTile * kRowBytes,
                 valid + (stage ^ 1) * kTile, status);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    // dequantise raw[stage] -> Vs (fp16)
    {
      const uint8_t* rs = raw + stage * kTile * kRowBytes;
      for (int u = tid; u < kTile * (kD / 16); u += kThreads) {
        const int r = u / (kD / 16), blk = u % (kD / 16);
        const uint2 codes = *reinterpret_cast<const uint2*>(rs + r * kRowBytes + blk * 8);
        const uint32_t sb = rs[r * kRowBytes + kCodeBytes + blk];
        const uint32_t s2 = e4m3x2_to_f16x2((uint16_t)(sb | (sb << 8)));
        const __half2 sc = *reinterpret_cast<const __half2*>(&s2);
        uint32_t o[8];
        uint32_t cw[2] = {codes.x, codes.y};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t v2 = e2m1x2_to_f16x2((cw[i >> 2] >> (8 * (i & 3))) & 0xFF);
          __half2 h = __hmul2(*reinterpret_cast<__half2*>(&v2), sc);
          o[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        uint4* dst = reinterpret_cast<uint4*>(Vs + r * kRowH + blk * 16);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
    __syncthreads();

    // S = Q V^T for heads [16 hg, 16 hg + 16) x entries [EW part, EW part + EW)
    float s_acc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) s_acc[i][0] = s_acc[i][1] = s_acc[i][2] = s_acc[i][3] = 0.f;
    {
      const int arow = hg * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
      const int acol = 8 * (lane >> 4);
      const uint32_t a_addr = q_base + (arow * kRowH + acol) * 2;
#pragma unroll 4
      for (int kk = 0; kk < kD / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(a_addr + kk * 32, a0, a1, a2, a3);
        if constexpr (NT == 1) {
          const int brow = part * EW + (lane & 7);
          const int bcol = 8 * ((lane >> 3) & 1);
          uint32_t b0, b1;
          ldsm_x2(v_base + (brow * kRowH + bcol) * 2 + kk * 32, b0, b1);
          mma16816(s_acc[0], a0, a1, a2, a3, b0, b1);
        } else {
#pragma unroll
          for (int np = 0; np < NT / 2; ++np) {
            const int brow = part * EW + np * 16 + (lane & 7) + 8 * (lane >> 4);
            const int bcol = 8 * ((lane >> 3) & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(v_base + (brow * kRowH + bcol) * 2 + kk * 32, b0, b1, b2, b3);
            mma16816(s_acc[2 * np], a0, a1, a2, a3, b0, b1);
            mma16816(s_acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
          }
        }
      }
    }

    // mask, tile max per row
    const int32_t* vld = valid + stage * kTile;
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const int e = part * EW + i * 8 + 2 * t4;
      const bool v0 = vld[e] != 0, v1 = vld[e + 1] != 0;
      if (!v0) { s_acc[i][0] = -INFINITY; s_acc[i][2] = -INFINITY; }
      if (!v1) { s_acc[i][1] = -INFINITY; s_acc[i][3] = -INFINITY; }
      tmax[0] = fmaxf(tmax[0], fmaxf(s_acc[i][0], s_acc[i][1]));
      tmax[1] = fmaxf(tmax[1], fmaxf(s_acc[i][2], s_acc[i][3]));
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 1));
      tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 2));
    }
    if (WP > 1) {
      if (t4 == 0) {
        red[part * H + hg * 16 + g] = tmax[0];
        red[part * H + hg * 16 + g + 8] = tmax[1];
      }
      __syncthreads();
#pragma unroll
      for (int p = 0; p < WP; ++p) {
        tmax[0] = fmaxf(tmax[0], red[p * H + hg * 16 + g]);
        tmax[1] = fmaxf(tmax[1], red[p * H + hg * 16 + g + 8]);
      }
    }
    float alpha[2], mref[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float m_new = fmaxf(m_run[r], tmax[r]);
      if (m_new == -INFINITY) {
        alpha[r] = 1.f;
        mref[r] = 0.f;  // every logit so far is -inf: p = exp2(-inf) = 0
      } else {
        alpha[r] = exp2f((m_run[r] - m_new) * scale_log2);
        mref[r] = m_new * scale_log2;
      }
      m_run[r] = m_new;
      l_run[r] *= alpha[r];
    }
    // P = exp2(scale_log2 * s - scale_log2 * m), rounded to fp16 into Ps
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const int e = part * EW + i * 8 + 2 * t4;
      float p0 = exp2f(fmaf(s_acc[i][0], scale_log2, -mref[0]));
      float p1 = exp2f(fmaf(s_acc[i][1], scale_log2, -mref[0]));
      float p2 = exp2f(fmaf(s_acc[i][2], scale_log2, -mref[1]));
      float p3 = exp2f(fmaf(s_acc[i][3], scale_log2, -mref[1]));
      l_run[0] += p0 + p1;
      l_run[1] += p2 + p3;
      *reinterpret_cast<uint32_t*>(Ps + (hg * 16 + g) * kPRowH + e) = pack_half2(p0, p1);
      *reinterpret_cast<uint32_t*>(Ps + (hg * 16 + g + 8) * kPRowH + e) = pack_half2(p2, p3);
    }
#pragma unroll
    for (int i = 0; i < CNT; ++i) {
      o_acc[i][0] *= alpha[0];
      o_acc[i][1] *= alpha[0];
      o_acc[i][2] *= alpha[1];
      o_acc[i][3] *= alpha[1];
    }
    __syncthreads();

    // O += P V for heads [16 hg, +16) x channels [CW part, +CW)
    {
      const int arow = hg * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
      const int acol = 8 * (lane >> 4);
      const uint32_t a_addr = p_base + (arow * kPRowH + acol) * 2;
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(a_addr + kk * 32, a0, a1, a2, a3);
        const int vrow = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int vcol = part * CW + 8 * (lane >> 4);
        const uint32_t vb = v_base + (vrow * kRowH + vcol) * 2;
#pragma unroll
        for (int np = 0; np < CNT / 2; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + np * 32, b0, b1, b2, b3);
          mma16816(o_acc[2 * np], a0, a1, a2, a3, b0, b1);
          mma16816(o_acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();
  }

  // finish the row sums: quad, then across the warps of the head group
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
  }
  if (t4 == 0) {
    red[part * H + hg * 16 + g] = l_run[0];
    red[part * H + hg * 16 + g + 8] = l_run[1];
  }
  __syncthreads();
  float l_tot[2] = {0.f, 0.f};
#pragma unroll
  for (int p = 0; p < WP; ++p) {
    l_tot[0] += red[p * H + hg * 16 + g];
    l_tot[1] += red[p * H + hg * 16 + g + 8];
  }
  const float ln2 = 0.69314718055994530942f;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int h = hg * 16 + g + 8 * r;
    const bool empty = !(l_tot[r] > 0.f);
    const float inv = empty ? 0.f : 1.f / l_tot[r];
    const float lse_v = empty ? -INFINITY : (m_run[r] * scale_log2 + log2f(l_tot[r])) * ln2;
    float* orow;
    if (nsplit == 1) {
      orow = out + ((int64_t)b * H + h) * kD;
      if (lse && part == 0 && t4 == 0) lse[(int64_t)b * H + h] = lse_v;
    } else {
      orow = part_o + (((int64_t)b * nsplit + split) * H + h) * kD;
      if (part == 0 && t4 == 0) part_lse[((int64_t)b * nsplit + split) * H + h] = lse_v;
    }
#pragma unroll
    for (int i = 0; i < CNT; ++i) {
      const int c = part * CW + i * 8 + 2 * t4;
      *reinterpret_cast<float2*>(orow + c) =
          make_float2(o_acc[i][2 * r] * inv, o_acc[i][2 * r + 1] * inv);
    }
  }
}

// Merge the per-chunk (o, lse) partials of each (query, head).
__global__ void __launch_bounds__(128)
attn_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse, int H,
                    int nsplit, float* __restrict__ out, float* __restrict__ lse) {
  const int h = blockIdx.x, b = blockIdx.y;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part_lse[((int64_t)b * nsplit + s) * H + h]);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float L = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < nsplit; ++s) {
      const float ls = part_lse[((int64_t)b * nsplit + s) * H + h];
      const float w = expf(ls - M);
      L += w;
      const float4 v = *reinterpret_cast<const float4*>(
          part_o + (((int64_t)b * nsplit + s) * H + h) * kD + 4 * threadIdx.x);
      acc[0] = fmaf(w, v.x, acc[0]);
      acc[1] = fmaf(w, v.y, acc[1]);
      acc[2] = fmaf(w, v.z, acc[2]);
      acc[3] = fmaf(w, v.w, acc[3]);
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  *reinterpret_cast<float4*>(out + ((int64_t)b * H + h) * kD + 4 * threadIdx.x) =
      make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
  if (lse && threadIdx.x == 0) lse[(int64_t)b * H + h] = (L > 0.f) ? M + logf(L) : -INFINITY;
}

constexpr int kSplitTile = 128;  // entries per tile of the tensor-core kernel

int choose_splits(int B, int k) {
  const int sms = device_sm_count();
  int max_split = (k + kSplitTile - 1) / kSplitTile;
  int s = sms / (B > 0 ? B : 1);
  if (s < 1) s = 1;
  if (s > max_split) s = max_split;
  // round chunk to whole tiles, then recount
  int chunk = ((k + s - 1) / s + kSplitTile - 1) / kSplitTile * kSplitTile;
  return (k + chunk - 1) / chunk;
}

cudaError_t launch_attn(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H, int64_t N,
                        int64_t kv_seq_stride, int q_per_seq, const int32_t* idx, int k,
                        float softmax_scale, float* out, float* lse, void* scratch,
                        int32_t* status, cudaStream_t stream) {
  const int nsplit = choose_splits(B, k);
  const int chunk = ((k + nsplit - 1) / nsplit + kSplitTile - 1) / kSplitTile * kSplitTile;
  float* part_o = nullptr;
  float* part_lse = nullptr;
  if (nsplit > 1) {
    part_o = reinterpret_cast<float*>(scratch);
    part_lse = part_o + (size_t)B * nsplit * H * kD;
  }
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  cudaError_t e = launch_sparse_attn_tc(q_bf16, kv_fp4, B, H, N, kv_seq_stride, q_per_seq, idx, k,
                                        nsplit, chunk, scale_log2, out, lse, part_o, part_lse,
                                        status, stream);
  if (e != cudaSuccess || nsplit == 1) return e;
  attn_combine_kernel<<<dim3((unsigned)H, (unsigned)B), 128, 0, stream>>>(part_o, part_lse, H,
                                                                         nsplit, out, lse);
  return cudaGetLastError();
}

}  // namespace

int attn_launches(int B, int k) {
  if (B <= 0 || k <= 0) return 0;
  return choose_splits(B, k) > 1 ? 2 : 1;
}

size_t attn_scratch_bytes(int B, int H, int k) {
  if (B <= 0 || H <= 0 || k <= 0) return 0;
  const int nsplit = choose_splits(B, k);
  if (nsplit <= 1) return 0;
  return align_up((size_t)B * nsplit * H * kD * 4 + (size_t)B * nsplit * H * 4, 256);
}

cudaError_t launch_sparse_attn(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H,
                               int64_t N, int64_t kv_seq_stride, int q_per_seq, const int32_t* idx,
                               int k, float softmax_scale, float* out, float* lse, void* scratch,
                               int32_t* status, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  return launch_attn(q_bf16, kv_fp4, B, H, N, kv_seq_stride, q_per_seq, idx, k, softmax_scale, out,
                     lse, scratch, status, stream);
}

}  // namespace csa2
