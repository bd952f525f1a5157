// Split-k bookkeeping of the sparse attention (DeepSeek-V4.1-Flash paper
// walkthrough, 1.(4) "CSA2": each query attends its selected entries).  The
// tensor-core kernel (attention_tc.cu) processes one query x one chunk of its
// selected slots per CTA; when a query's slots are split over several CTAs,
// each writes its normalised partial output (fp16, [channel][head]) and
// log-sum-exp (fp32), and attn_combine_kernel merges them in fp32:
// out = sum_s exp(lse_s - LSE) o_s with LSE = log sum_s exp(lse_s).
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

// Merge the per-chunk (o, lse) partials.  CTA (g, b) covers channels
// 64 g .. 64 g + 63 of query b for every head: the fp16 partials are
// [split][channel][head], so thread (channel, 8 heads) reads 16 contiguous
// bytes per split; the weights exp(lse_s - M) / L per (split, head) are
// computed once in shared memory, and the result goes out through a
// shared-memory transpose as [head][channel] rows.
__global__ void __launch_bounds__(512)
attn_combine_kernel(const __half* __restrict__ part_o, const float* __restrict__ part_lse, int H,
                    int nsplit, float* __restrict__ out, float* __restrict__ lse) {
  extern __shared__ float msm[];  // weights [nsplit][64], then the [64][64] tile
  pdl_trigger();  // the next layer's attention may start its query prologue
  pdl_wait();     // the partials come from the attention kernel before
  float* wts = msm;
  float* tile = msm + 64 * nsplit;  // [head][64 channels + 1 pad]
  const int b = blockIdx.y, c0 = blockIdx.x * 64, t = threadIdx.x;
  const float* pl = part_lse + (int64_t)b * nsplit * H;
  if (t < H) {
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, pl[(int64_t)s * H + t]);
    float L = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float w = M == -INFINITY ? 0.f : expf(pl[(int64_t)s * H + t] - M);
      wts[s * 64 + t] = w;
      L += w;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int s = 0; s < nsplit; ++s) wts[s * 64 + t] *= inv;
    if (lse && blockIdx.x == 0) lse[(int64_t)b * H + t] = (L > 0.f) ? M + logf(L) : -INFINITY;
  }
  __syncthreads();
  const int ch = t >> 3, hg = (t & 7) * 8;  // channel c0 + ch, heads hg .. hg + 7
  if (hg < H) {
    const uint4* po = reinterpret_cast<const uint4*>(part_o + ((int64_t)b * nsplit * kD + c0 + ch) * H + hg);
    const int64_t step = (int64_t)kD * H / 8;  // 16-byte vectors between consecutive splits
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < nsplit; s0 += 8) {
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = s0 + i < nsplit ? po[(s0 + i) * step] : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (s0 + i >= nsplit) break;
        const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = half2_bits_to_float2(u[j]);
          acc[2 * j] = fmaf(wts[(s0 + i) * 64 + hg + 2 * j], f.x, acc[2 * j]);
          acc[2 * j + 1] = fmaf(wts[(s0 + i) * 64 + hg + 2 * j + 1], f.y, acc[2 * j + 1]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) tile[(hg + j) * 65 + ch] = acc[j];
  }
  __syncthreads();
  // rows: head h, channels c0 .. c0 + 63 (16 float4 per head)
  for (int f = t; f < H * 16; f += 512) {
    const int h = f >> 4, c4 = f & 15;
    const float* src = tile + h * 65 + 4 * c4;
    reinterpret_cast<float4*>(out + ((int64_t)b * H + h) * kD + c0)[c4] =
        make_float4(src[0], src[1], src[2], src[3]);
  }
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

// fp16 partial outputs, then fp32 partial lse
size_t partial_bytes(int B, int H, int nsplit) {
  if (nsplit <= 1) return 0;
  return align_up((size_t)B * nsplit * H * kD * 2, 256) + align_up((size_t)B * nsplit * H * 4, 256);
}

cudaError_t launch_attn(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H, int64_t N,
                        int64_t kv_seq_stride, int q_per_seq, const int32_t* idx, int k,
                        float softmax_scale, float* out, float* lse, void* scratch,
                        int32_t* status, cudaStream_t stream, bool pdl, const SwaArgs* swa,
                        int32_t* idx_copy) {
  const int nsplit = choose_splits(B, k);
  const int chunk = ((k + nsplit - 1) / nsplit + kSplitTile - 1) / kSplitTile * kSplitTile;
  __half* part_o = nullptr;
  float* part_lse = nullptr;
  if (nsplit > 1) {
    part_o = reinterpret_cast<__half*>(scratch);
    part_lse = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(scratch) +
                                        align_up((size_t)B * nsplit * H * kD * 2, 256));
  }
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  cudaError_t e = launch_sparse_attn_tc(q_bf16, kv_fp4, B, H, N, kv_seq_stride, q_per_seq, idx, k,
                                        nsplit, chunk, scale_log2, out, lse, part_o, part_lse,
                                        status, swa, idx_copy, stream, pdl);
  if (e != cudaSuccess || nsplit == 1) return e;
  const size_t smem = (size_t)(64 * nsplit + 64 * 65) * sizeof(float);
  if (smem > 48 * 1024 &&
      (e = cudaFuncSetAttribute(attn_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem)) != cudaSuccess)
    return e;
  return launch_kernel(attn_combine_kernel, dim3((unsigned)(kD / 64), (unsigned)B), dim3(512), smem,
                       stream, true, part_o, part_lse, H, nsplit, out, lse);
}

}  // namespace

int attn_launches(int B, int k) {
  if (B <= 0 || k <= 0) return 0;
  return choose_splits(B, k) > 1 ? 2 : 1;
}

size_t attn_scratch_bytes(int B, int H, int k) {
  if (B <= 0 || H <= 0 || k <= 0) return 0;
  return partial_bytes(B, H, choose_splits(B, k));
}

cudaError_t launch_sparse_attn(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H,
                               int64_t N, int64_t kv_seq_stride, int q_per_seq, const int32_t* idx,
                               int k, float softmax_scale, float* out, float* lse, void* scratch,
                               int32_t* status, cudaStream_t stream, bool pdl, const SwaArgs* swa,
                               int32_t* idx_copy) {
  if (B == 0) return cudaSuccess;
  return launch_attn(q_bf16, kv_fp4, B, H, N, kv_seq_stride, q_per_seq, idx, k, softmax_scale, out,
                     lse, scratch, status, stream, pdl, swa, idx_copy);
}

}  // namespace csa2
