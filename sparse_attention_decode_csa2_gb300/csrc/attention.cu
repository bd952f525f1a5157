// Split-k bookkeeping of the sparse attention (DeepSeek-V4.1-Flash paper
// walkthrough, 1.(4) "CSA2": each query attends its selected entries).  The
// tensor-core kernel (attention_tc.cu) processes one query x one chunk of its
// selected slots per CTA; when a query's slots are split over several CTAs,
// each writes its normalised partial output and log-sum-exp, and
// attn_combine_kernel merges them: out = sum_s exp(lse_s - LSE) o_s with
// LSE = log sum_s exp(lse_s).
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

// Merge the per-chunk (o, lse) partials of each (query, head).
__global__ void __launch_bounds__(128)
attn_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse, int H,
                    int nsplit, float* __restrict__ out, float* __restrict__ lse) {
  pdl_trigger();  // the next layer's attention may start its query prologue
  pdl_wait();     // the partials come from the attention kernel before
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

size_t partial_bytes(int B, int H, int nsplit) {
  if (nsplit <= 1) return 0;
  return align_up((size_t)B * nsplit * H * kD * 4 + (size_t)B * nsplit * H * 4, 256);
}

cudaError_t launch_attn(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H, int64_t N,
                        int64_t kv_seq_stride, int q_per_seq, const int32_t* idx, int k,
                        float softmax_scale, float* out, float* lse, void* scratch,
                        int32_t* status, cudaStream_t stream, bool pdl, const SwaArgs* swa,
                        int32_t* idx_copy) {
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
                                        status, swa, idx_copy, stream, pdl);
  if (e != cudaSuccess || nsplit == 1) return e;
  return launch_kernel(attn_combine_kernel, dim3((unsigned)H, (unsigned)B), dim3(128), 0, stream,
                       true, part_o, part_lse, H, nsplit, out, lse);
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
