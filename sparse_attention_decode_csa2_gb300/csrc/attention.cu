// Split-k bookkeeping of the sparse attention (DeepSeek-V4.1-Flash paper
// walkthrough, 1.(4) "CSA2": each query attends its selected entries).  The
// tensor-core kernel (attention_tc.cu) processes one query x one chunk of its
// selected slots per CTA; when a query's slots are split over several CTAs
// (a thread-block cluster), each writes its partial log-sum-exp (fp32) to the
// workspace and hands its normalised partial output (fp16) to the cluster's
// other CTAs through shared memory; they merge in fp32:
// out = sum_s exp(lse_s - LSE) o_s with LSE = log sum_s exp(lse_s).
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kSplitTile = 128;  // entries per tile of the tensor-core kernel
constexpr int kMaxSplit = 8;     // a query's splits form one (portable-size) cluster

// Splits per query: about SMs / B, a power of two (the cluster's merge gives
// each split 8 / nsplit of the eight 64-channel blocks), at most 8, and
// chunks of whole tiles.
int choose_splits(int B, int k) {
  const int sms = device_sm_count();
  const int max_split = (k + kSplitTile - 1) / kSplitTile;
  int lim = sms / (B > 0 ? B : 1);
  if (lim > kMaxSplit) lim = kMaxSplit;
  if (lim > max_split) lim = max_split;
  int s = 1;
  while (2 * s <= lim) s *= 2;
  for (; s > 1; s /= 2) {
    const int chunk = ((k + s - 1) / s + kSplitTile - 1) / kSplitTile * kSplitTile;
    if ((k + chunk - 1) / chunk == s) return s;
  }
  return 1;
}

// fp32 partial lse [B][nsplit][H] (the partial outputs stay in shared memory)
size_t partial_bytes(int B, int H, int nsplit) {
  if (nsplit <= 1) return 0;
  return align_up((size_t)B * nsplit * H * 4, 256);
}

cudaError_t launch_attn(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H, int64_t N,
                        int64_t kv_seq_stride, int q_per_seq, const int32_t* idx, int k,
                        float softmax_scale, float* out, float* lse, void* scratch,
                        int32_t* status, cudaStream_t stream, bool pdl, const SwaArgs* swa,
                        int32_t* idx_copy) {
  const int nsplit = choose_splits(B, k);
  const int chunk = ((k + nsplit - 1) / nsplit + kSplitTile - 1) / kSplitTile * kSplitTile;
  float* part_lse = nsplit > 1 ? reinterpret_cast<float*>(scratch) : nullptr;
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  return launch_sparse_attn_tc(q_bf16, kv_fp4, B, H, N, kv_seq_stride, q_per_seq, idx, k, nsplit,
                               chunk, scale_log2, out, lse, part_lse, status, swa,
                               idx_copy, stream, pdl);
}

}  // namespace

int attn_launches(int B, int k) {
  if (B <= 0 || k <= 0) return 0;
  return 1;
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
