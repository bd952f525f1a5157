// csa2_sparse_attn_fp4_noalloc: the sparse-attention entry point for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or own a workspace: code running while a
// stream is being captured into a CUDA graph (allocation is not a stream
// operation and would break the capture), plug-ins hosted by a runtime that
// owns every device allocation, and latency-critical serving loops that must
// never hit the allocator (cudaMalloc may synchronise the device).  This entry
// point runs exactly the same kernels as csa2_sparse_attn_fp4, but its split
// partials (the per-split log-sum-exp; the partial outputs themselves never
// leave shared memory) live in a fixed, file-scope device array instead of a
// caller workspace.  That array is kNoallocScratchBytes (256 KiB: a query's
// splits never outnumber the SMs, so 64 heads x 4 bytes per SM suffice for
// any GPU of up to 1024 SMs) and is held by every GPU that loads the library
// until the process exits.
#include <mutex>

#include "csa2_internal.cuh"

// Scratch for the split-k partial log-sum-exps.  In host code this name is only a
// host-side stand-in; kernels receive the device address obtained below.
static __device__ __align__(256) uint8_t g_csa2_attn_scratch[256u << 10];

namespace csa2 {
namespace {

constexpr size_t kNoallocScratchBytes = sizeof(g_csa2_attn_scratch);

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_csa2_attn_scratch on the current device, looked up once per
// device (under a lock) with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_csa2_attn_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" csa2_status csa2_sparse_attn_fp4_noalloc(const uint16_t* q_bf16, const uint8_t* kv_fp4,
                                                   int B, int H, int D, int64_t N,
                                                   int64_t kv_seq_stride, int q_per_seq,
                                                   const int32_t* idx, int k,
                                                   float softmax_scale, float* out, float* lse,
                                                   cudaStream_t stream) {
  if (B < 0 || N < 0 || N > INT32_MAX - 1 || q_per_seq < 1 || kv_seq_stride < 0 ||
      (kv_seq_stride > 0 && kv_seq_stride < N))
    return CSA2_ERR_INVALID_ARG;
  if (B > 0 && (!q_bf16 || !kv_fp4 || !out || !idx)) return CSA2_ERR_INVALID_ARG;
  if (D != kD) return CSA2_ERR_UNSUPPORTED;
  if (H != 16 && H != 32 && H != 64) return CSA2_ERR_UNSUPPORTED;
  if (k < 1) return CSA2_ERR_INVALID_ARG;
  if (k > 16384) return CSA2_ERR_UNSUPPORTED;
  if (!(softmax_scale > 0.0f) || !(softmax_scale < INFINITY)) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(q_bf16) || !aligned16(kv_fp4) || !aligned16(out)) return CSA2_ERR_INVALID_ARG;
  if (attn_scratch_bytes(B, H, k) > kNoallocScratchBytes) return CSA2_ERR_WORKSPACE;
  if (B == 0) return CSA2_OK;
  void* scratch = nullptr;
  csa2_status s = check_launch(scratch_address(&scratch));
  if (s != CSA2_OK) return s;
  // The partials are fully written before they are read, so nothing needs
  // clearing between calls.  No status word: indices outside [-1, N) are
  // skipped exactly as in csa2_sparse_attn_fp4, and a bounded device wait
  // that gives up ends its CTA early, but neither is reported.
  return check_launch(launch_sparse_attn(q_bf16, kv_fp4, B, H, N, kv_seq_stride, q_per_seq, idx,
                                         k, softmax_scale, out, lse, scratch, nullptr, stream));
}
