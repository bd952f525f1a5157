// Internal declarations shared by the CUDA translation units of libcsa2.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "csa2.h"

namespace csa2 {

// Device status bits (first word of the workspace).
constexpr int32_t kStatusBadIndex = 1;
constexpr int32_t kStatusTimeout = 2;
constexpr size_t kStatusBytes = 256;

constexpr int kD = 512;                      // latent channels
constexpr int kRowBytes = kD / 2 + kD / 16;  // 288 bytes per FP4 row
constexpr int kCodeBytes = kD / 2;           // 256

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

// Two E4M3 bytes (low byte = element 0) -> two fp16 values (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

// One byte holding two E2M1 codes (low nibble = element 0) -> two fp16 values (exact).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(r)
      : "r"(byte));
  return r;
}

// fp32 -> E4M3 byte, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint32_t f32_to_e4m3_satfinite(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;  // low byte holds the second source operand
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t h2) {
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Order-preserving map of a (non-NaN) float to uint32; -0 maps like +0.
__device__ __forceinline__ uint32_t float_to_ordered(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Number of entries visible to a query at token position pos:
// entry j is visible iff ratio*j + ratio - 1 <= pos, i.e. j < (pos+1)/ratio.
__device__ __forceinline__ int64_t n_visible(const int32_t* q_pos, int q, int ratio, int64_t N) {
  if (q_pos == nullptr) return N;
  int64_t pos = q_pos[q];
  if (pos < 0) return 0;
  int64_t n = (pos + 1) / ratio;
  return n < N ? n : N;
}

__device__ __forceinline__ void set_status(int32_t* status, int32_t bits) {
  if (status) atomicOr(status, bits);
}

// Programmatic dependent launch.  A kernel launched with `pdl` set may begin
// while the previous kernel of its stream is still running: it calls
// pdl_wait() before it reads anything that kernel writes (without the launch
// attribute the wait returns at once).  Kernels call pdl_trigger() as they
// start, so that the next kernel's CTAs may be scheduled onto SMs they leave
// free and run their independent set-up early.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Kernel launch with an optional programmatic-dependent-launch attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// Launchers (each returns cudaGetLastError() of its launch)
// ---------------------------------------------------------------------------

cudaError_t launch_quantize_kv_fp4(const float* x, int64_t n_rows, uint8_t* out,
                                   cudaStream_t stream);

cudaError_t launch_index_scores(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I,
                                int D_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                const int32_t* q_pos, int ratio, float* scores, int32_t* status,
                                cudaStream_t stream);

// Tensor-core indexer (TMA + tcgen05 kind::f8f6f4); cudaErrorNotSupported for
// shapes it does not cover.
cudaError_t launch_index_scores_tc(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I,
                                   int D_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                   const int32_t* q_pos, int ratio, float* scores,
                                   int32_t* status, cudaStream_t stream);

// Scores pool entries: pool_scores[b][p] for valid pool[b][p], -inf for -1 padding.
// Flags a pool that is not strictly ascending with -1 only at the tail.
cudaError_t launch_pool_scores(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I,
                               int D_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                               const int32_t* pool, int P, float* pool_scores, int32_t* status,
                               cudaStream_t stream);

// MXFP4 indexer (rows of D_I = 128: 64 code bytes + 4 E8M0 scale bytes).
cudaError_t launch_quantize_mxfp4(const float* x, int64_t n_rows, int d, uint8_t* out,
                                  cudaStream_t stream);
cudaError_t launch_index_scores_mxfp4(const uint8_t* q_mx, const uint8_t* k_mx, int B, int H_I,
                                      int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                      const int32_t* q_pos, int ratio, float* scores,
                                      int32_t* status, cudaStream_t stream);
cudaError_t launch_pool_scores_mxfp4(const uint8_t* q_mx, const uint8_t* k_mx, int B, int H_I,
                                     int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                     const int32_t* pool, int P, float* pool_scores,
                                     int32_t* status, cudaStream_t stream);

// Where a top-k's selected entries are read next: their FP4 rows (row j of
// query b at kv + (b / q_per_seq) * seq_bytes + j * kRowBytes, j < n; kv
// 16-byte aligned), which the top-k requests into L2 as it writes the
// indices.  kv == nullptr: no requests.
struct RowPrefetch {
  const uint8_t* kv = nullptr;
  int64_t seq_bytes = 0;
  int64_t n = 0;
  int q_per_seq = 1;
};

// Top-k over rows of `scores` [B][N].  The number of candidates of row b is
// n_visible(q_pos, b, ratio, N) when n_valid is null, else n_valid[b].  When
// `map` is non-null the selected position p is written as map[b*N + p].
// pdl: launched as a programmatic dependent of the kernel before it.
// Rows longer than 32768 entries are selected in three launches when
// `scratch` holds topk_scratch_bytes(B, N, k) bytes, else by one slower
// kernel.  `pf`: the rows to request into L2 (none by default).
cudaError_t launch_topk(const float* scores, int B, int64_t N, int k, const int32_t* q_pos,
                        int ratio, const int32_t* n_valid, const int32_t* map, int32_t* idx,
                        cudaStream_t stream, bool pdl = false, void* scratch = nullptr,
                        size_t scratch_bytes = 0, const RowPrefetch& pf = RowPrefetch{});
size_t topk_scratch_bytes(int B, int64_t N, int k);
int topk_launches(int B, int64_t N, int k, size_t scratch_bytes);

// Blockwise candidate pool of the Hierarchical Sparse Indexer: scores [B][N]
// -> pool [B][n_blocks * block] (ascending entries of the kept blocks, -1
// padded).  scratch: block_pool_scratch(...).bytes bytes.
struct BlockPoolScratch {
  float* bscores;    // [B][ceil(N / block)]
  int32_t* n_valid;  // [B] blocks holding a visible entry
  int32_t* blk;      // [B][n_blocks] kept blocks
  size_t bytes;
};
BlockPoolScratch block_pool_scratch(void* base, int B, int64_t N, int block, int n_blocks);
size_t block_pool_scratch_bytes(int B, int64_t N, int block, int n_blocks);
cudaError_t launch_block_pool(const float* scores, int B, int64_t N, const int32_t* q_pos,
                              int ratio, int block, int n_blocks, int32_t* pool, void* scratch,
                              cudaStream_t stream, bool pdl);

// The sliding window of a layer's SWA KV that a call also attends.
struct SwaArgs {
  const uint8_t* kv;     // E4M3 [S][ring][512]
  int64_t ring;
  int n_win;
  const int32_t* q_pos;  // [B] query token positions
};

// Sparse attention (+ the SWA window when swa is non-null).  scratch:
// attn_scratch_bytes(B, H, k) bytes (split-k partials).  idx_copy non-null:
// the kernel also writes the slots it reads to idx_copy [B][k].  Before
// waiting on the previous kernel (programmatic dependent launch) the kernel
// reads only q_bf16, so every launch of it may be a dependent one.
size_t attn_scratch_bytes(int B, int H, int k);
int attn_launches(int B, int k);  // kernels one call launches
cudaError_t launch_sparse_attn(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H,
                               int64_t N, int64_t kv_seq_stride, int q_per_seq, const int32_t* idx,
                               int k, float softmax_scale, float* out, float* lse, void* scratch,
                               int32_t* status, cudaStream_t stream, bool pdl = false,
                               const SwaArgs* swa = nullptr, int32_t* idx_copy = nullptr);

// tcgen05 kernel of one sparse-attention call.  With nsplit > 1 (a power of
// two, at most 8) a query's nsplit CTAs form one thread-block cluster that
// writes partial lse part_lse [B][nsplit][H], exchanges its fp16 partial
// outputs through shared memory and merges them into `out` / `lse`.
cudaError_t launch_sparse_attn_tc(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H,
                                  int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                  const int32_t* idx, int k, int nsplit, int chunk,
                                  float scale_log2, float* out, float* lse, float* part_lse,
                                  int32_t* status, const SwaArgs* swa, int32_t* idx_copy,
                                  cudaStream_t stream, bool pdl);

// csa2_upload: the copy of the packed buffer and the kernel that places its
// segments (work_units: 16-byte units and rows of all segments, for sizing).
cudaError_t launch_upload(const void* host_packed, size_t bytes, int n_segs, void* dev_stage,
                          int64_t work_units, cudaStream_t stream);

int device_sm_count();

// CSA2_OK for cudaSuccess; otherwise keeps cudaGetErrorString(e) for
// csa2_last_cuda_error() (per host thread) and returns CSA2_ERR_CUDA.
csa2_status check_launch(cudaError_t e);

}  // namespace csa2
