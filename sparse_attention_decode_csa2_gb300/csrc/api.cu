// C ABI of libcsa2.so: argument validation, workspace layout and the
// Full / Reindex / Reuse layer schedule (DeepSeek-V4.1-Flash paper
// walkthrough, 1.(4).1 "Cross-Layer KV and Index Reuse" and 1.(4).2
// "Hierarchical Sparse Indexer").  Every compute step runs in the kernels of
// the other translation units; this file only checks arguments, carves the
// caller's workspace and enqueues launches.
#include <stdio.h>

#include "csa2_internal.cuh"

namespace csa2 {

int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return sms > 0 ? sms : 148;
}

thread_local const char* g_last_cuda_error = "no error";

csa2_status check_launch(cudaError_t e) {
  if (e == cudaSuccess) return CSA2_OK;
  g_last_cuda_error = cudaGetErrorString(e);
  return CSA2_ERR_CUDA;
}

namespace {

struct WsLayout {
  size_t status = 0;       // 256 B
  size_t scores = 0;       // [B][N] fp32
  size_t pool_scores = 0;  // [B][P] fp32
  size_t attn = 0;         // attention partials
  size_t bpool = 0;        // blockwise-pool scratch (blocks of 2 or more entries)
  size_t topk = 0;         // chunked selection of rows longer than 32768 entries
  size_t topk_bytes = 0;
  size_t total = 0;
};

WsLayout layout(int B, int64_t N, int k, int H, int P) {
  WsLayout w;
  size_t off = kStatusBytes;
  w.scores = off;
  off += align_up((size_t)(B > 0 ? B : 0) * (size_t)(N > 0 ? N : 0) * 4, 256);
  w.pool_scores = off;
  off += align_up((size_t)(B > 0 ? B : 0) * (size_t)(P > 0 ? P : 0) * 4, 256);
  w.attn = off;
  off += attn_scratch_bytes(B, H, k);
  w.bpool = off;
  if (P > 0) off += block_pool_scratch_bytes(B, N, 2, P / 2 > 0 ? P / 2 : 1);
  w.topk = off;
  w.topk_bytes = topk_scratch_bytes(B, N, k);
  if (P > 0 && topk_scratch_bytes(B, N, P) > w.topk_bytes) w.topk_bytes = topk_scratch_bytes(B, N, P);
  off += w.topk_bytes;
  w.total = off;
  return w;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

csa2_status check_seq(int B, int64_t N, int64_t kv_seq_stride, int q_per_seq) {
  if (B < 0 || N < 0 || N > INT32_MAX - 1) return CSA2_ERR_INVALID_ARG;
  if (q_per_seq < 1 || kv_seq_stride < 0) return CSA2_ERR_INVALID_ARG;
  if (kv_seq_stride > 0 && kv_seq_stride < N) return CSA2_ERR_INVALID_ARG;
  return CSA2_OK;
}

csa2_status check_indexer(const uint8_t* q, const uint8_t* k, int B, int H_I, int D_I, int ratio) {
  if (B > 0 && (!q || !k)) return CSA2_ERR_INVALID_ARG;
  if (ratio < 1 || H_I < 1) return CSA2_ERR_INVALID_ARG;
  if (D_I != 32 && D_I != 64 && D_I != 128) return CSA2_ERR_UNSUPPORTED;
  if (H_I > 32) return CSA2_ERR_UNSUPPORTED;
  if (!aligned16(k)) return CSA2_ERR_INVALID_ARG;
  return CSA2_OK;
}

// The full E4M3 scan reads indexer K through 2D tensor-map coordinates, which
// are 32-bit: every row it may touch, (sequences - 1) * kv_seq_stride + N of
// them, must have an index below 2^31.
csa2_status check_scan_rows(int B, int64_t N, int64_t kv_seq_stride, int q_per_seq) {
  if (B <= 0) return CSA2_OK;
  const int64_t S = ((int64_t)B + q_per_seq - 1) / q_per_seq;
  const int64_t rows = (S - 1) * kv_seq_stride + N;
  return rows > (int64_t)INT32_MAX ? CSA2_ERR_UNSUPPORTED : CSA2_OK;
}

// MXFP4 indexer rows (68 bytes at D_I = 128): a sequence's rows must start
// on a 16-byte boundary for the bulk copies of the full scan.
csa2_status check_indexer_mx(const uint8_t* q, const uint8_t* k, int B, int H_I, int D_I,
                             int ratio, int64_t kv_seq_stride, int q_per_seq) {
  if (B > 0 && (!q || !k)) return CSA2_ERR_INVALID_ARG;
  if (ratio < 1 || H_I < 1) return CSA2_ERR_INVALID_ARG;
  if (D_I != 128 || H_I > 64) return CSA2_ERR_UNSUPPORTED;  // the kernels stage <= 64 rows
  if (!aligned16(k)) return CSA2_ERR_INVALID_ARG;
  if (B > q_per_seq && kv_seq_stride % 4 != 0) return CSA2_ERR_UNSUPPORTED;
  return CSA2_OK;
}

csa2_status check_indexer_fmt(int fmt, const uint8_t* q, const uint8_t* k, int B, int H_I,
                              int D_I, int ratio, int64_t kv_seq_stride, int q_per_seq) {
  if (fmt == CSA2_INDEXER_E4M3) return check_indexer(q, k, B, H_I, D_I, ratio);
  if (fmt == CSA2_INDEXER_MXFP4)
    return check_indexer_mx(q, k, B, H_I, D_I, ratio, kv_seq_stride, q_per_seq);
  return CSA2_ERR_INVALID_ARG;
}

csa2_status check_attn(const uint16_t* q, const uint8_t* kv, int B, int H, int D, int k,
                       float scale, const float* out) {
  if (B > 0 && (!q || !kv || !out)) return CSA2_ERR_INVALID_ARG;
  if (D != kD) return CSA2_ERR_UNSUPPORTED;
  if (H != 16 && H != 32 && H != 64) return CSA2_ERR_UNSUPPORTED;
  if (k < 1) return CSA2_ERR_INVALID_ARG;
  if (k > 16384) return CSA2_ERR_UNSUPPORTED;
  if (!(scale > 0.0f) || !(scale < INFINITY)) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || ((uintptr_t)out & 15u)) return CSA2_ERR_INVALID_ARG;
  return CSA2_OK;
}

int32_t* status_ptr(void* ws) { return reinterpret_cast<int32_t*>(ws); }

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" {

const char* csa2_status_string(csa2_status s) {
  switch (s) {
    case CSA2_OK: return "CSA2_OK";
    case CSA2_ERR_INVALID_ARG: return "CSA2_ERR_INVALID_ARG";
    case CSA2_ERR_UNSUPPORTED: return "CSA2_ERR_UNSUPPORTED";
    case CSA2_ERR_WORKSPACE: return "CSA2_ERR_WORKSPACE";
    case CSA2_ERR_CUDA: return "CSA2_ERR_CUDA";
    case CSA2_ERR_BAD_INDEX: return "CSA2_ERR_BAD_INDEX";
    case CSA2_ERR_TIMEOUT: return "CSA2_ERR_TIMEOUT";
  }
  return "CSA2_ERR_UNKNOWN";
}

int csa2_version(void) { return 100; }

const char* csa2_last_cuda_error(void) { return g_last_cuda_error; }

size_t csa2_workspace_size(int B, int64_t N, int k, int H, int P) {
  return layout(B, N, k, H, P).total;
}

csa2_status csa2_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!ws || ws_bytes < kStatusBytes) return CSA2_ERR_WORKSPACE;
  return check_launch(cudaMemsetAsync(ws, 0, kStatusBytes, stream));
}

csa2_status csa2_read_status(void* ws, cudaStream_t stream, int32_t* device_bits) {
  if (!ws) return CSA2_ERR_WORKSPACE;
  int32_t bits = 0;
  csa2_status s = check_launch(cudaMemcpyAsync(&bits, ws, 4, cudaMemcpyDeviceToHost, stream));
  if (s == CSA2_OK) s = check_launch(cudaMemsetAsync(ws, 0, 4, stream));
  if (s == CSA2_OK) s = check_launch(cudaStreamSynchronize(stream));
  if (s != CSA2_OK) return s;
  if (device_bits) *device_bits = bits;
  if (bits & kStatusBadIndex) return CSA2_ERR_BAD_INDEX;
  if (bits & kStatusTimeout) return CSA2_ERR_TIMEOUT;
  return CSA2_OK;
}

csa2_status csa2_quantize_kv_fp4(const float* x, int64_t n_rows, int d, uint8_t* out,
                                 cudaStream_t stream) {
  if (n_rows < 0) return CSA2_ERR_INVALID_ARG;
  if (n_rows > 0 && (!x || !out)) return CSA2_ERR_INVALID_ARG;
  if (d != kD) return CSA2_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(out)) return CSA2_ERR_INVALID_ARG;
  return check_launch(launch_quantize_kv_fp4(x, n_rows, out, stream));
}

csa2_status csa2_upload(const void* host_packed, size_t bytes, int n_segs, void* dev_stage,
                        size_t stage_bytes, cudaStream_t stream) {
  static_assert(sizeof(csa2_upload_seg) == 48, "upload table entry");
  if (n_segs < 0 || !host_packed || !dev_stage || !aligned16(dev_stage)) return CSA2_ERR_INVALID_ARG;
  const size_t table = (size_t)n_segs * sizeof(csa2_upload_seg);
  if (bytes < table || stage_bytes < bytes) return CSA2_ERR_INVALID_ARG;
  const csa2_upload_seg* segs = reinterpret_cast<const csa2_upload_seg*>(host_packed);
  int64_t work = 0;
  for (int i = 0; i < n_segs; ++i) {
    const csa2_upload_seg& g = segs[i];
    if (g.reserved != 0 || (g.src_off & 15u) != 0 || g.src_off < table) return CSA2_ERR_INVALID_ARG;
    if (g.rows == 0) continue;
    if (g.dst == 0 || g.row_bytes == 0 || g.row_bytes > bytes || g.rows > bytes / g.row_bytes)
      return CSA2_ERR_INVALID_ARG;
    const uint64_t payload = g.rows * g.row_bytes;
    if (g.src_off > bytes || payload > bytes - g.src_off) return CSA2_ERR_INVALID_ARG;
    if (g.kind == CSA2_UPLOAD_KV_FP4) {
      if (g.row_bytes != (uint64_t)kD * 4 || ((g.dst | g.dst_stride) & 15u) != 0 ||
          (g.rows > 1 && g.dst_stride < (uint64_t)kRowBytes))
        return CSA2_ERR_INVALID_ARG;
      work += (int64_t)g.rows * 32;
    } else if (g.kind == CSA2_UPLOAD_RAW) {
      if (g.rows > 1 && g.dst_stride < g.row_bytes) return CSA2_ERR_INVALID_ARG;
      work += (int64_t)((payload + 15) / 16);
    } else {
      return CSA2_ERR_INVALID_ARG;
    }
  }
  return check_launch(launch_upload(host_packed, bytes, n_segs, dev_stage, work, stream));
}

csa2_status csa2_index_scores(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I, int D_I,
                              int64_t N, int64_t kv_seq_stride, int q_per_seq,
                              const int32_t* q_pos, int ratio, float* scores,
                              cudaStream_t stream) {
  csa2_status s = check_seq(B, N, kv_seq_stride, q_per_seq);
  if (s != CSA2_OK) return s;
  if ((s = check_indexer(q_fp8, k_fp8, B, H_I, D_I, ratio)) != CSA2_OK) return s;
  if ((s = check_scan_rows(B, N, kv_seq_stride, q_per_seq)) != CSA2_OK) return s;
  if (B > 0 && N > 0 && !scores) return CSA2_ERR_INVALID_ARG;
  return check_launch(launch_index_scores(q_fp8, k_fp8, B, H_I, D_I, N, kv_seq_stride, q_per_seq,
                                          q_pos, ratio, scores, nullptr, stream));
}

csa2_status csa2_quantize_mxfp4(const float* x, int64_t n_rows, int d, uint8_t* out,
                               cudaStream_t stream) {
  if (n_rows < 0 || d < 32 || d % 32 != 0 || d > 4096) return CSA2_ERR_INVALID_ARG;
  if (n_rows > 0 && (!x || !out)) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(x)) return CSA2_ERR_INVALID_ARG;
  return check_launch(launch_quantize_mxfp4(x, n_rows, d, out, stream));
}

csa2_status csa2_index_scores_mxfp4(const uint8_t* q_mx, const uint8_t* k_mx, int B, int H_I,
                                    int D_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                    const int32_t* q_pos, int ratio, float* scores,
                                    cudaStream_t stream) {
  csa2_status s = check_seq(B, N, kv_seq_stride, q_per_seq);
  if (s != CSA2_OK) return s;
  if ((s = check_indexer_mx(q_mx, k_mx, B, H_I, D_I, ratio, kv_seq_stride, q_per_seq)) != CSA2_OK)
    return s;
  if (B > 0 && N > 0 && !scores) return CSA2_ERR_INVALID_ARG;
  return check_launch(launch_index_scores_mxfp4(q_mx, k_mx, B, H_I, N, kv_seq_stride, q_per_seq,
                                                q_pos, ratio, scores, nullptr, stream));
}

csa2_status csa2_topk(const float* scores, int B, int64_t N, int k, const int32_t* q_pos,
                      int ratio, int32_t* idx, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (B < 0 || N < 0 || N > INT32_MAX - 1 || k < 1 || ratio < 1) return CSA2_ERR_INVALID_ARG;
  if (B > 0 && (!idx || (N > 0 && !scores))) return CSA2_ERR_INVALID_ARG;
  if (!ws || ws_bytes < kStatusBytes) return CSA2_ERR_WORKSPACE;
  // a workspace of csa2_workspace_size(B, N, k, 0, 0) bytes enables the
  // chunked selection of long rows; a smaller one falls back to one kernel
  const WsLayout w = layout(B, N, k, 0, 0);
  uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
  const bool room = ws_bytes >= w.total;
  return check_launch(launch_topk(scores, B, N, k, q_pos, ratio, nullptr, nullptr, idx, stream,
                                  false, room ? wsb + w.topk : nullptr, room ? w.topk_bytes : 0));
}

size_t csa2_block_pool_workspace_size(int B, int64_t N, int block, int n_blocks) {
  return block_pool_scratch_bytes(B, N, block, n_blocks);
}

csa2_status csa2_block_pool(const float* scores, int B, int64_t N, const int32_t* q_pos,
                            int ratio, int block, int n_blocks, int32_t* pool, void* ws,
                            size_t ws_bytes, cudaStream_t stream) {
  if (B < 0 || N < 0 || N > INT32_MAX - 1 || ratio < 1 || block < 1 || n_blocks < 1)
    return CSA2_ERR_INVALID_ARG;
  if ((int64_t)n_blocks * block > INT32_MAX) return CSA2_ERR_INVALID_ARG;
  if (B > 0 && (!pool || (N > 0 && !scores))) return CSA2_ERR_INVALID_ARG;
  if (B == 0) return CSA2_OK;
  if (!ws || ws_bytes < block_pool_scratch_bytes(B, N, block, n_blocks)) return CSA2_ERR_WORKSPACE;
  return check_launch(
      launch_block_pool(scores, B, N, q_pos, ratio, block, n_blocks, pool, ws, stream, false));
}

csa2_status csa2_hier_pool_index(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I,
                                 int D_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                 const int32_t* pool, int P, int k, int32_t* idx, void* ws,
                                 size_t ws_bytes, cudaStream_t stream) {
  csa2_status s = check_seq(B, N, kv_seq_stride, q_per_seq);
  if (s != CSA2_OK) return s;
  if ((s = check_indexer(q_fp8, k_fp8, B, H_I, D_I, 1)) != CSA2_OK) return s;
  if (P < 1 || k < 1) return CSA2_ERR_INVALID_ARG;
  if (B > 0 && (!pool || !idx)) return CSA2_ERR_INVALID_ARG;
  WsLayout w = layout(B, 0, 0, 0, P);
  if (!ws || ws_bytes < w.total) return CSA2_ERR_WORKSPACE;
  uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
  float* pscores = reinterpret_cast<float*>(wsb + w.pool_scores);
  cudaError_t e = launch_pool_scores(q_fp8, k_fp8, B, H_I, D_I, N, kv_seq_stride, q_per_seq, pool,
                                     P, pscores, status_ptr(ws), stream);
  if (e != cudaSuccess) return check_launch(e);
  return check_launch(
      launch_topk(pscores, B, P, k, nullptr, 1, nullptr, pool, idx, stream, /*pdl=*/true));
}

csa2_status csa2_hier_pool_index_mxfp4(const uint8_t* q_mx, const uint8_t* k_mx, int B, int H_I,
                                       int D_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                       const int32_t* pool, int P, int k, int32_t* idx, void* ws,
                                       size_t ws_bytes, cudaStream_t stream) {
  csa2_status s = check_seq(B, N, kv_seq_stride, q_per_seq);
  if (s != CSA2_OK) return s;
  if ((s = check_indexer_mx(q_mx, k_mx, B, H_I, D_I, 1, kv_seq_stride, q_per_seq)) != CSA2_OK)
    return s;
  if (P < 1 || k < 1) return CSA2_ERR_INVALID_ARG;
  if (B > 0 && (!pool || !idx)) return CSA2_ERR_INVALID_ARG;
  WsLayout w = layout(B, 0, 0, 0, P);
  if (!ws || ws_bytes < w.total) return CSA2_ERR_WORKSPACE;
  uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
  float* pscores = reinterpret_cast<float*>(wsb + w.pool_scores);
  cudaError_t e = launch_pool_scores_mxfp4(q_mx, k_mx, B, H_I, N, kv_seq_stride, q_per_seq, pool,
                                           P, pscores, status_ptr(ws), stream);
  if (e != cudaSuccess) return check_launch(e);
  return check_launch(
      launch_topk(pscores, B, P, k, nullptr, 1, nullptr, pool, idx, stream, /*pdl=*/true));
}

csa2_status csa2_sparse_attn_fp4(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H,
                                 int D, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                 const int32_t* idx, int k, float softmax_scale, float* out,
                                 float* lse, void* ws, size_t ws_bytes, cudaStream_t stream) {
  csa2_status s = check_seq(B, N, kv_seq_stride, q_per_seq);
  if (s != CSA2_OK) return s;
  if ((s = check_attn(q_bf16, kv_fp4, B, H, D, k, softmax_scale, out)) != CSA2_OK) return s;
  if (B > 0 && !idx) return CSA2_ERR_INVALID_ARG;
  WsLayout w = layout(B, 0, k, H, 0);
  if (!ws || ws_bytes < w.total) return CSA2_ERR_WORKSPACE;
  uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
  return check_launch(launch_sparse_attn(q_bf16, kv_fp4, B, H, N, kv_seq_stride, q_per_seq, idx,
                                         k, softmax_scale, out, lse, wsb + w.attn,
                                         status_ptr(ws), stream));
}

csa2_status csa2_sparse_attn_fp4_swa(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H,
                                     int D, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                     const int32_t* idx, int k, const uint8_t* swa_kv,
                                     int64_t swa_ring, int n_win, const int32_t* q_pos,
                                     float softmax_scale, float* out, float* lse, void* ws,
                                     size_t ws_bytes, cudaStream_t stream) {
  csa2_status s = check_seq(B, N, kv_seq_stride, q_per_seq);
  if (s != CSA2_OK) return s;
  if ((s = check_attn(q_bf16, kv_fp4, B, H, D, k, softmax_scale, out)) != CSA2_OK) return s;
  if (B > 0 && (!idx || !swa_kv || !q_pos)) return CSA2_ERR_INVALID_ARG;
  if (n_win < 1 || swa_ring < n_win || !aligned16(swa_kv)) return CSA2_ERR_INVALID_ARG;
  WsLayout w = layout(B, 0, k, H, 0);
  if (!ws || ws_bytes < w.total) return CSA2_ERR_WORKSPACE;
  uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
  const SwaArgs swa{swa_kv, swa_ring, n_win, q_pos};
  return check_launch(launch_sparse_attn(q_bf16, kv_fp4, B, H, N, kv_seq_stride, q_per_seq, idx,
                                         k, softmax_scale, out, lse, wsb + w.attn,
                                         status_ptr(ws), stream, false, &swa));
}

int csa2_layer_group_launches(const csa2_layer* layers, int n_layers, const csa2_group_args* g) {
  if (!layers || !g || n_layers < 1 || layers[0].mode != CSA2_FULL) return -1;
  if (g->B == 0) return 0;
  int n = 0;
  for (int l = 0; l < n_layers; ++l) {
    const int m = layers[l].mode;
    if (m == CSA2_FULL)
      n += 1 + topk_launches(g->B, g->N, g->k, (size_t)-1) +
           (g->pool_size > 0 ? (g->pool_block > 1 ? 3 : topk_launches(g->B, g->N, g->pool_size,
                                                                        (size_t)-1))
                             : 0);
    else if (m == CSA2_REINDEX) n += 2;
    else if (m != CSA2_REUSE) return -1;
    n += attn_launches(g->B, g->k);
  }
  return n;
}

csa2_status csa2_layer_group(const csa2_layer* layers, int n_layers, const csa2_group_args* g,
                             void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!layers || !g || n_layers < 1) return CSA2_ERR_INVALID_ARG;
  if (layers[0].mode != CSA2_FULL) return CSA2_ERR_INVALID_ARG;
  csa2_status s = check_seq(g->B, g->N, g->kv_seq_stride, g->q_per_seq);
  if (s != CSA2_OK) return s;
  if (g->pool_size < 0) return CSA2_ERR_INVALID_ARG;
  if (g->pool_size > 0 && g->B > 0 && !g->pool_out) return CSA2_ERR_INVALID_ARG;
  if (g->pool_size > 0 && g->pool_size < g->k) return CSA2_ERR_INVALID_ARG;
  if (g->pool_block < 0 || (g->pool_block > 1 && g->pool_size % g->pool_block != 0))
    return CSA2_ERR_INVALID_ARG;
  if (g->n_win < 0 || (g->n_win > 0 && (g->swa_ring < g->n_win || (g->B > 0 && !g->q_pos))))
    return CSA2_ERR_INVALID_ARG;
  // validate every layer before launching anything
  for (int l = 0; l < n_layers; ++l) {
    const csa2_layer& L = layers[l];
    if (L.mode != CSA2_FULL && L.mode != CSA2_REINDEX && L.mode != CSA2_REUSE)
      return CSA2_ERR_INVALID_ARG;
    if (g->n_win > 0 && L.swa_kv && !aligned16(L.swa_kv)) return CSA2_ERR_INVALID_ARG;
    if ((s = check_attn(L.q_bf16, g->kv_fp4, g->B, g->H, g->D, g->k, g->softmax_scale, L.out)) !=
        CSA2_OK)
      return s;
    if (L.mode == CSA2_REUSE) {
      if (L.qi_fp8) return CSA2_ERR_INVALID_ARG;
    } else {
      if ((s = check_indexer_fmt(g->indexer_fmt, L.qi_fp8, g->ki_fp8, g->B, g->H_I, g->D_I,
                                 g->ratio, g->kv_seq_stride, g->q_per_seq)) != CSA2_OK)
        return s;
      if (g->indexer_fmt == CSA2_INDEXER_E4M3 &&
          (s = check_scan_rows(g->B, g->N, g->kv_seq_stride, g->q_per_seq)) != CSA2_OK)
        return s;
      if (g->B > 0 && !L.idx_out) return CSA2_ERR_INVALID_ARG;
    }
  }
  WsLayout w = layout(g->B, g->N, g->k, g->H, g->pool_size);
  if (!ws || ws_bytes < w.total) return CSA2_ERR_WORKSPACE;
  if (g->B == 0) return CSA2_OK;
  uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
  int32_t* status = status_ptr(ws);
  float* scores = reinterpret_cast<float*>(wsb + w.scores);
  float* pscores = reinterpret_cast<float*>(wsb + w.pool_scores);
  const int32_t* latest = nullptr;
  const bool mx = g->indexer_fmt == CSA2_INDEXER_MXFP4;
  cudaError_t e = cudaSuccess;
  // A layer's top-k requests the FP4 rows it selects into L2 while it writes
  // them, so that the attention's first tiles find their rows there; only
  // when the selected rows of the batch take at most half of L2 (not for
  // many queries over one shared context, whose rows repeat).
  RowPrefetch pf;
  if ((reinterpret_cast<uintptr_t>(g->kv_fp4) & 15u) == 0 &&
      (int64_t)g->B * g->k * kRowBytes <= (int64_t)64 << 20) {
    pf.kv = g->kv_fp4;
    pf.seq_bytes = g->kv_seq_stride * kRowBytes;
    pf.n = g->N;
    pf.q_per_seq = g->q_per_seq;
  }
  bool q_waited = false;
  for (int l = 0; l < n_layers && e == cudaSuccess; ++l) {
    const csa2_layer& L = layers[l];
    const int32_t* use = nullptr;
    if (L.mode == CSA2_FULL || (L.mode == CSA2_REINDEX && g->pool_size == 0)) {
      e = mx ? launch_index_scores_mxfp4(L.qi_fp8, g->ki_fp8, g->B, g->H_I, g->N,
                                         g->kv_seq_stride, g->q_per_seq, g->q_pos, g->ratio,
                                         scores, status, stream)
             : launch_index_scores(L.qi_fp8, g->ki_fp8, g->B, g->H_I, g->D_I, g->N,
                                   g->kv_seq_stride, g->q_per_seq, g->q_pos, g->ratio, scores,
                                   status, stream);
      if (e == cudaSuccess && L.mode == CSA2_FULL && g->pool_size > 0) {
        if (g->pool_block > 1)  // blockwise pool (a one-entry block pool is the flat one)
          e = launch_block_pool(scores, g->B, g->N, g->q_pos, g->ratio, g->pool_block,
                                g->pool_size / g->pool_block, g->pool_out, wsb + w.bpool, stream,
                                /*pdl=*/true);
        else
          e = launch_topk(scores, g->B, g->N, g->pool_size, g->q_pos, g->ratio, nullptr, nullptr,
                          g->pool_out, stream, /*pdl=*/true, wsb + w.topk, w.topk_bytes);
      }
      if (e == cudaSuccess)
        e = launch_topk(scores, g->B, g->N, g->k, g->q_pos, g->ratio, nullptr, nullptr, L.idx_out,
                        stream, /*pdl=*/true, wsb + w.topk, w.topk_bytes, pf);
      use = L.idx_out;
    } else if (L.mode == CSA2_REINDEX) {
      e = mx ? launch_pool_scores_mxfp4(L.qi_fp8, g->ki_fp8, g->B, g->H_I, g->N,
                                        g->kv_seq_stride, g->q_per_seq, g->pool_out,
                                        g->pool_size, pscores, status, stream)
             : launch_pool_scores(L.qi_fp8, g->ki_fp8, g->B, g->H_I, g->D_I, g->N,
                                  g->kv_seq_stride, g->q_per_seq, g->pool_out, g->pool_size,
                                  pscores, status, stream);
      if (e == cudaSuccess)
        e = launch_topk(pscores, g->B, g->pool_size, g->k, nullptr, 1, nullptr, g->pool_out,
                        L.idx_out, stream, /*pdl=*/true, nullptr, 0, pf);
      use = L.idx_out;
    } else {  // REUSE: the attention kernel writes the copy of the reused indices
      use = latest;
    }
    if (e != cudaSuccess) break;
    latest = use;
    // The attention starts early (programmatic dependent launch): it loads Q
    // and sets up while the kernel before it (this layer's top-k, or the
    // previous layer's merge) finishes.
    if (g->q_ready && !q_waited) {  // the main queries may arrive on another stream
      e = cudaStreamWaitEvent(stream, g->q_ready, 0);
      q_waited = true;
      if (e != cudaSuccess) break;
    }
    const SwaArgs swa{L.swa_kv, g->swa_ring, g->n_win, g->q_pos};
    const bool with_swa = g->n_win > 0 && L.swa_kv;
    e = launch_sparse_attn(L.q_bf16, g->kv_fp4, g->B, g->H, g->N, g->kv_seq_stride, g->q_per_seq,
                           use, g->k, g->softmax_scale, L.out, L.lse, wsb + w.attn, status,
                           stream, /*pdl=*/true, with_swa ? &swa : nullptr,
                           L.mode == CSA2_REUSE ? L.idx_out : nullptr);
  }
  return check_launch(e);
}

}  // extern "C"
