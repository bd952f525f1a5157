/*
 * csa2.h -- C ABI of libcsa2.so, the GB300 (sm_103a) implementation of the
 * CSA2 compressed-sparse-attention hot path of DeepSeek-V4.1-Flash.
 *
 * The operations follow the method as described on these pages:
 *  - modelscope.csdn.net DeepSeek-V4.1-Flash release summary, section "CSA2"
 *    (three static layer modes sharing main KV and indexer K; FP4 E2M1 main
 *    KV with one E4M3 scale per 16 channels);
 *  - wkq9411.github.io DeepSeek-V4.1-Flash paper walkthrough, sections
 *    1.(4) "CSA2" (indexer scores entries, per-query top-k, each query attends
 *    its selected entries), 1.(4).1 "Cross-Layer KV and Index Reuse",
 *    1.(4).2 "Hierarchical Sparse Indexer", 1.(5).4 "FP4 Main KV Cache",
 *    3.(2).1 "Model settings" (64 query heads x 512).
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers, allocated and owned by the
 *    caller; the library never allocates device memory and keeps no state.
 *  - Layouts are dense row-major, innermost dimension last.
 *  - Every call is asynchronous on `stream` and never synchronises, except
 *    csa2_read_status.  Arguments are validated on the host before any
 *    launch; an invalid call returns an error and launches nothing.
 *  - Sequences: query q reads sequence s = q / q_per_seq, whose entries start
 *    at entry offset s * kv_seq_stride of the KV and indexer-K arrays
 *    (kv_seq_stride = 0: every query shares one context).
 *  - Causal visibility: with q_pos non-NULL, entry j is visible to query q
 *    iff ratio * j + ratio - 1 <= q_pos[q] (the entry's last token is not in
 *    the query's future); q_pos NULL makes every entry visible.
 *  - Scratch memory is passed as (ws, ws_bytes).  Its first 256 bytes hold a
 *    device status word that kernels set when they meet a bad index or give
 *    up a bounded wait; csa2_workspace_init clears it and csa2_read_status
 *    reads and clears it.  Calls that overlap on the GPU must not share a
 *    workspace.
 *  - Supported shapes on the GPU path: D = 512, D_I in {32, 64, 128},
 *    H in {16, 32, 64}, 1 <= H_I <= 32, 1 <= k <= 16384,
 *    N < 2^31; MXFP4 indexer rows: D_I = 128, 1 <= H_I <= 64.  Other shapes
 *    return CSA2_ERR_UNSUPPORTED.
 */
#ifndef CSA2_H_
#define CSA2_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum csa2_status {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad schedule */
  CSA2_ERR_UNSUPPORTED = 2,   /* shape outside what the kernels are built for */
  CSA2_ERR_WORKSPACE = 3,     /* ws NULL or ws_bytes too small */
  CSA2_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  CSA2_ERR_BAD_INDEX = 5,     /* (device status) an index was outside [-1, N) */
  CSA2_ERR_TIMEOUT = 6        /* (device status) a bounded device wait gave up */
} csa2_status;

typedef enum csa2_mode {
  CSA2_FULL = 0,     /* own indexer q; scores every visible entry; new top-k */
  CSA2_REINDEX = 1,  /* own indexer q; re-scores the shared indexer K (or the pool) */
  CSA2_REUSE = 2     /* no indexer; reuses the latest FULL/REINDEX indices */
} csa2_mode;

/* Formats of the indexer query and key rows of a layer group. */
typedef enum csa2_indexer_fmt {
  CSA2_INDEXER_E4M3 = 0,   /* E4M3 [D_I] bytes per row */
  CSA2_INDEXER_MXFP4 = 1   /* OCP MXFP4 rows of CSA2_MXFP4_ROW_BYTES(D_I) bytes */
} csa2_indexer_fmt;

/* Bytes of one MXFP4 indexer row of d elements: d/2 E2M1 code bytes then d/32
 * E8M0 scale bytes (68 bytes at d = 128). */
#define CSA2_MXFP4_ROW_BYTES(d) ((d) / 2 + (d) / 32)

/* Bytes of one FP4 main-KV row of d channels: d/2 code bytes then d/16 scale bytes. */
#define CSA2_FP4_ROW_BYTES(d) ((d) / 2 + (d) / 16)

/* Human-readable name of a status code (static string). */
const char* csa2_status_string(csa2_status s);

/* Library version: major * 10000 + minor * 100 + patch. */
int csa2_version(void);

/* Message of the last CUDA error that made a call of this thread return
 * CSA2_ERR_CUDA (static string; "no error" if none). */
const char* csa2_last_cuda_error(void);

/*
 * csa2_quantize_kv_fp4 -- writes FP4 main-KV rows (walkthrough 1.(5).4
 * "FP4 Main KV Cache": E2M1 codes, one E4M3 scale per 16 channels, no global
 * scale; release summary "CSA2").
 *   x      fp32 [n_rows][d], finite values
 *   out    uint8 [n_rows][d/2 + d/16]; byte j of a row holds channel 2j in its
 *          low nibble and channel 2j+1 in its high nibble; then one E4M3 byte
 *          per 16-channel block b (channels 16b..16b+15)
 *   Per block: scale = E4M3(absmax / 6) rounded to nearest even, saturating
 *   at 448; each code = the E2M1 value nearest to the exact |x| / scale (ties
 *   to the even code), sign bit = sign bit of x; a zero scale gives zero
 *   magnitudes.  Bit-exact.  d must be 512; x and out 16-byte aligned.
 */
csa2_status csa2_quantize_kv_fp4(const float* x, int64_t n_rows, int d, uint8_t* out,
                                 cudaStream_t stream);

/*
 * csa2_upload -- a decode step's host inputs in one host-to-device copy.
 * The pages have no counterpart: this is the serving-side transfer of a
 * step's inputs into the resident buffers the other calls read.
 *   host_packed  host buffer of `bytes` bytes (pinned for an asynchronous
 *                copy): n_segs csa2_upload_seg entries at offset 0, then the
 *                segments' payloads at the offsets the entries give
 *   dev_stage    device staging area, >= bytes, 16-byte aligned; the whole
 *                buffer is copied there (one cudaMemcpyAsync), then one kernel
 *                writes each segment's rows to its destination:
 *     CSA2_UPLOAD_RAW     rows x row_bytes payload bytes, row r to
 *                         dst + r * dst_stride
 *     CSA2_UPLOAD_KV_FP4  rows x 512 fp32 latent channels (row_bytes = 2048),
 *                         each packed exactly as csa2_quantize_kv_fp4 packs it
 *                         into the 288-byte FP4 row at dst + r * dst_stride
 *                         (dst and dst_stride multiples of 16, dst_stride >= 288)
 *   Segments are applied in table order (a later segment overwriting the same
 *   bytes wins).  Payload offsets must be 16-byte aligned and lie inside
 *   `bytes`; the table is validated on the host before anything is enqueued
 *   (CSA2_ERR_INVALID_ARG).  Destinations are device addresses owned by the
 *   caller; the staging area must not be reused until the stream has passed
 *   the kernel.
 */
typedef enum csa2_upload_kind { CSA2_UPLOAD_RAW = 0, CSA2_UPLOAD_KV_FP4 = 1 } csa2_upload_kind;

typedef struct csa2_upload_seg {
  uint64_t dst;         /* device address of destination row 0 */
  uint64_t src_off;     /* byte offset of the payload in the packed buffer */
  uint64_t rows;        /* rows of the segment */
  uint64_t row_bytes;   /* payload bytes per row (2048 for CSA2_UPLOAD_KV_FP4) */
  uint64_t dst_stride;  /* bytes between destination rows */
  uint32_t kind;        /* csa2_upload_kind */
  uint32_t reserved;    /* 0 */
} csa2_upload_seg;      /* 48 bytes */

csa2_status csa2_upload(const void* host_packed, size_t bytes, int n_segs, void* dev_stage,
                        size_t stage_bytes, cudaStream_t stream);

/*
 * csa2_index_scores -- the lightweight indexer (walkthrough 1.(4) "CSA2":
 * indexer Q and indexer K score main-KV entries).
 *   q_fp8    E4M3 [B][H_I][D_I] indexer queries
 *   k_fp8    E4M3 [S][N][D_I] indexer keys, one per entry, shared by all
 *            indexer heads (sequence s at entry offset s * kv_seq_stride)
 *   scores   fp32 [B][N]: scores[q][j] = sum_h sum_d q[q][h][d] * k[s][j][d]
 *            for visible j, -inf for invisible j
 *   Arithmetic: the tensor-core scan forms each head's D_I-term dot
 *   product with exact E4M3 x E4M3 products accumulated in fp32, then adds
 *   the H_I per-head fp32 sums in fp32.  Every step is exact whenever every
 *   partial sum is fp32-representable (e.g. integer inputs, where |score| <=
 *   H_I * D_I * 64 < 2^24); otherwise each sum carries ordinary fp32
 *   rounding.  (The pool re-index of csa2_hier_pool_index forms the head sum
 *   of the query first, in two f16 parts: exact for integer inputs.)
 *   k_fp8 must be 16-byte aligned.
 *   Returns CSA2_ERR_UNSUPPORTED when the rows the scan reads,
 *   (S - 1) * kv_seq_stride + N with S = ceil(B / q_per_seq), number 2^31 or
 *   more (the scan addresses them with 32-bit tensor coordinates); the
 *   E4M3 layers of csa2_layer_group have the same limit.
 */
csa2_status csa2_index_scores(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I, int D_I,
                              int64_t N, int64_t kv_seq_stride, int q_per_seq,
                              const int32_t* q_pos, int ratio, float* scores,
                              cudaStream_t stream);

/*
 * csa2_quantize_mxfp4 -- writes MXFP4 indexer rows (walkthrough 1.(5).4: the
 * indexer query and key are FP4 in the OCP MXFP4 format: blocks of 32 E2M1
 * elements sharing one E8M0 power-of-two scale).
 *   x      fp32 [n_rows][d], finite values; d a multiple of 32, <= 4096;
 *          16-byte aligned
 *   out    uint8 [n_rows][d/2 + d/32]: byte j of a row holds element 2j in its
 *          low nibble and 2j+1 in its high nibble; then one E8M0 byte per
 *          32-element block b (2^(byte - 127))
 *   Per block: shared exponent e = floor(log2(absmax)) - 2 (2 is the largest
 *   E2M1 exponent) clamped to >= -127, scale byte e + 127 (0 for an all-zero
 *   block); each code = the E2M1 value nearest to the exact |x| / 2^e (ties to
 *   the even code), saturating at 6; sign bit = sign bit of x.  Bit-exact.
 */
csa2_status csa2_quantize_mxfp4(const float* x, int64_t n_rows, int d, uint8_t* out,
                                cudaStream_t stream);

/*
 * csa2_index_scores_mxfp4 -- the lightweight indexer with MXFP4 query and key
 * (walkthrough 1.(4) "CSA2" and 1.(5).4).
 *   q_mx     MXFP4 [B][H_I][68] indexer queries (D_I = 128)
 *   k_mx     MXFP4 [S][N][68] indexer keys (sequence s at entry offset
 *            s * kv_seq_stride); 16-byte aligned, and kv_seq_stride a multiple
 *            of 4 when there is more than one sequence
 *   scores   fp32 [B][N]: sum_h sum_d value(q[q][h][d]) * value(k[s][j][d]) for
 *            visible j, -inf for invisible j
 *   The head sum of the decoded query is formed first (compensated fp32
 *   summation); the dot product with each key accumulates fp32 products of
 *   exact decoded values, scaled per 32-element block.  Scores are therefore
 *   fp32 approximations of the exact sum (relative error of the order of
 *   2^-20 of the sum of absolute products).  D_I must be 128, 1 <= H_I <= 64.
 */
csa2_status csa2_index_scores_mxfp4(const uint8_t* q_mx, const uint8_t* k_mx, int B, int H_I,
                                    int D_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                    const int32_t* q_pos, int ratio, float* scores,
                                    cudaStream_t stream);

/*
 * csa2_topk -- per-query top-k selection (walkthrough 1.(4) "CSA2": the top-k
 * entries per query).
 *   scores   fp32 [B][N] (NaN not allowed; -0 and +0 compare equal)
 *   idx      int32 [B][k]: the min(k, visible) visible entries with the
 *            largest scores, ties broken towards the lower index, written in
 *            ascending index order and padded with -1.  Bit-exact.
 *   ws       at least csa2_workspace_size(B, N, k, 0, 0) bytes.
 */
csa2_status csa2_topk(const float* scores, int B, int64_t N, int k, const int32_t* q_pos,
                      int ratio, int32_t* idx, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * csa2_block_pool -- blockwise candidate pool of the Hierarchical Sparse
 * Indexer (walkthrough 1.(4).2 "Hierarchical Sparse Indexer": the Full
 * layer's index score of a block is the largest score among its positions,
 * the top-scoring blocks are chosen and the positions they cover form the
 * candidate pool that later Reindex layers score).
 *   scores   fp32 [B][N] index scores (as csa2_index_scores writes them);
 *            only the visible entries of each query count (q_pos, ratio as
 *            in csa2_index_scores)
 *   block    entries per block (>= 1): aligned runs [block*b, block*b+block)
 *   n_blocks blocks kept per query (>= 1), ranked by (block score desc,
 *            block index asc); a block without a visible entry is no candidate
 *   pool     int32 [B][n_blocks * block]: the visible entries of the kept
 *            blocks in ascending order, padded with -1 (the layout
 *            csa2_hier_pool_index takes).  Bit-exact.
 *   ws       device scratch, at least
 *            csa2_block_pool_workspace_size(B, N, block, n_blocks) bytes,
 *            owned by the caller; contents need no initialisation.
 * Returns CSA2_ERR_INVALID_ARG for negative sizes, block or n_blocks < 1 or
 * missing pointers, CSA2_ERR_WORKSPACE for a short workspace.
 */
csa2_status csa2_block_pool(const float* scores, int B, int64_t N, const int32_t* q_pos,
                            int ratio, int block, int n_blocks, int32_t* pool, void* ws,
                            size_t ws_bytes, cudaStream_t stream);

/* Scratch bytes csa2_block_pool needs for these dimensions. */
size_t csa2_block_pool_workspace_size(int B, int64_t N, int block, int n_blocks);

/*
 * csa2_hier_pool_index -- a Reindex layer of the Hierarchical Sparse Indexer
 * (walkthrough 1.(4).2): scores only the candidate-pool entries with this
 * layer's indexer q and keeps its own top-k inside the pool.
 *   pool     int32 [B][P] entry ids, strictly ascending, -1 padding only at
 *            the end (the layout csa2_topk writes); a violation sets the
 *            CSA2_ERR_BAD_INDEX status and the row's result is unspecified
 *   idx      int32 [B][k] selected entry ids, ascending, -1 padded; ranking
 *            by (score desc, entry id asc).  Bit-exact given exact scores.
 *   Scores: the head sum of the query (exact in fp32 for H_I <= 32) is split
 *   into two f16 parts (22 significant bits: exact for integer inputs) and
 *   dotted with the gathered rows on tensor cores in fp32.
 *   ws       at least csa2_workspace_size(B, N, k, 0, P) bytes.
 */
csa2_status csa2_hier_pool_index(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I,
                                 int D_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                 const int32_t* pool, int P, int k, int32_t* idx, void* ws,
                                 size_t ws_bytes, cudaStream_t stream);

/*
 * csa2_hier_pool_index_mxfp4 -- csa2_hier_pool_index with MXFP4 indexer rows
 * (q_mx, k_mx as in csa2_index_scores_mxfp4); same pool, idx and workspace
 * rules.
 */
csa2_status csa2_hier_pool_index_mxfp4(const uint8_t* q_mx, const uint8_t* k_mx, int B, int H_I,
                                       int D_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                       const int32_t* pool, int P, int k, int32_t* idx, void* ws,
                                       size_t ws_bytes, cudaStream_t stream);

/*
 * csa2_sparse_attn_fp4 -- gathers the selected FP4 entries, dequantises them
 * and runs MQA softmax attention over them (walkthrough 1.(4) "CSA2";
 * 1.(5).4: the cache is dequantised before attention; 3.(2).1: 64 heads x
 * 512).  K = V = the dequantised latent, shared by all heads.
 *   q_bf16   bf16 [B][H][D] main queries (16-byte aligned)
 *   kv_fp4   uint8 [S][N][D/2 + D/16] FP4 rows (16-byte aligned)
 *   idx      int32 [B][k] entry ids; -1 slots are skipped; ids outside
 *            [-1, N) are skipped and set CSA2_ERR_BAD_INDEX in the status
 *   out      fp32 [B][H][D]: softmax(softmax_scale * q . v_j) weighted sum of v_j
 *   lse      fp32 [B][H] log-sum-exp of the scaled logits, or NULL
 *   A row with no valid slot yields out = 0 and lse = -inf.
 *   ws       at least csa2_workspace_size(B, 0, k, H, 0) bytes.
 */
csa2_status csa2_sparse_attn_fp4(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H,
                                 int D, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                 const int32_t* idx, int k, float softmax_scale, float* out,
                                 float* lse, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * csa2_sparse_attn_fp4_swa -- csa2_sparse_attn_fp4 with the query's sliding
 * window of the layer's SWA KV in the same softmax (walkthrough 1.(4): every
 * query attends the selected entries and its layer's own SWA KV; 1.(5).4:
 * SWA KV stays FP8; 3.(2).1: window n_win = 128).
 *   swa_kv   E4M3 [S][swa_ring][D] one latent per token (plain E4M3, no
 *            scale), per sequence a ring: token t at row t mod swa_ring
 *            (16-byte aligned)
 *   swa_ring rows per sequence, >= n_win; when several queries share a
 *            sequence the ring must hold all of their windows
 *   n_win    window length (>= 1): the query at q_pos[b] attends tokens
 *            max(0, q_pos[b] - n_win + 1) .. q_pos[b] (none when q_pos[b] < 0)
 *   q_pos    int32 [B] token positions (required)
 *   out, lse as csa2_sparse_attn_fp4, over the union of both sets: K = V, one
 *            softmax with the same scale.
 *   ws       at least csa2_workspace_size(B, 0, k, H, 0) bytes.
 * Errors as csa2_sparse_attn_fp4; CSA2_ERR_INVALID_ARG for a missing swa_kv /
 * q_pos, n_win < 1 or swa_ring < n_win.
 */
csa2_status csa2_sparse_attn_fp4_swa(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H,
                                     int D, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                     const int32_t* idx, int k, const uint8_t* swa_kv,
                                     int64_t swa_ring, int n_win, const int32_t* q_pos,
                                     float softmax_scale, float* out, float* lse, void* ws,
                                     size_t ws_bytes, cudaStream_t stream);

/*
 * csa2_sparse_attn_fp4_noalloc -- csa2_sparse_attn_fp4 for callers that cannot
 * allocate device memory.  The pages have no counterpart: this is a deployment
 * variant, not part of the method.
 *   Who needs it: code that enqueues work while its stream is being captured
 *   into a CUDA graph (an allocation is not a stream operation and breaks the
 *   capture), plug-ins inside a runtime that owns every device allocation, and
 *   latency-critical loops that must never call cudaMalloc (it can synchronise
 *   the device).  Such callers still pass their inputs and outputs, but no
 *   workspace.
 *   Arguments, layouts and results are those of csa2_sparse_attn_fp4 (same
 *   kernels).  The split partials (per-split log-sum-exps) live in a fixed
 *   256 KiB device array inside the library, held by every GPU that loads the
 *   library until the process exits.  A call whose partials would not fit
 *   (csa2_workspace_size(B, 0, k, H, 0) - 256 bytes > 256 KiB) returns
 *   CSA2_ERR_WORKSPACE and launches nothing; with splits never outnumbering
 *   the SMs, that needs a GPU of more than 1024 SMs.  No cudaMalloc, cudaFree or
 *   allocating library routine is called.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, once per device, under a lock); make that first
 *   call before any stream capture.  All calls share the array, which keeps
 *   the last call's contents (nothing needs to start cleared): calls that
 *   overlap on the GPU (other streams, other host threads) race on it and must
 *   be serialised by the caller.  There is no status word: indices outside
 *   [-1, N) are skipped as in csa2_sparse_attn_fp4, and a bounded device wait
 *   that gives up (about 2 s) ends its CTA early, but neither is reported.
 *   A failing CUDA call returns CSA2_ERR_CUDA and leaves its message for
 *   csa2_last_cuda_error().
 */
csa2_status csa2_sparse_attn_fp4_noalloc(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B,
                                         int H, int D, int64_t N, int64_t kv_seq_stride,
                                         int q_per_seq, const int32_t* idx, int k,
                                         float softmax_scale, float* out, float* lse,
                                         cudaStream_t stream);

/* One layer of a CSA2 layer group. */
typedef struct csa2_layer {
  int mode;                /* csa2_mode */
  const uint16_t* q_bf16;  /* bf16 [B][H][D] this layer's main query */
  const uint8_t* qi_fp8;   /* [B][H_I][row] indexer query in the group's indexer format
                              (E4M3 [D_I] or MXFP4 rows); NULL for REUSE */
  float* out;              /* fp32 [B][H][D] */
  float* lse;              /* fp32 [B][H] or NULL */
  int32_t* idx_out;        /* int32 [B][k]: indices this layer attended.  Required for
                              FULL and REINDEX; for REUSE, NULL or a buffer that
                              receives a copy of the reused indices */
  const uint8_t* swa_kv;   /* E4M3 [S][swa_ring][D] this layer's SWA KV (see
                              csa2_sparse_attn_fp4_swa), or NULL: no window */
} csa2_layer;

/* What the layers of one group share (walkthrough 1.(4).1). */
typedef struct csa2_group_args {
  const uint8_t* kv_fp4;   /* [S][N][D/2 + D/16] shared FP4 main KV */
  const uint8_t* ki_fp8;   /* [S][N][row] shared indexer K in the indexer format */
  int B, H, H_I, D, D_I;
  int64_t N, kv_seq_stride;
  int q_per_seq;
  const int32_t* q_pos;    /* [B] or NULL */
  int ratio;
  int k;
  int pool_size;           /* 0: flat indexer; P > 0: FULL layers build a P-entry pool and
                              REINDEX layers select inside it (walkthrough 1.(4).2) */
  int32_t* pool_out;       /* int32 [B][pool_size] when pool_size > 0 */
  float softmax_scale;
  int pool_block;          /* how FULL layers build the pool: 0 or 1: the top pool_size
                              entries; b > 1: the blockwise pool of pool_size / b blocks
                              of b entries (csa2_block_pool; pool_size % b == 0) */
  int64_t swa_ring;        /* rows per sequence of the layers' SWA KV rings */
  int n_win;               /* SWA window; 0: no layer attends a window.  With n_win > 0
                              each layer with swa_kv also attends its window (q_pos
                              required, swa_ring >= n_win) */
  int indexer_fmt;         /* csa2_indexer_fmt of qi_fp8 and ki_fp8 */
  cudaEvent_t q_ready;     /* NULL, or an event the group's attention launches wait for
                              (cudaStreamWaitEvent before the first one): the layers'
                              main queries may still be arriving on another stream while
                              the indexer and top-k run */
} csa2_group_args;

/*
 * csa2_layer_group -- runs a static schedule of CSA2 layers over one shared
 * FP4 main KV and indexer K (walkthrough 1.(4).1, 1.(4).2):
 *   FULL    scores all visible entries with its own indexer q, takes top-k
 *           (and builds the pool when pool_size > 0: see pool_block), attends;
 *   REINDEX re-scores the shared indexer K (only the pool when pool_size > 0)
 *           with its own indexer q, takes top-k, attends;
 *   REUSE   attends with the indices of the nearest preceding FULL/REINDEX.
 * Every layer attends with its own main query.  layers[0] must be FULL.
 *   ws   at least csa2_workspace_size(B, N, k, H, pool_size) bytes.
 */
csa2_status csa2_layer_group(const csa2_layer* layers, int n_layers, const csa2_group_args* g,
                             void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Number of kernel launches csa2_layer_group enqueues for these arguments
 * (-1 if they are invalid).  Host-only; useful to size CUDA-graph captures
 * and to account for launches.
 */
int csa2_layer_group_launches(const csa2_layer* layers, int n_layers, const csa2_group_args* g);

/*
 * Scratch bytes for csa2_layer_group with these dimensions (pass 0 for
 * dimensions a call does not use).  The same number is enough for every
 * individual call made with the same or smaller dimensions.  Depends on the
 * current device's SM count.
 */
size_t csa2_workspace_size(int B, int64_t N, int k, int H, int P);

/* Clears the workspace's device status word (asynchronous, on `stream`). */
csa2_status csa2_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Synchronises `stream`, reads and clears the device status word.  Writes
 * the raw bits to *device_bits (if non-NULL): bit 0 bad index, bit 1 bounded
 * wait timed out.  Returns CSA2_OK, CSA2_ERR_BAD_INDEX or CSA2_ERR_TIMEOUT;
 * CSA2_ERR_WORKSPACE for a NULL ws, CSA2_ERR_CUDA if the copy, the clear or
 * the synchronisation fails (csa2_last_cuda_error names the cause).
 */
csa2_status csa2_read_status(void* ws, cudaStream_t stream, int32_t* device_bits);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H_ */
