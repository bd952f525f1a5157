// Indexer scores on the tensor cores (DeepSeek-V4.1-Flash paper walkthrough,
// 1.(4) "CSA2": indexer q and indexer K score the main-KV entries).
//
//   D[e][n] = sum_d KI[e][d] * B[n][d]   (tcgen05.mma kind::f8f6f4, E4M3 x E4M3,
//                                         fp32 accumulate, M = 128 entries)
//   score[q][e] = sum_h D[e][(q - q0) * H_I + h]
// B holds the indexer heads of QG queries that share one context (QG = 1 for
// decode: the heads padded to N = 16 or 32; QG = 16 for the prefill-shaped
// case: N = 16 * H_I), so one pass over the K tile scores every head of every
// query in the group.  FP8 products are exact; each head's 64-term sum and
// the head sum accumulate in fp32 (exact for integer-valued inputs).
//
// Roles (192 threads): warp 0 lane 0 streams 128-entry K tiles with 2D TMA
// (swizzle matching the UMMA layout) into an 8-stage ring; warp 1 owns the
// TMEM accumulator (two buffers) and lane 0 issues the MMAs; warps 2-5 (one
// thread per TMEM lane = entry) sum the head columns, apply causal
// visibility and store the scores.  Tiles wholly past every query's visible
// prefix are not loaded; their scores are written as -inf directly.
#include <cuda.h>

#include "csa2_internal.cuh"
#include "tc_common.cuh"

namespace csa2 {
namespace {

using namespace tc;

constexpr int kIdxThreads = 192;
constexpr int kStages = 8;
constexpr int kTile = 128;

struct IdxCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
  int32_t nvis[16];
};

template <int D_I>
struct IdxLayout {
  static constexpr uint32_t tile_bytes = kTile * D_I;
  static constexpr uint32_t k_off = 0;
  static constexpr uint32_t b_off = k_off + kStages * tile_bytes;  // up to 256 rows x D_I
  static constexpr uint32_t b_bytes = 256 * D_I;
  static constexpr uint32_t ctl_off = b_off + b_bytes;
  static constexpr uint32_t bytes = ctl_off + 512;
  static constexpr uint32_t alloc = bytes + 1024;
};

// One CTA: query group [q0, q0 + QG) (one sequence) x tiles [t0, t0 + nt) of 128 entries.
template <int D_I>
__global__ void __launch_bounds__(kIdxThreads, 1)
index_tc_kernel(const __grid_constant__ CUtensorMap tmap, const uint8_t* __restrict__ q_fp8,
                int B, int H_I, int64_t N, int64_t kv_seq_stride, int q_per_seq, int QG, int NB,
                int tiles_per_cta, const int32_t* __restrict__ q_pos, int ratio,
                float* __restrict__ scores, int32_t* status) {
  using L = IdxLayout<D_I>;
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = su32(smem_raw);
  const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_s + pad;
  IdxCtl& ctl = *reinterpret_cast<IdxCtl*>(smem + L::ctl_off);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q0 = blockIdx.y * QG;
  const int nq = min(QG, B - q0);
  const int64_t total_tiles = (N + kTile - 1) / kTile;
  const int64_t t0 = (int64_t)blockIdx.x * tiles_per_cta;
  const int nt = (int)(total_tiles - t0 < tiles_per_cta ? total_tiles - t0 : tiles_per_cta);
  const int64_t row0 = (int64_t)(q0 / q_per_seq) * kv_seq_stride;  // first row of the sequence

  // ---- prologue: B operand (heads of the group's queries), barriers, TMEM ----
  for (int i = tid; i < 256 * D_I / 16; i += kIdxThreads) {
    const int n = i / (D_I / 16), c = i % (D_I / 16);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < NB) {
      const int qq = n / H_I, h = n % H_I;
      if (qq < nq)
        v = __ldg(reinterpret_cast<const uint4*>(q_fp8 + ((int64_t)(q0 + qq) * H_I + h) * D_I) +
                  c);
    }
    *reinterpret_cast<uint4*>(smem + L::b_off + swz_off(n, c * 16, D_I)) = v;
  }
  if (tid < 16) ctl.nvis[tid] = (tid < nq) ? (int)n_visible(q_pos, q0 + tid, ratio, N) : 0;
  if (warp == 1) {
    const uint32_t cols = NB <= 16 ? 32u : (NB <= 32 ? 64u : (NB <= 64 ? 128u : (NB <= 128 ? 256u : 512u)));
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(&ctl.tmem_base)),
                 "r"(cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(su32(&ctl.full[s]), 1);
      mbar_init(su32(&ctl.empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(su32(&ctl.acc_full[i]), 1);
      mbar_init(su32(&ctl.acc_empty[i]), 4);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  proxy_fence();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  int nvis_max = 0;
#pragma unroll 1
  for (int i = 0; i < nq; ++i) nvis_max = max(nvis_max, ctl.nvis[i]);
  // tiles [t0, t0 + n_live) hold visible entries of some query
  const int64_t live_end = (nvis_max + kTile - 1) / kTile;
  const int64_t live_n = live_end - t0 < nt ? live_end - t0 : nt;
  const int n_live = (int)(live_n > 0 ? live_n : 0);

  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < n_live; ++i) {
        const int s = i % kStages;
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        if (!mbar_wait(su32(&ctl.empty[s]), ph ^ 1u, status)) break;
        mbar_expect_tx(su32(&ctl.full[s]), L::tile_bytes);
        tma_load_2d(sbase + L::k_off + s * L::tile_bytes, &tmap, 0,
                    (int)(row0 + (t0 + i) * kTile), su32(&ctl.full[s]));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_e4m3(NB);
      const uint64_t dA0 = swz_desc(sbase + L::k_off, D_I);
      const uint64_t dB0 = swz_desc(sbase + L::b_off, D_I);
      bool alive = true;
      for (int i = 0; i < n_live && alive; ++i) {
        const int s = i % kStages;
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        const int ab = i & 1;
        if (!mbar_wait(su32(&ctl.full[s]), ph, status) ||
            !mbar_wait(su32(&ctl.acc_empty[ab]), (((uint32_t)i >> 1) & 1u) ^ 1u, status)) {
          alive = false;
          break;
        }
        tc_fence_after();
        const uint64_t da0 = dA0 + ((uint32_t)(s * L::tile_bytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D_I / 32; ++kk)
          mma_e4m3(tmem + ab * NB, da0 + ((kk * 32) >> 4), dB0 + ((kk * 32) >> 4), idesc,
                   kk > 0 ? 1u : 0u);
        mma_commit(su32(&ctl.acc_full[ab]));
        mma_commit(su32(&ctl.empty[s]));
      }
      if (alive && n_live > 0)
        mbar_wait(su32(&ctl.acc_full[(n_live - 1) & 1]), (((uint32_t)(n_live - 1)) >> 1) & 1u,
                  status);
    }
  } else {
    // epilogue: thread = TMEM lane = entry row of the tile
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    bool alive = true;
    for (int i = 0; i < nt; ++i) {
      const int64_t e = (t0 + i) * kTile + r;
      if (i < n_live && alive) {
        const int ab = i & 1;
        if (!mbar_wait(su32(&ctl.acc_full[ab]), ((uint32_t)i >> 1) & 1u, status)) {
          alive = false;
        } else {
          tc_fence_after();
          for (int qq = 0; qq < nq; ++qq) {
            // this query's H_I head columns
            float acc = 0.0f;
            int h = 0;
            for (; h + 16 <= H_I; h += 16) {
              float v[16];
              tmem_ld16(tmem + lane_base + ab * NB + qq * H_I + h, v);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) acc += v[j];
            }
            if (h < H_I) {
              float v[16];
              // 16 columns starting at this query's remaining heads (stays inside NB:
              // NB is a multiple of 16 and QG * H_I <= NB)
              const int cbase = min(qq * H_I + h, NB - 16);
              tmem_ld16(tmem + lane_base + ab * NB + cbase, v);
              tmem_wait_ld();
              const int off = qq * H_I + h - cbase;
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (j >= off && j < off + (H_I - h)) acc += v[j];
            }
            if (e < N) scores[(int64_t)(q0 + qq) * N + e] = (e < ctl.nvis[qq]) ? acc : -INFINITY;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(su32(&ctl.acc_empty[ab]));
          continue;
        }
      }
      if (e < N)
        for (int qq = 0; qq < nq; ++qq) scores[(int64_t)(q0 + qq) * N + e] = -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    const uint32_t cols = NB <= 16 ? 32u : (NB <= 32 ? 64u : (NB <= 64 ? 128u : (NB <= 128 ? 256u : 512u)));
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(cols));
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

template <int D_I>
cudaError_t launch_t(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I, int64_t N,
                     int64_t kv_seq_stride, int q_per_seq, int QG, int NB, const int32_t* q_pos,
                     int ratio, float* scores, int32_t* status, cudaStream_t stream) {
  using L = IdxLayout<D_I>;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int64_t n_seq = (B + q_per_seq - 1) / q_per_seq;
  const int64_t rows = kv_seq_stride > 0 ? (n_seq - 1) * kv_seq_stride + N : N;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)D_I, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D_I};
  const cuuint32_t box[2] = {(cuuint32_t)D_I, (cuuint32_t)kTile};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = D_I == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                           : (D_I == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                        : CU_TENSOR_MAP_SWIZZLE_32B);
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(k_fp8), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int64_t total_tiles = (N + kTile - 1) / kTile;
  const int groups = (B + QG - 1) / QG;
  const int64_t target = 3LL * device_sm_count();
  int64_t per = (total_tiles * groups + target - 1) / target;
  if (per < 4) per = 4;
  if (per > total_tiles) per = total_tiles;
  const int64_t gx = (total_tiles + per - 1) / per;
  // Co-resident CTAs must never need more than the SM's 512 TMEM columns (an
  // allocation would block): request enough shared memory to cap residency.
  const uint32_t cols = NB <= 16 ? 32u : (NB <= 32 ? 64u : (NB <= 64 ? 128u : (NB <= 128 ? 256u : 512u)));
  const uint32_t max_ctas = 512u / cols;
  uint32_t smem = L::alloc;
  const uint32_t cap_smem = 232448u / max_ctas - 1024u;  // leaves room for the runtime's reservation
  if (max_ctas < 16 && smem < cap_smem) smem = cap_smem;
  cudaError_t e = cudaFuncSetAttribute(index_tc_kernel<D_I>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  index_tc_kernel<D_I><<<dim3((unsigned)gx, (unsigned)groups), kIdxThreads, smem, stream>>>(
      map, q_fp8, B, H_I, N, kv_seq_stride, q_per_seq, QG, NB, (int)per, q_pos, ratio, scores,
      status);
  return cudaGetLastError();
}

}  // namespace

// Returns cudaErrorNotSupported when the shape has no tensor-core variant.
cudaError_t launch_index_scores_tc(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I,
                                   int D_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                   const int32_t* q_pos, int ratio, float* scores,
                                   int32_t* status, cudaStream_t stream) {
  int QG, NB;
  if (q_per_seq >= 16 && q_per_seq % 16 == 0 && 16 * H_I <= 256 && (H_I % 4) == 0) {
    QG = 16;
    NB = 16 * H_I;  // multiple of 64
  } else if (H_I <= 32) {
    QG = 1;
    NB = H_I <= 16 ? 16 : 32;
  } else {
    return cudaErrorNotSupported;
  }
  switch (D_I) {
    case 32:
      return launch_t<32>(q_fp8, k_fp8, B, H_I, N, kv_seq_stride, q_per_seq, QG, NB, q_pos, ratio,
                          scores, status, stream);
    case 64:
      return launch_t<64>(q_fp8, k_fp8, B, H_I, N, kv_seq_stride, q_per_seq, QG, NB, q_pos, ratio,
                          scores, status, stream);
    case 128:
      return launch_t<128>(q_fp8, k_fp8, B, H_I, N, kv_seq_stride, q_per_seq, QG, NB, q_pos,
                           ratio, scores, status, stream);
    default:
      return cudaErrorNotSupported;
  }
}

}  // namespace csa2
