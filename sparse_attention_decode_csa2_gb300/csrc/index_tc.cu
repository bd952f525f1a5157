// Indexer scores on the tensor cores (DeepSeek-V4.1-Flash paper walkthrough,
// 1.(4) "CSA2": indexer q and indexer K score the main-KV entries).
//
//   D[e][n] = sum_d KI[e][d] * B[n][d]   (tcgen05.mma kind::f8f6f4, E4M3 x E4M3,
//                                         fp32 accumulate, M = 128 entries)
//   score[q][e] = sum_h D[e][(q - q0) * H_I + h]
// B holds the indexer heads of QG queries that share one context (QG = 1 for
// decode: the heads padded to N = 16 or 32; up to QG = 16 for the prefill-shaped
// case: N = QG * H_I <= 256), so one pass over the K tile scores every head of
// every query in the group.  FP8 products are exact; each head's 64-term sum and
// the head sum accumulate in fp32 (exact for integer-valued inputs).
//
// Work split: the (query group, 128-entry tile) items of the whole call are
// cut into one contiguous range per CTA, and the grid holds no more CTAs than
// fit on the GPU at once, so every SM streams K tiles for the whole kernel
// (no second, partly empty wave).  A range spans at most two query groups;
// both groups' B operands are kept.
//
// Roles (192 threads): warp 0 lane 0 streams K tiles with 2D TMA (swizzle
// matching the UMMA layout) into an 8-stage ring, the first 8 requested
// before the queries' visibility is known; warp 1 owns the TMEM accumulator (two buffers) and lane 0
// issues the MMAs; warps 2-5 first stage the B operands and the queries'
// visible lengths (signalled on an mbarrier), then, one thread per TMEM lane
// = entry, sum the head columns, apply causal visibility and store the
// scores.  Tiles wholly past every query's visible prefix are not loaded
// (beyond the first ring's worth, which is requested speculatively); their
// scores are written as -inf directly.
#include <cuda.h>

#include "csa2_internal.cuh"
#include "tc_common.cuh"

namespace csa2 {
namespace {

using namespace tc;

// warps 0, 1 (TMA producer, MMA issuer) + EW epilogue warps; EW = 8 when a
// tile's accumulator holds 256 head columns per entry (the epilogue, summing
// them, bounds those shapes), each quadrant of tensor-memory lanes read by
// two warps that split the group's queries; EW = 4 otherwise
template <int EW>
constexpr int idx_threads() { return (2 + EW) * 32; }
constexpr int kStages = 8;
constexpr int kTile = 128;

struct IdxCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t meta;           // B operands, visible lengths and live_end staged
  uint32_t tmem_base;
  int32_t live_end[2];     // per group of the range: tiles holding any visible entry
  int32_t nvis[2][16];
};

template <int D_I>
struct IdxLayout {
  static constexpr uint32_t tile_bytes = kTile * D_I;
  static constexpr uint32_t k_off = 0;
  static constexpr uint32_t b_off = k_off + kStages * tile_bytes;
  static constexpr uint32_t b_max = 256 * D_I;  // one group's B: up to 256 rows x D_I
  // B stride for NB rows, whole 8-row swizzle atoms, 1 KiB aligned
  __host__ __device__ static uint32_t b_stride(int NB) {
    return (uint32_t)((NB * D_I + 1023) / 1024 * 1024);
  }
  __host__ __device__ static uint32_t ctl_off(int NB) { return b_off + 2 * b_stride(NB); }
  __host__ __device__ static uint32_t alloc(int NB) { return ctl_off(NB) + 512 + 1024; }
};

__device__ __forceinline__ uint32_t idx_tmem_cols(int NB) {
  return NB <= 16 ? 32u : (NB <= 32 ? 64u : (NB <= 64 ? 128u : (NB <= 128 ? 256u : 512u)));
}

// A tile's scores from its accumulator columns (thread = entry e of the tile,
// taddr = its TMEM lane at the buffer's first column): query qq's score is the
// sum, in column order, of its HI head columns qq * HI .. +HI; 32 columns per
// tensor-memory round trip.  `srow` = the group's first score row.
template <int HI>
__device__ __forceinline__ void score_columns(uint32_t taddr, int nq, int64_t e, int64_t N,
                                              const int32_t* nv, float* srow) {
  const int ncols = nq * HI;
  for (int c0 = 0; c0 < ncols; c0 += 32) {
    float v[32];
    tmem_ld16(taddr + c0, v);
    if (c0 + 16 < ncols) tmem_ld16(taddr + c0 + 16, v + 16);
    tmem_wait_ld();
#pragma unroll
    for (int qn = 0; qn < 32 / HI; ++qn) {
      const int qq = c0 / HI + qn;
      if (qq < nq) {
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < HI; ++j) acc += v[HI * qn + j];
        if (e < N) srow[qq * N + e] = (e < nv[qq]) ? acc : -INFINITY;
      }
    }
  }
}

// One CTA: items [w0, w1) of the call, item w = (group w / T, tile w % T).
template <int D_I, int EW>
__global__ void __launch_bounds__(idx_threads<EW>(), EW == 4 ? 3 : 2)
index_tc_kernel(const __grid_constant__ CUtensorMap tmap, const uint8_t* __restrict__ q_fp8,
                int B, int H_I, int64_t N, int64_t kv_seq_stride, int q_per_seq, int QG, int NB,
                int64_t T, int64_t W, const int32_t* __restrict__ q_pos, int ratio,
                float* __restrict__ scores, int32_t* status) {
  using L = IdxLayout<D_I>;
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = su32(smem_raw);
  const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_s + pad;
  const uint32_t bstride = L::b_stride(NB);
  IdxCtl& ctl = *reinterpret_cast<IdxCtl*>(smem + L::ctl_off(NB));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t C = gridDim.x;
  const int64_t w0 = (int64_t)blockIdx.x * W / C, w1 = ((int64_t)blockIdx.x + 1) * W / C;
  const int nitems = (int)(w1 - w0);
  const int64_t g0 = w0 / T;  // first group of the range (the range ends in g0 or g0 + 1)
  const uint32_t cols = idx_tmem_cols(NB);
  const int ng = (int)((w1 - 1) / T - g0) + 1;  // groups in the range: 1 or 2
  if (warp >= 2) {
    // The heads and positions of the range's queries are requested first,
    // ahead of the K stream in the memory queues (read again, from L2, below).
    const int et = tid - 64;
    for (int gi = 0; gi < ng; ++gi) {
      const int64_t q0 = (g0 + gi) * QG;
      const int nq = (int)min((int64_t)QG, (int64_t)B - q0);
      const uint8_t* qb = q_fp8 + q0 * H_I * D_I;
      for (int off = et * 128; off < nq * H_I * D_I; off += EW * 32 * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(qb + off));
      if (q_pos && et < nq) asm volatile("prefetch.global.L2 [%0];" ::"l"(q_pos + q0 + et));
    }
  }

  if (warp == 1) {
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
      mbar_init(su32(&ctl.acc_empty[i]), EW);
    }
    mbar_init(su32(&ctl.meta), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // first row of the sequence of group g0 + gi
  const int64_t row_g0 = ((g0 * QG) / q_per_seq) * kv_seq_stride;
  const int64_t row_g1 = (((g0 + 1) * QG) / q_per_seq) * kv_seq_stride;
  const int n_spec = nitems < kStages ? nitems : kStages;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  // item i of the range is loaded, multiplied and read back iff it is in the
  // first (speculative) ring's worth or its tile holds a visible entry
  auto processed = [&](int i, int64_t g, int64_t t) {
    return i < n_spec || t < ctl.live_end[g - g0];
  };

  if (warp == 0) {
    if (lane == 0) {
      // the first ring's worth is requested at once (speculatively: the
      // visible lengths may still be on their way)
      int n = 0;
      bool meta = false;
      int64_t g = g0, t = w0 - g0 * T;
      for (int i = 0; i < nitems; ++i, t = (t + 1 == T) ? (++g, 0) : t + 1) {
        if (i >= n_spec) {
          if (!meta && !(meta = mbar_wait(su32(&ctl.meta), 0, status))) break;
          if (!processed(i, g, t)) continue;
        }
        const int s = n % kStages;
        const uint32_t ph = (uint32_t)(n / kStages) & 1u;
        if (!mbar_wait(su32(&ctl.empty[s]), ph ^ 1u, status)) break;
        mbar_expect_tx(su32(&ctl.full[s]), L::tile_bytes);
        tma_load_2d(sbase + L::k_off + s * L::tile_bytes, &tmap, 0,
                    (int)((g == g0 ? row_g0 : row_g1) + t * kTile), su32(&ctl.full[s]));
        ++n;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_e4m3(NB);
      const uint64_t dA0 = swz_desc(sbase + L::k_off, D_I);
      const uint64_t dB0 = swz_desc(sbase + L::b_off, D_I);
      bool alive = mbar_wait(su32(&ctl.meta), 0, status);
      int n = 0;
      int64_t g = g0, t = w0 - g0 * T;
      for (int i = 0; i < nitems && alive; ++i, t = (t + 1 == T) ? (++g, 0) : t + 1) {
        if (!processed(i, g, t)) continue;
        const int s = n % kStages;
        const uint32_t ph = (uint32_t)(n / kStages) & 1u;
        const int ab = n & 1;
        if (!mbar_wait(su32(&ctl.full[s]), ph, status) ||
            !mbar_wait(su32(&ctl.acc_empty[ab]), (((uint32_t)n >> 1) & 1u) ^ 1u, status)) {
          alive = false;
          break;
        }
        tc_fence_after();
        const uint64_t da0 = dA0 + ((uint32_t)(s * L::tile_bytes) >> 4);
        const uint64_t db0 = dB0 + ((uint32_t)((g - g0) * bstride) >> 4);
#pragma unroll
        for (int kk = 0; kk < D_I / 32; ++kk)
          mma_e4m3(tmem + ab * NB, da0 + ((kk * 32) >> 4), db0 + ((kk * 32) >> 4), idesc,
                   kk > 0 ? 1u : 0u);
        mma_commit(su32(&ctl.acc_full[ab]));
        mma_commit(su32(&ctl.empty[s]));
        ++n;
      }
      if (alive && n > 0)
        mbar_wait(su32(&ctl.acc_full[(n - 1) & 1]), (((uint32_t)(n - 1)) >> 1) & 1u, status);
    }
  } else {
    // ---- stage the B operands (heads of each group's queries) and the visible lengths ----
    const int et = tid - 64;  // 0 .. 32 EW - 1
    for (int gi = 0; gi < ng; ++gi) {
      const int64_t q0 = (g0 + gi) * QG;
      const int nq = (int)min((int64_t)QG, (int64_t)B - q0);
      for (int i = et; i < NB * D_I / 16; i += EW * 32) {
        const int nrow = i / (D_I / 16), c = i % (D_I / 16);
        uint4 v = make_uint4(0, 0, 0, 0);
        const int qq = nrow / H_I, h = nrow % H_I;
        if (qq < nq)
          v = __ldg(reinterpret_cast<const uint4*>(q_fp8 + ((q0 + qq) * H_I + h) * D_I) + c);
        *reinterpret_cast<uint4*>(smem + L::b_off + gi * bstride + swz_off(nrow, c * 16, D_I)) = v;
      }
      if (et < 16) ctl.nvis[gi][et] = (et < nq) ? (int)n_visible(q_pos, (int)(q0 + et), ratio, N) : 0;
    }
    proxy_fence();
    asm volatile("bar.sync 1, %0;" ::"n"(EW * 32) : "memory");
    if (et == 0) {
      for (int gi = 0; gi < 2; ++gi) {
        int m = 0;
        if (gi < ng)
          for (int i = 0; i < 16; ++i) m = max(m, ctl.nvis[gi][i]);
        ctl.live_end[gi] = (int)((m + kTile - 1) / kTile);
      }
      mbar_arrive(su32(&ctl.meta));
    }
    asm volatile("bar.sync 1, %0;" ::"n"(EW * 32) : "memory");

    // ---- epilogue: thread = TMEM lane = entry row of the tile; with eight
    //      epilogue warps, warps 2-5 take the first half of the group's
    //      queries and warps 6-9 the second (multiples of four queries) ----
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int cg = (warp - 2) >> 2;  // column group
    bool alive = true;
    int n = 0;
    int64_t g = g0, t = w0 - g0 * T;
    for (int i = 0; i < nitems; ++i, t = (t + 1 == T) ? (++g, 0) : t + 1) {
      const int64_t e = t * kTile + r;
      const int64_t qg0 = g * QG;
      const int nq_g = (int)min((int64_t)QG, (int64_t)B - qg0);
      // this warp's queries of the group: [q_lo, q_lo + nq)
      const int per = EW == 4 ? nq_g : ((nq_g + 1) / 2 + 3) / 4 * 4;
      const int q_lo = min(nq_g, cg * per);
      const int nq = min(nq_g, q_lo + per) - q_lo;
      const int64_t q0 = qg0 + q_lo;
      const int32_t* nv = ctl.nvis[g - g0] + q_lo;
      const uint32_t col0 = (uint32_t)(q_lo * H_I);  // this warp's first accumulator column
      if (processed(i, g, t)) {
        const int ab = n & 1;
        const uint32_t ph = ((uint32_t)n >> 1) & 1u;
        ++n;
        if (alive && !mbar_wait(su32(&ctl.acc_full[ab]), ph, status)) alive = false;
        if (alive && (H_I == 8 || H_I == 16 || H_I == 32)) {
          // 8, 16 or 32 heads per query: the group's head columns 32 per
          // tensor-memory round trip, each query's H_I columns summed in
          // column order
          tc_fence_after();
          if (H_I == 8)
            score_columns<8>(tmem + lane_base + ab * NB + col0, nq, e, N, nv, scores + q0 * N);
          else if (H_I == 16)
            score_columns<16>(tmem + lane_base + ab * NB + col0, nq, e, N, nv, scores + q0 * N);
          else
            score_columns<32>(tmem + lane_base + ab * NB + col0, nq, e, N, nv, scores + q0 * N);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(su32(&ctl.acc_empty[ab]));
          continue;
        }
        if (alive) {
          tc_fence_after();
          for (int qq = 0; qq < nq; ++qq) {
            // this query's H_I head columns
            float acc = 0.0f;
            int h = 0;
            for (; h + 16 <= H_I; h += 16) {
              float v[16];
              tmem_ld16(tmem + lane_base + ab * NB + col0 + qq * H_I + h, v);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) acc += v[j];
            }
            if (h < H_I) {
              float v[16];
              // 16 columns starting at this query's remaining heads (stays inside NB:
              // NB is a multiple of 16 and QG * H_I <= NB)
              const int cbase = min((int)col0 + qq * H_I + h, NB - 16);
              tmem_ld16(tmem + lane_base + ab * NB + cbase, v);
              tmem_wait_ld();
              const int off = (int)col0 + qq * H_I + h - cbase;
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (j >= off && j < off + (H_I - h)) acc += v[j];
            }
            if (e < N) scores[(q0 + qq) * N + e] = (e < nv[qq]) ? acc : -INFINITY;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(su32(&ctl.acc_empty[ab]));
          continue;
        }
      }
      if (e < N)
        for (int qq = 0; qq < nq; ++qq) scores[(q0 + qq) * N + e] = -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(cols));
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once (a function-local static is
// initialised exactly once even when several host threads launch at the same time).
EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
  }();
  return fn;
}

template <int D_I, int EW>
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
  const int64_t T = (N + kTile - 1) / kTile;  // tiles per query group
  const int64_t groups = (B + QG - 1) / QG;
  const int64_t W = groups * T;                // items of the call
  // Co-resident CTAs must never need more than the SM's 512 TMEM columns (an
  // allocation would block): request enough shared memory to cap residency.
  const uint32_t cols = NB <= 16 ? 32u : (NB <= 32 ? 64u : (NB <= 64 ? 128u : (NB <= 128 ? 256u : 512u)));
  const uint32_t max_ctas = 512u / cols;
  uint32_t smem = L::alloc(NB);
  const uint32_t cap_smem = 232448u / max_ctas - 1024u;  // leaves room for the runtime's reservation
  if (max_ctas < 16 && smem < cap_smem) smem = cap_smem;
  cudaError_t e = cudaFuncSetAttribute(index_tc_kernel<D_I, EW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // one wave: as many CTAs as fit at once, but each range within two groups
  e = cudaFuncSetAttribute(index_tc_kernel<D_I, EW>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           100);
  if (e != cudaSuccess) return e;
  int dev = 0, smem_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
      cudaSuccess)
    return e;
  int per_sm = smem_sm / (int)(smem + 1024);  // the runtime reserves 1 KiB per CTA
  if (per_sm > 4) per_sm = 4;
  if (per_sm > 12 / EW) per_sm = 12 / EW;  // registers: 3 CTAs of 6 warps or 2 of 10
  if (per_sm < 1) per_sm = 1;
  int64_t C = (int64_t)per_sm * device_sm_count();
  if (C > W) C = W;
  if (C < groups) C = groups;  // W / C <= T: no range spans more than two groups
  return launch_kernel(index_tc_kernel<D_I, EW>, dim3((unsigned)C), dim3(idx_threads<EW>()), smem, stream,
                       false, map, q_fp8, B, H_I, N, kv_seq_stride, q_per_seq, QG, NB, T, W, q_pos,
                       ratio, scores, status);
}

}  // namespace

// Returns cudaErrorNotSupported when the shape has no tensor-core variant.
cudaError_t launch_index_scores_tc(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I,
                                   int D_I, int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                   const int32_t* q_pos, int ratio, float* scores,
                                   int32_t* status, cudaStream_t stream) {
  // queries sharing a context share each K tile: the largest group of
  // QG <= 16 queries whose QG * H_I heads fit one MMA (N <= 256, a multiple of 16)
  int QG = 0, NB = 0;
  for (int qg = 16; qg >= 2 && QG == 0; qg >>= 1)
    if (q_per_seq % qg == 0 && qg * H_I <= 256 && (qg * H_I) % 16 == 0) QG = qg;
  if (QG > 0) {
    NB = QG * H_I;
  } else if (H_I <= 32) {
    QG = 1;
    NB = H_I <= 16 ? 16 : 32;
  } else {
    return cudaErrorNotSupported;
  }
  // eight epilogue warps when a tile's accumulator has 256 head columns per
  // entry (query groups of 32-head queries: the epilogue bounds those); four
  // otherwise (measured: with 128 columns the split epilogue was slower)
  const bool wide = NB >= 256;
#define CSA2_IDX_LAUNCH(DI)                                                                     \
  return wide ? launch_t<DI, 8>(q_fp8, k_fp8, B, H_I, N, kv_seq_stride, q_per_seq, QG, NB,    \
                                q_pos, ratio, scores, status, stream)                          \
              : launch_t<DI, 4>(q_fp8, k_fp8, B, H_I, N, kv_seq_stride, q_per_seq, QG, NB,    \
                                q_pos, ratio, scores, status, stream)
  switch (D_I) {
    case 32:
      CSA2_IDX_LAUNCH(32);
    case 64:
      CSA2_IDX_LAUNCH(64);
    case 128:
      CSA2_IDX_LAUNCH(128);
    default:
      return cudaErrorNotSupported;
  }
#undef CSA2_IDX_LAUNCH
}

}  // namespace csa2
