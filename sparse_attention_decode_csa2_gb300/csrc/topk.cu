// Per-query top-k selection (DeepSeek-V4.1-Flash paper walkthrough, 1.(4)
// "CSA2": the indexer keeps the top-k entries of each query).  Ties go to
// the lower index; the result is written in ascending index order and padded
// with -1 when fewer than k entries are candidates.
//
// One 1024-thread CTA per row.  Scores map to order-preserving uint32 keys
// (-0 folded onto +0).  A three-pass MSB radix select (11 + 11 + 10 bits,
// shared-memory histograms with warp-aggregated atomics) finds the exact k-th
// largest key T and how many keys equal to T are still needed.  A final
// in-order sweep over 1024-element rounds (warp ballots for ranks) writes
// every key > T and the first `need` keys == T, in ascending position.  Rows
// whose candidates fit in shared memory keep their keys there; longer rows
// re-read the scores (L2-resident) on every pass.
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kSmemKeyCap = 40960;  // 160 KiB of keys

struct TopkShared {
  int32_t hist[2048];
  int32_t warp_a[kWarps];
  int32_t warp_b[kWarps];
  int32_t digit;
  int32_t above;
  int32_t n;
  int32_t out_pos;
  int32_t eq_taken;
};

template <bool kSmem>
struct KeySource {
  const float* row;
  const uint32_t* keys;
  __device__ __forceinline__ uint32_t operator()(int j) const {
    if (kSmem) return keys[j];
    return float_to_ordered(row[j]);
  }
};

// Exclusive scan over the block of one int per thread; returns the exclusive
// prefix, writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int32_t* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = warp_tot[lane];
    int s = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_tot[lane] = s - t;  // exclusive warp offsets
    if (lane == 31) warp_tot[kWarps] = s;
  }
  __syncthreads();
  int r = warp_tot[warp] + x - v;
  *total = warp_tot[kWarps];
  __syncthreads();
  return r;
}

template <bool kSmem>
__global__ void __launch_bounds__(kThreads, 1)
topk_kernel(const float* __restrict__ scores, int64_t N, int k, const int32_t* __restrict__ q_pos,
            int ratio, const int32_t* __restrict__ n_valid, const int32_t* __restrict__ map,
            int32_t* __restrict__ idx) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  TopkShared& sh = *reinterpret_cast<TopkShared*>(smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + align_up(sizeof(TopkShared), 16));
  // warp_tot scratch for scans needs kWarps + 1 slots
  __shared__ int32_t scan_tot[kWarps + 1];

  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const float* row = scores + (int64_t)b * N;
  const int32_t* mrow = map ? map + (int64_t)b * N : nullptr;
  int32_t* out = idx + (int64_t)b * k;

  // number of candidates
  int n;
  if (map) {
    // candidates are the valid (>= 0) leading positions of the map row
    int c = 0;
    for (int64_t j = tid; j < N; j += kThreads) c += (mrow[j] >= 0);
    int tot;
    block_exclusive_scan(c, scan_tot, &tot);
    n = tot;
  } else if (n_valid) {
    n = n_valid[b];
  } else {
    n = (int)n_visible(q_pos, b, ratio, N);
  }

  if (n <= k) {
    for (int j = tid; j < k; j += kThreads) {
      int32_t v = -1;
      if (j < n) v = mrow ? mrow[j] : j;
      out[j] = v;
    }
    return;
  }

  if (kSmem) {
    for (int j = tid; j < n; j += kThreads) keys[j] = float_to_ordered(row[j]);
  }
  KeySource<kSmem> key{row, keys};

  uint32_t prefix = 0, mask = 0;
  int need = k;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nbins = pass == 2 ? 1024 : 2048;
    for (int i = tid; i < 2048; i += kThreads) sh.hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < n; base += kThreads) {
      const int j = base + tid;
      bool act = false;
      uint32_t d = 0;
      if (j < n) {
        uint32_t kk = key(j);
        act = (kk & mask) == prefix;
        d = (kk >> shift) & (uint32_t)(nbins - 1);
      }
      // warp-aggregated atomics: one add per distinct bin in the warp
      unsigned am = __ballot_sync(0xffffffffu, act);
      if (act) {
        unsigned peers = __match_any_sync(am, d);
        int leader = __ffs(peers) - 1;
        if (lane == leader) atomicAdd(&sh.hist[d], __popc(peers));
      }
    }
    __syncthreads();
    // find the digit holding the need-th largest key: scan bins from the top
    const int per = nbins / kThreads;  // 2 or 1
    int cnt = 0;
    int dtop = nbins - 1 - tid * per;
    for (int i = 0; i < per; ++i) cnt += sh.hist[dtop - i];
    int tot;
    int before = block_exclusive_scan(cnt, scan_tot, &tot);
    if (before < need && before + cnt >= need) {
      int acc = before;
      for (int i = 0; i < per; ++i) {
        int h = sh.hist[dtop - i];
        if (acc + h >= need) {
          sh.digit = dtop - i;
          sh.above = acc;
          break;
        }
        acc += h;
      }
    }
    __syncthreads();
    need -= sh.above;
    prefix |= (uint32_t)sh.digit << shift;
    mask |= (uint32_t)(nbins - 1) << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;

  // in-order compaction
  if (tid == 0) {
    sh.out_pos = 0;
    sh.eq_taken = 0;
  }
  __syncthreads();
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = 0; base < n; base += kThreads) {
    const int j = base + tid;
    uint32_t kk = j < n ? key(j) : 0u;
    const bool gt = j < n && kk > T;
    const bool eq = j < n && kk == T;
    unsigned eqm = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) sh.warp_a[warp] = __popc(eqm);
    __syncthreads();
    int eq_before = sh.eq_taken;
    for (int w = 0; w < warp; ++w) eq_before += sh.warp_a[w];
    eq_before += __popc(eqm & lt_mask);
    const bool take = gt || (eq && eq_before < need);
    unsigned tm = __ballot_sync(0xffffffffu, take);
    if (lane == 0) sh.warp_b[warp] = __popc(tm);
    __syncthreads();
    int pos = sh.out_pos;
    for (int w = 0; w < warp; ++w) pos += sh.warp_b[w];
    pos += __popc(tm & lt_mask);
    if (take && pos < k) out[pos] = mrow ? mrow[j] : j;
    __syncthreads();
    if (tid == 0) {
      int te = 0, tt = 0;
      for (int w = 0; w < kWarps; ++w) {
        te += sh.warp_a[w];
        tt += sh.warp_b[w];
      }
      sh.eq_taken += te;
      sh.out_pos += tt;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_topk(const float* scores, int B, int64_t N, int k, const int32_t* q_pos,
                        int ratio, const int32_t* n_valid, const int32_t* map, int32_t* idx,
                        cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const size_t base = align_up(sizeof(TopkShared), 16);
  if (N <= kSmemKeyCap) {
    size_t smem = base + (size_t)N * 4;
    static bool attr_set = false;
    if (!attr_set) {
      cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)(base + (size_t)kSmemKeyCap * 4));
      attr_set = true;
    }
    topk_kernel<true><<<B, kThreads, smem, stream>>>(scores, N, k, q_pos, ratio, n_valid, map,
                                                     idx);
  } else {
    topk_kernel<false><<<B, kThreads, base, stream>>>(scores, N, k, q_pos, ratio, n_valid, map,
                                                      idx);
  }
  return cudaGetLastError();
}

}  // namespace csa2
