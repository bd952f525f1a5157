// Per-query top-k selection (DeepSeek-V4.1-Flash paper walkthrough, 1.(4)
// "CSA2": the indexer keeps the top-k entries of each query).  Ties go to
// the lower index; the result is written in ascending index order and padded
// with -1 when fewer than k entries are candidates.
//
// Scores map to order-preserving uint32 keys (-0 folded onto +0).  An MSB
// radix select finds the exact k-th largest key class and how many of its
// members are still needed; an ordered sweep then writes every larger key
// and the first `need` members of the class, in ascending position.
//
// Rows of up to 32768 candidates (topk_reg_kernel, one 512-thread CTA per
// row): each thread holds KPT consecutive keys in registers, so the ordered
// sweep needs only two block scans.  The radix passes start at the highest
// bit where the row's min and max keys differ and take 8-bit digits counted
// in per-warp private histograms (rows with few distinct scores, such as
// integer-valued ones, would otherwise serialise on a handful of shared
// bins); they stop as soon as the threshold bin is consumed exactly.
// Longer rows (topk_long_kernel, 1024 threads): keys are re-read from the
// (L2-resident) scores on every pass, three 11/11/10-bit passes, and the
// ordered sweep runs in 1024-element rounds with warp ballots.
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

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

constexpr int kRegThreads = 512;
constexpr int kRegWarps = kRegThreads / 32;
constexpr int kRegMaxKeys = kRegThreads * 64;

// Exclusive scan of one int per thread over a kRegThreads block.
__device__ __forceinline__ int reg_block_scan(int v, int32_t* tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = lane < kRegWarps ? tot[lane] : 0;
    int s = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kRegWarps) tot[lane] = s - t;
    if (lane == kRegWarps - 1) tot[kRegWarps] = s;
  }
  __syncthreads();
  const int r = tot[warp] + x - v;
  *total = tot[kRegWarps];
  __syncthreads();
  return r;
}

template <int KPT>
__global__ void __launch_bounds__(kRegThreads, 1)
topk_reg_kernel(const float* __restrict__ scores, int64_t N, int k,
                const int32_t* __restrict__ q_pos, int ratio, const int32_t* __restrict__ n_valid,
                const int32_t* __restrict__ map, int32_t* __restrict__ idx) {
  __shared__ int32_t whist[kRegWarps * 256];  // per-warp 8-bit digit histograms
  __shared__ int32_t tot[kRegWarps + 1];
  __shared__ uint32_t red_min[kRegWarps], red_max[kRegWarps];
  __shared__ int32_t s_digit, s_above, s_cnt;

  pdl_trigger();
  pdl_wait();  // scores, n_valid and map come from the kernel before
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* row = scores + (int64_t)b * N;
  const int32_t* mrow = map ? map + (int64_t)b * N : nullptr;
  int32_t* out = idx + (int64_t)b * k;

  int n;
  if (map) {
    int c = 0;
    for (int64_t j = tid; j < N; j += kRegThreads) c += (mrow[j] >= 0);
    int t;
    reg_block_scan(c, tot, &t);
    n = t;
  } else if (n_valid) {
    n = n_valid[b];
  } else {
    n = (int)n_visible(q_pos, b, ratio, N);
  }
  if (n <= k) {
    for (int j = tid; j < k; j += kRegThreads) out[j] = (j < n) ? (mrow ? mrow[j] : j) : -1;
    return;
  }

  // keys of positions [tid*KPT, tid*KPT + KPT) in registers
  const int base = tid * KPT;
  uint32_t key[KPT];
  const bool vec = ((N & 3) == 0) && ((reinterpret_cast<uintptr_t>(scores) & 15u) == 0);
#pragma unroll
  for (int i = 0; i < KPT; i += 4) {
    const int j = base + i;
    float v[4];
    if (vec && j + 3 < n) {
      const float4 f = *reinterpret_cast<const float4*>(row + j);
      v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = (j + e < n) ? row[j + e] : 0.0f;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) key[i + e] = float_to_ordered(v[e]);
  }

  // highest bit where the row's keys differ
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    if (base + i < n) {
      kmin = min(kmin, key[i]);
      kmax = max(kmax, key[i]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) {
    red_min[warp] = kmin;
    red_max[warp] = kmax;
  }
  __syncthreads();
  kmin = red_min[0];
  kmax = red_max[0];
#pragma unroll
  for (int w = 1; w < kRegWarps; ++w) {
    kmin = min(kmin, red_min[w]);
    kmax = max(kmax, red_max[w]);
  }

  uint32_t prefix, mask;
  int cur_hi;
  const uint32_t diff = kmin ^ kmax;
  if (diff == 0u) {
    prefix = kmax;
    mask = 0xFFFFFFFFu;
    cur_hi = -1;
  } else {
    const int hb = 31 - __clz(diff);
    mask = ~((2u << hb) - 1u);  // hb = 31: 2u << 31 wraps to 0, mask = 0
    prefix = kmax & mask;
    cur_hi = hb;
  }
  int need = k;
  bool done = cur_hi < 0;
  int32_t* my_hist = whist + warp * 256;  // this warp's private histogram
  while (!done) {
    const int nbits = min(8, cur_hi + 1);
    const int shift = cur_hi + 1 - nbits;
    const uint32_t dmask = (1u << nbits) - 1u;
    for (int i = tid; i < kRegWarps * 256; i += kRegThreads) whist[i] = 0;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      if (base + i < n && (key[i] & mask) == prefix)
        atomicAdd(&my_hist[(key[i] >> shift) & dmask], 1);
    }
    __syncthreads();
    // thread t < 256 owns digit 255 - t (descending order for the scan)
    int cnt = 0;
    if (tid < 256) {
      const int d = 255 - tid;
#pragma unroll
      for (int w = 0; w < kRegWarps; ++w) cnt += whist[w * 256 + d];
    }
    int total;
    const int before = reg_block_scan(cnt, tot, &total);
    if (tid < 256 && before < need && before + cnt >= need) {
      s_digit = 255 - tid;
      s_above = before;
      s_cnt = cnt;
    }
    __syncthreads();
    need -= s_above;
    prefix |= (uint32_t)s_digit << shift;
    mask |= dmask << shift;
    cur_hi = shift - 1;
    done = (cur_hi < 0) || (s_cnt == need);
    __syncthreads();
  }

  // ordered write: keys above the class, then the first `need` class members
  int gt = 0, eq = 0;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    if (base + i < n) {
      const uint32_t km = key[i] & mask;
      gt += km > prefix;
      eq += km == prefix;
    }
  }
  int tot_eq, tot_sel;
  const int eq_before = reg_block_scan(eq, tot, &tot_eq);
  const int take_eq = max(0, min(eq, need - eq_before));
  int off = reg_block_scan(gt + take_eq, tot, &tot_sel);
  int taken = 0;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    if (base + i < n) {
      const uint32_t km = key[i] & mask;
      const bool is_eq = km == prefix;
      const bool t = (km > prefix) || (is_eq && taken < take_eq);
      taken += (is_eq && t);
      if (t && off < k) {
        out[off] = mrow ? mrow[base + i] : base + i;
        ++off;
      }
    }
  }
}

template <bool kSmem>
__global__ void __launch_bounds__(kThreads, 1)
topk_long_kernel(const float* __restrict__ scores, int64_t N, int k, const int32_t* __restrict__ q_pos,
            int ratio, const int32_t* __restrict__ n_valid, const int32_t* __restrict__ map,
            int32_t* __restrict__ idx) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  TopkShared& sh = *reinterpret_cast<TopkShared*>(smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + align_up(sizeof(TopkShared), 16));
  // warp_tot scratch for scans needs kWarps + 1 slots
  __shared__ int32_t scan_tot[kWarps + 1];

  pdl_trigger();
  pdl_wait();  // scores, n_valid and map come from the kernel before
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
                        cudaStream_t stream, bool pdl) {
  if (B == 0) return cudaSuccess;
  const dim3 grid((unsigned)B);
  if (N <= kRegMaxKeys) {
    if (N <= kRegThreads * 8)
      return launch_kernel(topk_reg_kernel<8>, grid, dim3(kRegThreads), 0, stream, pdl, scores, N,
                           k, q_pos, ratio, n_valid, map, idx);
    if (N <= kRegThreads * 16)
      return launch_kernel(topk_reg_kernel<16>, grid, dim3(kRegThreads), 0, stream, pdl, scores,
                           N, k, q_pos, ratio, n_valid, map, idx);
    if (N <= kRegThreads * 32)
      return launch_kernel(topk_reg_kernel<32>, grid, dim3(kRegThreads), 0, stream, pdl, scores,
                           N, k, q_pos, ratio, n_valid, map, idx);
    return launch_kernel(topk_reg_kernel<64>, grid, dim3(kRegThreads), 0, stream, pdl, scores, N,
                         k, q_pos, ratio, n_valid, map, idx);
  }
  const size_t base = align_up(sizeof(TopkShared), 16);
  return launch_kernel(topk_long_kernel<false>, grid, dim3(kThreads), base, stream, pdl, scores, N,
                       k, q_pos, ratio, n_valid, map, idx);
}

}  // namespace csa2
