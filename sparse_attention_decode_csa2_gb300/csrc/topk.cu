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
// row; topk_cluster_kernel, a cluster of 2, 4 or 8 such CTAs per row when the
// batch alone would leave SMs idle): each thread holds KPT consecutive
// keys in registers.  The radix
// passes take 8-bit digits from the highest bit where the row's min and max
// keys differ down to the lowest bit that differs between two keys of the
// selected sign (OR ^ AND per sign; integer-valued scores skip their zero
// low mantissa),
// counted in per-warp private histograms (rows with few distinct scores
// would otherwise serialise on a handful of shared bins), and stop as soon
// as the threshold bin is consumed exactly.  The histograms are
// double-buffered (one is cleared while the other is summed) and every warp
// picks the digit from the summed counts itself: two barriers per pass.  The
// ordered sweep builds above / class bit masks, needs one block scan, and is
// staged in shared memory so that the output is written coalesced.
// Longer rows (topk_long_kernel, 1024 threads): keys are re-read from the
// (L2-resident) scores on every pass, three 11/11/10-bit passes, and the
// ordered sweep runs in 1024-element rounds with warp ballots.
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// The FP4 row of selected entry j of row b, requested into L2 for the
// attention launched next (every 128-byte line the row touches; no effect on
// the result).
__device__ __forceinline__ void prefetch_row(const RowPrefetch& pf, int b, int32_t j) {
  if (pf.kv != nullptr && j >= 0 && j < pf.n) {
    const uint8_t* r = pf.kv + (int64_t)(b / pf.q_per_seq) * pf.seq_bytes + (int64_t)j * kRowBytes;
#pragma unroll
    for (int off = 0; off < kRowBytes; off += 128)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(r + off));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(r + kRowBytes - 1));
  }
}

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

// Warp-wide choice of the radix digit that holds the need-th largest key:
// csum[t] = number of keys with digit 255 - t (descending digit order).
// Every warp runs it on the same counts and reaches the same answer, so no
// broadcast (and no barrier) is needed.  Returns the digit; *above = keys in
// larger digits, *cnt = keys with this digit.
__device__ __forceinline__ int select_digit(const int32_t* csum, int need, int* above, int* cnt) {
  const int lane = threadIdx.x & 31;
  const int4 a = reinterpret_cast<const int4*>(csum)[2 * lane];
  const int4 b = reinterpret_cast<const int4*>(csum)[2 * lane + 1];
  const int c[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  int local = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) local += c[j];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int before = incl - local;
  int hit = -1, hit_before = 0, hit_cnt = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (hit < 0 && before < need && before + c[j] >= need) {
      hit = j;
      hit_before = before;
      hit_cnt = c[j];
    }
    before += c[j];
  }
  const unsigned m = __ballot_sync(0xffffffffu, hit >= 0);
  const int src = __ffs(m) - 1;
  const int t = __shfl_sync(0xffffffffu, 8 * lane + hit, src);
  *above = __shfl_sync(0xffffffffu, hit_before, src);
  *cnt = __shfl_sync(0xffffffffu, hit_cnt, src);
  return 255 - t;
}

// The low n bits of a W-bit mask (1 <= n <= W <= 64).
template <int W>
__device__ __forceinline__ uint64_t lo_bits(int n) {
  return n >= 64 ? ~0ull : ((1ull << n) - 1ull);
}
// A W-bit mask (W a power of two, 8..64) rotated left by r (0 <= r < W).
template <int W>
__device__ __forceinline__ uint64_t rot_bits(uint64_t m, int r) {
  if (r == 0) return m;
  const uint64_t all = lo_bits<W>(W);
  return ((m << r) | (m >> (W - r))) & all;
}

// chunk == 0: CTA b selects row b.  chunk > 0 (map must be null): CTA (c, b)
// selects among the candidates [c*chunk, (c+1)*chunk) of row b and writes
// their positions in the row to idx[b][c][0..k) (one level of the long-row
// selection).
template <int KPT>
__global__ void __launch_bounds__(kRegThreads, 1)
topk_reg_kernel(const float* __restrict__ scores, int64_t N, int k,
                const int32_t* __restrict__ q_pos, int ratio, const int32_t* __restrict__ n_valid,
                const int32_t* __restrict__ map, int32_t* __restrict__ idx, int chunk,
                RowPrefetch pf) {
  // two sets of per-warp 8-bit digit histograms: one is counted into while
  // the other is cleared for the next pass; reused to stage the output
  __shared__ __align__(16) int32_t whist[2][kRegWarps * 256];
  __shared__ __align__(16) int32_t csum[256];
  __shared__ int32_t tot[kRegWarps + 1];
  __shared__ uint32_t red[4][kRegWarps];
  __shared__ __align__(8) uint64_t row_bar;  // the row's bulk copy into shared memory
  extern __shared__ __align__(16) uint32_t row_s[];  // KPT * kRegThreads keys (bulk path)

  pdl_trigger();
  pdl_wait();  // scores, n_valid and map come from the kernel before
  const int b = chunk ? blockIdx.y : blockIdx.x;
  const int64_t pos0 = chunk ? (int64_t)blockIdx.x * chunk : 0;  // first entry of the chunk
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* row = scores + (int64_t)b * N + pos0;
  const int32_t* mrow = map ? map + (int64_t)b * N : nullptr;
  int32_t* out = idx + ((int64_t)b * (chunk ? gridDim.x : 1) + (chunk ? blockIdx.x : 0)) * k;

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
  if (chunk) n = (int)max((int64_t)0, min((int64_t)chunk, (int64_t)n - pos0));
  if (n <= k) {
    for (int j = tid; j < k; j += kRegThreads) {
      const int32_t v = (j < n) ? (mrow ? mrow[j] : (int32_t)(pos0 + j)) : -1;
      out[j] = v;
      prefetch_row(pf, b, v);
    }
    return;
  }

  // keys of positions [tid*KPT, tid*KPT + KPT) in registers.  A 16-byte
  // aligned row comes into shared memory with bulk copies (the copy engine
  // fetches it far faster than the threads' own 16-byte loads, each of which
  // touches 32 rows' worth of lines); thread t then reads its 16-byte chunks
  // starting at chunk t mod (KPT / 4), so that eight consecutive threads hit
  // eight different bank groups: key[4 g + e] is position base + 4 ((g + rot)
  // mod (KPT / 4)) + e
  const int base = tid * KPT;
  constexpr int kCh = KPT / 4;  // 16-byte chunks per thread
  uint32_t key[KPT];
  const bool vec = ((N & 3) == 0) && ((reinterpret_cast<uintptr_t>(scores) & 15u) == 0);
  const bool bulk = vec && ((reinterpret_cast<uintptr_t>(row) & 15u) == 0);
  bool staged_row = false;
  if (bulk) {
    const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(&row_bar));
    if (tid == 0) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar));
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const uint32_t bytes = (uint32_t)((n * 4 + 15) & ~15);  // within the row (N % 4 == 0)
    if (tid == 0) {
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                   : "memory");
      const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(row_s));
      for (uint32_t off = 0; off < bytes; off += 16384u) {
        const uint32_t len = min(16384u, bytes - off);
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
            ::"r"(dst + off), "l"(reinterpret_cast<const uint8_t*>(row) + off), "r"(len), "r"(bar)
            : "memory");
      }
    }
    // bounded wait (about 2 s); on a timeout the keys are read from global memory
    const uint64_t t0 = clock64();
    bool done = false;
    while (!done) {
      uint32_t ok;
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(ok)
          : "r"(bar), "r"(0u)
          : "memory");
      done = ok != 0;
      if (!done && clock64() - t0 > 4000000000ll) break;
    }
    staged_row = __syncthreads_and(done);
  }
  const int rot = staged_row ? tid : 0;
  // key-order bits <-> position-order bits: a rotation by whole chunks of the
  // KPT-bit masks (bit 4 g + e of key order is bit 4 ((g + rot) mod kCh) + e
  // of position order)
  auto to_pos = [&](uint64_t m) { return rot_bits<KPT>(m, 4 * (rot & (kCh - 1))); };
  auto to_key = [&](uint64_t m) {
    return rot_bits<KPT>(m, (KPT - 4 * (rot & (kCh - 1))) & (KPT - 1));
  };
  // the valid keys (positions below n), in key order
  const int nv_here = n - base;
  const uint64_t vpos = nv_here >= KPT ? lo_bits<KPT>(KPT)
                                       : (nv_here <= 0 ? 0ull : lo_bits<KPT>(nv_here));
  const uint64_t vkey = to_key(vpos);
  if (staged_row) {
#pragma unroll
    for (int g = 0; g < kCh; ++g) {
      const uint4 u = *reinterpret_cast<const uint4*>(row_s + base + 4 * ((g + rot) & (kCh - 1)));
      key[4 * g + 0] = float_to_ordered(__uint_as_float(u.x));
      key[4 * g + 1] = float_to_ordered(__uint_as_float(u.y));
      key[4 * g + 2] = float_to_ordered(__uint_as_float(u.z));
      key[4 * g + 3] = float_to_ordered(__uint_as_float(u.w));
    }
  } else {
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
  }

  // OR / AND of the keys, per sign of the score.  Over the whole row they
  // give the highest differing bit (where the passes start) and the common
  // prefix above it.  Once the sign is decided (the first pass covers it when
  // both occur), bits below the lowest one that differs among keys of that
  // sign (the zero low mantissa of integer-valued scores, say) are never
  // counted.
  uint32_t por = 0u, pand = 0xFFFFFFFFu, nor = 0u, nand = 0xFFFFFFFFu;  // >= 0 / < 0
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const uint32_t valid = ((vkey >> i) & 1u) ? 0xFFFFFFFFu : 0u;
    const uint32_t pos = valid & (0u - (key[i] >> 31));  // all ones for a valid key >= 0
    const uint32_t neg = valid & ~pos;
    por |= key[i] & pos;
    pand &= key[i] | ~pos;
    nor |= key[i] & neg;
    nand &= key[i] | ~neg;
  }
  por = __reduce_or_sync(0xffffffffu, por);
  pand = __reduce_and_sync(0xffffffffu, pand);
  nor = __reduce_or_sync(0xffffffffu, nor);
  nand = __reduce_and_sync(0xffffffffu, nand);
  if (lane == 0) {
    red[0][warp] = por;
    red[1][warp] = pand;
    red[2][warp] = nor;
    red[3][warp] = nand;
  }
  for (int i = tid; i < kRegWarps * 256; i += kRegThreads) whist[0][i] = 0;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kRegWarps; ++w) {
    por |= red[0][w];
    pand &= red[1][w];
    nor |= red[2][w];
    nand &= red[3][w];
  }
  // lowest differing bit among the keys of one sign (32: they are all equal)
  const int lo_pos = (por ^ pand) ? __ffs(por ^ pand) - 1 : 32;
  const int lo_neg = (nor ^ nand) ? __ffs(nor ^ nand) - 1 : 32;
  const uint32_t kor = por | nor, kand = pand & nand;  // over the whole row

  uint32_t prefix = kand, mask = 0xFFFFFFFFu;  // all keys equal: one class
  int cur_hi = -1, lo = 0;
  if (kor != kand) {
    cur_hi = 31 - __clz(kor ^ kand);
    mask = ~((2u << cur_hi) - 1u);  // cur_hi = 31: 2u << 31 wraps to 0, mask = 0
    prefix = kand & mask;
    // both signs present: bit 31 itself differs, so the first pass covers it
    lo = min(cur_hi, cur_hi == 31 ? min(lo_pos, lo_neg) : ((kor >> 31) ? lo_pos : lo_neg));
  }
  int need = k;
  for (int pass = 0; cur_hi >= lo; ++pass) {
    const int nbits = min(8, cur_hi + 1 - lo);
    const int shift = cur_hi + 1 - nbits;
    const uint32_t dmask = (1u << nbits) - 1u;
    int32_t* hist = whist[pass & 1];
    int32_t* my_hist = hist + warp * 256;  // this warp's private histogram
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      if (((vkey >> i) & 1u) && (key[i] & mask) == prefix)
        atomicAdd(&my_hist[(key[i] >> shift) & dmask], 1);
    }
    __syncthreads();
    if (tid < 256) {
      // thread t sums digit 255 - t over the warps (descending order for the scan)
      const int d = 255 - tid;
      int c = 0;
#pragma unroll
      for (int w = 0; w < kRegWarps; ++w) c += hist[w * 256 + d];
      csum[tid] = c;
    } else {
      int32_t* next = whist[(pass + 1) & 1];
      for (int i = tid - 256; i < kRegWarps * 256; i += kRegThreads - 256) next[i] = 0;
    }
    __syncthreads();
    int above, cnt;
    const int digit = select_digit(csum, need, &above, &cnt);
    need -= above;
    prefix |= (uint32_t)digit << shift;
    mask |= dmask << shift;
    cur_hi = shift - 1;
    lo = (prefix >> 31) ? lo_pos : lo_neg;  // the sign bit is decided now
    if (cnt == need) break;  // the whole class is taken
  }
  // (keys agree on every bit below `lo`, so comparing on the bits of `mask`
  // orders them completely)

  // ordered write: every key above the class (key & mask > prefix), then the
  // first `need` class members in position order.  One scan of the two
  // counts packed in 16-bit halves (n <= 32768) gives both prefixes; the
  // class members taken before this thread are min(eq_before, need).
  // key-order masks, then bit b: position base + b (the chunk rotation undone)
  uint64_t g64 = 0u, e64 = 0u;
#pragma unroll
  for (int ii = 0; ii < KPT; ++ii) {
    const uint32_t km = key[ii] & mask;
    g64 |= (uint64_t)(km > prefix) << ii;
    e64 |= (uint64_t)(km == prefix) << ii;
  }
  g64 = to_pos(g64 & vkey);
  e64 = to_pos(e64 & vkey);
  uint32_t gtm[(KPT + 31) / 32], eqm[(KPT + 31) / 32];
  int gt = 0, eq = 0;
#pragma unroll
  for (int w = 0; w < (KPT + 31) / 32; ++w) {
    gtm[w] = (uint32_t)(g64 >> (32 * w));
    eqm[w] = (uint32_t)(e64 >> (32 * w));
    gt += __popc(gtm[w]);
    eq += __popc(eqm[w]);
  }
  int tot_packed;
  const int before = reg_block_scan((gt << 16) | eq, tot, &tot_packed);
  const int eq_before = before & 0xFFFF;
  int take = max(0, min(eq, need - eq_before));
  int off = (before >> 16) + min(eq_before, need);
  const bool staged = k <= 2 * kRegWarps * 256;
  int32_t* stage = &whist[0][0];
#pragma unroll
  for (int w = 0; w < (KPT + 31) / 32; ++w) {
    uint32_t sel = gtm[w];
    for (uint32_t c = eqm[w]; take > 0 && c != 0u; --take) {
      sel |= c & (~c + 1u);  // lowest remaining class member
      c &= c - 1u;
    }
    while (sel != 0u && off < k) {
      const int p = base + 32 * w + __ffs(sel) - 1;
      sel &= sel - 1u;
      if (staged) {
        stage[off] = p;
      } else {
        const int32_t v = mrow ? mrow[p] : (int32_t)(pos0 + p);
        out[off] = v;
        prefetch_row(pf, b, v);
      }
      ++off;
    }
  }
  if (staged) {
    __syncthreads();
    for (int j = tid; j < k; j += kRegThreads) {
      const int32_t p = stage[j];
      const int32_t v = mrow ? mrow[p] : (int32_t)(pos0 + p);
      out[j] = v;
      prefetch_row(pf, b, v);
    }
  }
}

// ---------------------------------------------------------------------------
// Cluster variant for batches too small to fill the GPU one row per CTA: a
// cluster of CL CTAs shares a row, CTA r holding the KPT * kRegThreads keys
// from position r * KPT * kRegThreads on.  Every step that needs the whole row
// (OR / AND of the keys, each pass's digit counts, the counts of keys above
// and inside the threshold class before each CTA) is exchanged through
// distributed shared memory: a CTA publishes its values in its own shared
// memory, one cluster barrier (release / acquire) makes them visible, and
// every CTA reads all CL copies, so all of them take the same decisions.  The
// per-pass counts are double-buffered: a buffer is rewritten two passes
// later, after the next barrier has shown that every peer has read it.  From
// the same per-peer counts each CTA also accumulates how many keys above the
// class, and inside it, its lower-ranked peers hold: its output offsets.  The
// last barrier is split: a CTA arrives once it has read its peers for the
// last time and waits (so that its own shared memory outlives their reads)
// only after writing its output.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Sum of one int per thread over the first 256 threads (8 warps) of the
// block; `scratch` holds 8 ints.  Every thread gets the total.  Ends with a
// barrier of the whole block.
__device__ __forceinline__ int sum256(int v, int32_t* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_add_sync(0xffffffffu, v);
  if (warp < 8 && lane == 0) scratch[warp] = v;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) t += scratch[w];
  __syncthreads();
  return t;
}

// The shared-memory word at `p` (this CTA's address) in cluster CTA `rank`.
__device__ __forceinline__ uint32_t ld_peer(const void* p, uint32_t rank) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p)), ra, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
  return v;
}

template <int KPT, int CL>
__global__ void __launch_bounds__(kRegThreads, 1)
topk_cluster_kernel(const float* __restrict__ scores, int64_t N, int k,
                    const int32_t* __restrict__ q_pos, int ratio,
                    const int32_t* __restrict__ n_valid, const int32_t* __restrict__ map,
                    int32_t* __restrict__ idx, RowPrefetch pf) {
  __shared__ __align__(16) int32_t whist[2][kRegWarps * 256];
  __shared__ __align__(16) int32_t csum[256];
  __shared__ __align__(16) int32_t pub[2][256];  // this CTA's digit counts (descending digits)
  __shared__ uint32_t pub_bits[4];               // this CTA's OR / AND per sign
  __shared__ uint32_t all_bits[4 * CL];
  __shared__ int32_t red8[1][8];
  __shared__ int32_t tot[kRegWarps + 1];
  __shared__ uint32_t red[4][kRegWarps];

  pdl_trigger();
  pdl_wait();  // scores, n_valid and map come from the kernel before
  const int b = blockIdx.y;
  const uint32_t rank = cluster_ctarank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* row = scores + (int64_t)b * N;
  const int32_t* mrow = map ? map + (int64_t)b * N : nullptr;
  int32_t* out = idx + (int64_t)b * k;

  const int base = (int)rank * (KPT * kRegThreads) + tid * KPT;  // row position of key[0]
  uint32_t key[KPT];
  const bool vec = ((N & 3) == 0) && ((reinterpret_cast<uintptr_t>(scores) & 15u) == 0);
  // the whole row range (entries n .. N - 1 are read, never counted): the
  // loads need not wait for the candidate count
#pragma unroll
  for (int i = 0; i < KPT; i += 4) {
    const int j = base + i;
    float v[4];
    if (vec && j + 3 < N) {
      const float4 f = *reinterpret_cast<const float4*>(row + j);
      v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = (j + e < N) ? row[j + e] : 0.0f;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) key[i + e] = float_to_ordered(v[e]);
  }

  int n;  // candidates of the row, the same in every CTA of the cluster
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
  if (n <= k) {  // the whole cluster leaves here together
    if (rank == 0)
      for (int j = tid; j < k; j += kRegThreads) {
        const int32_t v = (j < n) ? (mrow ? mrow[j] : j) : -1;
        out[j] = v;
        prefetch_row(pf, b, v);
      }
    return;
  }

  // OR / AND of the keys per sign (see topk_reg_kernel), over the cluster.
  // They travel with the first pass, which takes the fixed top digit (bits
  // 31..24) of every candidate: one cluster exchange fewer than finding the
  // differing bit range first.
  uint32_t por = 0u, pand = 0xFFFFFFFFu, nor = 0u, nand = 0xFFFFFFFFu;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const uint32_t valid = base + i < n ? 0xFFFFFFFFu : 0u;
    const uint32_t pos = valid & (0u - (key[i] >> 31));
    const uint32_t neg = valid & ~pos;
    por |= key[i] & pos;
    pand &= key[i] | ~pos;
    nor |= key[i] & neg;
    nand &= key[i] | ~neg;
  }
  por = __reduce_or_sync(0xffffffffu, por);
  pand = __reduce_and_sync(0xffffffffu, pand);
  nor = __reduce_or_sync(0xffffffffu, nor);
  nand = __reduce_and_sync(0xffffffffu, nand);
  if (lane == 0) {
    red[0][warp] = por;
    red[1][warp] = pand;
    red[2][warp] = nor;
    red[3][warp] = nand;
  }
  for (int i = tid; i < kRegWarps * 256; i += kRegThreads) whist[0][i] = 0;
  __syncthreads();
  {
    int32_t* my_hist = whist[0] + warp * 256;
#pragma unroll
    for (int i = 0; i < KPT; ++i)
      if (base + i < n) atomicAdd(&my_hist[key[i] >> 24], 1);
  }
  if (tid < 4) {
    uint32_t v = (tid & 1) ? 0xFFFFFFFFu : 0u;
#pragma unroll
    for (int w = 0; w < kRegWarps; ++w) v = (tid & 1) ? (v & red[tid][w]) : (v | red[tid][w]);
    pub_bits[tid] = v;
  }

  int need = k;
  // this thread's share (digit 255 - tid) of the keys above the class / inside
  // it held by the lower-ranked CTAs, summed over the block after the passes
  int gt_part = 0, eq_part = 0;
  bool any_pass = false;
  uint32_t prefix = 0u, mask = 0u;
  int cur_hi = 31, lo = 0;
  for (int pass = 0; cur_hi >= lo; ++pass) {
    const int nbits = pass == 0 ? 8 : min(8, cur_hi + 1 - lo);
    const int shift = cur_hi + 1 - nbits;
    const uint32_t dmask = (1u << nbits) - 1u;
    int32_t* hist = whist[pass & 1];
    if (pass > 0) {
      int32_t* my_hist = hist + warp * 256;
#pragma unroll
      for (int i = 0; i < KPT; ++i) {
        if (base + i < n && (key[i] & mask) == prefix)
          atomicAdd(&my_hist[(key[i] >> shift) & dmask], 1);
      }
    }
    __syncthreads();
    if (tid < 256) {
      const int d = 255 - tid;
      int c = 0;
#pragma unroll
      for (int w = 0; w < kRegWarps; ++w) c += hist[w * 256 + d];
      pub[pass & 1][tid] = c;
    } else {
      int32_t* next = whist[(pass + 1) & 1];
      for (int i = tid - 256; i < kRegWarps * 256; i += kRegThreads - 256) next[i] = 0;
    }
    cluster_barrier();
    if (pass == 0 && tid >= 256 && tid < 256 + 4 * CL)
      all_bits[tid - 256] = ld_peer(&pub_bits[(tid - 256) & 3], (uint32_t)((tid - 256) >> 2));
    int lower = 0;  // this digit's count in the lower-ranked CTAs
    if (tid < 256) {
      int c = 0;
#pragma unroll
      for (int r = 0; r < CL; ++r) {
        const int v = (int)ld_peer(&pub[pass & 1][tid], (uint32_t)r);
        c += v;
        if (r < (int)rank) lower += v;
      }
      csum[tid] = c;
    }
    __syncthreads();
    int above, cnt;
    const int digit = select_digit(csum, need, &above, &cnt);
    const int tsel = 255 - digit;
    gt_part += tid < tsel ? lower : 0;
    eq_part = tid == tsel ? lower : 0;
    any_pass = true;
    need -= above;
    prefix |= (uint32_t)digit << shift;
    mask |= dmask << shift;
    cur_hi = shift - 1;
    if (pass == 0) {  // the lowest bit that differs between two keys, per sign
      por = 0u; pand = 0xFFFFFFFFu; nor = 0u; nand = 0xFFFFFFFFu;
#pragma unroll
      for (int r = 0; r < CL; ++r) {
        por |= all_bits[4 * r];
        pand &= all_bits[4 * r + 1];
        nor |= all_bits[4 * r + 2];
        nand &= all_bits[4 * r + 3];
      }
    }
    const int lo_pos = (por ^ pand) ? __ffs(por ^ pand) - 1 : 32;
    const int lo_neg = (nor ^ nand) ? __ffs(nor ^ nand) - 1 : 32;
    lo = (prefix >> 31) ? lo_pos : lo_neg;
    if (cnt == need) break;
  }
  cluster_arrive_relaxed();  // this CTA reads no peer any more
  // both sums are below 2^15 (the lower ranks hold fewer than 32768 keys),
  // so one packed reduction carries them; with no pass (all keys equal) the
  // class is every valid key
  const int packed = sum256((gt_part << 16) | eq_part, red8[0]);
  const int gt_lower = packed >> 16;
  const int eq_lower =
      any_pass ? (packed & 0xFFFF) : (int)min((int64_t)n, (int64_t)rank * (KPT * kRegThreads));

  // ordered write (see topk_reg_kernel), offset by the keys above / inside
  // the class held by the lower-ranked CTAs of the cluster
  uint32_t gtm[(KPT + 31) / 32], eqm[(KPT + 31) / 32];
  int gt = 0, eq = 0;
#pragma unroll
  for (int w = 0; w < (KPT + 31) / 32; ++w) {
    uint32_t g = 0u, e = 0u;
#pragma unroll
    for (int i = 0; i < 32 && 32 * w + i < KPT; ++i) {
      const int ii = 32 * w + i;
      const uint32_t km = key[ii] & mask;
      const bool valid = base + ii < n;
      g |= (uint32_t)(valid && km > prefix) << i;
      e |= (uint32_t)(valid && km == prefix) << i;
    }
    gtm[w] = g;
    eqm[w] = e;
    gt += __popc(g);
    eq += __popc(e);
  }
  int tot_packed;
  const int before = reg_block_scan((gt << 16) | eq, tot, &tot_packed);
  const int eq_before = eq_lower + (before & 0xFFFF);
  int take = max(0, min(eq, need - eq_before));
  int off = gt_lower + (before >> 16) + min(eq_before, need);
#pragma unroll
  for (int w = 0; w < (KPT + 31) / 32; ++w) {
    uint32_t sel = gtm[w];
    for (uint32_t c = eqm[w]; take > 0 && c != 0u; --take) {
      sel |= c & (~c + 1u);
      c &= c - 1u;
    }
    while (sel != 0u && off < k) {
      const int p = base + 32 * w + __ffs(sel) - 1;
      sel &= sel - 1u;
      const int32_t v = mrow ? mrow[p] : p;
      out[off] = v;
      prefetch_row(pf, b, v);
      ++off;
    }
  }
  cluster_wait();  // the peers' last reads of this CTA's shared memory are done
}

template <bool kSmem>
__global__ void __launch_bounds__(kThreads, 1)
topk_long_kernel(const float* __restrict__ scores, int64_t N, int k, const int32_t* __restrict__ q_pos,
            int ratio, const int32_t* __restrict__ n_valid, const int32_t* __restrict__ map,
            int32_t* __restrict__ idx, RowPrefetch pf) {
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
      prefetch_row(pf, b, v);
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
    if (take && pos < k) {
      const int32_t v = mrow ? mrow[j] : j;
      out[pos] = v;
      prefetch_row(pf, b, v);
    }
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

namespace {

// One level of the long-row selection, second half: the chunks' selections
// (each a valid prefix of k positions, -1 after) are packed in chunk order --
// so in ascending position order -- with their scores and entry ids
// (ids_in[pos], or pos itself at the first level); slots past the packed
// count get id -1.  count[b] = packed candidates of row b.
__global__ void __launch_bounds__(256)
topk_pack_kernel(const float* __restrict__ scores, int64_t M_in, const int32_t* __restrict__ ids_in,
                 const int32_t* __restrict__ sel, int C, int k, float* __restrict__ score_out,
                 int32_t* __restrict__ id_out, int32_t* __restrict__ count) {
  pdl_trigger();
  pdl_wait();  // the chunk selections come from the kernel before
  __shared__ int32_t off[65];
  const int b = blockIdx.x;
  const int32_t* s = sel + (int64_t)b * C * k;
  if (threadIdx.x < C) {
    // valid prefix length of chunk c: binary search for the first -1
    const int32_t* sc = s + (int64_t)threadIdx.x * k;
    int lo = 0, hi = k;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sc[mid] >= 0) lo = mid + 1; else hi = mid;
    }
    off[threadIdx.x + 1] = lo;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    off[0] = 0;
    for (int c = 0; c < C; ++c) off[c + 1] += off[c];
    count[b] = off[C];
  }
  __syncthreads();
  const int M = C * k;
  float* so = score_out + (int64_t)b * M;
  int32_t* io = id_out + (int64_t)b * M;
  for (int j = threadIdx.x; j < M; j += blockDim.x) {
    const int c = j / k, t = j % k;
    if (t < off[c + 1] - off[c]) {
      const int32_t pos = s[j];
      so[off[c] + t] = scores[(int64_t)b * M_in + pos];
      io[off[c] + t] = ids_in ? ids_in[(int64_t)b * M_in + pos] : pos;
    }
    if (j >= off[C]) io[j] = -1;
  }
}

// Rows longer than one register CTA holds are cut into chunks of kRegMaxKeys
// entries: every member of the row's top-k is in its chunk's top-k (the
// ranking inside a chunk is the row's ranking), so the top-k of the union of
// the chunk selections, taken in entry order, is the row's top-k.  Levels
// repeat until the union fits one CTA (each shrinks the row by at least
// kRegMaxKeys / k >= 2 for k <= 16384).
int long_chunks(int64_t N) { return (int)((N + kRegMaxKeys - 1) / kRegMaxKeys); }
bool chunked_ok(int64_t N, int k) {
  return N > kRegMaxKeys && long_chunks(N) <= 64 && k <= kRegMaxKeys / 2;
}

template <int KPT>
cudaError_t launch_reg(dim3 grid, const float* scores, int64_t N, int k, const int32_t* q_pos,
                       int ratio, const int32_t* n_valid, const int32_t* map, int32_t* idx,
                       int chunk, cudaStream_t stream, bool pdl, const RowPrefetch& pf) {
  // the row's keys staged in shared memory (bulk copies)
  const size_t row_bytes = (size_t)KPT * kRegThreads * 4;
  cudaError_t e = cudaFuncSetAttribute(topk_reg_kernel<KPT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)row_bytes);
  if (e != cudaSuccess) return e;
  return launch_kernel(topk_reg_kernel<KPT>, grid, dim3(kRegThreads), row_bytes, stream, pdl,
                       scores, N, k, q_pos, ratio, n_valid, map, idx, chunk, pf);
}

template <int KPT, int CL>
cudaError_t launch_cluster(int B, const float* scores, int64_t N, int k, const int32_t* q_pos,
                           int ratio, const int32_t* n_valid, const int32_t* map, int32_t* idx,
                           cudaStream_t stream, bool pdl, const RowPrefetch& pf) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, (unsigned)B);
  cfg.blockDim = dim3(kRegThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, topk_cluster_kernel<KPT, CL>, scores, N, k, q_pos, ratio,
                            n_valid, map, idx, pf);
}

template <int CL>
cudaError_t launch_cluster_kpt(int kpt, int B, const float* scores, int64_t N, int k,
                               const int32_t* q_pos, int ratio, const int32_t* n_valid,
                               const int32_t* map, int32_t* idx, cudaStream_t stream, bool pdl,
                               const RowPrefetch& pf) {
  switch (kpt) {
    case 4: return launch_cluster<4, CL>(B, scores, N, k, q_pos, ratio, n_valid, map, idx, stream, pdl, pf);
    case 8: return launch_cluster<8, CL>(B, scores, N, k, q_pos, ratio, n_valid, map, idx, stream, pdl, pf);
    case 16: return launch_cluster<16, CL>(B, scores, N, k, q_pos, ratio, n_valid, map, idx, stream, pdl, pf);
    default: return launch_cluster<32, CL>(B, scores, N, k, q_pos, ratio, n_valid, map, idx, stream, pdl, pf);
  }
}

// Rows of <= 32768 candidates when one CTA per row leaves SMs idle: a cluster
// of 8 (B <= SMs / 8), 4 (B <= SMs / 4) or 2 (B <= SMs / 2) CTAs per row.
// Rows too short to give every CTA 2048 keys use fewer CTAs (or one): below
// that the cluster barriers cost more than the split saves.  Returns false
// when the shape does not qualify.
bool cluster_launch(int B, const float* scores, int64_t N, int k, const int32_t* q_pos,
                    int ratio, const int32_t* n_valid, const int32_t* map, int32_t* idx,
                    cudaStream_t stream, bool pdl, cudaError_t* err, const RowPrefetch& pf) {
  const int sms = device_sm_count();
  int CL = 0;
  for (int c = 8; c >= 2 && CL == 0; c >>= 1)
    if (B * c <= sms && N >= (int64_t)c * 2048) CL = c;
  if (CL == 0 || N > kRegMaxKeys) return false;
  const int64_t per = (N + CL - 1) / CL;  // keys per CTA
  int kpt = 4;
  while ((int64_t)kpt * kRegThreads < per) kpt *= 2;
  if (kpt > 32) return false;
  *err = CL == 8 ? launch_cluster_kpt<8>(kpt, B, scores, N, k, q_pos, ratio, n_valid, map, idx,
                                          stream, pdl, pf)
       : CL == 4 ? launch_cluster_kpt<4>(kpt, B, scores, N, k, q_pos, ratio, n_valid, map, idx,
                                          stream, pdl, pf)
                 : launch_cluster_kpt<2>(kpt, B, scores, N, k, q_pos, ratio, n_valid, map, idx,
                                          stream, pdl, pf);
  return true;
}

cudaError_t launch_reg_any(dim3 grid, const float* scores, int64_t N, int64_t keys, int k,
                           const int32_t* q_pos, int ratio, const int32_t* n_valid,
                           const int32_t* map, int32_t* idx, int chunk, cudaStream_t stream,
                           bool pdl, const RowPrefetch& pf) {
  if (keys <= kRegThreads * 8)
    return launch_reg<8>(grid, scores, N, k, q_pos, ratio, n_valid, map, idx, chunk, stream, pdl, pf);
  if (keys <= kRegThreads * 16)
    return launch_reg<16>(grid, scores, N, k, q_pos, ratio, n_valid, map, idx, chunk, stream, pdl, pf);
  if (keys <= kRegThreads * 32)
    return launch_reg<32>(grid, scores, N, k, q_pos, ratio, n_valid, map, idx, chunk, stream, pdl, pf);
  return launch_reg<64>(grid, scores, N, k, q_pos, ratio, n_valid, map, idx, chunk, stream, pdl, pf);
}

struct LongScratch {
  int32_t* sel;        // [B][C1 * k] chunk selections
  float* score[2];     // ping-pong packed candidates
  int32_t* id[2];
  int32_t* count[2];   // [B]
};

size_t long_scratch(void* base, int B, int64_t N, int k, LongScratch* ls) {
  const size_t M = (size_t)long_chunks(N) * k;
  const size_t a = align_up((size_t)B * M * 4, 256), c = align_up((size_t)B * 4, 256);
  if (ls) {
    uint8_t* p = reinterpret_cast<uint8_t*>(base);
    ls->sel = reinterpret_cast<int32_t*>(p);
    for (int i = 0; i < 2; ++i) {
      ls->score[i] = reinterpret_cast<float*>(p + a + i * (2 * a + c));
      ls->id[i] = reinterpret_cast<int32_t*>(p + 2 * a + i * (2 * a + c));
      ls->count[i] = reinterpret_cast<int32_t*>(p + 3 * a + i * (2 * a + c));
    }
  }
  return a + 2 * (2 * a + c);
}

}  // namespace

size_t topk_scratch_bytes(int B, int64_t N, int k) {
  if (B <= 0 || k < 1 || !chunked_ok(N, k)) return 0;
  return long_scratch(nullptr, B, N, k, nullptr);
}

int topk_launches(int B, int64_t N, int k, size_t scratch_bytes) {
  if (B <= 0) return 0;
  const size_t need = topk_scratch_bytes(B, N, k);
  if (need == 0 || scratch_bytes < need) return 1;
  int n = 1;
  for (int64_t M = N; M > kRegMaxKeys; M = (int64_t)long_chunks(M) * k) n += 2;
  return n;
}

cudaError_t launch_topk(const float* scores, int B, int64_t N, int k, const int32_t* q_pos,
                        int ratio, const int32_t* n_valid, const int32_t* map, int32_t* idx,
                        cudaStream_t stream, bool pdl, void* scratch, size_t scratch_bytes,
                        const RowPrefetch& pf) {
  if (B == 0) return cudaSuccess;
  if (N <= kRegMaxKeys) {
    cudaError_t e;
    if (cluster_launch(B, scores, N, k, q_pos, ratio, n_valid, map, idx, stream, pdl, &e, pf))
      return e;
    return launch_reg_any(dim3((unsigned)B), scores, N, N, k, q_pos, ratio, n_valid, map, idx, 0,
                          stream, pdl, pf);
  }
  const size_t need = topk_scratch_bytes(B, N, k);
  if (!map && need > 0 && scratch && scratch_bytes >= need) {
    LongScratch ls;
    long_scratch(scratch, B, N, k, &ls);
    const float* cur_score = scores;
    const int32_t* cur_id = nullptr;       // ids of the current candidates (null: positions)
    const int32_t* cur_count = n_valid;    // candidates per row (null: visibility via q_pos)
    const int32_t* cur_pos = q_pos;
    int cur_ratio = ratio;
    int64_t M = N;
    cudaError_t e = cudaSuccess;
    for (int lvl = 0; M > kRegMaxKeys; ++lvl) {
      const int C = long_chunks(M);
      e = launch_reg_any(dim3((unsigned)C, (unsigned)B), cur_score, M, kRegMaxKeys, k, cur_pos,
                         cur_ratio, cur_count, nullptr, ls.sel, kRegMaxKeys, stream,
                         lvl == 0 ? pdl : true, RowPrefetch{});
      if (e != cudaSuccess) return e;
      const int o = lvl & 1;
      e = launch_kernel(topk_pack_kernel, dim3((unsigned)B), dim3(256), 0, stream, true, cur_score,
                        M, cur_id, ls.sel, C, k, ls.score[o], ls.id[o], ls.count[o]);
      if (e != cudaSuccess) return e;
      cur_score = ls.score[o];
      cur_id = ls.id[o];
      cur_count = ls.count[o];
      cur_pos = nullptr;
      cur_ratio = 1;
      M = (int64_t)C * k;
    }
    // the packed ids serve as the map: the selected candidates' entry ids
    if (cluster_launch(B, cur_score, M, k, nullptr, 1, nullptr, cur_id, idx, stream, true, &e, pf))
      return e;
    return launch_reg_any(dim3((unsigned)B), cur_score, M, M, k, nullptr, 1, nullptr, cur_id, idx,
                          0, stream, true, pf);
  }
  const size_t base = align_up(sizeof(TopkShared), 16);
  return launch_kernel(topk_long_kernel<false>, dim3((unsigned)B), dim3(kThreads), base, stream,
                       pdl, scores, N, k, q_pos, ratio, n_valid, map, idx, pf);
}

}  // namespace csa2
