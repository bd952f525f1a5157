// Sparse MQA attention over the selected FP4 entries on the 5th-generation
// tensor cores (DeepSeek-V4.1-Flash paper walkthrough, 1.(4) "CSA2": each
// query attends its selected main-KV entries; 1.(5).4: the FP4 cache is
// dequantised before attention; 2.(2).1: 64 query heads x 512).  K = V = the
// dequantised 512-channel latent shared by the heads.
//
// One CTA = one query x a chunk of its selected slots, in tiles of 128
// entries.  The problem is computed transposed so that the 128 entries of a
// tile fill the M = 128 rows of a tcgen05.mma:
//   S^T[e][h]  = sum_c V[e][c] Q[h][c]         A = V tile (K-major, SW128)
//   O^T[c][h] += sum_e V[e][c] P[h][e]         A = the same V bytes read as an
//                                              MN-major operand, 4 x 128 rows
// B operands (Q, P) are K-major SW128 tiles in shared memory; both
// accumulators live in tensor memory (O^T: 4 x H columns, S^T: H columns).
//
// Warp roles (512 threads):
//   warps 0-7   softmax + epilogue: thread = TMEM lane = entry (S) / channel
//               (O), warps w and w + 4 share lanes and split the 64 heads;
//               warp 0 allocates TMEM and its lane 0 issues every MMA
//   warps 8-15  dequantisers: each thread loads half of one FP4 row (144 B)
//               straight from global memory one tile ahead, converts E2M1 x
//               E4M3 to fp16 (exact) and stores it into the swizzled V tile
// Per tile: dequant V (per 64-channel atom, signalled by mbarriers) -> S^T
// MMAs -> online softmax (fp32, exp2, lazy rescale: the reference max moves
// only when a tile max exceeds it by more than 2^8 in the exp2 domain, so P
// <= 256 stays in fp16 range and O is rarely touched) -> P (fp16) to smem ->
// O^T MMAs -> next tile.  All mbarrier waits are bounded (about 2 s of
// %globaltimer); a wait that gives up sets the timeout status bit and the CTA
// drains and exits, freeing its tensor memory.
#include "csa2_internal.cuh"
#include "tc_common.cuh"

namespace csa2 {
namespace {

using namespace tc;

constexpr int kSoftWarps = 8;                  // warps 0-7 (warp 0 lane 0 also issues the MMAs)
constexpr int kDeqWarp0 = 8;                   // warps 8-15
constexpr int kThreadsTc = 16 * 32;
constexpr int kTileE = 128;
constexpr int kHN = 64;                        // MMA N: heads, zero-padded to 64
constexpr int kIdxCache = 2048;                // slots of the CTA's chunk kept in smem

struct TcLayout {
  static constexpr uint32_t q_atom = kHN * 128;           // [8 atoms][64 rows][128 B]
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t v_atom = kTileE * 128;        // [8 atoms][128 rows][128 B]
  static constexpr uint32_t v_off = q_off + 8 * q_atom;
  static constexpr uint32_t p_off = v_off + 8 * v_atom;   // [128 rows][128 B] (MN-major B)
  static constexpr uint32_t idx_off = p_off + kTileE * 128;
  static constexpr uint32_t ctl_off = idx_off + kIdxCache * 4;
  static constexpr uint32_t bytes = ctl_off + 4096;
  static constexpr uint32_t alloc = bytes + 1024;         // slack to align the base to 1 KiB
};

struct TcCtl {
  uint64_t bar_v[8];    // V atom a of the current tile written (4 dequant-warp arrivals)
  uint64_t bar_s;       // S^T MMAs done (commit)
  uint64_t bar_p;       // P written and O rescaled (8 softmax-warp arrivals)
  uint64_t bar_o[4];    // O^T MMAs of M-block mb done (commit)
  uint32_t tmem_base;
  int32_t exceed[2];    // some logit of the tile passed its head's reference max (+ margin)
  int32_t rescale;
  float red[4][kHN];    // per entry-warp partial max / sum per head
  float mref[kHN];      // reference max per head (raw logit units)
  float alpha[kHN];     // rescale factor of the current tile per head
  float linv[kHN];      // 1 / row sum per head (epilogue)
};

// Butterfly transpose-reduce of 32 values over the 32 lanes of a warp: lane l
// ends up with element l reduced over all lanes.
template <bool kMax>
__device__ __forceinline__ float warp_reduce32(float* v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < o) {
        const float mine = upper ? v[i + o] : v[i];
        const float send = upper ? v[i] : v[i + o];
        const float other = __shfl_xor_sync(0xffffffffu, send, o);
        v[i] = kMax ? fmaxf(mine, other) : mine + other;
      }
    }
  }
  return v[0];
}

__device__ __forceinline__ void softmax_bar() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// SWA branch (swa_kv non-null): the CTA of the last chunk of query b also
// attends the query's sliding window of the layer's SWA KV (E4M3 rows, per
// sequence a ring with token t at row t mod swa_ring; window
// max(0, pos - n_win + 1) .. pos) as extra tiles after its selected entries,
// in the same online softmax; the split-k merge then combines everything
// into one softmax over both sets.
template <int H>
__global__ void __launch_bounds__(kThreadsTc, 1)
sparse_attn_tc_kernel(const uint16_t* __restrict__ q_bf16, const uint8_t* __restrict__ kv_fp4,
                      int64_t N, int64_t kv_seq_stride, int q_per_seq,
                      const int32_t* __restrict__ idx, int k, int chunk, float scale_log2,
                      float* __restrict__ out, float* __restrict__ lse, float* __restrict__ part_o,
                      float* __restrict__ part_lse, int32_t* status,
                      const uint8_t* __restrict__ swa_kv, int64_t swa_ring, int n_win,
                      const int32_t* __restrict__ q_pos, int32_t* __restrict__ idx_copy) {
  using L = TcLayout;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = su32(smem_raw);
  const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_s + pad;
  TcCtl& ctl = *reinterpret_cast<TcCtl*>(smem + L::ctl_off);
  int32_t* idx_s = reinterpret_cast<int32_t*>(smem + L::idx_off);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.y, split = blockIdx.x, nsplit = gridDim.x;
  const int s0 = split * chunk;
  const int s1 = min(k, s0 + chunk);
  const int cnt = max(0, s1 - s0);
  const int nmain = (cnt + kTileE - 1) / kTileE;  // tiles of selected entries
  // the query's SWA window: tiles [nmain, ntiles) of the last chunk's CTA
  int64_t w0 = 0;
  int wcnt = 0;
  if (swa_kv && split == nsplit - 1) {
    const int64_t pos = q_pos[b];
    w0 = pos - n_win + 1 > 0 ? pos - n_win + 1 : 0;
    wcnt = pos >= 0 ? (int)(pos - w0 + 1) : 0;
  }
  const int ntiles = nmain + (wcnt + kTileE - 1) / kTileE;
  const uint8_t* swaseq = swa_kv ? swa_kv + (int64_t)(b / q_per_seq) * swa_ring * kD : nullptr;
  const int32_t* slots = idx + (int64_t)b * k + s0;
  const uint8_t* kvseq = kv_fp4 + (int64_t)(b / q_per_seq) * kv_seq_stride * kRowBytes;
  const uint32_t q_s = sbase + L::q_off, v_s = sbase + L::v_off, p_s = sbase + L::p_off;
  // slot s of this chunk (s < cnt): entry id, -1 if empty
  auto slot_at = [&](int s) -> int32_t { return s < kIdxCache ? idx_s[s] : slots[s]; };

  pdl_trigger();
  // ---- prologue: Q (bf16 -> fp16, swizzled, zero-padded to 64 rows), TMEM,
  //      barriers; then (once the kernel that selected them has finished) the
  //      slot indices ----
  {
    constexpr int kQChunks = kHN * (kD / 8);
    constexpr int kPer = (kQChunks + kThreadsTc - 1) / kThreadsTc;
    const uint4* qsrc = reinterpret_cast<const uint4*>(q_bf16 + (int64_t)b * H * kD);
    uint4 qv[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int c = tid + i * kThreadsTc;
      qv[i] = (c < H * (kD / 8)) ? __ldg(qsrc + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int c = tid + i * kThreadsTc;
      if (c < kQChunks) {
        const int h = c / (kD / 8), col = (c % (kD / 8)) * 8;
        const uint32_t w[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          o[j] = pack_f16x2(bf16_bits_to_float((uint16_t)(w[j] & 0xFFFFu)),
                            bf16_bits_to_float((uint16_t)(w[j] >> 16)));
        *reinterpret_cast<uint4*>(smem + L::q_off + sw128_off(h, col, L::q_atom)) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
        su32(&ctl.tmem_base)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int a = 0; a < 8; ++a) mbar_init(su32(&ctl.bar_v[a]), 4);
    mbar_init(su32(&ctl.bar_s), 1);
    mbar_init(su32(&ctl.bar_p), kSoftWarps);
    for (int mb = 0; mb < 4; ++mb) mbar_init(su32(&ctl.bar_o[mb]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    ctl.exceed[0] = ctl.exceed[1] = 0;
    ctl.rescale = 0;
  }
  if (tid < kHN) ctl.mref[tid] = -INFINITY;
  pdl_wait();
  for (int i = tid; i < min(cnt, kIdxCache); i += kThreadsTc) idx_s[i] = slots[i];
  if (idx_copy) {  // the caller's copy of the slots this CTA reads
    int32_t* dst = idx_copy + (int64_t)b * k + s0;
    for (int i = tid; i < cnt; i += kThreadsTc) dst[i] = slots[i];
  }
  proxy_fence();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const uint32_t tm_o = tmem;          // columns [0, 256): 4 M-blocks x 64 heads
  const uint32_t tm_s = tmem + 256;    // columns [256, 320)

  if (warp >= kDeqWarp0) {
    // ================= dequantisers =================
    const int dt = tid - kDeqWarp0 * 32;
    const int e = dt & 127, half = dt >> 7;
    uint4 raw[9];
    auto load_row = [&](int t, uint4* r) {
      const int s = t * kTileE + e;
      const int32_t j = (s < cnt) ? slot_at(s) : -1;
      const bool ok = (j >= 0) && (j < N);
      if (half == 0 && (j >= N || j < -1)) set_status(status, kStatusBadIndex);
      if (ok) {
        const uint4* src = reinterpret_cast<const uint4*>(kvseq + (int64_t)j * kRowBytes);
#pragma unroll
        for (int i = 0; i < 8; ++i) r[i] = __ldg(src + half * 8 + i);
        r[8] = __ldg(src + 16 + half);
      } else {
#pragma unroll
        for (int i = 0; i < 9; ++i) r[i] = make_uint4(0, 0, 0, 0);
      }
    };
    // this thread's 256 bytes of window row sw*128 + e (tile sw of the window)
    auto swa_row = [&](int sw) -> const uint4* {
      const int sl = sw * kTileE + e;
      return sl < wcnt ? reinterpret_cast<const uint4*>(swaseq + ((w0 + sl) % swa_ring) * kD) +
                             16 * half
                       : nullptr;
    };
    if (nmain > 0) load_row(0, raw);
    bool alive = true;
    for (int t = 0; t < ntiles && alive; ++t) {
      if (t >= nmain) {
        // ---- a tile of the SWA window: E4M3 -> fp16 (exact), two atoms per load ----
        const uint4* src = swa_row(t - nmain);
        if (t + 1 < ntiles)
          if (const uint4* nx = swa_row(t + 1 - nmain))
            for (int i = 0; i < 2; ++i) asm volatile("prefetch.global.L2 [%0];" ::"l"(nx + 8 * i));
#pragma unroll 1
        for (int ap = 0; ap < 2 && alive; ++ap) {
          uint4 wv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) wv[i] = src ? __ldg(src + 8 * ap + i) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int aj = 0; aj < 2; ++aj) {
            const int ai = 2 * ap + aj;
            const int a = half * 4 + ai;
            if (t > 0 && aj == 0 && !mbar_wait(su32(&ctl.bar_o[a >> 1]), (t - 1) & 1, status)) {
              alive = false;
              break;
            }
#pragma unroll
            for (int ci = 0; ci < 8; ++ci) {
              // channels 8 ci .. 8 ci + 7 of atom a: bytes 8 (ci & 1) .. of wv[4 aj + ci / 2]
              const uint4 u = wv[4 * aj + (ci >> 1)];
              const uint32_t lo = (ci & 1) ? u.z : u.x, hi = (ci & 1) ? u.w : u.y;
              const uint32_t off = L::v_off + (uint32_t)a * L::v_atom +
                                   (uint32_t)(e >> 3) * 1024u + (uint32_t)(e & 7) * 128u +
                                   (uint32_t)((ci ^ (e & 7)) << 4);
              *reinterpret_cast<uint4*>(smem + off) =
                  make_uint4(e4m3x2_to_f16x2((uint16_t)(lo & 0xFFFFu)),
                             e4m3x2_to_f16x2((uint16_t)(lo >> 16)),
                             e4m3x2_to_f16x2((uint16_t)(hi & 0xFFFFu)),
                             e4m3x2_to_f16x2((uint16_t)(hi >> 16)));
            }
            proxy_fence();
            __syncwarp();
            if (lane == 0) mbar_arrive(su32(&ctl.bar_v[a]));
          }
        }
        continue;
      }
      uint4 nxt[9];
      if (t + 1 < nmain) {
        load_row(t + 1, nxt);
      } else {
        if (t + 1 < ntiles)  // the window follows: bring its rows into L2 meanwhile
          if (const uint4* nx = swa_row(0))
            for (int i = 0; i < 2; ++i) asm volatile("prefetch.global.L2 [%0];" ::"l"(nx + 8 * i));
#pragma unroll
        for (int i = 0; i < 9; ++i) nxt[i] = make_uint4(0, 0, 0, 0);
      }
      const uint32_t sc_words[4] = {raw[8].x, raw[8].y, raw[8].z, raw[8].w};
#pragma unroll
      for (int ai = 0; ai < 4; ++ai) {
        const int a = half * 4 + ai;
        // atom a feeds the O^T M-block a / 2 of the previous tile
        if (t > 0 && (ai & 1) == 0 && !mbar_wait(su32(&ctl.bar_o[a >> 1]), (t - 1) & 1, status)) {
          alive = false;
          break;
        }
        const uint32_t cw[8] = {raw[2 * ai].x,     raw[2 * ai].y,     raw[2 * ai].z,
                                raw[2 * ai].w,     raw[2 * ai + 1].x, raw[2 * ai + 1].y,
                                raw[2 * ai + 1].z, raw[2 * ai + 1].w};
#pragma unroll
        for (int ci = 0; ci < 8; ++ci) {
          // 8 channels (8 ci .. 8 ci + 7 of atom a) = 4 code bytes; scale of block 2 ai + ci / 2
          const uint32_t sb = (sc_words[ai] >> (8 * (ci >> 1))) & 0xFFu;
          const uint32_t s2 = e4m3x2_to_f16x2((uint16_t)(sb | (sb << 8)));
          const __half2 sc = *reinterpret_cast<const __half2*>(&s2);
          uint32_t o[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t v2 = e2m1x2_to_f16x2((cw[ci] >> (8 * q4)) & 0xFFu);
            __half2 hv = __hmul2(*reinterpret_cast<__half2*>(&v2), sc);
            o[q4] = *reinterpret_cast<uint32_t*>(&hv);
          }
          const uint32_t off = L::v_off + (uint32_t)a * L::v_atom + (uint32_t)(e >> 3) * 1024u +
                               (uint32_t)(e & 7) * 128u + (uint32_t)((ci ^ (e & 7)) << 4);
          *reinterpret_cast<uint4*>(smem + off) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        proxy_fence();
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&ctl.bar_v[a]));
      }
#pragma unroll
      for (int i = 0; i < 9; ++i) raw[i] = nxt[i];
    }
  } else {
    // ================= softmax (warps 0-7) =================
    // thread = TMEM lane = entry e of the tile; warp w covers heads 32 (w / 4) .. +32
    const int e = (warp & 3) * 32 + lane;
    const int hh = warp >> 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float c = scale_log2;
    const float tau_raw = 8.0f / c;  // lazy-rescale margin in raw logit units
    float m_own = -INFINITY;         // reference max of head tid (tid < 64)
    float l_part[32];                // this thread's share of the row sums of its 32 heads
#pragma unroll
    for (int i = 0; i < 32; ++i) l_part[i] = 0.0f;
    // S^T: A = V (K-major), B = Q (K-major).  O^T: A = V (MN-major), B = P (MN-major).
    const uint32_t id_s = (1u << 4) | ((uint32_t)(kHN >> 3) << 17) | ((128u >> 4) << 24);
    const uint32_t id_o = id_s | (1u << 15) | (1u << 16);
    // Base descriptors; each MMA only adds a compile-time offset (in 16-byte
    // units) to the start-address field, so issuing costs a few instructions.
    const uint64_t dS_a = sw128_desc(v_s, 16, 1024);
    const uint64_t dS_b = sw128_desc(q_s, 16, 1024);
    const uint64_t dO_a = sw128_desc(v_s, L::v_atom, 1024);
    const uint64_t dO_b = sw128_desc(p_s, L::v_atom, 1024);
    const bool issuer = (tid == 0);
    bool alive = true;
    for (int t = 0; t < ntiles && alive; ++t) {
      if (issuer) {
        // S^T(t) over the 8 channel atoms as the dequantisers finish them
#pragma unroll
        for (int a = 0; a < 8; ++a) {
          if (!alive) break;
          if (!mbar_wait(su32(&ctl.bar_v[a]), t & 1, status)) {
            alive = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
            mma_f16(tm_s, dS_a + ((a * L::v_atom + jj * 32) >> 4),
                    dS_b + ((a * L::q_atom + jj * 32) >> 4), id_s, (a | jj) != 0 ? 1u : 0u);
        }
        if (alive) mma_commit(su32(&ctl.bar_s));
      }
      __syncwarp();
      if (!mbar_wait(su32(&ctl.bar_s), t & 1, status)) {
        alive = false;
        break;
      }
      tc_fence_after();
      float s[32];
      tmem_ld16(tm_s + lane_base + hh * 32, s);
      tmem_ld16(tm_s + lane_base + hh * 32 + 16, s + 16);
      tmem_wait_ld();
      {
        const int sl = t * kTileE + e;
        bool valid;
        if (t < nmain) {
          const int32_t j = sl < cnt ? slot_at(sl) : -1;
          valid = j >= 0 && j < N;
        } else {
          valid = (t - nmain) * kTileE + e < wcnt;  // a window row
        }
        if (!valid) {
#pragma unroll
          for (int i = 0; i < 32; ++i) s[i] = -INFINITY;
        }
      }
      // does any logit pass its head's reference max by more than the margin?
      bool ex = false;
#pragma unroll
      for (int i = 0; i < 32; ++i) ex |= s[i] > ctl.mref[hh * 32 + i] + tau_raw;
      if (__any_sync(0xffffffffu, ex) && lane == 0) ctl.exceed[t & 1] = 1;
      softmax_bar();
      if (tid == 0) ctl.exceed[(t + 1) & 1] = 0;  // every thread has read the previous tile's flag
      if (ctl.exceed[t & 1]) {
        // exact tile max per head, new reference where it moved past the margin
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = s[i];
        ctl.red[warp & 3][hh * 32 + lane] = warp_reduce32<true>(v);
        softmax_bar();
        if (tid < kHN) {
          const float mt = fmaxf(fmaxf(ctl.red[0][tid], ctl.red[1][tid]),
                                 fmaxf(ctl.red[2][tid], ctl.red[3][tid]));
          float a = 1.0f;
          if (mt > m_own + tau_raw) {
            a = exp2f((m_own - mt) * c);  // 0 while m_own = -inf
            m_own = mt;
            if (t > 0) ctl.rescale = 1;
          }
          ctl.mref[tid] = m_own;
          ctl.alpha[tid] = a;
        }
        softmax_bar();
        if (ctl.rescale) {
#pragma unroll
          for (int i = 0; i < 32; ++i) l_part[i] *= ctl.alpha[hh * 32 + i];
          // every earlier O^T MMA is complete: this tile's S^T was issued after them
#pragma unroll 1
          for (int mb = 0; mb < 4; ++mb) {
#pragma unroll 1
            for (int c16 = 0; c16 < 2; ++c16) {
              float o16[16];
              const uint32_t ta = tm_o + lane_base + mb * kHN + hh * 32 + c16 * 16;
              tmem_ld16(ta, o16);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) o16[i] *= ctl.alpha[hh * 32 + c16 * 16 + i];
              tmem_st16(ta, o16);
            }
          }
          tmem_wait_st();
        }
        softmax_bar();
        if (tid == 0) ctl.rescale = 0;
      }
      // P = exp2(c s - c m_ref), fp16, into row e of the MN-major P tile
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float m0 = ctl.mref[hh * 32 + i], m1 = ctl.mref[hh * 32 + i + 1];
        const float p0 = exp2f(fmaf(s[i], c, m0 == -INFINITY ? 0.0f : -m0 * c));
        const float p1 = exp2f(fmaf(s[i + 1], c, m1 == -INFINITY ? 0.0f : -m1 * c));
        l_part[i] += p0;
        l_part[i + 1] += p1;
        pk[i >> 1] = pack_f16x2(p0, p1);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int chunk = hh * 4 + j;  // heads 8 chunk .. +8
        const uint32_t off = L::p_off + (uint32_t)(e >> 3) * 1024u + (uint32_t)(e & 7) * 128u +
                             (uint32_t)((chunk ^ (e & 7)) << 4);
        *reinterpret_cast<uint4*>(smem + off) =
            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
      }
      proxy_fence();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(su32(&ctl.bar_p));
      if (issuer) {
        // O^T(t) once every softmax warp has written its part of P
        if (!mbar_wait(su32(&ctl.bar_p), t & 1, status)) {
          alive = false;
        } else {
          tc_fence_after();
          const uint32_t acc0 = t > 0 ? 1u : 0u;
#pragma unroll
          for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
            for (int kk = 0; kk < kTileE / 16; ++kk) {
              // A = V^T rows 128 mb .. +128 (channels) x entries 16 kk .. +16;
              // B = P entries 16 kk .. +16 x 64 heads
              mma_f16(tm_o + mb * kHN, dO_a + ((2 * mb * L::v_atom + kk * 2048) >> 4),
                      dO_b + ((kk * 2048) >> 4), id_o, kk > 0 ? 1u : acc0);
            }
            mma_commit(su32(&ctl.bar_o[mb]));
          }
        }
      }
      __syncwarp();
    }
    // ---- epilogue ----
    if (alive && ntiles > 0) alive = mbar_wait(su32(&ctl.bar_o[3]), (ntiles - 1) & 1, status);
    tc_fence_after();
    ctl.red[warp & 3][hh * 32 + lane] = warp_reduce32<false>(l_part);
    softmax_bar();
    const float ln2 = 0.69314718055994530942f;
    if (tid < kHN) {
      const float l = (ctl.red[0][tid] + ctl.red[1][tid]) + (ctl.red[2][tid] + ctl.red[3][tid]);
      const bool empty = !(l > 0.0f);
      ctl.linv[tid] = empty ? 0.0f : 1.0f / l;
      if (tid < H) {
        const float lse_v = empty ? -INFINITY : (m_own * c + log2f(l)) * ln2;
        if (nsplit == 1) {
          if (lse) lse[(int64_t)b * H + tid] = lse_v;
        } else {
          part_lse[((int64_t)b * nsplit + split) * H + tid] = lse_v;
        }
      }
    }
    softmax_bar();
    float* obase = (nsplit == 1) ? out + (int64_t)b * H * kD
                                 : part_o + ((int64_t)b * nsplit + split) * H * kD;
#pragma unroll 1
    for (int mb = 0; mb < 4; ++mb) {
      const int ch = mb * 128 + e;  // this thread's channel
#pragma unroll 1
      for (int c16 = 0; c16 < 2; ++c16) {
        const int h0 = hh * 32 + c16 * 16;
        if (h0 >= H) continue;
        float o16[16];
        if (alive && ntiles > 0) {
          tmem_ld16(tm_o + lane_base + mb * kHN + h0, o16);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) o16[i] = 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) obase[(int64_t)(h0 + i) * kD + ch] = o16[i] * ctl.linv[h0 + i];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}

}  // namespace

template <int H>
static cudaError_t launch_tc_t(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int64_t N,
                               int64_t kv_seq_stride, int q_per_seq, const int32_t* idx, int k,
                               int nsplit, int chunk, float scale_log2, float* out, float* lse,
                               float* part_o, float* part_lse, int32_t* status,
                               const SwaArgs* swa, int32_t* idx_copy, cudaStream_t stream,
                               bool pdl) {
  using L = TcLayout;
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_tc_kernel<H>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::alloc);
  if (e != cudaSuccess) return e;
  return launch_kernel(sparse_attn_tc_kernel<H>, dim3((unsigned)nsplit, (unsigned)B),
                       dim3(kThreadsTc), L::alloc, stream, pdl, q_bf16, kv_fp4, N, kv_seq_stride,
                       q_per_seq, idx, k, chunk, scale_log2, out, lse, part_o, part_lse, status,
                       swa ? swa->kv : nullptr, swa ? swa->ring : (int64_t)0, swa ? swa->n_win : 0,
                       swa ? swa->q_pos : nullptr, idx_copy);
}

cudaError_t launch_sparse_attn_tc(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H,
                                  int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                  const int32_t* idx, int k, int nsplit, int chunk,
                                  float scale_log2, float* out, float* lse, float* part_o,
                                  float* part_lse, int32_t* status, const SwaArgs* swa,
                                  int32_t* idx_copy, cudaStream_t stream, bool pdl) {
  switch (H) {
    case 16:
      return launch_tc_t<16>(q_bf16, kv_fp4, B, N, kv_seq_stride, q_per_seq, idx, k, nsplit,
                             chunk, scale_log2, out, lse, part_o, part_lse, status, swa, idx_copy,
                             stream, pdl);
    case 32:
      return launch_tc_t<32>(q_bf16, kv_fp4, B, N, kv_seq_stride, q_per_seq, idx, k, nsplit,
                             chunk, scale_log2, out, lse, part_o, part_lse, status, swa, idx_copy,
                             stream, pdl);
    default:
      return launch_tc_t<64>(q_bf16, kv_fp4, B, N, kv_seq_stride, q_per_seq, idx, k, nsplit,
                             chunk, scale_log2, out, lse, part_o, part_lse, status, swa, idx_copy,
                             stream, pdl);
  }
}

}  // namespace csa2
