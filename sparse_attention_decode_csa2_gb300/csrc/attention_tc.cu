// Sparse MQA attention over the selected FP4 entries on the 5th-generation
// tensor cores (DeepSeek-V4.1-Flash paper walkthrough, 1.(4) "CSA2": each
// query attends its selected main-KV entries; 1.(5).4: the FP4 cache is
// dequantised before attention; 3.(2).1: 64 query heads x 512).  K = V = the
// dequantised 512-channel latent shared by the heads.
//
// One CTA = one query x a chunk of its selected slots, in tiles of 128
// entries:
//   S[h][e]    = sum_c Q[h][c] V[e][c]     M = 64 heads, N = 128 entries
//                                          (A = Q, B = V tile, both K-major SW128)
//   O^T[c][h] += sum_e V[e][c] P[h][e]    M = 4 x 128 channels, N = 64 heads,
//                                          K = 128 entries (A = the same V bytes
//                                          read MN-major, B = P K-major)
// Both accumulators live in tensor memory: O^T in 4 x 64 columns, S (one head
// per TMEM lane of the M = 64 layout: heads 16q .. 16q + 15 in lanes 32q ..
// 32q + 15) in two buffers of 128 columns.  A tcgen05.mma of this shape costs
// about the same whether it covers 64 or 128 entries, so the tile is as wide
// as shared memory allows.
//
// Pipeline.  There is one V buffer, handed over in two halves of four
// 64-channel atoms: O^T(t) M-blocks 2h, 2h + 1 read atoms 4h .. 4h + 3 of
// V(t); once they complete the dequantisers write those atoms of V(t + 1),
// and S(t + 1) consumes each half as it arrives.  The tensor pipe thus runs
// O^T(t) and S(t + 1) back to back and idles only while the softmax of t + 1
// runs.  Warp roles (512 threads):
//   warps 0-3   softmax: warp q holds heads 16q .. 16q + 15; a paired 16-lane
//               load gives lane l head 16q + l % 16 and half of the tile's
//               entries (lanes l and l ^ 16 share a head), so a head's max and
//               sum need one shuffle.  Online softmax in fp32 with exp2 and a
//               lazy per-head reference max (it moves only when a logit passes
//               it by more than 2^8 in the exp2 domain, so P <= 256 stays in
//               fp16 range and O is rarely rescaled)
//   warps 4-11  dequantisers: for half h a lane converts atom 4 h + lane / 8
//               of rows 16 w + 8 i + lane % 8 (E2M1 x E4M3 -> fp16, exact),
//               from registers loaded a tile ahead; each load instruction of
//               a warp reads 128 contiguous bytes of eight rows, each 16-byte
//               store phase writes eight consecutive rows of one atom
//               (conflict-free); the next tile's rows are requested after the
//               tile's handovers
//   warp 12     TMEM allocation; lane 0 issues every MMA
//   warp 13     prefetcher: requests the selected rows of tiles 1, 2, ... (and
//               the SWA window) into L2 with bulk prefetches, up to 16 tiles
//               ahead of the dequantisers
//   warps 14-15 join the epilogue
// (Measured alternatives that were slower: staging rows in shared memory, since
// the tensor cores read their operands from shared memory and its bandwidth
// bounds a tile; one cp.async.bulk copy per 288-byte row, bounded by the copy
// engine's per-request cost; one row per lane in each load, bounded by the
// SM's outstanding-request tracking; S^T at M = 128 with eight softmax warps,
// whose softmax and MN-major P^T operand cost more than they saved.)
// The chunk's slot ids are read once at the start: the first kIdxCache into
// shared memory, the validity of every slot into a bit mask.
// SWA branch: the CTA of a query's last chunk also attends the query's sliding
// window (E4M3 rows of the layer's SWA ring) as extra tiles after its selected
// entries, in the same online softmax.
// Epilogue: every warp reads one M-block x 32 channels of O^T from tensor
// memory.  With one split it writes the output ([head][channel] fp32); with
// several, the query's splits form one thread-block cluster that merges them
// (staged fp16 blocks pushed into their owners' shared memory by bulk copies:
// see below).
// Every mbarrier wait is bounded (about 2 s of %globaltimer): a wait that
// gives up sets the timeout status bit and the CTA drains, frees its tensor
// memory and exits.
#include "csa2_internal.cuh"
#include "tc_common.cuh"

namespace csa2 {
namespace {

using namespace tc;

constexpr int kThreadsTc = 16 * 32;
constexpr int kTileE = 128;         // entries per tile
constexpr int kHN = 64;             // heads, zero-padded to 64
constexpr int kSoftWarps = 4;       // warps 0-3
constexpr int kDeqWarp0 = 4;        // warps 4-11
constexpr int kDeqWarps = 8;
constexpr int kIssuerWarp = 12;
constexpr int kPrefWarp = 13;
constexpr int kAheadTiles = 16;     // tiles requested into L2 ahead of the dequantisers
constexpr int kIdxCache = 2048;     // slot ids kept in shared memory
constexpr int kMaxSlots = 16384;    // validity bits kept for a chunk
constexpr int kMaxSplitTc = 8;      // splits of a query (one cluster), a power of two

struct TcLayout {
  static constexpr uint32_t q_atom = 64 * 128;            // [64 heads][128 B]
  static constexpr uint32_t v_atom = kTileE * 128;        // [128 entries][128 B]
  static constexpr uint32_t p_atom = 64 * 128;            // [64 heads][64 entries x 2 B]
  static constexpr uint32_t q_off = 0;                    // 8 atoms
  static constexpr uint32_t v_off = q_off + 8 * q_atom;   // 8 atoms
  static constexpr uint32_t p_off = v_off + 8 * v_atom;   // 2 atoms
  static constexpr uint32_t idx_off = p_off + 2 * p_atom;
  static constexpr uint32_t mask_off = idx_off + kIdxCache * 4;
  static constexpr uint32_t ctl_off = mask_off + kMaxSlots / 8;
  static constexpr uint32_t bytes = ctl_off + 1024;
  static constexpr uint32_t alloc = bytes + 1024;         // slack to align the base to 1 KiB
};
static_assert(TcLayout::alloc <= 232448, "shared memory");

struct TcCtl {
  float alpha[kHN];      // rescale factor of O^T per head (rare)
  float linv[kHN];       // 1 / row sum per head (epilogue)
  uint64_t v_ready[2];   // atoms 4h .. 4h + 3 of the current V tile written (8 warps)
  uint64_t s_full[2];    // S of a tile in S buffer (commit)
  uint64_t o_half[2];    // O^T(t) M-blocks 2h, 2h + 1 done: atoms 4h .. 4h + 3 free (commit)
  uint64_t p_half[2];    // P entries 64 j .. 64 j + 63 written (4 softmax warps)
  uint64_t recv;         // the split merge's partial blocks have arrived (bulk copies)
  uint32_t tmem_base;
  int32_t abort;         // a bounded wait gave up somewhere in the CTA
  int32_t tiles_done;    // tiles the first dequantiser warp has written
};
static_assert(sizeof(TcCtl) <= 1024, "control block");

__device__ __forceinline__ void softmax_bar() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Barrier of the softmax warps that also returns the OR of a predicate over
// their threads: every warp takes the same decision.
__device__ __forceinline__ bool softmax_bar_or(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p)
      : "memory");
  return r != 0;
}

// 16 TMEM columns of 16 lanes, twice: lanes 0-15 of the warp read lanes
// base + l at columns [col, col + 16), lanes 16-31 read lanes base + l - 16 at
// columns [col + 32, col + 48).
__device__ __forceinline__ void tmem_ld16_pair32(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15}, [%16], 32;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Requests `bytes` bytes at `row` (16-byte aligned, a multiple of 16) into
// L2 through the bulk-copy unit: no load/store-unit traffic, which the
// softmax and dequantiser warps of the SM share.
__device__ __forceinline__ void prefetch_l2(const uint8_t* row, int bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(row), "r"((uint32_t)bytes)
               : "memory");
}

// This CTA's shared-memory address `a` as seen in cluster CTA `rank`.
__device__ __forceinline__ uint32_t peer_smem(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
// Bulk copy of `bytes` from this CTA's shared memory into another CTA's of
// the cluster, completing on that CTA's mbarrier `bar` (both addresses from
// peer_smem, 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_push(uint32_t dst, uint32_t src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst),
      "r"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// The same bounded wait for every lane of a warp, with one answer for all of
// them (the warp's later .sync.aligned instructions need every lane).
__device__ __forceinline__ bool warp_wait(TcCtl& ctl, uint64_t* bar, uint32_t parity,
                                          int32_t* status) {
  bool ok = mbar_wait(su32(bar), parity, status);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) *reinterpret_cast<volatile int32_t*>(&ctl.abort) = 1;
  return ok;
}

__device__ __forceinline__ bool aborted(TcCtl& ctl) {
  return *reinterpret_cast<volatile int32_t*>(&ctl.abort) != 0;
}

// 32 bytes of read-only global data into two uint4: one 256-bit load when
// the address is 32-byte aligned (fewer requests in flight per SM), two
// 128-bit loads otherwise.
__device__ __forceinline__ void ld32(const uint8_t* p, bool wide, uint4& lo, uint4& hi) {
  if (wide) {
    asm volatile("ld.global.nc.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y),
                   "=r"(hi.z), "=r"(hi.w)
                 : "l"(p));
  } else {
    lo = __ldg(reinterpret_cast<const uint4*>(p));
    hi = __ldg(reinterpret_cast<const uint4*>(p) + 1);
  }
}

// 8 fp16 channels from 8 E2M1 codes (one 32-bit word) times a scale (f16x2).
__device__ __forceinline__ uint4 dequant8(uint32_t w, __half2 sc) {
  uint32_t o[4];
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    uint32_t v2 = e2m1x2_to_f16x2((w >> (8 * q4)) & 0xFFu);
    __half2 hv = __hmul2(*reinterpret_cast<__half2*>(&v2), sc);
    o[q4] = *reinterpret_cast<uint32_t*>(&hv);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Byte offset of the 16-byte chunk ci (channels 8 ci .. 8 ci + 7 of atom a)
// of row e in the V tile (K-major SW128 atoms of 128 rows).
__device__ __forceinline__ uint32_t v_chunk_off(int a, int e, int ci) {
  return (uint32_t)a * TcLayout::v_atom + (uint32_t)(e >> 3) * 1024u + (uint32_t)(e & 7) * 128u +
         (uint32_t)((ci ^ (e & 7)) << 4);
}

// One atom of a row held by a dequantiser: 32 code bytes.
struct Eighth {
  uint4 cw[2];
};

template <int H>
__global__ void __launch_bounds__(kThreadsTc, 1)
sparse_attn_tc_kernel(const uint16_t* __restrict__ q_bf16, const uint8_t* __restrict__ kv_fp4,
                      int64_t N, int64_t kv_seq_stride, int q_per_seq,
                      const int32_t* __restrict__ idx, int k, int chunk, float scale_log2,
                      float* __restrict__ out, float* __restrict__ lse,
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
  uint32_t* mask_s = reinterpret_cast<uint32_t*>(smem + L::mask_off);

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

  pdl_trigger();
  // ---- prologue: Q (bf16 -> fp16, swizzled, zero-padded to 64 rows), TMEM,
  //      barriers; the slot ids are read only after the kernel that selected
  //      them has finished ----
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
  if (warp == kIssuerWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
        su32(&ctl.tmem_base)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(su32(&ctl.v_ready[i]), kDeqWarps);
      mbar_init(su32(&ctl.o_half[i]), 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(su32(&ctl.s_full[i]), 1);
    for (int i = 0; i < 2; ++i) mbar_init(su32(&ctl.p_half[i]), kSoftWarps);
    mbar_init(su32(&ctl.recv), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    ctl.abort = 0;
    ctl.tiles_done = 0;
  }
  pdl_wait();
  // ---- the chunk's slot ids (all threads): bad ids raise the status bit, the
  //      Reuse layers' copy of the slots is written, the first kIdxCache ids
  //      are kept in shared memory and every slot's validity in a bit mask ----
  {
    constexpr int kUnroll = kIdxCache / kThreadsTc;
    for (int base = 0; base < cnt; base += kUnroll * kThreadsTc) {
      int32_t j[kUnroll];
#pragma unroll
      for (int i = 0; i < kUnroll; ++i) {
        const int s = base + i * kThreadsTc + tid;
        j[i] = s < cnt ? slots[s] : -1;
      }
#pragma unroll
      for (int i = 0; i < kUnroll; ++i) {
        const int s = base + i * kThreadsTc + tid;
        if (s < cnt) {
          if (j[i] >= N || j[i] < -1) set_status(status, kStatusBadIndex);
          if (idx_copy) idx_copy[(int64_t)b * k + s0 + s] = j[i];
          if (s < kIdxCache) idx_s[s] = j[i];
        }
        const uint32_t m = __ballot_sync(0xffffffffu, s < cnt && j[i] >= 0 && j[i] < N);
        if (lane == 0 && s < cnt) mask_s[s >> 5] = m;
      }
    }
  }
  proxy_fence();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const uint32_t tm_o = tmem;          // columns [0, 256): 4 M-blocks x 64 heads
  const uint32_t tm_s = tmem + 256;    // columns [256, 512): 2 S buffers x 128 entries
  auto slot_id = [&](int s) -> int32_t { return s < kIdxCache ? idx_s[s] : slots[s]; };
  auto slot_ok = [&](int s) -> bool { return (mask_s[s >> 5] >> (s & 31)) & 1u; };
  bool alive = true;

  if (warp == kPrefWarp) {
    // ================= prefetcher =================
    // the window rows first (small), then tile t's 128 rows (four per lane)
    // once the dequantisers have written fewer than kAheadTiles tiles before it
    for (int r = lane; r < wcnt; r += 32)
      prefetch_l2(swaseq + ((w0 + r) % swa_ring) * kD, kD);
    uint64_t t_idle = 0;
    for (int t = 1; t < nmain && !aborted(ctl);) {  // the dequantisers load tile 0 themselves
      const int done = *reinterpret_cast<volatile int32_t*>(&ctl.tiles_done);
      if (t >= done + kAheadTiles) {
        if (t_idle == 0) t_idle = globaltimer();
        if (globaltimer() - t_idle > kWaitLimitNs) break;  // the consumer has stopped
        __nanosleep(256);
        continue;
      }
      t_idle = 0;
#pragma unroll
      for (int i = 0; i < kTileE / 32; ++i) {
        const int s = t * kTileE + lane + 32 * i;
        if (s < cnt && slot_ok(s)) prefetch_l2(kvseq + (int64_t)slot_id(s) * kRowBytes, kRowBytes);
      }
      ++t;
    }
  } else if (warp >= kDeqWarp0 && warp < kDeqWarp0 + kDeqWarps) {
    // ================= dequantisers =================
    // V is handed over in two halves of four 64-channel atoms.  For half h a
    // lane converts atom 4 h + lane / 8 of rows 16 w + 8 i + lane % 8 (i = 0,
    // 1; w = the dequantiser warp): each load instruction of a warp reads 128
    // contiguous bytes of eight rows (a few cache lines per row instead of one
    // per lane), and the eight lanes of each phase of a 16-byte shared-memory
    // store write eight consecutive rows of one atom, i.e. eight different
    // 16-byte slots of the swizzle.
    const int dt = tid - kDeqWarp0 * 32;  // 0..255
    const int dw = dt >> 5, sub = lane >> 3, rsub = lane & 7;
    // 256-bit loads need a 32-byte aligned cache (rows are 288 = 9 x 32 bytes)
    const bool wide = (reinterpret_cast<uintptr_t>(kv_fp4) & 31u) == 0;
    uint8_t* vt = smem + L::v_off;
    Eighth cur[2][2];   // [half][i]: 32 code bytes of the lane's atom of a row
    uint32_t scw[2][2];  // [half][i]: the atom's 4 scale bytes
    auto load_tile = [&](int t) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int sl = t * kTileE + 16 * dw + 8 * i + rsub;
        const uint8_t* src = (t < nmain && sl < cnt && slot_ok(sl))
                                 ? kvseq + (int64_t)slot_id(sl) * kRowBytes
                                 : nullptr;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int a = 4 * h + sub;
          if (src) {
            ld32(src + 32 * a, wide, cur[h][i].cw[0], cur[h][i].cw[1]);
            scw[h][i] = __ldg(reinterpret_cast<const uint32_t*>(src + kCodeBytes + 4 * a));
          } else {
            cur[h][i].cw[0] = cur[h][i].cw[1] = make_uint4(0, 0, 0, 0);
            scw[h][i] = 0u;
          }
        }
      }
    };
    load_tile(0);
    for (int t = 0; t < ntiles && alive; ++t) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // atoms 4h .. 4h + 3 are free once O^T(t - 1) M-blocks 2h, 2h + 1 have read them
        if (t >= 1 && !warp_wait(ctl, &ctl.o_half[h], (uint32_t)(t - 1) & 1u, status)) {
          alive = false;
          break;
        }
        const int a = 4 * h + sub;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int e = 16 * dw + 8 * i + rsub;
          if (t < nmain) {
            // word w of code vector u: channels 64 a + 32 u + 8 w .. +8,
            // scale byte 2 u + w / 2 of the atom, 16-byte chunk 4 u + w
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint32_t sbytes = (scw[h][i] >> (16 * u)) & 0xFFFFu;
              const uint32_t s_lo = e4m3x2_to_f16x2((uint16_t)((sbytes & 0xFFu) * 0x101u));
              const uint32_t s_hi = e4m3x2_to_f16x2((uint16_t)((sbytes >> 8) * 0x101u));
              const __half2 h_lo = *reinterpret_cast<const __half2*>(&s_lo);
              const __half2 h_hi = *reinterpret_cast<const __half2*>(&s_hi);
              const uint4 w = cur[h][i].cw[u];
              *reinterpret_cast<uint4*>(vt + v_chunk_off(a, e, 4 * u + 0)) = dequant8(w.x, h_lo);
              *reinterpret_cast<uint4*>(vt + v_chunk_off(a, e, 4 * u + 1)) = dequant8(w.y, h_lo);
              *reinterpret_cast<uint4*>(vt + v_chunk_off(a, e, 4 * u + 2)) = dequant8(w.z, h_hi);
              *reinterpret_cast<uint4*>(vt + v_chunk_off(a, e, 4 * u + 3)) = dequant8(w.w, h_hi);
            }
          } else {
            // a tile of the SWA window: E4M3 row from global (in L2), -> fp16 (exact)
            const int sl = (t - nmain) * kTileE + e;
            uint4 wv[4];
            if (sl < wcnt) {
              const uint4* src =
                  reinterpret_cast<const uint4*>(swaseq + ((w0 + sl) % swa_ring) * kD) + 4 * a;
#pragma unroll
              for (int j = 0; j < 4; ++j) wv[j] = __ldg(src + j);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j) wv[j] = make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int ci = 0; ci < 8; ++ci) {
              // channels 8 ci .. 8 ci + 7 of atom a: bytes 8 (ci & 1) .. of wv[ci / 2]
              const uint4 u = wv[ci >> 1];
              const uint32_t lo = (ci & 1) ? u.z : u.x, hi = (ci & 1) ? u.w : u.y;
              *reinterpret_cast<uint4*>(vt + v_chunk_off(a, e, ci)) =
                  make_uint4(e4m3x2_to_f16x2((uint16_t)(lo & 0xFFFFu)),
                             e4m3x2_to_f16x2((uint16_t)(lo >> 16)),
                             e4m3x2_to_f16x2((uint16_t)(hi & 0xFFFFu)),
                             e4m3x2_to_f16x2((uint16_t)(hi >> 16)));
            }
          }
        }
        proxy_fence();  // the tensor cores read V through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&ctl.v_ready[h]));
      }
      if (warp == kDeqWarp0 && lane == 0)
        *reinterpret_cast<volatile int32_t*>(&ctl.tiles_done) = t + 1;
      // the next tile's rows, requested only now: an arrive (release) waits
      // for the loads its thread has in flight, so loads issued before the
      // arrives above would hold this tile's handovers for a memory round trip
      if (alive && t + 1 < nmain) load_tile(t + 1);
    }
  } else if (warp == kIssuerWarp) {
    // ================= MMA issuer =================
    if (lane == 0 && ntiles > 0) {
      // S: A = Q (K-major, 64 rows), B = V (K-major, 128 rows).  O^T: A = V
      // (MN-major: channels), B = P (K-major, 64 head rows).  Each MMA adds a
      // compile-time offset (16-byte units) to a base descriptor.
      const uint32_t id_s = (1u << 4) | ((uint32_t)(kTileE >> 3) << 17) | ((64u >> 4) << 24);
      const uint32_t id_o =
          (1u << 4) | ((uint32_t)(kHN >> 3) << 17) | ((128u >> 4) << 24) | (1u << 15);
      const uint64_t dS_a = sw128_desc(q_s, 16, 1024);
      const uint64_t dS_b = sw128_desc(v_s, 16, 1024);
      const uint64_t dO_a = sw128_desc(v_s, L::v_atom, 1024);
      const uint64_t dO_b = sw128_desc(p_s, 16, 1024);
      uint64_t* last = nullptr;  // barrier of the last commit, and its phase parity
      uint32_t last_par = 0;
      bool ok = true;
      for (int t = 0; t < ntiles && ok; ++t) {
        const uint32_t d_s = tm_s + (uint32_t)(t & 1) * kTileE;
        // S(t), half by half as the dequantisers finish them
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!mbar_wait(su32(&ctl.v_ready[h]), (uint32_t)t & 1u, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int a = 4 * h; a < 4 * h + 4; ++a)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
              mma_f16(d_s, dS_a + ((a * L::q_atom + jj * 32) >> 4),
                      dS_b + ((a * L::v_atom + jj * 32) >> 4), id_s, (a | jj) != 0 ? 1u : 0u);
        }
        if (!ok) break;
        mma_commit(su32(&ctl.s_full[t & 1]));
        last = &ctl.s_full[t & 1];
        last_par = ((uint32_t)t >> 1) & 1u;
        // O^T(t): entries 0-63 once their P is written (the softmax is
        // still on entries 64-127), then entries 64-127 M-block by M-block, so
        // that M-block p's atoms are freed as early as possible
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (!mbar_wait(su32(&ctl.p_half[hf]), (uint32_t)t & 1u, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
            for (int kk = 4 * hf; kk < 4 * hf + 4; ++kk)
              // A = V^T channels 128 mb .. +128 x entries 16 kk .. +16;
              // B = P heads x entries 16 kk .. +16 (atom kk / 4)
              mma_f16(tm_o + mb * kHN, dO_a + ((2 * mb * L::v_atom + kk * 2048) >> 4),
                      dO_b + (((kk >> 2) * L::p_atom + (kk & 3) * 32) >> 4), id_o,
                      (t > 0 || kk > 0) ? 1u : 0u);
            if (hf == 1 && (mb & 1)) mma_commit(su32(&ctl.o_half[mb >> 1]));
          }
        }
        if (!ok) break;
        last = &ctl.o_half[1];
        last_par = (uint32_t)t & 1u;
      }
      if (!ok) *reinterpret_cast<volatile int32_t*>(&ctl.abort) = 1;
      // the MMAs complete in order: once the last commit has arrived none is
      // in flight, whatever the other roles did (tensor memory is freed below)
      if (last) mbar_wait(su32(last), last_par, status);
    }
    __syncwarp();
  } else if (warp < kSoftWarps) {
    // ================= softmax (warps 0-3) =================
    // lane l of warp q: head 16 q + l % 16; entries col0 + 32 (l / 16) + 0..15
    // for col0 in {0, 16, 64, 80}
    const int qd = warp, h = qd * 16 + (lane & 15), hs = lane >> 4;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const float c = scale_log2;
    const float tau_raw = 8.0f / c;  // lazy-rescale margin in raw logit units
    float m_ref = -INFINITY;         // reference max of head h (raw logit units)
    float l_acc = 0.0f;              // this thread's share of head h's row sum
    for (int t = 0; t < ntiles; ++t) {
      const int sb = t & 1;
      // validity of this thread's 64 entries of the tile (bit i: entry i of the thread)
      uint64_t vmask = 0;
#pragma unroll
      for (int bi = 0; bi < 4; ++bi) {
        const int col0 = (bi < 2 ? 16 * bi : 64 + 16 * (bi - 2)) + 32 * hs;
        uint32_t m16;
        if (t < nmain) {
          const int sbase_i = t * kTileE + col0;  // a multiple of 16
          m16 = sbase_i < cnt ? (mask_s[sbase_i >> 5] >> (sbase_i & 31)) & 0xFFFFu : 0u;
        } else {
          const int wr = (t - nmain) * kTileE + col0;  // window rows wr .. wr + 15
          const int nv = min(16, max(0, wcnt - wr));
          m16 = nv >= 16 ? 0xFFFFu : ((1u << nv) - 1u);
        }
        vmask |= (uint64_t)m16 << (16 * bi);
      }
      if (!warp_wait(ctl, &ctl.s_full[sb], ((uint32_t)t >> 1) & 1u, status)) alive = false;
      float s[64];
      if (alive) {
        tc_fence_after();
        const uint32_t ta = tm_s + sb * kTileE + lane_base;
        tmem_ld16_pair32(ta + 0, s);
        tmem_ld16_pair32(ta + 16, s + 16);
        tmem_ld16_pair32(ta + 64, s + 32);
        tmem_ld16_pair32(ta + 80, s + 48);
        tmem_wait_ld();
      }
      if (!alive || vmask != ~0ull) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (!alive || !((vmask >> i) & 1u)) s[i] = -INFINITY;
      }
      float mx4[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) mx4[j] = s[j];
#pragma unroll
      for (int i = 4; i < 64; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], s[i]);
      float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      // a new reference max for this head when the tile's max passes it by
      // more than the margin; O^T's column needs rescaling only if the head
      // already has a contribution
      float alpha = 1.0f;
      bool resc = false;
      if (mx > m_ref + tau_raw) {
        resc = m_ref != -INFINITY;
        alpha = resc ? exp2f((m_ref - mx) * c) : 0.0f;
        m_ref = mx;
      }
      l_acc *= alpha;
      if (softmax_bar_or(resc || aborted(ctl))) {
        if (softmax_bar_or(aborted(ctl))) {  // every softmax warp leaves together
          alive = false;
          break;
        }
        if (lane < 16) ctl.alpha[h] = resc ? alpha : 1.0f;
        softmax_bar();
        // O^T(t - 1), the last product into O, must be complete; O^T rows are
        // channels: this warp rescales all 256 columns of its quadrant's lanes
        if (warp_wait(ctl, &ctl.o_half[1], (uint32_t)(t - 1) & 1u, status)) {
          tc_fence_after();
#pragma unroll 1
          for (int c4 = 0; c4 < 64; ++c4) {
            uint32_t o4[4];
            const uint32_t ta = tm_o + lane_base + c4 * 4;
            asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(o4[0]), "=r"(o4[1]), "=r"(o4[2]), "=r"(o4[3])
                         : "r"(ta));
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 4; ++i)
              o4[i] = __float_as_uint(__uint_as_float(o4[i]) * ctl.alpha[(c4 & 15) * 4 + i]);
            asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(ta),
                         "r"(o4[0]), "r"(o4[1]), "r"(o4[2]), "r"(o4[3])
                         : "memory");
          }
          tmem_wait_st();
        }
      }
      // P is free once O^T(t - 1) has read it
      if (t > 0 && !warp_wait(ctl, &ctl.o_half[1], (uint32_t)(t - 1) & 1u, status)) alive = false;
      // P = exp2(c s - c m_ref), fp16, into row h of the K-major P tile
      const float mneg = m_ref == -INFINITY ? 0.0f : -m_ref * c;
      float lsum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      // blocks 0, 1 hold entries 0-63 (P atom 0), blocks 2, 3 entries 64-127
#pragma unroll
      for (int bi = 0; bi < 4; ++bi) {
        const int col0 = (bi < 2 ? 16 * bi : 64 + 16 * (bi - 2)) + 32 * hs;  // first entry
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const float p0 = exp2f(fmaf(s[16 * bi + i], c, mneg));
          const float p1 = exp2f(fmaf(s[16 * bi + i + 1], c, mneg));
          lsum[(i >> 1) & 3] += p0 + p1;
          pk[i >> 1] = pack_f16x2(p0, p1);
        }
        if (alive) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int e0 = col0 + 8 * half;  // entries e0 .. e0 + 7: atom e0 / 64, chunk (e0 % 64) / 8
            const uint32_t off = L::p_off + (uint32_t)(e0 >> 6) * L::p_atom +
                                 (uint32_t)(h >> 3) * 1024u + (uint32_t)(h & 7) * 128u +
                                 (uint32_t)((((e0 & 63) >> 3) ^ (h & 7)) << 4);
            *reinterpret_cast<uint4*>(smem + off) =
                make_uint4(pk[4 * half], pk[4 * half + 1], pk[4 * half + 2], pk[4 * half + 3]);
          }
        }
        if (bi & 1) {  // entries 64 (bi / 2) .. +64 written by this warp
          proxy_fence();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(su32(&ctl.p_half[bi >> 1]));
        }
      }
      l_acc += (lsum[0] + lsum[1]) + (lsum[2] + lsum[3]);
    }
    // ---- row sums, lse ----
    const float l = l_acc + __shfl_xor_sync(0xffffffffu, l_acc, 16);
    if (lane < 16) {
      const float ln2 = 0.69314718055994530942f;
      const bool empty = !(l > 0.0f);
      ctl.linv[h] = empty ? 0.0f : 1.0f / l;
      if (h < H) {
        const float lse_v = empty ? -INFINITY : (m_ref * c + log2f(l)) * ln2;
        if (nsplit == 1) {
          if (lse) lse[(int64_t)b * H + h] = lse_v;
        } else {
          part_lse[((int64_t)b * nsplit + split) * H + h] = lse_v;
        }
      }
    }
  }

  // ---- epilogue: every warp reads one M-block x 32 channels of O^T from
  //      tensor memory (a thread holds one channel of every head) and scales
  //      it by 1 / row sum.  One split: the output [head][channel] fp32 (for
  //      each head a warp stores one 128-byte line).  Several: this split's
  //      partial, staged in shared memory (V is no longer read) as eight
  //      64-channel blocks [block][channel][head] fp16, 16-byte chunks of a
  //      row swizzled by the channel (a thread's heads are one row: wide
  //      conflict-free stores) ----
  __syncthreads();
  bool have_o = ntiles > 0 && !aborted(ctl);
  if (have_o)
    have_o = __all_sync(0xffffffffu, mbar_wait(su32(&ctl.o_half[1]),
                                               (uint32_t)(ntiles - 1) & 1u, status));
  tc_fence_after();
  constexpr int kCr = H / 8;                        // 16-byte chunks per staged row
  const uint32_t blk_bytes = (uint32_t)H * 64u * 2u;  // one fp16 partial block
  auto chunk_off = [&](int j, int ch, int c) -> uint32_t {  // staged block j, row ch, chunk c
    return (uint32_t)j * blk_bytes + (uint32_t)ch * (H * 2) + (uint32_t)((c ^ (ch & (kCr - 1))) << 4);
  };
  {
    const int qd = warp & 3, mb = warp >> 2;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const int ch = mb * 128 + qd * 32 + lane;  // this thread's channel
    float o[kHN];
    if (have_o) {  // all of the thread's columns: one tensor-memory round trip
#pragma unroll
      for (int h0 = 0; h0 < H; h0 += 16) tmem_ld16(tm_o + lane_base + mb * kHN + h0, o + h0);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int i = 0; i < kHN; ++i) o[i] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < H; i += 4) {
      const float4 li = *reinterpret_cast<const float4*>(&ctl.linv[i]);
      o[i] *= li.x;
      o[i + 1] *= li.y;
      o[i + 2] *= li.z;
      o[i + 3] *= li.w;
    }
    if (nsplit == 1) {
      float* orow = out + (int64_t)b * H * kD + ch;
#pragma unroll
      for (int i = 0; i < H; ++i) orow[(int64_t)i * kD] = o[i];
    } else {
#pragma unroll
      for (int c = 0; c < kCr; ++c)
        *reinterpret_cast<uint4*>(smem + L::v_off + chunk_off(ch >> 6, ch & 63, c)) =
            make_uint4(pack_f16x2(o[8 * c], o[8 * c + 1]), pack_f16x2(o[8 * c + 2], o[8 * c + 3]),
                       pack_f16x2(o[8 * c + 4], o[8 * c + 5]), pack_f16x2(o[8 * c + 6], o[8 * c + 7]));
    }
  }
  proxy_fence();  // the bulk copies read the staged blocks through the async proxy
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kIssuerWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));

  if (nsplit > 1) {
    // ---- merge of the query's splits (the cluster is the query's nsplit
    //      CTAs, nsplit a power of two): CTA `split` owns the 64-channel
    //      blocks j = split, split + nsplit, ...  Past a cluster barrier
    //      (every CTA's MMAs are done with V, whose upper part receives the
    //      blocks), each CTA pushes the blocks it does not own into their
    //      owners' shared memory with bulk copies that complete on the
    //      owner's mbarrier, then forms o = sum_s exp(lse_s - lse) o_s over
    //      its own blocks, lse the log-sum-exp of the lse_s ----
    const int n_own = 8 / nsplit;
    const uint32_t recv_s = sbase + L::v_off + 8 * blk_bytes;  // [source][own block]
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (tid == 0) {
      mbar_expect_tx(su32(&ctl.recv), (uint32_t)(nsplit - 1) * n_own * blk_bytes);
      for (int j = 0; j < 8; ++j) {
        const int owner = j % nsplit;
        if (owner == split) continue;
        // this split's slot among the owner's sources, block j / nsplit of the owner's
        const int slot = (split < owner ? split : split - 1) * n_own + j / nsplit;
        bulk_push(peer_smem(recv_s + (uint32_t)slot * blk_bytes, (uint32_t)owner),
                  sbase + L::v_off + j * blk_bytes, blk_bytes,
                  peer_smem(su32(&ctl.recv), (uint32_t)owner));
      }
    }
    // weights exp(lse_s - M) / sum (per split and head), in the free Q region
    float* wts = reinterpret_cast<float*>(smem + L::q_off);
    if (tid >= 32 && tid < 32 + H) {
      const int hh = tid - 32;
      const float* pl = part_lse + (int64_t)b * nsplit * H + hh;
      float lv[kMaxSplitTc];
#pragma unroll
      for (int s2 = 0; s2 < kMaxSplitTc; ++s2)
        lv[s2] = s2 < nsplit ? __ldcg(pl + (int64_t)s2 * H) : -INFINITY;
      float m = -INFINITY;
#pragma unroll
      for (int s2 = 0; s2 < kMaxSplitTc; ++s2) m = fmaxf(m, lv[s2]);
      float sum = 0.0f;
#pragma unroll
      for (int s2 = 0; s2 < kMaxSplitTc; ++s2) {
        lv[s2] = m == -INFINITY ? 0.0f : expf(lv[s2] - m);
        sum += lv[s2];
      }
      const float inv = sum > 0.0f ? 1.0f / sum : 0.0f;
#pragma unroll
      for (int s2 = 0; s2 < kMaxSplitTc; ++s2)
        if (s2 < nsplit) wts[s2 * 64 + hh] = lv[s2] * inv;
      if (split == 0 && lse) lse[(int64_t)b * H + hh] = sum > 0.0f ? m + logf(sum) : -INFINITY;
    }
    __syncthreads();
    const bool got = __all_sync(0xffffffffu, mbar_wait(su32(&ctl.recv), 0u, status));
    // every block pushed to this CTA has landed; the matching wait below keeps
    // this CTA's staged blocks alive until every peer's have too
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    // warp w: channels 32 (w & 1) .. +32 of a block (lane = channel), heads
    // 8 (w >> 1) .. +8; for each head the warp stores one 128-byte line
    const int cc = 32 * (warp & 1) + lane, c8 = warp >> 1;
    if (c8 < kCr) {
      for (int kk = 0; kk < n_own; ++kk) {
        const int j = split + kk * nsplit;
        float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        for (int s2 = 0, slot = 0; s2 < nsplit; ++s2) {
          uint32_t off;
          if (s2 == split) {
            off = L::v_off + chunk_off(j, cc, c8);
          } else {
            off = L::v_off + 8 * blk_bytes + (uint32_t)(slot * n_own + kk) * blk_bytes +
                  chunk_off(0, cc, c8);
            ++slot;
          }
          const uint4 v = *reinterpret_cast<const uint4*>(smem + off);
          const float4 w0 = *reinterpret_cast<const float4*>(wts + s2 * 64 + 8 * c8);
          const float4 w1 = *reinterpret_cast<const float4*>(wts + s2 * 64 + 8 * c8 + 4);
          const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = half2_bits_to_float2(u[q]);
            acc[2 * q] = fmaf(got ? wv[2 * q] : 0.0f, f.x, acc[2 * q]);
            acc[2 * q + 1] = fmaf(got ? wv[2 * q + 1] : 0.0f, f.y, acc[2 * q + 1]);
          }
        }
        float* orow = out + ((int64_t)b * H + 8 * c8) * kD + 64 * j + cc;
#pragma unroll
        for (int i = 0; i < 8; ++i) orow[(int64_t)i * kD] = acc[i];
      }
    }
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  }
}

}  // namespace

template <int H>
static cudaError_t launch_tc_t(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int64_t N,
                               int64_t kv_seq_stride, int q_per_seq, const int32_t* idx, int k,
                               int nsplit, int chunk, float scale_log2, float* out, float* lse,
                               float* part_lse, int32_t* status,
                               const SwaArgs* swa, int32_t* idx_copy, cudaStream_t stream,
                               bool pdl) {
  using L = TcLayout;
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_tc_kernel<H>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::alloc);
  if (e != cudaSuccess) return e;
  // a query's splits run as one thread-block cluster, which merges them
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nsplit, (unsigned)B);
  cfg.blockDim = dim3(kThreadsTc);
  cfg.dynamicSmemBytes = L::alloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  if (nsplit > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)nsplit;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, sparse_attn_tc_kernel<H>, q_bf16, kv_fp4, N, kv_seq_stride,
                            q_per_seq, idx, k, chunk, scale_log2, out, lse, part_lse,
                            status, swa ? swa->kv : nullptr, swa ? swa->ring : (int64_t)0,
                            swa ? swa->n_win : 0, swa ? swa->q_pos : nullptr, idx_copy);
}

cudaError_t launch_sparse_attn_tc(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H,
                                  int64_t N, int64_t kv_seq_stride, int q_per_seq,
                                  const int32_t* idx, int k, int nsplit, int chunk,
                                  float scale_log2, float* out, float* lse, float* part_lse,
                                  int32_t* status, const SwaArgs* swa, int32_t* idx_copy,
                                  cudaStream_t stream, bool pdl) {
  switch (H) {
    case 16:
      return launch_tc_t<16>(q_bf16, kv_fp4, B, N, kv_seq_stride, q_per_seq, idx, k, nsplit,
                             chunk, scale_log2, out, lse, part_lse, status, swa, idx_copy,
                             stream, pdl);
    case 32:
      return launch_tc_t<32>(q_bf16, kv_fp4, B, N, kv_seq_stride, q_per_seq, idx, k, nsplit,
                             chunk, scale_log2, out, lse, part_lse, status, swa, idx_copy,
                             stream, pdl);
    default:
      return launch_tc_t<64>(q_bf16, kv_fp4, B, N, kv_seq_stride, q_per_seq, idx, k, nsplit,
                             chunk, scale_log2, out, lse, part_lse, status, swa, idx_copy,
                             stream, pdl);
  }
}

}  // namespace csa2
