// Blockwise candidate pool of the Hierarchical Sparse Indexer (DeepSeek-V4.1-
// Flash paper walkthrough, 1.(4).2): the first Full layer scores every
// visible entry; a block's score is the largest score among its entries; the
// best blocks are kept and the entries they cover form the pool that later
// Reindex layers score.  Blocks are aligned runs of `block` entries; only
// visible entries count; ties keep the lower block index; the pool lists the
// visible entries of the kept blocks in ascending order, padded with -1.
//
// Three launches: block maxima (+ the number of blocks holding a visible
// entry), the radix top-k over block scores, and the expansion of the kept
// blocks into entries.  Only the last visible block can be partly visible and
// it is the highest kept block, so its missing entries fall at the tail.
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kBpThreads = 256;

__global__ void __launch_bounds__(kBpThreads)
block_max_kernel(const float* __restrict__ scores, int64_t N, const int32_t* __restrict__ q_pos,
                 int ratio, int block, int64_t nblk, float* __restrict__ bscores,
                 int32_t* __restrict__ n_valid) {
  pdl_trigger();
  pdl_wait();  // the scores come from the kernel before
  const int b = blockIdx.y;
  const int64_t nv = n_visible(q_pos, b, ratio, N);
  const int64_t nb = (nv + block - 1) / block;
  const int64_t j = (int64_t)blockIdx.x * kBpThreads + threadIdx.x;
  if (blockIdx.x == 0 && threadIdx.x == 0) n_valid[b] = (int32_t)nb;
  if (j >= nblk) return;
  float m = -INFINITY;
  if (j < nb) {
    const float* row = scores + (int64_t)b * N;
    const int64_t e1 = min((j + 1) * block, nv);
    for (int64_t e = j * block; e < e1; ++e) m = fmaxf(m, row[e]);
  }
  bscores[(int64_t)b * nblk + j] = m;
}

__global__ void __launch_bounds__(kBpThreads)
pool_expand_kernel(const int32_t* __restrict__ blk, int n_blocks, int block, int64_t N,
                   const int32_t* __restrict__ q_pos, int ratio, int32_t* __restrict__ pool) {
  pdl_trigger();
  pdl_wait();  // the kept blocks come from the kernel before
  const int b = blockIdx.y;
  const int64_t P = (int64_t)n_blocks * block;
  const int64_t s = (int64_t)blockIdx.x * kBpThreads + threadIdx.x;
  if (s >= P) return;
  const int64_t nv = n_visible(q_pos, b, ratio, N);
  const int32_t kb = blk[(int64_t)b * n_blocks + s / block];
  const int64_t e = (int64_t)kb * block + s % block;
  pool[(int64_t)b * P + s] = (kb >= 0 && e < nv) ? (int32_t)e : -1;
}

}  // namespace

size_t block_pool_scratch_bytes(int B, int64_t N, int block, int n_blocks) {
  if (B <= 0 || N < 0 || block < 1 || n_blocks < 1) return 0;
  const int64_t nblk = (N + block - 1) / block;
  return align_up((size_t)B * nblk * 4, 256) + align_up((size_t)B * 4, 256) +
         align_up((size_t)B * n_blocks * 4, 256);
}

BlockPoolScratch block_pool_scratch(void* base, int B, int64_t N, int block, int n_blocks) {
  BlockPoolScratch s;
  uint8_t* p = reinterpret_cast<uint8_t*>(base);
  const int64_t nblk = (N + block - 1) / block;
  s.bscores = reinterpret_cast<float*>(p);
  p += align_up((size_t)B * nblk * 4, 256);
  s.n_valid = reinterpret_cast<int32_t*>(p);
  p += align_up((size_t)B * 4, 256);
  s.blk = reinterpret_cast<int32_t*>(p);
  p += align_up((size_t)B * n_blocks * 4, 256);
  s.bytes = (size_t)(p - reinterpret_cast<uint8_t*>(base));
  return s;
}

cudaError_t launch_block_pool(const float* scores, int B, int64_t N, const int32_t* q_pos,
                              int ratio, int block, int n_blocks, int32_t* pool, void* scratch,
                              cudaStream_t stream, bool pdl) {
  if (B == 0) return cudaSuccess;
  const BlockPoolScratch s = block_pool_scratch(scratch, B, N, block, n_blocks);
  const int64_t nblk = (N + block - 1) / block;
  cudaError_t e = launch_kernel(block_max_kernel,
                                dim3((unsigned)((nblk + kBpThreads - 1) / kBpThreads), (unsigned)B),
                                dim3(kBpThreads), 0, stream, pdl, scores, N, q_pos, ratio, block,
                                nblk, s.bscores, s.n_valid);
  if (e != cudaSuccess) return e;
  e = launch_topk(s.bscores, B, nblk, n_blocks, nullptr, 1, s.n_valid, nullptr, s.blk, stream,
                  true);
  if (e != cudaSuccess) return e;
  const int64_t P = (int64_t)n_blocks * block;
  return launch_kernel(pool_expand_kernel,
                       dim3((unsigned)((P + kBpThreads - 1) / kBpThreads), (unsigned)B),
                       dim3(kBpThreads), 0, stream, true, s.blk, n_blocks, block, N, q_pos, ratio,
                       pool);
}

}  // namespace csa2
