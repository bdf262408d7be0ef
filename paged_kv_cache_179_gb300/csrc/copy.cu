// copy.cu -- whole-block copies inside the paged pools.
//
// "rvLLM: High-performance LLM inference in Rust", CUDA Kernels table,
// "Block Copy" (KV cache block copy for beam search) and Architecture,
// rvllm-block-manager (block allocation, copy-on-write, prefix sharing):
// when a sequence forks (a beam, a parallel sample, a shared prefix that is
// about to be written), the block manager gives the writer a fresh physical
// block and the cache contents of the shared one are copied into it.
//
// For each pair (src, dst) of block_mapping, every kv head's 16 rows of K
// and of V (and, for E4M3 pools, the block's K and V scales) are copied from
// physical block src to physical block dst.  HBM-bound: one read and one
// write of each byte.  One CTA per (pair, K|V) streams the block with
// coalesced 16-byte loads and stores that bypass L1 and mark the lines
// evict-first (the copied data is not read again by this kernel).
#include "pa_launch.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                   float* __restrict__ k_scale, float* __restrict__ v_scale,
                   const int64_t* __restrict__ pairs, int64_t chunks_per_block, int Hkv,
                   int64_t num_blocks, unsigned* status) {
  const int64_t pair = blockIdx.x >> 1;
  const int kv = blockIdx.x & 1;
  const int64_t src = __ldg(pairs + 2 * pair);
  const int64_t dst = __ldg(pairs + 2 * pair + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && kv == 0) atomicOr(status, kStatusBadBlock);
    return;
  }
  if (src == dst) return;
  uint4* pool = kv ? v_cache : k_cache;
  const uint4* from = pool + src * chunks_per_block;
  uint4* to = pool + dst * chunks_per_block;
  // up to four loads in flight per thread before its stores
  for (int64_t base = 0; base < chunks_per_block; base += 4 * kCopyThreads) {
    uint4 r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t i = base + threadIdx.x + j * kCopyThreads;
      if (i < chunks_per_block) r[j] = __ldcs(from + i);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t i = base + threadIdx.x + j * kCopyThreads;
      if (i < chunks_per_block) __stcs(to + i, r[j]);
    }
  }
  float* scales = kv ? v_scale : k_scale;
  if (scales != nullptr && threadIdx.x < Hkv)
    scales[dst * Hkv + threadIdx.x] = scales[src * Hkv + threadIdx.x];
}

}  // namespace

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                               const int64_t* pairs, int num_pairs, int Hkv, int row_bytes,
                               int block_size, int64_t num_blocks, unsigned* status,
                               cudaStream_t s) {
  const int64_t chunks = static_cast<int64_t>(Hkv) * block_size * row_bytes / 16;
  copy_blocks_kernel<<<static_cast<unsigned>(2 * static_cast<int64_t>(num_pairs)), kCopyThreads,
                       0, s>>>(static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                               k_scale, v_scale, pairs, chunks, Hkv, num_blocks, status);
  return cudaGetLastError();
}

}  // namespace pa
