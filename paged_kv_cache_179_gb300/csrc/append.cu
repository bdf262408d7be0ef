// append.cu -- K1: scatter the step's new K/V rows into the paged pools.
//
// "rvLLM: High-performance LLM inference in Rust", CUDA Kernels table,
// "Reshape and Cache": write the new K/V into the paged cache; "rvllm - A
// Small LLM Inference Engine in Rust", How it's put together: every forward
// takes explicit write positions computed from the block table.  The FP8 form
// encodes the row as E4M3 with a per-(page, kv head) scale (rvLLM, "FP8 KV
// Cache" row; "LLM Serving Kernels", Projects row 05).
//
// Both kernels move a few hundred KB per decode step; they are launch- and
// latency-bound, so they are written for few instructions per byte and fully
// coalesced 16-byte accesses, nothing more.
#include "pa_e4m3.cuh"
#include "pa_launch.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

// One thread per 16-byte chunk of one (token, kv head) row, K and V together.
__global__ void __launch_bounds__(256)
append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
              uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
              const int64_t* __restrict__ slots, int T, int Hkv, int chunks_per_row,
              int block_size, int64_t num_slots, unsigned* status) {
  // a decode launched next with an early prologue may start its prologue now
  // (it waits for this launch to complete before reading the pools)
  griddep_launch_dependents();
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t per_tok = static_cast<int64_t>(Hkv) * chunks_per_row;
  if (idx >= per_tok * T) return;
  const int64_t i = idx / per_tok;
  const int64_t rem = idx - i * per_tok;
  const int64_t h = rem / chunks_per_row;
  const int64_t c = rem - h * chunks_per_row;
  const int64_t s = slots[i];
  if (s < 0) return;                       // padding token
  if (s >= num_slots) {
    if (h == 0 && c == 0) atomicOr(status, kStatusBadSlot);
    return;
  }
  const int64_t blk = s / block_size, row = s - blk * block_size;
  const int64_t dst = ((blk * Hkv + h) * block_size + row) * chunks_per_row + c;
  const int64_t src = (i * Hkv + h) * chunks_per_row + c;
  k_cache[dst] = k_new[src];
  v_cache[dst] = v_new[src];
}

// One warp per (token, kv head, K|V) row of head_dim 16-bit values; a row
// that would saturate under its page's scale re-scales the page first.
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
append_fp8_kernel(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                  uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                  float* __restrict__ k_scale, float* __restrict__ v_scale,
                  const int64_t* __restrict__ slots, int T, int Hkv, int block_size,
                  int64_t num_slots, unsigned* status) {
  griddep_launch_dependents();   // as in append_kernel
  const int lane = threadIdx.x & 31;
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (w >= static_cast<int64_t>(T) * Hkv * 2) return;
  const int kv = static_cast<int>(w & 1);
  const int64_t th = w >> 1;
  const int64_t i = th / Hkv, h = th - i * Hkv;
  const int64_t s = slots[i];
  if (s < 0) return;
  if (s >= num_slots) {
    if (lane == 0 && kv == 0 && h == 0) atomicOr(status, kStatusBadSlot);
    return;
  }
  const int64_t blk = s / block_size, row = s - blk * block_size;
  const RowF16<D> x = load_row<D, BF16>((kv ? v_new : k_new) + (i * Hkv + h) * D, lane);
  float* scales = kv ? v_scale : k_scale;
  const int64_t tile = blk * Hkv + h;
  uint8_t* page = (kv ? v_cache : k_cache) + tile * block_size * D;
  const float amax = e4m3_row_amax<D>(x);
  float scale;
  if (row == 0) {
    scale = e4m3_page_scale(amax);
    if (lane == 0) scales[tile] = scale;
  } else {
    scale = scales[tile];
    if (e4m3_saturates(amax, scale)) {   // re-scale the page's earlier rows first
      const float s_new = e4m3_page_scale(amax);
      e4m3_rescale_rows<D, true>(page, page, nullptr, static_cast<int>(row), scale, s_new, lane);
      scale = s_new;
      if (lane == 0) scales[tile] = scale;
    }
  }
  store_row_codes<D>(page + row * D, lane, e4m3_row_codes<D>(x, scale));
}

}  // namespace

cudaError_t launch_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                          const int64_t* slots, int T, int Hkv, int row_bytes, int block_size,
                          int64_t num_blocks, unsigned* status, cudaStream_t s) {
  const int chunks = row_bytes / 16;
  const int64_t n = static_cast<int64_t>(T) * Hkv * chunks;
  const int threads = 256;
  const int64_t grid = (n + threads - 1) / threads;
  append_kernel<<<static_cast<unsigned>(grid), threads, 0, s>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slots, T, Hkv, chunks,
      block_size, num_blocks * block_size, status);
  return cudaGetLastError();
}

cudaError_t launch_append_fp8(const void* k_new, const void* v_new, uint8_t* k_cache,
                              uint8_t* v_cache, float* k_scale, float* v_scale,
                              const int64_t* slots, int T, int Hkv, int D, int block_size,
                              int64_t num_blocks, bool bf16, unsigned* status, cudaStream_t s) {
  const int64_t warps = static_cast<int64_t>(T) * Hkv * 2;
  const int threads = 256;
  const unsigned grid = static_cast<unsigned>((warps * 32 + threads - 1) / threads);
  const auto* kn = static_cast<const uint16_t*>(k_new);
  const auto* vn = static_cast<const uint16_t*>(v_new);
  const int64_t ns = num_blocks * block_size;
#define PA_APPEND_FP8(DD, BB)                                                              \
  append_fp8_kernel<DD, BB><<<grid, threads, 0, s>>>(kn, vn, k_cache, v_cache, k_scale, v_scale, \
                                                     slots, T, Hkv, block_size, ns, status)
  if (D == 128) {
    if (bf16) PA_APPEND_FP8(128, true);
    else PA_APPEND_FP8(128, false);
  } else {
    if (bf16) PA_APPEND_FP8(64, true);
    else PA_APPEND_FP8(64, false);
  }
#undef PA_APPEND_FP8
  return cudaGetLastError();
}

}  // namespace pa
