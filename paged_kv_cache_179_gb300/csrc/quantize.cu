// quantize.cu -- K2: bulk E4M3 page quantisation of an fp16 pool, and the
// bare E4M3 encoder.
//
// "rvLLM: High-performance LLM inference in Rust", CUDA Kernels table, "FP8
// KV Cache" (E4M3 quantisation of the KV cache) and feature list "per-head
// scaling"; "LLM Serving Kernels", Projects table, row 05 ("E4M3 storage,
// page scales").  One scale per (physical block, kv head) tile:
//   scale = amax / 448 (fp32; 1 when amax == 0), code = E4M3_RNE_sat(x / scale)
// with the quotient rounded to fp32 (IEEE division, never a reciprocal).
//
// HBM-bound: 2 bytes read and 1 byte written per element.  One warp owns a
// tile (16 rows x head_dim), reads it with coalesced 16-byte loads, reduces
// amax with shuffles and writes the codes with coalesced 8-byte stores.
#include "pa_launch.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

template <int CHUNKS>   // 16-byte chunks per lane: tile_elems / 256
__global__ void __launch_bounds__(256)
quantize_fp8_kernel(const uint4* __restrict__ src, uint2* __restrict__ codes,
                    float* __restrict__ scales, int64_t num_tiles) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       t < num_tiles; t += warps_total) {
    const uint4* tile = src + t * (CHUNKS * 32);
    uint4 v[CHUNKS];
#pragma unroll
    for (int k = 0; k < CHUNKS; ++k) v[k] = __ldcs(tile + lane + 32 * k);
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < CHUNKS; ++k) {
      const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    if (lane == 0) scales[t] = scale;
    uint2* out = codes + t * (CHUNKS * 32);
#pragma unroll
    for (int k = 0; k < CHUNKS; ++k) {
      const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
      uint32_t c[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
        c[j] = f32x2_to_e4m3x2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale));
      }
      __stcs(out + lane + 32 * k, make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16)));
    }
  }
}

__global__ void __launch_bounds__(256)
e4m3_encode_kernel(const float* __restrict__ x, uint8_t* __restrict__ codes, int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t n4 = n / 4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += stride) {
    const float4 v = reinterpret_cast<const float4*>(x)[i];
    const uint32_t lo = f32x2_to_e4m3x2(v.x, v.y), hi = f32x2_to_e4m3x2(v.z, v.w);
    reinterpret_cast<uint32_t*>(codes)[i] = lo | (hi << 16);
  }
  const int64_t tail = n4 * 4 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (tail < n) codes[tail] = static_cast<uint8_t>(f32x2_to_e4m3x2(x[tail], 0.f));
}

}  // namespace

cudaError_t launch_quantize_fp8(const void* src, uint8_t* codes, float* scales,
                                int64_t num_tiles, int tile_elems, cudaStream_t s) {
  if (num_tiles == 0) return cudaSuccess;
  const int threads = 256, warps_per_cta = threads / 32;
  const int64_t want = (num_tiles + warps_per_cta - 1) / warps_per_cta;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  const auto* in = static_cast<const uint4*>(src);
  auto* out = reinterpret_cast<uint2*>(codes);
  if (tile_elems == 16 * 128)
    quantize_fp8_kernel<8><<<grid, threads, 0, s>>>(in, out, scales, num_tiles);
  else
    quantize_fp8_kernel<4><<<grid, threads, 0, s>>>(in, out, scales, num_tiles);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_encode(const float* x, uint8_t* codes, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t want = (n / 4 + threads) / threads;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 32;
  const unsigned grid = static_cast<unsigned>(want < cap ? (want > 0 ? want : 1) : cap);
  e4m3_encode_kernel<<<grid, threads, 0, s>>>(x, codes, n);
  return cudaGetLastError();
}

}  // namespace pa
