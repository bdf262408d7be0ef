// pa_e4m3.cuh -- the E4M3 row quantiser shared by the append kernels and the
// fused append + decode kernel, so both store bit-identical codes and scales.
//
// A row of D fp16 values is spread over a warp, D/32 values per lane.  A row
// that opens its page sets the page scale amax(|row|)/448 (fp32, IEEE
// division; 1 when amax is 0); later rows reuse the stored scale.  Codes are
// E4M3(x / scale): the quotient rounded to fp32 by IEEE division, the code
// rounded to nearest even and saturated at +-448 ("rvLLM: High-performance
// LLM inference in Rust", CUDA Kernels table, "FP8 KV Cache"; "LLM Serving
// Kernels", Projects table, row 05).
#pragma once

#include "pa_ptx.cuh"

namespace pa {

template <int D>
struct RowF16 {
  static constexpr int PER_LANE = D / 32;   // 2 or 4 values per lane
  float x[PER_LANE];
};

// Lane's D/32 values of an fp16 row at `src` (the row base).
template <int D>
__device__ __forceinline__ RowF16<D> load_row_f16(const __half* row, int lane) {
  RowF16<D> r;
  const __half* src = row + lane * RowF16<D>::PER_LANE;
  if constexpr (RowF16<D>::PER_LANE == 4) {
    const uint2 raw = *reinterpret_cast<const uint2*>(src);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    r.x[0] = a.x; r.x[1] = a.y; r.x[2] = b.x; r.x[3] = b.y;
  } else {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(src));
    r.x[0] = a.x; r.x[1] = a.y;
  }
  return r;
}

// Page scale a row sets when it opens its page (all lanes get it).
template <int D>
__device__ __forceinline__ float e4m3_row_scale(const RowF16<D>& r) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < RowF16<D>::PER_LANE; ++j) amax = fmaxf(amax, fabsf(r.x[j]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  return amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
}

// The lane's codes packed low byte first (4 bytes for D=128, 2 for D=64).
template <int D>
__device__ __forceinline__ uint32_t e4m3_row_codes(const RowF16<D>& r, float scale) {
  const uint32_t c01 = f32x2_to_e4m3x2(__fdiv_rn(r.x[0], scale), __fdiv_rn(r.x[1], scale));
  if constexpr (RowF16<D>::PER_LANE == 4) {
    const uint32_t c23 = f32x2_to_e4m3x2(__fdiv_rn(r.x[2], scale), __fdiv_rn(r.x[3], scale));
    return c01 | (c23 << 16);
  } else {
    return c01;
  }
}

template <int D>
__device__ __forceinline__ void store_row_codes(uint8_t* row, int lane, uint32_t codes) {
  if constexpr (RowF16<D>::PER_LANE == 4)
    *reinterpret_cast<uint32_t*>(row + 4 * lane) = codes;
  else
    *reinterpret_cast<uint16_t*>(row + 2 * lane) = static_cast<uint16_t>(codes);
}

}  // namespace pa
