// pa_e4m3.cuh -- the E4M3 row quantiser shared by the append kernels and the
// fused append + decode kernel, so both store bit-identical codes and scales.
//
// A row of D values (fp16 or bf16) is spread over a warp, D/32 values per
// lane.  Per page (block, kv head) and pool:
//   - a row that opens its page sets the page scale amax(|row|) / 448 (fp32,
//     IEEE division; 1 when amax is 0);
//   - a later row is encoded with the stored scale s when fl32(amax / s) <= 448
//     (no element saturates);
//   - otherwise the page is re-scaled first: s' = amax / 448, and each code c of
//     the page's earlier rows becomes E4M3(fl32(fl32(e4m3(c) * s) / s')).
// Codes are E4M3(x / scale): the quotient rounded to fp32 by IEEE division, the
// code rounded to nearest even and saturated at +-448 ("rvLLM: High-performance
// LLM inference in Rust", CUDA Kernels table, "FP8 KV Cache"; "LLM Serving
// Kernels", Projects table, row 05, E4M3 storage with page scales).
#pragma once

#include "pa_ptx.cuh"

namespace pa {

template <int D>
struct RowF16 {
  static constexpr int PER_LANE = D / 32;   // 2 or 4 values per lane
  float x[PER_LANE];
};

template <bool BF16>
__device__ __forceinline__ float2 bits2_to_float2(uint32_t w) {
  if constexpr (BF16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
}

// The lane's D/32 values of a row whose 16-bit bits the lane holds (two
// values per 32-bit word, low half first).
template <int D, bool BF16>
__device__ __forceinline__ RowF16<D> row_from_bits(uint2 raw) {
  RowF16<D> r;
  const float2 a = bits2_to_float2<BF16>(raw.x);
  r.x[0] = a.x;
  r.x[1] = a.y;
  if constexpr (RowF16<D>::PER_LANE == 4) {
    const float2 b = bits2_to_float2<BF16>(raw.y);
    r.x[2] = b.x;
    r.x[3] = b.y;
  }
  return r;
}

// Lane's D/32 values of a 16-bit row at `row` (the row base).
template <int D, bool BF16>
__device__ __forceinline__ RowF16<D> load_row(const uint16_t* row, int lane) {
  const uint16_t* src = row + lane * RowF16<D>::PER_LANE;
  uint2 raw = make_uint2(0, 0);
  if constexpr (RowF16<D>::PER_LANE == 4)
    raw = *reinterpret_cast<const uint2*>(src);
  else
    raw.x = *reinterpret_cast<const uint32_t*>(src);
  return row_from_bits<D, BF16>(raw);
}

// amax(|row|) over the warp (all lanes get it).
template <int D>
__device__ __forceinline__ float e4m3_row_amax(const RowF16<D>& r) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < RowF16<D>::PER_LANE; ++j) amax = fmaxf(amax, fabsf(r.x[j]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  return amax;
}

__device__ __forceinline__ float e4m3_page_scale(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
}

// Whether a row with this amax would saturate under page scale s.
__device__ __forceinline__ bool e4m3_saturates(float amax, float s) {
  return __fdiv_rn(amax, s) > 448.f;
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
__device__ __forceinline__ uint32_t load_row_codes(const uint8_t* row, int lane) {
  if constexpr (RowF16<D>::PER_LANE == 4)
    return *reinterpret_cast<const uint32_t*>(row + 4 * lane);
  else
    return *reinterpret_cast<const uint16_t*>(row + 2 * lane);
}

template <int D>
__device__ __forceinline__ void store_row_codes(uint8_t* row, int lane, uint32_t codes) {
  if constexpr (RowF16<D>::PER_LANE == 4)
    *reinterpret_cast<uint32_t*>(row + 4 * lane) = codes;
  else
    *reinterpret_cast<uint16_t*>(row + 2 * lane) = static_cast<uint16_t>(codes);
}

// Two codes from scale s_old to scale s_new.
__device__ __forceinline__ uint32_t e4m3x2_rescale(uint32_t two, float s_old, float s_new) {
  const uint32_t h = e4m3x2_to_f16x2(two);
  const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&h));
  return f32x2_to_e4m3x2(__fdiv_rn(__fmul_rn(v.x, s_old), s_new),
                         __fdiv_rn(__fmul_rn(v.y, s_old), s_new));
}

// Re-encode rows [0, nrows) of a page (nrows < 16; D codes a row, rows
// contiguous) from s_old to s_new.  Reads src, writes dst and, when non-null,
// dst2 (src may equal dst: each lane rewrites only its own bytes).  From
// global memory (BATCH) all rows are read before any is written, so the
// reads are in flight together; from shared memory one row at a time.
template <int D, bool BATCH>
__device__ __forceinline__ void e4m3_rescale_rows(const uint8_t* src, uint8_t* dst, uint8_t* dst2,
                                                  int nrows, float s_old, float s_new, int lane) {
  auto rescale = [&](uint32_t c) {
    uint32_t n = e4m3x2_rescale(c & 0xffffu, s_old, s_new);
    if constexpr (RowF16<D>::PER_LANE == 4) n |= e4m3x2_rescale(c >> 16, s_old, s_new) << 16;
    return n;
  };
  if constexpr (BATCH) {
    uint32_t c[15];
#pragma unroll
    for (int j = 0; j < 15; ++j) c[j] = j < nrows ? load_row_codes<D>(src + j * D, lane) : 0u;
#pragma unroll
    for (int j = 0; j < 15; ++j) {
      if (j >= nrows) break;
      const uint32_t n = rescale(c[j]);
      store_row_codes<D>(dst + j * D, lane, n);
      if (dst2 != nullptr) store_row_codes<D>(dst2 + j * D, lane, n);
    }
  } else {
    for (int j = 0; j < nrows; ++j) {
      const uint32_t n = rescale(load_row_codes<D>(src + j * D, lane));
      store_row_codes<D>(dst + j * D, lane, n);
      if (dst2 != nullptr) store_row_codes<D>(dst2 + j * D, lane, n);
    }
  }
}

}  // namespace pa
