// decode.cu -- K3/K4: split-K paged GQA decode (16-bit and E4M3 pools) and
// K5: the log-sum-exp merge of partitions.
//
// What is computed ("rvLLM: High-performance LLM inference in Rust", CUDA
// Kernels table, "PagedAttention V2": attention with block-table
// indirection and online softmax; "LLM Serving Kernels", Projects row 04:
// page tables, GQA/MQA, online softmax; row 05: fused E4M3 dequantisation;
// "rvllm - A Small LLM Inference Engine in Rust", How it's put together: each
// KV head serves a group of query heads):
//   out[b][hq] = sum_t softmax_t(scale * q[b][hq] . K_t) V_t,
//   t < context_lens[b], K_t in block block_tables[b][t/16], row t%16,
//   kv head hq / group.
//
// Design (sm_103a, one GB300):
//  * One CTA = one (sequence, kv head, context partition).  It serves the
//    whole query group, so every K/V byte is read from HBM once.
//  * Four warps split the partition's blocks round-robin.  Each warp owns a
//    private ring of STAGES shared-memory slots; lane 0 fetches one (block,
//    kv head) K tile and V tile per slot with two bulk asynchronous copies
//    (the TMA engine, cp.async.bulk) that complete on the slot's mbarrier.
//    No cross-warp synchronisation inside the main loop.
//  * Per 16-token block the warp computes S^T = K Q^T (16 tokens x 8 query
//    heads) and O^T += V^T P^T (head_dim x 8) with mma.sync m16n8k16,
//    fp32 accumulation.  The query group (<= 8 heads) is the N=8 side, so no
//    tensor-core row is wasted on padding beyond G < 8.  The online softmax
//    runs on the S fragments (max across lanes with shuffles, exp2 on the
//    SFU); P goes from accumulator to operand layout with movmatrix.
//    For E4M3 pools the codes are widened to f16 in registers (exact) right
//    before the MMA; the page scales are folded into the score scale (K) and
//    into P (V).
//  * The warps' partial (max, sum, acc) are combined in shared memory; a
//    sequence with one partition writes its output directly, otherwise the
//    partial goes to the workspace and merge_kernel combines partitions.
//
// Bounds: block ids outside [0, num_blocks) and context lengths above their
// bounds are never dereferenced; they set a status bit.  Every mbarrier wait
// is bounded (kWaitLimit) and reports kStatusTimeout instead of hanging.
#include <cfloat>
#include <type_traits>

#include "pa_launch.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kGroupMax = 8;          // query heads per kv head served by one MMA N=8 tile
constexpr float kLog2e = 1.4426950408889634f;
// E4M3 path: P * v_scale is scaled by 2^8 before rounding to f16 so small
// weights stay in f16's normal range; the fp32 result is scaled back.  With
// fp16-sourced pools v_scale <= 65504/448, so P' <= 146.3 * 256 < 65504.
constexpr float kPBoost = 256.f;

template <int D, bool FP8>
struct Tile {
  static constexpr int ROW = FP8 ? D : 2 * D;   // bytes of one token row of one kv head
  static constexpr int BYTES = 16 * ROW;        // one (block, kv head) tile
  static constexpr int STAGES = FP8 ? 4 : 3;    // ring slots per warp
  static constexpr int SLOT = 2 * BYTES;        // K tile + V tile
  static constexpr int RING = kWarps * STAGES * SLOT;
  static constexpr int MERGE = kWarps * kGroupMax * (D + 2) * 4;
  static_assert(MERGE <= RING, "merge area must fit in the ring");
};

// d index of the O^T fragment rows (m-tile i, lane row r): low (row r) and
// high (row r + 8) halves.  Chosen so each lane's V reads are one or two
// contiguous 16-byte chunks of a token row.
template <int D, bool FP8>
__device__ __forceinline__ int d_lo(int i, int r) {
  if constexpr (FP8 && D == 128) return 16 * r + i;
  else return 8 * r + i;
}
template <int D, bool FP8>
__device__ __forceinline__ int d_hi(int i, int r) {
  if constexpr (FP8 && D == 128) return 16 * r + 8 + i;
  else if constexpr (D == 128) return 64 + 8 * r + i;
  else return 8 * r + 4 + i;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int k) {
  return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}
__device__ __forceinline__ uint32_t word(const uint2& v, int k) { return k == 0 ? v.x : v.y; }

template <int D>
struct WarpAcc {
  float o[D / 16][4];   // O^T fragments: (d_lo, g=2c), (d_lo, 2c+1), (d_hi, 2c), (d_hi, 2c+1)
  float m0, m1;         // running max (log2 units) of query heads 2c, 2c+1
  float l0, l1;         // this lane's share of the running sums
};

// One 16-token block already in shared memory: K tile at kt, V tile at vt.
template <int D, bool FP8, bool BF16>
__device__ __forceinline__ void attend_block(WarpAcc<D>& st, const uint32_t (&qf)[D / 16][2],
                                             uint32_t kt, uint32_t vt, int n_valid, float sl2,
                                             float v_mul, int r, int c) {
  using TL = Tile<D, FP8>;
  // ---- S^T = K Q^T : 16 tokens x 8 query heads, k = head_dim
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (!FP8) {
    // lane (r, c) reads 16-byte chunk 4i+c of rows r and r+8: d = 32i + 8c + 0..7
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      const uint4 ka = lds128(kt + r * TL::ROW + (4 * i + c) * 16);
      const uint4 kb = lds128(kt + (r + 8) * TL::ROW + (4 * i + c) * 16);
      mma16816<BF16>(acc, ka.x, kb.x, ka.y, kb.y, qf[2 * i][0], qf[2 * i][1]);
      mma16816<BF16>(acc, ka.z, kb.z, ka.w, kb.w, qf[2 * i + 1][0], qf[2 * i + 1][1]);
    }
  } else {
    // lane (r, c) reads 16 codes at byte 64i + 16c of rows r and r+8
#pragma unroll
    for (int i = 0; i < D / 64; ++i) {
      const uint4 ka = lds128(kt + r * TL::ROW + 64 * i + 16 * c);
      const uint4 kb = lds128(kt + (r + 8) * TL::ROW + 64 * i + 16 * c);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint32_t wa = word(ka, q4), wb = word(kb, q4);
        mma16816<false>(acc, e4m3x2_to_f16x2(wa), e4m3x2_to_f16x2(wb),
                        e4m3x2_to_f16x2(wa >> 16), e4m3x2_to_f16x2(wb >> 16),
                        qf[4 * i + q4][0], qf[4 * i + q4][1]);
      }
    }
  }

  // ---- online softmax on the fragment: this lane holds tokens r, r+8 of heads 2c, 2c+1
  float s0 = acc[0] * sl2, s1 = acc[1] * sl2, s2 = acc[2] * sl2, s3 = acc[3] * sl2;
  if (r >= n_valid) s0 = s1 = -INFINITY;
  if (r + 8 >= n_valid) s2 = s3 = -INFINITY;
  float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, o));
    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, o));
  }
  const float mn0 = fmaxf(st.m0, bm0), mn1 = fmaxf(st.m1, bm1);
  const float a0 = fast_exp2(st.m0 - mn0), a1 = fast_exp2(st.m1 - mn1);
  st.m0 = mn0;
  st.m1 = mn1;
  const float p0 = fast_exp2(s0 - mn0), p1 = fast_exp2(s1 - mn1);
  const float p2 = fast_exp2(s2 - mn0), p3 = fast_exp2(s3 - mn1);
  st.l0 = st.l0 * a0 + (p0 + p2);
  st.l1 = st.l1 * a1 + (p1 + p3);
#pragma unroll
  for (int i = 0; i < D / 16; ++i) {
    st.o[i][0] *= a0;
    st.o[i][1] *= a1;
    st.o[i][2] *= a0;
    st.o[i][3] *= a1;
  }
  // P as the B operand (k = token, n = head): an 8x8 transpose per token half
  const uint32_t b0 = movmatrix_trans(pack2<BF16 && !FP8>(p0 * v_mul, p1 * v_mul));
  const uint32_t b1 = movmatrix_trans(pack2<BF16 && !FP8>(p2 * v_mul, p3 * v_mul));

  // ---- O^T += V^T P^T : lane needs tokens 2c, 2c+1, 2c+8, 2c+9
  const int tk0 = 2 * c, tk1 = 2 * c + 1, tk2 = 2 * c + 8, tk3 = 2 * c + 9;
  if constexpr (!FP8) {
    constexpr int U = D / 64;   // 16-byte chunks per token row for this lane
    uint4 v[4][U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      v[0][u] = lds128(vt + tk0 * TL::ROW + (8 * u + r) * 16);
      v[1][u] = lds128(vt + tk1 * TL::ROW + (8 * u + r) * 16);
      v[2][u] = lds128(vt + tk2 * TL::ROW + (8 * u + r) * 16);
      v[3][u] = lds128(vt + tk3 * TL::ROW + (8 * u + r) * 16);
    }
    if (n_valid < 16) {   // rows past the context may hold anything, NaN included
      const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (tk0 >= n_valid) v[0][u] = z;
        if (tk1 >= n_valid) v[1][u] = z;
        if (tk2 >= n_valid) v[2][u] = z;
        if (tk3 >= n_valid) v[3][u] = z;
      }
    }
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      const int elo = i, ulo = 0;
      const int ehi = (D == 128) ? i : 4 + i, uhi = (D == 128) ? 1 : 0;
      const uint32_t sl = (elo & 1) ? 0x7632u : 0x5410u;
      const uint32_t sh = (ehi & 1) ? 0x7632u : 0x5410u;
      const uint32_t x0 = __byte_perm(word(v[0][ulo], elo >> 1), word(v[1][ulo], elo >> 1), sl);
      const uint32_t x1 = __byte_perm(word(v[0][uhi], ehi >> 1), word(v[1][uhi], ehi >> 1), sh);
      const uint32_t x2 = __byte_perm(word(v[2][ulo], elo >> 1), word(v[3][ulo], elo >> 1), sl);
      const uint32_t x3 = __byte_perm(word(v[2][uhi], ehi >> 1), word(v[3][uhi], ehi >> 1), sh);
      mma16816<BF16>(st.o[i], x0, x1, x2, x3, b0, b1);
    }
  } else {
    using VT = typename std::conditional<D == 128, uint4, uint2>::type;
    constexpr int VB = D / 8;   // bytes per lane per token row: 16 (D=128) or 8 (D=64)
    VT v[4];
    if constexpr (D == 128) {
      v[0] = lds128(vt + tk0 * TL::ROW + VB * r);
      v[1] = lds128(vt + tk1 * TL::ROW + VB * r);
      v[2] = lds128(vt + tk2 * TL::ROW + VB * r);
      v[3] = lds128(vt + tk3 * TL::ROW + VB * r);
    } else {
      v[0] = lds64(vt + tk0 * TL::ROW + VB * r);
      v[1] = lds64(vt + tk1 * TL::ROW + VB * r);
      v[2] = lds64(vt + tk2 * TL::ROW + VB * r);
      v[3] = lds64(vt + tk3 * TL::ROW + VB * r);
    }
    if (n_valid < 16) {
      VT z{};
      if (tk0 >= n_valid) v[0] = z;
      if (tk1 >= n_valid) v[1] = z;
      if (tk2 >= n_valid) v[2] = z;
      if (tk3 >= n_valid) v[3] = z;
    }
#pragma unroll
    for (int i = 0; i < D / 16; i += 2) {
      const int elo = i, ehi = (D == 128) ? 8 + i : 4 + i;
      // bytes [x[e], y[e], x[e+1], y[e+1]] for e even
      const uint32_t sl = (elo & 3) | ((4 + (elo & 3)) << 4) | (((elo & 3) + 1) << 8) |
                          ((5 + (elo & 3)) << 12);
      const uint32_t sh = (ehi & 3) | ((4 + (ehi & 3)) << 4) | (((ehi & 3) + 1) << 8) |
                          ((5 + (ehi & 3)) << 12);
      const uint32_t x01l = __byte_perm(word(v[0], elo >> 2), word(v[1], elo >> 2), sl);
      const uint32_t x01h = __byte_perm(word(v[0], ehi >> 2), word(v[1], ehi >> 2), sh);
      const uint32_t x23l = __byte_perm(word(v[2], elo >> 2), word(v[3], elo >> 2), sl);
      const uint32_t x23h = __byte_perm(word(v[2], ehi >> 2), word(v[3], ehi >> 2), sh);
      mma16816<false>(st.o[i], e4m3x2_to_f16x2(x01l), e4m3x2_to_f16x2(x01h),
                      e4m3x2_to_f16x2(x23l), e4m3x2_to_f16x2(x23h), b0, b1);
      mma16816<false>(st.o[i + 1], e4m3x2_to_f16x2(x01l >> 16), e4m3x2_to_f16x2(x01h >> 16),
                      e4m3x2_to_f16x2(x23l >> 16), e4m3x2_to_f16x2(x23h >> 16), b0, b1);
    }
  }
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

template <int D, bool FP8, bool BF16>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const DecodeArgs a) {
  using TL = Tile<D, FP8>;
  using OutT = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TL::RING);
  int* s_ids = reinterpret_cast<int*>(smem + TL::RING + kWarps * TL::STAGES * 8);
  const int max_blk = a.part_tokens / 16;
  float* s_ks = reinterpret_cast<float*>(s_ids + max_blk);
  float* s_vs = s_ks + max_blk;

  const int p = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, c = lane & 3;
  const int G = a.group;
  OutT* out_rows = static_cast<OutT*>(a.out) + (static_cast<int64_t>(b) * a.Hq + h * G) * D;

  const int L = a.context_lens[b];
  if (L < 0 || L > a.max_context_len || L > a.mbs * 16) {
    if (p == 0) {
      if (tid == 0) atomicOr(a.status, kStatusBadLen);
      for (int i = tid; i < G * D; i += kThreads) out_rows[i] = from_f32<OutT>(0.f);
    }
    return;
  }
  if (L == 0) {
    if (p == 0)
      for (int i = tid; i < G * D; i += kThreads) out_rows[i] = from_f32<OutT>(0.f);
    return;
  }
  const int nparts = (L + a.part_tokens - 1) / a.part_tokens;
  if (p >= nparts) return;
  const int tok0 = p * a.part_tokens;
  const int ntok = min(a.part_tokens, L - tok0);
  const int nblk = (ntok + 15) / 16;
  const int blk0 = tok0 / 16;

  // ---- query fragments (B operand of S^T = K Q^T): row g = r of the group
  uint32_t qf[D / 16][2];
  {
    const uint4* qrow = reinterpret_cast<const uint4*>(
        static_cast<const uint16_t*>(a.q) + (static_cast<int64_t>(b) * a.Hq + h * G + r) * D);
    const bool live = r < G;
    if constexpr (!FP8) {
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        const uint4 v = live ? __ldg(qrow + 4 * i + c) : make_uint4(0, 0, 0, 0);
        qf[2 * i][0] = v.x;
        qf[2 * i][1] = v.y;
        qf[2 * i + 1][0] = v.z;
        qf[2 * i + 1][1] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < D / 64; ++i) {
        const uint4 lo = live ? __ldg(qrow + 8 * i + 2 * c) : make_uint4(0, 0, 0, 0);
        const uint4 hi = live ? __ldg(qrow + 8 * i + 2 * c + 1) : make_uint4(0, 0, 0, 0);
        qf[4 * i + 0][0] = lo.x; qf[4 * i + 0][1] = lo.y;
        qf[4 * i + 1][0] = lo.z; qf[4 * i + 1][1] = lo.w;
        qf[4 * i + 2][0] = hi.x; qf[4 * i + 2][1] = hi.y;
        qf[4 * i + 3][0] = hi.z; qf[4 * i + 3][1] = hi.w;
      }
    }
  }

  // ---- this partition's block ids (and page scales) into shared memory
  const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.mbs + blk0;
  for (int i = tid; i < nblk; i += kThreads) {
    int id = bt[i];
    if (id < 0 || id >= a.num_blocks) {
      atomicOr(a.status, kStatusBadBlock);
      id = -1;
    }
    s_ids[i] = id;
    if constexpr (FP8) {
      const int64_t tile = static_cast<int64_t>(id) * a.Hkv + h;
      s_ks[i] = id >= 0 ? a.k_scale[tile] : 0.f;
      s_vs[i] = id >= 0 ? a.v_scale[tile] : 0.f;
    }
  }
  const uint32_t ring = smem_u32(smem) + warp * TL::STAGES * TL::SLOT;
  const uint32_t wbar = smem_u32(bars) + warp * TL::STAGES * 8;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < TL::STAGES; ++s) mbar_init(wbar + 8 * s, 1);
    mbar_init_fence();
  }
  __syncthreads();

  // ---- per-warp pipeline over blocks warp, warp + 4, ...
  const int nb_w = warp < nblk ? (nblk - warp + kWarps - 1) / kWarps : 0;
  const uint8_t* kbase = static_cast<const uint8_t*>(a.k_cache);
  const uint8_t* vbase = static_cast<const uint8_t*>(a.v_cache);
  const uint64_t pol = l2_policy_evict_first();
  auto issue = [&](int k) {   // lane 0 only
    const int j = warp + k * kWarps;
    const int s = k % TL::STAGES;
    const uint32_t bar = wbar + 8 * s;
    const int id = s_ids[j];
    if (id >= 0) {
      const int64_t off = (static_cast<int64_t>(id) * a.Hkv + h) * TL::BYTES;
      mbar_arrive_expect_tx(bar, 2 * TL::BYTES);
      bulk_g2s(ring + s * TL::SLOT, kbase + off, TL::BYTES, bar, pol);
      bulk_g2s(ring + s * TL::SLOT + TL::BYTES, vbase + off, TL::BYTES, bar, pol);
    } else {
      mbar_arrive(bar);
    }
  };
  if (lane == 0)
    for (int k = 0; k < min(TL::STAGES, nb_w); ++k) issue(k);

  WarpAcc<D> st;
#pragma unroll
  for (int i = 0; i < D / 16; ++i) st.o[i][0] = st.o[i][1] = st.o[i][2] = st.o[i][3] = 0.f;
  st.m0 = st.m1 = -INFINITY;
  st.l0 = st.l1 = 0.f;
  const float sl2_base = a.scale_log2;

  for (int k = 0; k < nb_w; ++k) {
    const int s = k % TL::STAGES;
    const uint32_t parity = (k / TL::STAGES) & 1;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(wbar + 8 * s, parity));
    if (!ok) {
      // Report, then wait (bounded) for this warp's copies still in flight.
      if (lane == 0) atomicOr(a.status, kStatusTimeout);
      for (int kk = k + 1; kk < min(k + TL::STAGES, nb_w); ++kk)
        (void)mbar_wait(wbar + 8 * (kk % TL::STAGES), (kk / TL::STAGES) & 1);
      break;
    }
    const int j = warp + k * kWarps;
    if (s_ids[j] >= 0) {
      const int n_valid = min(16, ntok - j * 16);
      float sl2 = sl2_base, v_mul = 1.f;
      if constexpr (FP8) {
        sl2 *= s_ks[j];
        v_mul = s_vs[j] * kPBoost;
      }
      attend_block<D, FP8, BF16>(st, qf, ring + s * TL::SLOT, ring + s * TL::SLOT + TL::BYTES,
                                 n_valid, sl2, v_mul, r, c);
    }
    __syncwarp();
    if (lane == 0 && k + TL::STAGES < nb_w) issue(k + TL::STAGES);
  }

  // ---- combine the four warps, then write the output or the partition's partial
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, o);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, o);
  }
  __syncthreads();   // every warp is done with its ring: reuse it
  float* mo = reinterpret_cast<float*>(smem);                 // [warp][g][D]
  float* mm = mo + kWarps * kGroupMax * D;                    // [warp][g]
  float* ml = mm + kWarps * kGroupMax;                        // [warp][g]
  {
    float* wo = mo + warp * kGroupMax * D;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      const int dl = d_lo<D, FP8>(i, r), dh = d_hi<D, FP8>(i, r);
      wo[(2 * c) * D + dl] = st.o[i][0];
      wo[(2 * c + 1) * D + dl] = st.o[i][1];
      wo[(2 * c) * D + dh] = st.o[i][2];
      wo[(2 * c + 1) * D + dh] = st.o[i][3];
    }
    if (r == 0) {
      mm[warp * kGroupMax + 2 * c] = st.m0;
      mm[warp * kGroupMax + 2 * c + 1] = st.m1;
      ml[warp * kGroupMax + 2 * c] = st.l0;
      ml[warp * kGroupMax + 2 * c + 1] = st.l1;
    }
  }
  __syncthreads();
  const float unboost = FP8 ? 1.f / kPBoost : 1.f;
  for (int idx = tid; idx < G * D; idx += kThreads) {
    const int g = idx / D, d = idx - g * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mm[w * kGroupMax + g]);
    float sum = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float e = fast_exp2(mm[w * kGroupMax + g] - M);
        sum += e * ml[w * kGroupMax + g];
        acc += e * mo[(w * kGroupMax + g) * D + d];
      }
    }
    acc *= unboost;
    if (nparts == 1) {
      out_rows[idx] = from_f32<OutT>(sum > 0.f ? acc / sum : 0.f);
    } else {
      const int64_t row = ((static_cast<int64_t>(b) * a.Hq + h * G + g) * a.max_parts + p);
      a.ws_acc[row * D + d] = acc;
      if (d == 0) {
        a.ws_ml[row * 2] = M;
        a.ws_ml[row * 2 + 1] = sum;
      }
    }
  }
}

// K5: one warp per (sequence, query head) with more than one partition:
//   M = max_p m_p,  out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p.
template <int D, typename OutT>
__global__ void __launch_bounds__(256)
merge_kernel(const DecodeArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (w >= static_cast<int64_t>(a.B) * a.Hq) return;
  const int b = static_cast<int>(w / a.Hq);
  const int L = a.context_lens[b];
  if (L <= 0 || L > a.max_context_len || L > a.mbs * 16) return;   // written by decode_kernel
  const int nparts = (L + a.part_tokens - 1) / a.part_tokens;
  if (nparts <= 1) return;
  const float* ml = a.ws_ml + w * a.max_parts * 2;
  const float* acc = a.ws_acc + w * a.max_parts * D;
  float M = -INFINITY;
  for (int p = lane; p < nparts; p += 32) M = fmaxf(M, ml[2 * p]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  constexpr int PER = D / 32;
  float o_acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) o_acc[k] = 0.f;
  float sum = 0.f;
  for (int p0 = 0; p0 < nparts; p0 += 32) {
    const int p = p0 + lane;
    const float wp = p < nparts ? fast_exp2(ml[2 * p] - M) : 0.f;
    sum += p < nparts ? wp * ml[2 * p + 1] : 0.f;
    const int n = min(32, nparts - p0);
    for (int pp = 0; pp < n; ++pp) {
      const float e = __shfl_sync(0xffffffffu, wp, pp);
      const float* row = acc + static_cast<int64_t>(p0 + pp) * D;
#pragma unroll
      for (int k = 0; k < PER; ++k) o_acc[k] += e * row[lane + 32 * k];
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  OutT* out = static_cast<OutT*>(a.out) + w * D;
#pragma unroll
  for (int k = 0; k < PER; ++k) out[lane + 32 * k] = from_f32<OutT>(sum > 0.f ? o_acc[k] / sum : 0.f);
}

template <int D, bool FP8, bool BF16>
cudaError_t launch_one(const DecodeArgs& a, cudaStream_t s) {
  using TL = Tile<D, FP8>;
  using OutT = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  const int max_blk = a.part_tokens / 16;
  const size_t smem = TL::RING + kWarps * TL::STAGES * 8 + static_cast<size_t>(max_blk) * 4 * 3;
  auto* kern = decode_kernel<D, FP8, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(a.max_parts, a.Hkv, a.B);
  kern<<<grid, kThreads, smem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.max_parts <= 1) return e;
  const int64_t warps = static_cast<int64_t>(a.B) * a.Hq;
  const unsigned mgrid = static_cast<unsigned>((warps * 32 + 255) / 256);
  merge_kernel<D, OutT><<<mgrid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t decode_workspace_bytes(int B, int Hq, int D, int max_context_len, int part_tokens) {
  if (B <= 0 || Hq <= 0 || D <= 0 || part_tokens <= 0 || max_context_len < 0) return 0;
  const int64_t max_parts = (static_cast<int64_t>(max_context_len) + part_tokens - 1) / part_tokens;
  if (max_parts <= 1) return 0;
  const int64_t rows = static_cast<int64_t>(B) * Hq * max_parts;
  const size_t acc = ((static_cast<size_t>(rows) * D * 4) + 255) & ~static_cast<size_t>(255);
  return acc + static_cast<size_t>(rows) * 2 * 4;
}

void decode_workspace_split(const DecodeArgs& a, void* ws, float** acc, float** ml) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.Hq * a.max_parts;
  const size_t acc_bytes = ((static_cast<size_t>(rows) * a.D * 4) + 255) & ~static_cast<size_t>(255);
  *acc = static_cast<float*>(ws);
  *ml = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + acc_bytes);
}

cudaError_t launch_decode(const DecodeArgs& a, bool fp8, bool bf16, cudaStream_t s) {
  if (fp8) return a.D == 128 ? launch_one<128, true, false>(a, s) : launch_one<64, true, false>(a, s);
  if (bf16) return a.D == 128 ? launch_one<128, false, true>(a, s) : launch_one<64, false, true>(a, s);
  return a.D == 128 ? launch_one<128, false, false>(a, s) : launch_one<64, false, false>(a, s);
}

}  // namespace pa
