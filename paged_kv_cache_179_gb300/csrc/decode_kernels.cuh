// decode_kernels.cuh -- K3/K4: split-K paged GQA decode (16-bit and E4M3
// pools), K5, the log-sum-exp merge of the split partitions (merge_kernel),
// and their launch templates.  Included by the translation units that
// instantiate them: decode.cu (one tile of query columns per warp, and the
// host functions), decode_t2.cu and decode_t4_*.cu (two and four tiles).
// Everything here has internal linkage.
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
//  * The batch is one stream of (sequence, kv head, 16-token block) units.
//    The grid is persistent (two CTAs of four warps per SM for 16-bit pools,
//    three for E4M3) and every warp is an independent worker that takes an
//    equal contiguous share of the stream, so every warp moves the same
//    number of bytes whatever the spread of context lengths.  A warp's share
//    of one (sequence, kv head) is that sequence's context partition on this
//    worker: a short sequence lies inside one share and is attended whole, a
//    long one is split across consecutive workers (split-K).  Each worker
//    serves a whole query group per kv head, so every K/V byte is read from
//    HBM once.  The only CTA-wide step is the prologue: the prefix sums of
//    the per-sequence block counts, in shared memory.
//  * Each warp owns a ring of STAGES shared-memory slots; lane 0 fills a
//    slot with the K tile and V tile of one (block, kv head) by TMA copies
//    that complete on the slot's mbarrier: 16-bit tiles by tensor map
//    (boxes of 64 elements x 16 rows, 128-byte swizzle, so the fragment
//    reads below are free of bank conflicts), E4M3 tiles by one contiguous
//    bulk copy each.  The ring runs ahead across chunk and partition
//    boundaries.  Block ids (and E4M3 page scales) are prefetched into
//    registers, one per lane, two 32-block chunks ahead; the next
//    partition's query is prefetched too.
//  * Per block the warp computes S^T = K Q^T (16 tokens x 8 query rows) and
//    O^T += V^T P^T (head_dim x 8) with mma.sync m16n8k16 in fp32.  The query
//    rows of a (sequence, kv head) -- its group of G heads times n_q query
//    tokens -- are the N=8 side: one tile of 8 columns, or NT = 2 or 4 tiles
//    (up to 32 rows: multi-query groups, several query tokens), each K and V
//    fragment then serving every tile.  With one tile the query fragments
//    stay in registers; with more they are read from a per-warp buffer in
//    shared memory, filled by asynchronous copies when a piece starts.  The online softmax runs on the S
//    fragments (row max with shuffles, exp2 on the SFU); P moves from
//    accumulator to operand layout with movmatrix.  E4M3 codes are widened
//    to f16 in registers (exact) just before the MMA; the page scales fold
//    into the score scale (K) and into P (V).
//  * Partition end: a partition inside the worker's share writes its output
//    from registers; a split one writes its partial (running max, sum,
//    unnormalised acc) to the workspace, bit-inverted so that a zero word
//    means "not written".  The log-sum-exp merge is a second launch that
//    runs beside this grid (programmatic stream serialization) and merges
//    each split sequence as soon as its partials land.  No warp ever waits
//    for another.
//  * Optional fused append: the step's new K/V row is written to the pool
//    and into the tile just fetched by the warp that attends the sequence's
//    last block.  Optional early prologue: the launch may start while the
//    kernel before it ends; the prologue reads only context_lens and
//    block_tables and asks L2 for each warp's first tiles, and everything
//    else waits for griddepcontrol.wait.
//
// Bounds: block ids outside [0, num_blocks) and context lengths above their
// bounds are never dereferenced; they set a status bit.  Every mbarrier wait
// is bounded in time (DecodeArgs::wait_limit_ns) and reports kStatusTimeout
// instead of hanging.
#pragma once

#include <cfloat>
#include <climits>
#include <mutex>
#include <type_traits>

#include <cudaTypedefs.h>

#include "pa_e4m3.cuh"
#include "pa_launch.h"
#include "pa_ptx.cuh"

// Opt-in trace build (-DPA_TRACE): lane 0 of every worker warp records
// %globaltimer at its phases and its piece counts; pa_trace_read copies them.
// Slots per worker: 0 kernel entry, 1 first tile ready, 2 last block done,
// 3 end, 4 pieces, 5 split pieces, 6 blocks, 7 SM id.
#ifdef PA_TRACE
__device__ unsigned long long g_pa_trace[16384 * 8];
#define PA_TRACE_WARP(w, k, v)                                                   \
  do {                                                                           \
    if ((threadIdx.x & 31) == 0 && (w) < 16384) g_pa_trace[(w) * 8 + (k)] = (v);   \
  } while (0)
__device__ __forceinline__ unsigned long long pa_now() {
  unsigned long long t_;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));
  return t_;
}
__device__ __forceinline__ unsigned long long pa_smid() {
  unsigned v_;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(v_));
  return v_;
}
// per merge CTA: entry, layout known, end, pieces + 1000 x polling rounds
__device__ unsigned long long g_pa_trace_merge[16384 * 4];
extern "C" int pa_trace_read_merge(unsigned long long* host, int n_ctas) {
  const size_t n = static_cast<size_t>(n_ctas < 16384 ? n_ctas : 16384) * 4;
  return cudaMemcpyFromSymbol(host, g_pa_trace_merge, sizeof(unsigned long long) * n) ==
                 cudaSuccess ? 0 : 4;
}
extern "C" int pa_trace_read(unsigned long long* host, int n_workers) {
  const size_t n = static_cast<size_t>(n_workers < 16384 ? n_workers : 16384) * 8;
  return cudaMemcpyFromSymbol(host, g_pa_trace, sizeof(unsigned long long) * n) == cudaSuccess
             ? 0 : 4;
}
#define PA_TRACE_ONLY(x) x
#else
#define PA_TRACE_WARP(w, k, v) \
  do {                         \
  } while (0)
#define PA_TRACE_ONLY(x)
#endif

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kGroupMax = 8;     // query heads per kv head served by one MMA N=8 tile
// E4M3 path: P * v_scale is scaled by 2^8 before rounding to f16 so small
// weights stay in f16's normal range; the fp32 result is scaled back.  With
// fp16-sourced pools v_scale <= 65504/448, so P' <= 146.3 * 256 < 65504.
constexpr float kPBoost = 256.f;

template <int D, bool FP8, int STAGES>
struct Tile {
  static constexpr int ROW = FP8 ? D : 2 * D;   // bytes of one token row of one kv head
  static constexpr int BYTES = 16 * ROW;        // one (block, kv head) tile
  static constexpr int SLOT = 2 * BYTES;        // K tile + V tile
  static constexpr int RING = kWarps * STAGES * SLOT;
  // 16-bit tiles are copied by tensor map in boxes of 16 rows x 64 elements
  // with the 128-byte swizzle (see swz), which wants the ring on a 1024-byte
  // boundary: the layout reserves PAD bytes to align it.  E4M3 tiles are one
  // contiguous bulk copy each, stored as they are in the pool.
  static constexpr bool SWZ = !FP8;
  static constexpr int PAD = SWZ ? 1024 : 0;
};

// Byte offset, in a swizzled 16-bit tile, of 16-byte chunk j (elements
// 8j .. 8j+7) of token row t.  The tile is [D/64][16 rows][128 bytes]: the
// box of elements 64h .. 64h+63 of all 16 rows, then the next; chunk q of a
// 128-byte line t sits at q ^ (t % 8) (the TMA engine's 128-byte swizzle of a
// 1024-byte aligned box).
__device__ __forceinline__ uint32_t swz(int t, int j) {
  return static_cast<uint32_t>((j >> 3) * 2048 + t * 128 + (((j & 7) ^ (t & 7)) << 4));
}

__host__ __device__ constexpr int round16(int x) { return (x + 15) & ~15; }

// Dynamic shared-memory layout; the host sizes the launch with the same function.
struct Layout {
  int sbar, pf, len, misc, total;
};
__host__ __device__ inline Layout make_layout(int ring, int stages, int B) {
  Layout l{};
  int o = ring;
  l.sbar = o;  o += round16(kWarps * stages * 8);
  l.pf = o;    o += round16((B + 1) * 4);
  l.len = o;   o += round16(B * 4);
  l.misc = o;  o += 64;
  l.total = o;
  return l;
}

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
// The MMA's N = 8 columns are the query rows of one (sequence, kv head):
// row j is query token i_j = j / G (of n_q; position L - n_q + i_j) and head
// j % G of the group.  A lane holds columns 2c and 2c+1.  With positions
// taken relative to the first query's (L - n_q), column j attends relative
// positions in (i_j - window, i_j] (no lower bound without a window): the
// causal mask of several query tokens and the sliding window in one test.
struct ColMask {
  int ii;        // i_j of the lane's two columns, packed: column 2c + k in byte k
  int window;    // 0: no lower bound
  __device__ __forceinline__ bool sees(int e, int k) const {
    const int i = (ii >> (8 * k)) & 0xff;
    return e <= i && (window == 0 || e > i - window);
  }
};

// Swizzled byte offset of 16-byte chunk j of row t in a per-warp query
// buffer of ROWS rows (NT > 1): like a 16-bit K/V tile, [D/64][ROWS][128 B]
// with chunk q of line t at q ^ (t % 8), so the fragment reads of a quarter
// warp (rows t, t+1; four chunks of one parity each) hit 8 distinct 16-byte
// bank groups.
template <int ROWS>
__device__ __forceinline__ uint32_t qswz(int t, int j) {
  return static_cast<uint32_t>((j >> 3) * (ROWS * 128) + t * 128 + (((j & 7) ^ (t & 7)) << 4));
}

// The online-softmax step of one tile of 8 query columns for one 16-token
// block: scores from the S^T fragment acc (this lane: tokens r, r+8 of
// columns 2c, 2c+1), masked; running max, sum and accumulator rescaled; P
// returned in the B-operand layout of the PV product (b0: tokens 0-7, b1:
// tokens 8-15), multiplied by v_mul.
// GENERAL: a sliding window or several query tokens, masked per column with
// cm and e (the block's first position relative to the first query's);
// otherwise one query per sequence over its whole context, where only the
// rows past n_valid (the context's end) are masked.
template <int D, bool FP8, bool BF16, bool GENERAL>
__device__ __forceinline__ void softmax_tile(WarpAcc<D>& st, const float (&acc)[4],
                                             const ColMask& cm, int e, int n_valid, float sl2,
                                             float v_mul, int r, uint32_t& b0, uint32_t& b1) {
  float s0 = acc[0] * sl2, s1 = acc[1] * sl2, s2 = acc[2] * sl2, s3 = acc[3] * sl2;
  if constexpr (GENERAL) {
    // token rows r, r+8 sit at e + r, e + r + 8 relative to the first query's
    // position; column j attends relative positions (i_j - window, i_j]
    const int e0 = e + r, e1 = e0 + 8;
    if (!cm.sees(e0, 0)) s0 = -INFINITY;
    if (!cm.sees(e0, 1)) s1 = -INFINITY;
    if (!cm.sees(e1, 0)) s2 = -INFINITY;
    if (!cm.sees(e1, 1)) s3 = -INFINITY;
  } else {
    if (r >= n_valid) s0 = s1 = -INFINITY;
    if (r + 8 >= n_valid) s2 = s3 = -INFINITY;
  }
  float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, o));
    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, o));
  }
  const float mn0 = fmaxf(st.m0, bm0), mn1 = fmaxf(st.m1, bm1);
  // a column that has seen no token yet (a query before this block, with
  // several query tokens) keeps max -inf: exponentiate against 0 instead, so
  // its weights stay 0 rather than NaN
  const float x0 = GENERAL && mn0 == -INFINITY ? 0.f : mn0;
  const float x1 = GENERAL && mn1 == -INFINITY ? 0.f : mn1;
  const float a0 = fast_exp2(st.m0 - x0), a1 = fast_exp2(st.m1 - x1);
  st.m0 = mn0;
  st.m1 = mn1;
  const float p0 = fast_exp2(s0 - x0), p1 = fast_exp2(s1 - x1);
  const float p2 = fast_exp2(s2 - x0), p3 = fast_exp2(s3 - x1);
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
  b0 = movmatrix_trans(pack2<BF16 && !FP8>(p0 * v_mul, p1 * v_mul));
  b1 = movmatrix_trans(pack2<BF16 && !FP8>(p2 * v_mul, p3 * v_mul));
}

// O^T += V^T P^T for NT tiles of query columns that share the V tile at vt:
// each V fragment is read from shared memory once and multiplied into every
// tile's accumulator.  Lane (r, c) needs tokens 2c, 2c+1, 2c+8, 2c+9.
template <int D, bool FP8, bool BF16, int NT>
__device__ __forceinline__ void pv_tiles(WarpAcc<D> (&st)[NT], const uint32_t (&b0)[NT],
                                         const uint32_t (&b1)[NT], uint32_t vt, int n_valid,
                                         int r, int c) {
  constexpr int ROW = FP8 ? D : 2 * D;
  const int tk0 = 2 * c, tk1 = 2 * c + 1, tk2 = 2 * c + 8, tk3 = 2 * c + 9;
  if constexpr (!FP8) {
    // rows 2c, 2c+1, 2c+8, 2c+9 at chunk r: a quarter warp (r, r+1; c = 0..3)
    // reads 8 distinct bank groups through the swizzle
    constexpr int U = D / 64;   // 16-byte chunks per token row for this lane
    uint4 v[4][U];
#pragma unroll
    for (int u = 0; u < U; ++u) {   // chunk 8u + r: d = 64u + 8r .. +7
      v[0][u] = lds128(vt + swz(tk0, 8 * u + r));
      v[1][u] = lds128(vt + swz(tk1, 8 * u + r));
      v[2][u] = lds128(vt + swz(tk2, 8 * u + r));
      v[3][u] = lds128(vt + swz(tk3, 8 * u + r));
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
#pragma unroll
      for (int t = 0; t < NT; ++t) mma16816<BF16>(st[t].o[i], x0, x1, x2, x3, b0[t], b1[t]);
    }
  } else {
    using VT = typename std::conditional<D == 128, uint4, uint2>::type;
    constexpr int VB = D / 8;   // bytes per lane per token row: 16 (D=128) or 8 (D=64)
    VT v[4];
    if constexpr (D == 128) {
      v[0] = lds128(vt + tk0 * ROW + VB * r);
      v[1] = lds128(vt + tk1 * ROW + VB * r);
      v[2] = lds128(vt + tk2 * ROW + VB * r);
      v[3] = lds128(vt + tk3 * ROW + VB * r);
    } else {
      v[0] = lds64(vt + tk0 * ROW + VB * r);
      v[1] = lds64(vt + tk1 * ROW + VB * r);
      v[2] = lds64(vt + tk2 * ROW + VB * r);
      v[3] = lds64(vt + tk3 * ROW + VB * r);
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
      // (the conversions and MMAs are volatile asm, issued in this order:
      // with one tile each MMA follows its own four conversions)
      const uint32_t f0 = e4m3x2_to_f16x2(x01l), f1 = e4m3x2_to_f16x2(x01h);
      const uint32_t f2 = e4m3x2_to_f16x2(x23l), f3 = e4m3x2_to_f16x2(x23h);
#pragma unroll
      for (int t = 0; t < NT; ++t) mma16816<false>(st[t].o[i], f0, f1, f2, f3, b0[t], b1[t]);
      const uint32_t g0 = e4m3x2_to_f16x2(x01l >> 16), g1 = e4m3x2_to_f16x2(x01h >> 16);
      const uint32_t g2 = e4m3x2_to_f16x2(x23l >> 16), g3 = e4m3x2_to_f16x2(x23h >> 16);
#pragma unroll
      for (int t = 0; t < NT; ++t) mma16816<false>(st[t].o[i + 1], g0, g1, g2, g3, b0[t], b1[t]);
    }
  }
}

// One 16-token block already in shared memory (K tile at kt, V tile at vt),
// one tile of query columns whose fragments qf are held in registers.
template <int D, bool FP8, bool BF16, bool GENERAL>
__device__ __forceinline__ void attend_block(WarpAcc<D> (&st)[1], const uint32_t (&qf)[D / 16][2],
                                             uint32_t kt, uint32_t vt, const ColMask& cm,
                                             int e, int n_valid, float sl2,
                                             float v_mul, int r, int c) {
  constexpr int ROW = FP8 ? D : 2 * D;
  // ---- S^T = K Q^T : 16 tokens x 8 query heads, k = head_dim
  // two accumulators (even / odd k-steps) halve the dependent MMA chain
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (!FP8) {
    // lane (r, c) reads 16-byte chunk j = 8(i/2) + 2c + i%2 of rows r and r+8
    // (d = 8j .. 8j+7; the query fragments follow the same order).  A quarter
    // warp (rows r, r+1, c = 0..3) then reads chunks of one parity from row r
    // and of the other from row r+1, swizzled to 8 distinct bank groups.
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      const int j = 8 * (i >> 1) + 2 * c + (i & 1);
      const uint4 ka = lds128(kt + swz(r, j));
      const uint4 kb = lds128(kt + swz(r + 8, j));
      mma16816<BF16>(acc, ka.x, kb.x, ka.y, kb.y, qf[2 * i][0], qf[2 * i][1]);
      mma16816<BF16>(acc2, ka.z, kb.z, ka.w, kb.w, qf[2 * i + 1][0], qf[2 * i + 1][1]);
    }
  } else {
    // lane (r, c) reads 16 codes at byte 64i + 16c of rows r and r+8
#pragma unroll
    for (int i = 0; i < D / 64; ++i) {
      const uint4 ka = lds128(kt + r * ROW + 64 * i + 16 * c);
      const uint4 kb = lds128(kt + (r + 8) * ROW + 64 * i + 16 * c);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint32_t wa = word(ka, q4), wb = word(kb, q4);
        mma16816<false>(q4 & 1 ? acc2 : acc, e4m3x2_to_f16x2(wa), e4m3x2_to_f16x2(wb),
                        e4m3x2_to_f16x2(wa >> 16), e4m3x2_to_f16x2(wb >> 16),
                        qf[4 * i + q4][0], qf[4 * i + q4][1]);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] += acc2[k];
  uint32_t b0[1], b1[1];
  softmax_tile<D, FP8, BF16, GENERAL>(st[0], acc, cm, e, n_valid, sl2, v_mul, r, b0[0], b1[0]);
  pv_tiles<D, FP8, BF16, 1>(st, b0, b1, vt, n_valid, r, c);
}

// One 16-token block for NT > 1 tiles of query columns (8 NT rows), whose
// fragments are read from the warp's query buffer qbuf (qswz layout): each K
// fragment (and, for E4M3, its widening to f16) serves every tile, and each
// tile's MMA chain is independent of the others'.
template <int D, bool FP8, bool BF16, bool GENERAL, int NT>
__device__ __forceinline__ void attend_block_mt(WarpAcc<D> (&st)[NT], uint32_t qbuf, uint32_t kt,
                                                uint32_t vt, const ColMask (&cm)[NT], int e,
                                                int n_valid, float sl2, float v_mul, int r,
                                                int c) {
  constexpr int ROW = FP8 ? D : 2 * D;
  constexpr int ROWS = 8 * NT;
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  if constexpr (!FP8) {
    // the same d order as attend_block: chunk j = 8(i/2) + 2c + i%2
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      const int j = 8 * (i >> 1) + 2 * c + (i & 1);
      const uint4 ka = lds128(kt + swz(r, j));
      const uint4 kb = lds128(kt + swz(r + 8, j));
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const uint4 qv = lds128(qbuf + qswz<ROWS>(8 * t + r, j));
        mma16816<BF16>(acc[t], ka.x, kb.x, ka.y, kb.y, qv.x, qv.y);
        mma16816<BF16>(acc[t], ka.z, kb.z, ka.w, kb.w, qv.z, qv.w);
      }
    }
  } else {
    // 16 codes at byte 64i + 16c of rows r and r+8, against query chunks
    // 8i + 2c and 8i + 2c + 1 (fp16)
#pragma unroll
    for (int i = 0; i < D / 64; ++i) {
      const uint4 ka = lds128(kt + r * ROW + 64 * i + 16 * c);
      const uint4 kb = lds128(kt + (r + 8) * ROW + 64 * i + 16 * c);
      uint32_t f[4][4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint32_t wa = word(ka, q4), wb = word(kb, q4);
        f[q4][0] = e4m3x2_to_f16x2(wa);
        f[q4][1] = e4m3x2_to_f16x2(wb);
        f[q4][2] = e4m3x2_to_f16x2(wa >> 16);
        f[q4][3] = e4m3x2_to_f16x2(wb >> 16);
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const uint4 lo = lds128(qbuf + qswz<ROWS>(8 * t + r, 8 * i + 2 * c));
        const uint4 hi = lds128(qbuf + qswz<ROWS>(8 * t + r, 8 * i + 2 * c + 1));
        mma16816<false>(acc[t], f[0][0], f[0][1], f[0][2], f[0][3], lo.x, lo.y);
        mma16816<false>(acc[t], f[1][0], f[1][1], f[1][2], f[1][3], lo.z, lo.w);
        mma16816<false>(acc[t], f[2][0], f[2][1], f[2][2], f[2][3], hi.x, hi.y);
        mma16816<false>(acc[t], f[3][0], f[3][1], f[3][2], f[3][3], hi.z, hi.w);
      }
    }
  }
  uint32_t b0[NT], b1[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t)
    softmax_tile<D, FP8, BF16, GENERAL>(st[t], acc[t], cm[t], e, n_valid, sl2, v_mul, r, b0[t],
                                        b1[t]);
  pv_tiles<D, FP8, BF16, NT>(st, b0, b1, vt, n_valid, r, c);
}

// ------------------------------------------------------------ work split
// The batch is a stream of 16-token blocks ordered (sequence, kv head,
// block): segment (b, h) holds the ceil(L_b / 16) blocks of sequence b for
// kv head h, and starts at pf[b] + h * nblk_b where pf is the exclusive
// prefix sum of Hkv * nblk_b.  The N workers (warps of the grid) share the
// W blocks evenly: worker w takes blocks [w*W/N, (w+1)*W/N), and its share
// of a segment is one context partition ("piece").  A segment inside one
// worker's range is attended whole; one that crosses ranges is split into
// pieces whose partial results are merged.  A worker walks its range in
// chunks of at most kChunk blocks (CH), one block id per lane.
constexpr int kChunk = 32;

struct Chunk {
  int b, h;     // segment
  int cb0;      // first block of the chunk within the segment
  int nb;       // blocks in the chunk (0: past the end of the worker's range)
};

__device__ __forceinline__ int seg_blocks(const int* pf, int b, int Hkv) {
  return (pf[b + 1] - pf[b]) / Hkv;
}
__device__ __forceinline__ int64_t worker_lo(int64_t w, int64_t W, int64_t N) { return w * W / N; }
// The worker whose range holds block x.
__device__ __forceinline__ int worker_of(int64_t x, int64_t W, int64_t N) {
  return static_cast<int>(((x + 1) * N - 1) / W);
}

template <int CH = kChunk>
__device__ __forceinline__ Chunk first_chunk(int64_t lo, int64_t hi, const int* pf, int B,
                                             int Hkv) {
  Chunk x{0, 0, 0, 0};
  if (lo >= hi) return x;
  int l = 0, r = B;                        // pf[l] <= lo < pf[r]
  while (r - l > 1) {
    const int mid = (l + r) >> 1;
    if (pf[mid] <= lo) l = mid;
    else r = mid;
  }
  const int nbk = seg_blocks(pf, l, Hkv);
  x.b = l;
  x.h = static_cast<int>((lo - pf[l]) / nbk);
  const int64_t s0 = pf[l] + static_cast<int64_t>(x.h) * nbk;
  x.cb0 = static_cast<int>(lo - s0);
  x.nb = static_cast<int>(min(static_cast<int64_t>(CH), min(hi, s0 + nbk) - lo));
  return x;
}

template <int CH = kChunk>
__device__ __forceinline__ Chunk next_chunk(const Chunk& x, int64_t hi, const int* pf, int B,
                                            int Hkv) {
  Chunk y{0, 0, 0, 0};
  if (x.nb == 0) return y;
  int nbk = seg_blocks(pf, x.b, Hkv);
  int64_t s0 = pf[x.b] + static_cast<int64_t>(x.h) * nbk;
  const int pend = static_cast<int>(min(hi, s0 + nbk) - s0);
  const int n0 = x.cb0 + x.nb;
  if (n0 < pend) return Chunk{x.b, x.h, n0, min(CH, pend - n0)};
  int b = x.b, h = x.h + 1;
  if (h == Hkv) {
    h = 0;
    ++b;
    while (b < B && pf[b + 1] == pf[b]) ++b;
  }
  if (b >= B) return y;
  nbk = seg_blocks(pf, b, Hkv);
  s0 = pf[b] + static_cast<int64_t>(h) * nbk;
  if (s0 >= hi) return y;
  return Chunk{b, h, 0, static_cast<int>(min(static_cast<int64_t>(CH), min(hi, s0 + nbk) - s0))};
}

// The first block a sequence of L tokens attends: with a sliding window of
// `window` tokens the blocks before the first query's window are skipped.
// Segments and chunks count blocks from there.
__device__ __forceinline__ int window_first_block(int L, int window, int n_q) {
  const int first = L - (n_q - 1) - window;   // the first query's window start
  return window > 0 && first > 0 ? first >> 4 : 0;
}

// The context length a launch sees for a context_lens entry (-1: outside the
// stated bounds).  A launch serving query tokens q_first .. q_first+n_q-1 of
// q_tokens sees the cache up to its last query's position.
__device__ __forceinline__ int launch_len(const DecodeArgs& a, int raw) {
  const bool ok = raw >= 0 && raw <= a.max_context_len && raw <= a.mbs * 16;
  return ok ? max(0, raw - (a.q_tokens - a.q_first - a.n_q)) : -1;
}
// Blocks per kv head a sequence of launch length L puts in the block stream.
__device__ __forceinline__ int stream_blocks(const DecodeArgs& a, int L) {
  return L > 0 ? ((L + 15) >> 4) - window_first_block(L, a.window, a.n_q) : 0;
}
// Units per kv head it puts in the stream the workers share: its blocks,
// after a.seg_cost units that stand for a segment's fixed cost (a launch
// whose workers pay one per segment evens out the cost, not the blocks).
__device__ __forceinline__ int stream_units(const DecodeArgs& a, int L) {
  const int n = stream_blocks(a, L);
  return n > 0 ? n + a.seg_cost : 0;
}

// This lane's block id of chunk x (lane t holds block cb0 + t of the
// segment, block table entry fb + cb0 + t), -1 past its end.
__device__ __forceinline__ int load_chunk_id(const DecodeArgs& a, const Chunk& x, int fb,
                                             int lane) {
  if (lane >= x.nb) return -1;
  return __ldg(a.block_tables + static_cast<int64_t>(x.b) * a.mbs + fb + x.cb0 + lane);
}

// The query fragments of (sequence b, kv head h): the group's G rows, the
// MMA B operand.  Returns the factor the scores carry back: 1, except for a
// bf16 q over an E4M3 pool, which enters the fp16 products scaled by 2^k so
// that its largest element lies in [2^14, 2^15) (exact unless an element
// falls below fp16's subnormal range); the factor is then 2^-k.
template <int D, bool FP8, bool BF16>
__device__ __forceinline__ float load_query(uint32_t (&qf)[D / 16][2], const DecodeArgs& a, int b,
                                            int h, int r, int c) {
  // row r: query token q_first + r / G, head h*G + r % G; q is [B][q_tokens][Hq][D]
  const int G = a.group;
  const bool live = r < a.n_q * G;
  const uint4* qrow = reinterpret_cast<const uint4*>(
      static_cast<const uint16_t*>(a.q) +
      ((static_cast<int64_t>(b) * a.q_tokens + a.q_first + r / G) * a.Hq + h * G + r % G) * D);
  if constexpr (!FP8) {
    // k-step pair i holds chunk 8(i/2) + 2c + i%2, as the K fragments do
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      const uint4 v = live ? __ldg(qrow + 8 * (i >> 1) + 2 * c + (i & 1)) : make_uint4(0, 0, 0, 0);
      qf[2 * i][0] = v.x;
      qf[2 * i][1] = v.y;
      qf[2 * i + 1][0] = v.z;
      qf[2 * i + 1][1] = v.w;
    }
    return 1.f;
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
    if constexpr (!BF16) {
      return 1.f;
    } else {
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < D / 16; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float2 v = bits2_to_float2<true>(qf[i][j]);
          amax = fmaxf(amax, fmaxf(fabsf(v.x), fabsf(v.y)));
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      // amax = m * 2^e with m in [1, 2): k = 14 - e, kept within fp32's normal exponents
      const int e = amax > 0.f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xff) - 127 : 14;
      const int k = max(-126, min(126, 14 - e));
      const float up = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
#pragma unroll
      for (int i = 0; i < D / 16; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float2 v = bits2_to_float2<true>(qf[i][j]);
          const __half2 h2 = __floats2half2_rn(v.x * up, v.y * up);
          qf[i][j] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      return __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
    }
  }
}

// NT > 1: the query rows of (sequence b, kv head h) into the warp's buffer
// at qbuf (qswz layout, ROWS rows): row j is query token q_first + j / G,
// head h * G + j % G; rows at or past n_q * G are zero-filled.  The copies
// are asynchronous (16 bytes each, consecutive lanes on consecutive chunks);
// `pending` is set and the caller waits (cp_async_wait_all, __syncwarp)
// before the first fragment read.  A bf16 q over an E4M3 pool is then
// converted in place, as load_query does: to f16 scaled by a power of two
// 2^k per (sequence, kv head) so that the largest element lies in
// [2^14, 2^15); the factor 2^-k is returned (else 1).
template <int D, bool FP8, bool BF16, int ROWS>
__device__ __forceinline__ float fill_query_buffer(uint32_t qbuf, const DecodeArgs& a, int b,
                                                   int h, int lane, bool& pending) {
  constexpr int CH = D / 8;   // 16-byte chunks per row
  if (pending) cp_async_wait_all();   // never two fills of one buffer in flight
  const int G = a.group, live_rows = a.n_q * G;
  const uint16_t* q = static_cast<const uint16_t*>(a.q);
#pragma unroll 4
  for (int x = lane; x < ROWS * CH; x += 32) {
    const int j = x / CH, ch = x - j * CH;
    const bool live = j < live_rows;
    const int64_t row =
        live ? (static_cast<int64_t>(b) * a.q_tokens + a.q_first + j / G) * a.Hq + h * G + j % G
             : 0;
    cp_async16(qbuf + qswz<ROWS>(j, ch), q + row * D + ch * 8, live ? 16u : 0u);
  }
  pending = true;
  if constexpr (!(FP8 && BF16)) {
    return 1.f;
  } else {
    cp_async_wait_all();
    __syncwarp();
    pending = false;
    float amax = 0.f;
    for (int x = lane; x < ROWS * CH; x += 32) {
      const uint4 v = lds128(qbuf + qswz<ROWS>(x / CH, x % CH));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = bits2_to_float2<true>(word(v, k));
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    // amax = m * 2^e with m in [1, 2): k = 14 - e, kept within fp32's normal exponents
    const int e = amax > 0.f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xff) - 127 : 14;
    const int k = max(-126, min(126, 14 - e));
    const float up = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
    for (int x = lane; x < ROWS * CH; x += 32) {
      const uint32_t at = qbuf + qswz<ROWS>(x / CH, x % CH);
      uint4 v = lds128(at);
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = bits2_to_float2<true>(w[i]);
        const __half2 h2 = __floats2half2_rn(f.x * up, f.y * up);
        w[i] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      sts128(at, make_uint4(w[0], w[1], w[2], w[3]));
    }
    __syncwarp();
    return __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
  }
}

// NT > 1: ask L2 for the query rows of (sequence b, kv head h) ahead of their
// fill: one prefetch per query token (its G heads are contiguous).
template <int D>
__device__ __forceinline__ void prefetch_query_l2(const DecodeArgs& a, int b, int h, int lane) {
  if (lane < a.n_q)
    prefetch_l2(static_cast<const uint16_t*>(a.q) +
                    ((static_cast<int64_t>(b) * a.q_tokens + a.q_first + lane) * a.Hq + h * a.group) *
                        D,
                static_cast<uint32_t>(a.group * D * 2));
}

// Partial-result row of (worker w, piece slot k, query row g), with `rows`
// rows per piece (8 per tile of query columns the launch holds): slot 0 is
// the worker's first piece, slot 1 its last.
__device__ __forceinline__ int64_t piece_row(int w, int k, int g, int rows) {
  return (static_cast<int64_t>(w) * 2 + k) * rows + g;
}

// Write a whole piece's result from the warp's fragments: out = o / l.
// rows: the output of query row 0 of the (sequence, kv head); off: the
// offsets of the lane's columns 2c, 2c+1 from it (-1: not a query row).
template <int D, bool FP8, bool BF16>
__device__ __forceinline__ void store_output(const WarpAcc<D>& st, uint16_t* rows,
                                             const int (&off)[2], int r, int c, float unboost) {
  const float i0 = st.l0 > 0.f ? unboost / st.l0 : 0.f;
  const float i1 = st.l1 > 0.f ? unboost / st.l1 : 0.f;
#pragma unroll
  for (int i = 0; i < D / 16; i += 2) {
    const int dl = d_lo<D, FP8>(i, r), dh = d_hi<D, FP8>(i, r);   // d and d+1 with i, i+1
    if (off[0] >= 0) {
      *reinterpret_cast<uint32_t*>(rows + off[0] + dl) =
          pack2<BF16>(st.o[i][0] * i0, st.o[i + 1][0] * i0);
      *reinterpret_cast<uint32_t*>(rows + off[0] + dh) =
          pack2<BF16>(st.o[i][2] * i0, st.o[i + 1][2] * i0);
    }
    if (off[1] >= 0) {
      *reinterpret_cast<uint32_t*>(rows + off[1] + dl) =
          pack2<BF16>(st.o[i][1] * i1, st.o[i + 1][1] * i1);
      *reinterpret_cast<uint32_t*>(rows + off[1] + dh) =
          pack2<BF16>(st.o[i][3] * i1, st.o[i + 1][3] * i1);
    }
  }
}

// Partial results sit in the workspace bit-inverted, so that a zero word
// means "not written yet": no value the kernel computes has all 32 bits set
// (a NaN the GPU's arithmetic produces is 0x7fffffff).  A zero-filled
// workspace therefore holds no partial, and the merge launch, having read a
// partial, zeroes it again.
__device__ __forceinline__ uint32_t ws_enc(float x) { return ~__float_as_uint(x); }
__device__ __forceinline__ float ws_dec(uint32_t u) { return __uint_as_float(~u); }

// Write a split piece's partial (unnormalised acc, running max, sum) of
// query-column tile t to the workspace.
template <int D, bool FP8, int ROWS>
__device__ __forceinline__ void store_partial(const WarpAcc<D>& st, const DecodeArgs& a, int w,
                                              int slot, int r, int c, float unboost, int t) {
  const int g0 = 8 * t + 2 * c, g1 = g0 + 1;
  float* r0 = a.ws_acc + piece_row(w, slot, g0, ROWS) * D;
  float* r1 = a.ws_acc + piece_row(w, slot, g1, ROWS) * D;
#pragma unroll
  for (int i = 0; i < D / 16; i += 2) {
    const int dl = d_lo<D, FP8>(i, r), dh = d_hi<D, FP8>(i, r);
    if (g0 < a.n_q * a.group) {
      st_relaxed_v2(r0 + dl, ws_enc(st.o[i][0] * unboost), ws_enc(st.o[i + 1][0] * unboost));
      st_relaxed_v2(r0 + dh, ws_enc(st.o[i][2] * unboost), ws_enc(st.o[i + 1][2] * unboost));
    }
    if (g1 < a.n_q * a.group) {
      st_relaxed_v2(r1 + dl, ws_enc(st.o[i][1] * unboost), ws_enc(st.o[i + 1][1] * unboost));
      st_relaxed_v2(r1 + dh, ws_enc(st.o[i][3] * unboost), ws_enc(st.o[i + 1][3] * unboost));
    }
  }
  if (r == 0) {
    if (g0 < a.n_q * a.group)
      st_relaxed_v2(a.ws_ml + piece_row(w, slot, g0, ROWS) * 2, ws_enc(st.m0), ws_enc(st.l0));
    if (g1 < a.n_q * a.group)
      st_relaxed_v2(a.ws_ml + piece_row(w, slot, g1, ROWS) * 2, ws_enc(st.m1), ws_enc(st.l1));
  }
}

// Fused append: the new (this step's) row of one (sequence, kv head), the
// lane's D/16 bytes of it, and its slot.
struct NewRow {
  uint2 k, v;      // 16-bit values (D=64 uses .x only)
  int64_t slot;    // slot_mapping[b]; -2 when the chunk holds no sequence end
};

// Fused E4M3 append of sequence b's new row for kv head h into page `row`
// of physical block `blk`: the tile just fetched (ktile / vtile, 16 rows of D
// codes in shared memory) and the pool both get it.  Per pool, the page's
// first row sets its scale; a later row that would saturate re-scales the
// page's earlier rows in both copies.  Returns the K and V scales the page
// then has (ksc / vsc unchanged when nothing is appended: a padding slot, or
// a slot that is not position context_len - 1, which sets the status bit).
// Out of line and loading its own inputs: it runs once per sequence and kv
// head, and inlined, its registers would crowd the attention loop.
template <int D, bool BF16>
__device__ __noinline__ float2 append_e4m3_row(const uint16_t* k_new, const uint16_t* v_new,
                                               const int64_t* slots, uint8_t* ktile,
                                               uint8_t* vtile, uint8_t* k_pool, uint8_t* v_pool,
                                               float* k_scale, float* v_scale, unsigned* status,
                                               int b, int h, int Hkv, int blk, int row, float ksc,
                                               float vsc, int lane) {
  const int64_t slot = __ldg(slots + b);
  if (slot < 0) return make_float2(ksc, vsc);                      // padding: nothing appended
  if (slot != static_cast<int64_t>(blk) * 16 + row) {
    if (lane == 0) atomicOr(status, kStatusBadSlot);             // not a decode-step slot
    return make_float2(ksc, vsc);
  }
  const int64_t tile = static_cast<int64_t>(blk) * Hkv + h;
  const int64_t src = (static_cast<int64_t>(b) * Hkv + h) * D;
  float out[2];
#pragma unroll
  for (int kv = 0; kv < 2; ++kv) {
    uint8_t* t = kv ? vtile : ktile;
    uint8_t* page = (kv ? v_pool : k_pool) + tile * 16 * D;
    const RowF16<D> x = load_row<D, BF16>((kv ? v_new : k_new) + src, lane);
    const float amax = e4m3_row_amax<D>(x);
    float sc = kv ? vsc : ksc;
    if (row == 0 || e4m3_saturates(amax, sc)) {
      const float sn = e4m3_page_scale(amax);
      e4m3_rescale_rows<D, false>(t, t, page, row, sc, sn, lane);
      sc = sn;
      if (lane == 0) (kv ? v_scale : k_scale)[tile] = sc;
    }
    const uint32_t codes = e4m3_row_codes<D>(x, sc);
    store_row_codes<D>(t + row * D, lane, codes);
    store_row_codes<D>(page + row * D, lane, codes);
    out[kv] = sc;
  }
  __syncwarp();
  return make_float2(out[0], out[1]);
}

// The new row of chunk x's sequence and kv head when x holds the sequence's
// last block (the one the new token goes to), for this lane.
template <int D, bool APPEND>
__device__ __forceinline__ NewRow load_new_row(const DecodeArgs& a, const Chunk& x, const int* pf,
                                              int lane) {
  NewRow n;
  n.k = n.v = make_uint2(0, 0);
  n.slot = -2;
  if constexpr (APPEND) {
    if (x.nb > 0 && x.cb0 + x.nb == seg_blocks(pf, x.b, a.Hkv)) {
      n.slot = __ldg(a.slots + x.b);
      const int64_t off = (static_cast<int64_t>(x.b) * a.Hkv + x.h) * D * 2 + lane * (D / 16);
      const uint8_t* kr = static_cast<const uint8_t*>(a.k_new) + off;
      const uint8_t* vr = static_cast<const uint8_t*>(a.v_new) + off;
      if constexpr (D == 128) {
        n.k = __ldg(reinterpret_cast<const uint2*>(kr));
        n.v = __ldg(reinterpret_cast<const uint2*>(vr));
      } else {
        n.k.x = __ldg(reinterpret_cast<const uint32_t*>(kr));
        n.v.x = __ldg(reinterpret_cast<const uint32_t*>(vr));
      }
    }
  }
  return n;
}

// With an early prologue, each warp asks L2 for its first
// PA_EARLY_PREFETCH x STAGES tiles before it waits for the previous kernel,
// twice that when its share holds PA_EARLY_PREFETCH_LONG blocks or more;
// 0 turns this off.
#ifndef PA_EARLY_PREFETCH
#define PA_EARLY_PREFETCH 1
#endif
#ifndef PA_EARLY_PREFETCH_LONG
#define PA_EARLY_PREFETCH_LONG 32
#endif

template <int D, bool FP8, bool BF16, int STAGES, bool APPEND, bool GENERAL, int CTAS, int NT>
__global__ void __launch_bounds__(kThreads, CTAS)
decode_kernel(const __grid_constant__ DecodeArgs a) {
  using TL = Tile<D, FP8, STAGES>;
  constexpr int ROWS = 8 * NT;                      // query rows a warp holds
  constexpr int QBUF = NT > 1 ? ROWS * D * 2 : 0;   // bytes of a warp's query buffer (NT > 1)
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, c = lane & 3;
  const int B = a.B, Hkv = a.Hkv, Hq = a.Hq, G = a.group;
  // this lane's two columns of each tile (query rows 8t + 2c, 8t + 2c + 1):
  // the query token of each (a dead column, past the n_q * G rows, sees what
  // the last query sees)
  ColMask cm[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    cm[t].ii = 0;
    cm[t].window = a.window;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int j = 8 * t + 2 * c + k;
      cm[t].ii |= (j < a.n_q * G ? j / G : a.n_q - 1) << (8 * k);
    }
  }
  const Layout lay = make_layout(TL::RING + TL::PAD + kWarps * QBUF, STAGES, B);
  int* pf = reinterpret_cast<int*>(smem + lay.pf);
  int* len = reinterpret_cast<int*>(smem + lay.len);
  int* misc = reinterpret_cast<int*>(smem + lay.misc);   // [0..3] warp sums of the scan

  PA_TRACE_ONLY(const unsigned long long t_entry = pa_now());
  // ---- 0. with a device-side handshake, nothing of this step's inputs is
  // read before the copy that uploads them has completed: thread 0 waits
  // (bounded) for the word written after it.  A CTA that gives up reports
  // the timeout and returns without touching anything.
  if (a.ready != nullptr) {
    if (tid == 0) {
      bool ok = true;
      if (static_cast<int>(ld_acquire_b32(a.ready) - a.ready_value) < 0) {
        const uint64_t t0 = global_ns();
        while (static_cast<int>(ld_acquire_b32(a.ready) - a.ready_value) < 0) {
          __nanosleep(256);
          if (global_ns() - t0 > a.wait_limit_ns) {
            ok = false;
            break;
          }
        }
      }
      misc[4] = ok;
      if (!ok) atomicOr(a.status, kStatusTimeout);
    }
    __syncthreads();
    if (!misc[4]) return;
  }
  // ---- 1. blocks per sequence and their prefix sum (segments of Hkv * nblk)
  {
    const int per = (B + kThreads - 1) / kThreads;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) {
      const int L = launch_len(a, a.context_lens[b]);
      len[b] = L;
      sum += stream_blocks(a, L) * Hkv;
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane == 31) misc[warp] = inc;
    __syncthreads();
    int ex = inc - sum;
    for (int w = 0; w < warp; ++w) ex += misc[w];
    for (int b = b0; b < b1; ++b) {
      pf[b] = ex;
      ex += stream_blocks(a, len[b]) * Hkv;
    }
    if (tid == kThreads - 1) pf[B] = ex;
    __syncthreads();
  }
  const int64_t W = pf[B];
  const int cta = blockIdx.x;

  // The merge launch may be scheduled now: it waits for the partials it reads.
  griddep_launch_dependents();

  // ---- 2. the previous kernel on the stream.  With an early prologue this
  // launch may have started before it finished: the prologue above and the
  // block-table reads below touch only what that kernel does not write
  // (context_lens, block_tables); everything else waits for it here, except,
  // with early copies, the first K/V tiles of blocks before a sequence's last
  // two (which that kernel leaves alone, by the flag's contract).
  // Then sequences with nothing to attend get a zero output (one warp each).
  auto after_previous_kernel = [&]() {
    if (a.early) griddep_wait();
    for (int b = cta * kWarps + warp; b < B; b += static_cast<int>(gridDim.x) * kWarps) {
      const int L = len[b];
      if (L > 0) continue;
      if (L < 0 && lane == 0) atomicOr(a.status, kStatusBadLen);
      uint16_t* o = static_cast<uint16_t*>(a.out) +
                    (static_cast<int64_t>(b) * a.q_tokens + a.q_first) * Hq * D;
      for (int i = lane; i < a.n_q * Hq * D; i += 32) o[i] = 0;   // +0.0 in f16 and bf16
    }
  };

  // ---- 3. this warp's share of the block stream.  No CTA-wide barrier
  // follows: every warp is an independent worker from here on.  Never more
  // workers than blocks, so every worker owns at least one block (the piece
  // bookkeeping relies on it).
  const int64_t NW = min(static_cast<int64_t>(gridDim.x) * kWarps, W);
  const int gw = cta * kWarps + warp;
  if (gw >= NW) {
    after_previous_kernel();
    return;
  }
  const int64_t lo = worker_lo(gw, W, NW), hi = worker_lo(gw + 1, W, NW);

  uint32_t ring_at = 0;   // the rings start at the first 1024-byte boundary (swizzled tiles)
  if constexpr (TL::SWZ) ring_at = (1024u - (smem_u32(smem) & 1023u)) & 1023u;
  const uint32_t ring = smem_u32(smem) + ring_at + warp * STAGES * TL::SLOT;
  const uint32_t qbuf = smem_u32(smem) + ring_at + TL::RING + warp * QBUF;   // NT > 1
  const uint32_t sbar = smem_u32(smem + lay.sbar) + warp * STAGES * 8;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) mbar_init(sbar + 8 * s, 1);
    mbar_init_fence();
  }
  __syncwarp();

  // chunks k (being computed), k+1 and k+2, and this lane's block id in each
  Chunk ch0 = first_chunk(lo, hi, pf, B, Hkv);
  Chunk ch1 = next_chunk(ch0, hi, pf, B, Hkv);
  Chunk ch2 = next_chunk(ch1, hi, pf, B, Hkv);
  auto chunk_id = [&](const Chunk& x) {
    const int fb = GENERAL && x.nb > 0 ? window_first_block(len[x.b], a.window, a.n_q) : 0;
    return load_chunk_id(a, x, fb, lane);
  };
  int id0 = chunk_id(ch0);
  int id1 = chunk_id(ch1);
  int id2 = chunk_id(ch2);
  if (PA_EARLY_PREFETCH > 0 && a.early) {
    // While the previous kernel ends, warm L2 with the warp's first tiles
    // (lane t: block t of its first chunk), so that the first copies after
    // the wait are served from L2: a prefetch reads nothing into the SM, so
    // what that kernel writes before it completes is still what they read.
    // a long share (PA_EARLY_PREFETCH_LONG blocks or more) prefetches twice
    // as many: its first tiles are a small part of its work
    const int n_pf = PA_EARLY_PREFETCH * STAGES * (hi - lo >= PA_EARLY_PREFETCH_LONG ? 2 : 1);
    if (lane < n_pf && lane < ch0.nb && id0 >= 0 && id0 < a.num_blocks) {
      const int64_t tile = static_cast<int64_t>(id0) * Hkv + ch0.h;
      prefetch_l2(static_cast<const uint8_t*>(a.k_cache) + tile * TL::BYTES, TL::BYTES);
      prefetch_l2(static_cast<const uint8_t*>(a.v_cache) + tile * TL::BYTES, TL::BYTES);
    }
  }
  const uint8_t* kbase = static_cast<const uint8_t*>(a.k_cache);
  const uint8_t* vbase = static_cast<const uint8_t*>(a.v_cache);
  const uint64_t pol = l2_policy_evict_first();
  bool dead = false;            // a wait timed out: stop touching the pipeline
  int issued = 0, computed = 0;
  int ic = 0, it = 0;           // fetch cursor: chunk k+ic (ic in {0,1}), block it

  // Keeps STAGES copies in flight.  pre: before the wait for the previous
  // kernel (PA_DECODE_EARLY_COPIES), which may still write each sequence's
  // last two blocks: stop at the first block that is one of them.
  auto top_up = [&](bool pre) {
    while (!dead && issued - computed < STAGES) {
      const Chunk& x = ic == 0 ? ch0 : ch1;
      if (x.nb == 0) return;
      if (it >= x.nb) {
        if (ic == 1) return;    // never more than one chunk ahead
        ic = 1;
        it = 0;
        continue;
      }
      if (pre) {
        const int Ls = len[x.b];
        const int blk = (GENERAL ? window_first_block(Ls, a.window, a.n_q) : 0) + x.cb0 + it;
        if (blk + 2 >= (Ls + 15) / 16) return;
      }
      const int id = __shfl_sync(0xffffffffu, ic == 0 ? id0 : id1, it);
      const int s = issued % STAGES;
      const uint32_t bar = sbar + 8 * s;
      if (lane == 0) {
        if (id >= 0 && id < a.num_blocks) {
          const int64_t tile = static_cast<int64_t>(id) * Hkv + x.h;
          mbar_arrive_expect_tx(bar, 2 * TL::BYTES);
          if constexpr (TL::SWZ) {
            // boxes of 64 elements x 16 rows: D / 64 per tile
            const uint32_t kd = ring + s * TL::SLOT, vd = kd + TL::BYTES;
            const int ti = static_cast<int>(tile);
#pragma unroll
            for (int hb = 0; hb < D / 64; ++hb) {
              tensor3_g2s(kd + hb * 2048, &a.tm_k, 64 * hb, 0, ti, bar, pol);
              tensor3_g2s(vd + hb * 2048, &a.tm_v, 64 * hb, 0, ti, bar, pol);
            }
          } else {
            bulk_g2s(ring + s * TL::SLOT, kbase + tile * TL::BYTES, TL::BYTES, bar, pol);
            bulk_g2s(ring + s * TL::SLOT + TL::BYTES, vbase + tile * TL::BYTES, TL::BYTES, bar,
                     pol);
          }
        } else {
          atomicOr(a.status, kStatusBadBlock);
          mbar_arrive(bar);
        }
      }
      ++issued;
      ++it;
    }
  };
  if (a.early && a.early_copies) top_up(true);
  after_previous_kernel();
  float ks0 = 1.f, vs0 = 1.f, ks1 = 1.f, vs1 = 1.f;   // E4M3 page scales of chunks k, k+1
  if constexpr (FP8) {
    if (id0 >= 0 && id0 < a.num_blocks) {
      ks0 = __ldg(a.k_scale + static_cast<int64_t>(id0) * Hkv + ch0.h);
      vs0 = __ldg(a.v_scale + static_cast<int64_t>(id0) * Hkv + ch0.h);
    }
    if (id1 >= 0 && id1 < a.num_blocks) {
      ks1 = __ldg(a.k_scale + static_cast<int64_t>(id1) * Hkv + ch1.h);
      vs1 = __ldg(a.v_scale + static_cast<int64_t>(id1) * Hkv + ch1.h);
    }
  }
  // query fragments of the current piece and of the next one.  NT == 1: in
  // registers.  NT > 1: the current piece's rows in the warp's query buffer,
  // filled by asynchronous copies when the piece starts (waited for before
  // its first block); the next piece's rows are only asked of L2 ahead.
  constexpr int QF = NT == 1 ? D / 16 : 1;
  uint32_t qf[QF][2], qn[QF][2];
  uint8_t* const ring_ptr = smem + ring_at + warp * STAGES * TL::SLOT;   // generic address
  bool q_pending = false;   // NT > 1: copies into the query buffer in flight
  auto fill_query = [&](int b, int h) -> float {
    if constexpr (NT == 1)
      return load_query<D, FP8, BF16>(qf, a, b, h, r, c);
    else
      return fill_query_buffer<D, FP8, BF16, ROWS>(qbuf, a, b, h, lane, q_pending);
  };
  float q_mul = fill_query(ch0.b, ch0.h), qn_mul = 1.f;
  auto prefetch_next_query = [&](int b, int h) {
    ++h;
    if (h == Hkv) {
      h = 0;
      ++b;
      while (b < B && pf[b + 1] == pf[b]) ++b;
    }
    if (b < B && pf[b] + static_cast<int64_t>(h) * seg_blocks(pf, b, Hkv) < hi) {
      if constexpr (NT == 1)
        qn_mul = load_query<D, FP8, BF16>(qn, a, b, h, r, c);
      else
        prefetch_query_l2<D>(a, b, h, lane);
    }
  };
  prefetch_next_query(ch0.b, ch0.h);
  top_up(false);

  PA_TRACE_WARP(gw, 0, t_entry);
  PA_TRACE_ONLY(int tr_pieces = 0; int tr_split = 0);

  WarpAcc<D> st[NT];   // one per tile of 8 query columns
  auto reset_acc = [&]() {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
      for (int i = 0; i < D / 16; ++i)
        st[t].o[i][0] = st[t].o[i][1] = st[t].o[i][2] = st[t].o[i][3] = 0.f;
      st[t].m0 = st[t].m1 = -INFINITY;
      st[t].l0 = st[t].l1 = 0.f;
    }
  };
  reset_acc();

  const float unboost = FP8 ? 1.f / kPBoost : 1.f;
  int piece_no = 0;

  while (ch0.nb > 0) {
    const int L = len[ch0.b];
    const int fb0 = GENERAL ? window_first_block(L, a.window, a.n_q) : 0;
    // fused append: the new row, when this chunk ends its sequence.  Loaded
    // here rather than a chunk ahead: held across the loop it would cost the
    // E4M3 variant its third CTA per SM (or spills).
    const NewRow nt0 = load_new_row<D, APPEND && !FP8>(a, ch0, pf, lane);
    // fused append: index in this chunk of the sequence's last block, if any
    // (E4M3: the out-of-line append reads the slot and the row itself)
    const bool ends_seg = ch0.cb0 + ch0.nb == seg_blocks(pf, ch0.b, Hkv);
    const int t_last = (APPEND && ((FP8 && ends_seg) || nt0.slot >= 0)) ? ch0.nb - 1 : -1;
    for (int t = 0; t < ch0.nb && !dead; ++t) {
      const int s = computed % STAGES;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(sbar + 8 * s, (computed / STAGES) & 1, a.wait_limit_ns))) {
        if (lane == 0) atomicOr(a.status, kStatusTimeout);
        dead = true;
        break;
      }
      PA_TRACE_ONLY(if (computed == 0) PA_TRACE_WARP(gw, 1, pa_now()));
      const int id = __shfl_sync(0xffffffffu, id0, t);
      float sl2 = a.scale_log2 * q_mul, v_mul = 1.f;
      if constexpr (FP8) {
        sl2 *= __shfl_sync(0xffffffffu, ks0, t);
        v_mul = __shfl_sync(0xffffffffu, vs0, t) * kPBoost;
      }
      if constexpr (APPEND) {
        // This step's token of the sequence lands in its last block at row
        // (L-1) % 16: write it to the pool and into the tile just fetched
        // (which may predate the write), then attend.
        if (t == t_last && id >= 0 && id < a.num_blocks) {
          const int row = (L - 1) & 15;
          constexpr int ROWB = TL::BYTES / 16;
          uint8_t* ktile = ring_ptr + s * TL::SLOT;
          if constexpr (FP8) {
            const float2 sc = append_e4m3_row<D, BF16>(
                static_cast<const uint16_t*>(a.k_new), static_cast<const uint16_t*>(a.v_new),
                a.slots, ktile, ktile + TL::BYTES, static_cast<uint8_t*>(a.k_pool_w),
                static_cast<uint8_t*>(a.v_pool_w), a.k_scale_w, a.v_scale_w, a.status, ch0.b,
                ch0.h, Hkv, id, row, __shfl_sync(0xffffffffu, ks0, t),
                __shfl_sync(0xffffffffu, vs0, t), lane);
            sl2 = a.scale_log2 * q_mul * sc.x;
            v_mul = sc.y * kPBoost;
          } else if (nt0.slot != static_cast<int64_t>(id) * 16 + row) {
            if (lane == 0) atomicOr(a.status, kStatusBadSlot);   // not a decode-step slot
          } else {
            const int64_t prow = (static_cast<int64_t>(id) * Hkv + ch0.h) * 16 + row;
            uint8_t* kp = static_cast<uint8_t*>(a.k_pool_w) + prow * ROWB;
            uint8_t* vp = static_cast<uint8_t*>(a.v_pool_w) + prow * ROWB;
            // the lane's D/16 elements of the row, at their swizzled place in the tile
            const uint32_t so = D == 128 ? swz(row, lane >> 1) + 8 * (lane & 1)
                                         : swz(row, lane >> 2) + 4 * (lane & 3);
            uint8_t* kt = ktile + so;
            uint8_t* vt = kt + TL::BYTES;
            if constexpr (D == 128) {
              *reinterpret_cast<uint2*>(kt) = nt0.k;
              *reinterpret_cast<uint2*>(vt) = nt0.v;
              *reinterpret_cast<uint2*>(kp + 8 * lane) = nt0.k;
              *reinterpret_cast<uint2*>(vp + 8 * lane) = nt0.v;
            } else {
              *reinterpret_cast<uint32_t*>(kt) = nt0.k.x;
              *reinterpret_cast<uint32_t*>(vt) = nt0.v.x;
              *reinterpret_cast<uint32_t*>(kp + 4 * lane) = nt0.k.x;
              *reinterpret_cast<uint32_t*>(vp + 4 * lane) = nt0.v.x;
            }
            __syncwarp();
          }
        }
      }
      if (id >= 0 && id < a.num_blocks) {
        const int blk0 = (fb0 + ch0.cb0 + t) * 16;   // the block's first position
        const int n_valid = min(16, L - blk0);
        if constexpr (NT == 1) {
          attend_block<D, FP8, BF16, GENERAL>(
              st, qf, ring + s * TL::SLOT, ring + s * TL::SLOT + TL::BYTES,
              cm[0], blk0 - (L - a.n_q), n_valid, sl2, v_mul, r, c);
        } else {
          if (q_pending) {   // the piece's query rows, copied when it started
            cp_async_wait_all();
            __syncwarp();
            q_pending = false;
          }
          attend_block_mt<D, FP8, BF16, GENERAL, NT>(
              st, qbuf, ring + s * TL::SLOT, ring + s * TL::SLOT + TL::BYTES, cm,
              blk0 - (L - a.n_q), n_valid, sl2, v_mul, r, c);
        }
      }
      __syncwarp();
      ++computed;
      top_up(false);
    }

    // ---- does this chunk end its piece?  Then the warp's result is final.
    const int nbk = seg_blocks(pf, ch0.b, Hkv);
    const int64_t s0 = pf[ch0.b] + static_cast<int64_t>(ch0.h) * nbk;
    const bool piece_end = ch0.cb0 + ch0.nb == static_cast<int>(min(hi, s0 + nbk) - s0);
    if (piece_end) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          st[t].l0 += __shfl_xor_sync(0xffffffffu, st[t].l0, o);
          st[t].l1 += __shfl_xor_sync(0xffffffffu, st[t].l1, o);
        }
      }
      if (s0 >= lo && s0 + nbk <= hi) {
        uint16_t* rows = static_cast<uint16_t*>(a.out) +
                         ((static_cast<int64_t>(ch0.b) * a.q_tokens + a.q_first) * Hq +
                          ch0.h * G) * D;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          int col_off[2];   // output offsets of the lane's columns from query row 0
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int j = 8 * t + 2 * c + k;
            col_off[k] = j < a.n_q * G ? ((j / G) * Hq + j % G) * D : -1;
          }
          store_output<D, FP8, BF16>(st[t], rows, col_off, r, c, unboost);
        }
      } else if (a.ws_acc == nullptr) {
        if (lane == 0) atomicOr(a.status, kStatusNoWorkspace);   // never written through null
      } else {
        // a split segment: the merge launch, running beside this grid,
        // combines its pieces as soon as all are written
#pragma unroll
        for (int t = 0; t < NT; ++t)
          store_partial<D, FP8, ROWS>(st[t], a, gw, piece_no == 0 ? 0 : 1, r, c, unboost, t);
      }
      ++piece_no;
      PA_TRACE_ONLY(++tr_pieces; tr_split += !(s0 >= lo && s0 + nbk <= hi));
      reset_acc();
    }

    // ---- advance to chunk k+1
    ch0 = ch1;
    ch1 = ch2;
    ch2 = next_chunk(ch2, hi, pf, B, Hkv);
    id0 = id1;
    id1 = id2;
    id2 = chunk_id(ch2);
    if constexpr (FP8) {
      ks0 = ks1;
      vs0 = vs1;
      ks1 = vs1 = 1.f;
      if (ch1.nb > 0 && id1 >= 0 && id1 < a.num_blocks) {
        ks1 = __ldg(a.k_scale + static_cast<int64_t>(id1) * Hkv + ch1.h);
        vs1 = __ldg(a.v_scale + static_cast<int64_t>(id1) * Hkv + ch1.h);
      }
    }
    if (ic == 0) it = 0;        // the cursor had fetched all of chunk k
    ic = 0;
    if (piece_end && ch0.nb > 0) {
      if constexpr (NT == 1) {
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
          qf[i][0] = qn[i][0];
          qf[i][1] = qn[i][1];
        }
        q_mul = qn_mul;
      } else {
        __syncwarp();   // every lane has read the finished piece's rows
        q_mul = fill_query(ch0.b, ch0.h);
      }
      prefetch_next_query(ch0.b, ch0.h);
    }
    top_up(false);
  }
  PA_TRACE_WARP(gw, 2, pa_now());

  if constexpr (NT > 1) cp_async_wait_all();   // no query-buffer copy outlives the warp
  if (dead) {
    // Wait (bounded, never shorter than the default limit, whatever a test
    // set) for this warp's copies still in flight: none may land in shared
    // memory after the CTA has left it.
    const uint64_t drain = a.wait_limit_ns > kWaitLimitNs ? a.wait_limit_ns : kWaitLimitNs;
    for (; computed < issued; ++computed)
      (void)mbar_wait(sbar + 8 * (computed % STAGES), (computed / STAGES) & 1, drain);
  }

  PA_TRACE_WARP(gw, 3, pa_now());
  PA_TRACE_WARP(gw, 4, tr_pieces);
  PA_TRACE_WARP(gw, 5, tr_split);
  PA_TRACE_WARP(gw, 6, static_cast<unsigned long long>(hi - lo));
  PA_TRACE_WARP(gw, 7, pa_smid());
}

// ------------------------------------------------------------ merge launch
// The log-sum-exp merge of each split segment's pieces:
//   out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p
// (log2 units).  One CTA per (sequence, kv head, run of query rows); thread
// (j, g, d4) owns output columns 4*d4 .. 4*d4+3 of query row g within piece
// group j.  The segment's pieces are dealt in rounds of groups x kMergeBatch:
// group j takes pieces j*kMergeBatch .. of each round, so a round has the
// loads of up to 16 pieces in flight at once (a round costs about one L2
// round trip, however many of its pieces a thread folds).  Each group folds
// its pieces in order, rescaling its running state to each batch's maximum;
// at the end group 0 folds the other groups' states in group order: a fixed
// order, so results are deterministic.  Segments attended whole by one
// worker are skipped.
//
// The number of groups is the launch's (launch_merge): two only for
// partials of 8 rows (16 or 32 rows fill a CTA already, and their workers
// hold long shares, so few pieces), and only while the grid stays small
// (a batch of few sequences and kv heads, whose segments are split into
// many short pieces).  The kernel reads it from DecodeArgs::merge_groups and
// its rows per CTA from its grid.
//
// The launch runs beside the attention grid: it is scheduled once every
// attention CTA has passed its prologue, so it never holds resources an
// attention CTA waits for.  It finds the block stream's layout from the
// context lengths, as each attention CTA did, and reads its pieces as they
// are written (a zero word is a partial not written yet): a segment is
// merged as soon as its last piece lands, and only the segments of the last
// warps to finish are merged after the attention ends.  While a round is
// incomplete, warp 0 polls the first word of each missing piece (lane j:
// piece j of the round), so waiting costs one load per piece per poll.  The
// CTA zeroes the partials it read.  The last CTA ends with
// griddepcontrol.wait: the launch completes after the attention grid has
// completed and its writes are visible.
//
// A CTA has at most kMergeThreads threads and registers for two per SM, so
// that one fits beside an attention CTA that has not finished.
constexpr int kMergeThreads = 256;
#ifndef PA_MERGE_BATCH
#define PA_MERGE_BATCH 8
#endif
constexpr int kMergeBatch = PA_MERGE_BATCH;       // pieces a thread loads at once
constexpr int kMergeMaxGroups = 2;
static_assert(kMergeMaxGroups * kMergeBatch <= 32, "one poll lane per piece of a round");
// merge CTAs per SM the launch keeps to when it chooses several groups
constexpr int kMergeCtasPerSm = 4;

template <int D, bool BF16, int ROWS>
__global__ void __launch_bounds__(kMergeThreads, 2)
merge_kernel(const DecodeArgs a) {
  PA_TRACE_ONLY(const unsigned long long t_in = pa_now());
  // a decode launched after this one with an early prologue may start now:
  // it waits for this launch to complete before touching what it writes
  griddep_launch_dependents();
  constexpr int COLS = D / 4;
  constexpr int RG = kMergeThreads / (2 * COLS);   // rows per CTA at most, with 2+ groups
  __shared__ int red[kMergeThreads / 32][2];
  __shared__ unsigned want;
  __shared__ int fail;
  // the running state of groups 1.. at the end, for group 0 to fold
  __shared__ float gm[kMergeMaxGroups][RG], gs[kMergeMaxGroups][RG];
  __shared__ float4 gacc[kMergeMaxGroups - 1][RG][COLS];
  const int Hkv = a.Hkv, G = a.group;
  const int b = blockIdx.x / Hkv, h = blockIdx.x - b * Hkv;
  const int tid = threadIdx.x, lane = tid & 31;

  // ---- the block stream: its length W and the start of sequence b's segments
  int before = 0, total = 0;
  for (int i = tid; i < a.B; i += blockDim.x) {
    const int n = stream_units(a, launch_len(a, __ldg(a.context_lens + i))) * Hkv;
    total += n;
    before += i < b ? n : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  if (lane == 0) {
    red[tid >> 5][0] = before;
    red[tid >> 5][1] = total;
  }
  if (tid == 0) fail = 0;
  __syncthreads();
  before = total = 0;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
    before += red[w][0];
    total += red[w][1];
  }
  const int nbk = stream_blocks(a, launch_len(a, __ldg(a.context_lens + b)));
  int w0 = 0, np = 0, first_slot = 0;
  if (nbk > 0) {
    const int64_t W = total;
    const int64_t NW = min(a.workers > 0 ? static_cast<int64_t>(a.workers)
                                         : static_cast<int64_t>(a.split_ctas) * kWarps,
                           W);
    // the segment's units start at s0, its blocks at sb (after seg_cost units)
    const int64_t s0 = before + static_cast<int64_t>(h) * (nbk + a.seg_cost);
    const int64_t sb = s0 + a.seg_cost;
    w0 = worker_of(sb, W, NW);
    np = worker_of(sb + nbk - 1, W, NW) - w0 + 1;
    first_slot = s0 > worker_lo(w0, W, NW) ? 1 : 0;   // the segment is w0's last piece
  }
  PA_TRACE_ONLY(if (tid == 0 && blockIdx.x < 16384) {
    g_pa_trace_merge[blockIdx.x * 4 + 0] = t_in;
    g_pa_trace_merge[blockIdx.x * 4 + 1] = pa_now();
    g_pa_trace_merge[blockIdx.x * 4 + 2] = 0;
    g_pa_trace_merge[blockIdx.x * 4 + 3] = 0;
  });

  if (np > 1) {                                  // a split segment (np is CTA-uniform)
    // this launch's rows per CTA and piece groups: the live rows are spread
    // evenly over grid y, each row takes D/4 threads per group (the block is
    // rounded up to whole warps; threads past the groups hold no row)
    const int live = a.n_q * G;
    const int rows = (live + static_cast<int>(gridDim.y) - 1) / static_cast<int>(gridDim.y);
    const int groups = a.merge_groups > 0 ? a.merge_groups : 1;
    const int grp = tid / (rows * COLS);                 // the thread's piece group
    const int rl = (tid - grp * rows * COLS) / COLS;     // its row within the CTA
    const int d4 = tid % COLS;
    const int g0 = static_cast<int>(blockIdx.y) * rows;  // the CTA's first query row
    const int g = g0 + rl;                               // the thread's query row
    const bool row = grp < groups && g < live;
    // partial row of piece p for query row q
    auto prow = [&](int p, int q) {
      return piece_row(w0 + p, p == 0 ? first_slot : 0, q, ROWS);
    };
    const int kRound = groups * kMergeBatch;
    float M = -INFINITY, S = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    bool dirty = false;
    PA_TRACE_ONLY(int tr_waits = 0);
    for (int p0 = 0; p0 < np; p0 += kRound) {
      const int pr = min(kRound, np - p0);               // pieces of the round
      const int pg = p0 + grp * kMergeBatch;             // the group's first piece
      const int pn = max(0, min(kMergeBatch, np - pg));  // and its pieces in the round
      uint2 ml[kMergeBatch];
      uint4 v[kMergeBatch];
      // Issue every load of the batch before looking at any (they are in
      // flight together, with the other groups'); then note the pieces not
      // yet seen whole.  Piece pg + k sits 2 ROWS rows after piece pg + k - 1
      // (slot 0 of the next worker), except that the segment's first piece
      // may be its worker's slot 1.
      const int64_t rb = static_cast<int64_t>(w0 + pg) * 2 * ROWS + g;
      const float* mlb = a.ws_ml + rb * 2;
      const float* vb = a.ws_acc + rb * D + 4 * d4;
      const int s0x = pg == 0 ? first_slot * ROWS : 0;
      auto load = [&](int k) {
        const int dr = k == 0 ? s0x : 2 * ROWS * k;
        ml[k] = ld_relaxed_v2(mlb + dr * 2);
        v[k] = ld_relaxed_v4(vb + static_cast<int64_t>(dr) * D);
      };
      auto missing_of = [&](unsigned set) {
        unsigned m = 0;
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k)
          if ((set >> k & 1u) &&
              !(ml[k].x && ml[k].y && v[k].x && v[k].y && v[k].z && v[k].w))
            m |= 1u << k;
        return m;
      };
      const unsigned mine = row ? (1u << pn) - 1u : 0u;
#pragma unroll
      for (int k = 0; k < kMergeBatch; ++k)
        if (mine >> k & 1u) load(k);
      unsigned missing = missing_of(mine);       // pieces this thread has not seen whole
      if (__syncthreads_or(missing != 0u)) {
        // wait for the round's missing pieces (bounded), then read them again
        const uint64_t t0 = tid == 0 ? global_ns() : 0;
        for (;;) {
          if (tid == 0) want = 0u;
          __syncthreads();
          if (missing) atomicOr(&want, missing << (grp * kMergeBatch));
          __syncthreads();
          const unsigned need = want;
          if (need == 0u) break;
          PA_TRACE_ONLY(++tr_waits);
          if (tid < 32 && lane < pr && (need >> lane & 1u)) {
            const uint32_t* first =
                reinterpret_cast<const uint32_t*>(a.ws_ml + prow(p0 + lane, g0) * 2);
            const uint64_t tl = global_ns();
            while (ld_relaxed_b32(first) == 0u) {
              __nanosleep(64);
              if (global_ns() - tl > a.wait_limit_ns) {
                fail = 1;
                break;
              }
            }
          }
          if (tid == 0 && global_ns() - t0 > a.wait_limit_ns) fail = 1;
          __syncthreads();
          if (fail) break;
#pragma unroll
          for (int k = 0; k < kMergeBatch; ++k)
            if (missing >> k & 1u) load(k);
          missing = missing_of(missing);
        }
        if (fail) break;                         // (uniform: read after a barrier)
      }
      if (!row || pn == 0) continue;
      float mk[kMergeBatch];
      float mb = M;
#pragma unroll
      for (int k = 0; k < kMergeBatch; ++k) {
        mk[k] = k < pn ? ws_dec(ml[k].x) : -INFINITY;
        // a written piece has attended nothing (max -inf) or has a sum of at
        // least 1 (its largest score's own weight)
        if (k < pn && mk[k] != -INFINITY && ws_dec(ml[k].y) < 0.5f) dirty = true;
        mb = fmaxf(mb, mk[k]);
      }
      if (mb == -INFINITY) continue;             // nothing attended yet
      const float keep = fast_exp2(M - mb);
      acc.x *= keep;
      acc.y *= keep;
      acc.z *= keep;
      acc.w *= keep;
      S *= keep;
#pragma unroll
      for (int k = 0; k < kMergeBatch; ++k) {
        if (k >= pn) continue;
        const float e = fast_exp2(mk[k] - mb);
        S += e * ws_dec(ml[k].y);
        acc.x += e * ws_dec(v[k].x);
        acc.y += e * ws_dec(v[k].y);
        acc.z += e * ws_dec(v[k].z);
        acc.w += e * ws_dec(v[k].w);
      }
      M = mb;
    }
    if (fail) {
      if (tid == 0) atomicOr(a.status, kStatusTimeout);
    } else {
      // group 0 folds the other groups' states, in group order
      if (row && grp > 0) {
        gacc[grp - 1][rl][d4] = acc;
        if (d4 == 0) {
          gm[grp][rl] = M;
          gs[grp][rl] = S;
        }
      }
      __syncthreads();
      if (row && grp == 0) {
        for (int j = 1; j < groups; ++j) {
          const float mj = gm[j][rl];
          const float mb = fmaxf(M, mj);
          if (mb == -INFINITY) continue;         // neither has attended anything
          const float k0 = fast_exp2(M - mb), k1 = fast_exp2(mj - mb);
          const float4 aj = gacc[j - 1][rl][d4];
          S = S * k0 + gs[j][rl] * k1;
          acc.x = acc.x * k0 + aj.x * k1;
          acc.y = acc.y * k0 + aj.y * k1;
          acc.z = acc.z * k0 + aj.z * k1;
          acc.w = acc.w * k0 + aj.w * k1;
          M = mb;
        }
        const float inv = S > 0.f ? 1.f / S : 0.f;
        uint2 o;
        o.x = pack2<BF16>(acc.x * inv, acc.y * inv);
        o.y = pack2<BF16>(acc.z * inv, acc.w * inv);
        uint16_t* out = static_cast<uint16_t*>(a.out) +
                        ((static_cast<int64_t>(b) * a.q_tokens + a.q_first + g / G) * a.Hq +
                         h * G + g % G) * D;
        *reinterpret_cast<uint2*>(out + 4 * d4) = o;
      }
      if (row) {
        if (dirty) atomicOr(a.status, kStatusWsDirty);
        // leave the workspace zero-filled for the next call: each thread the
        // pieces its group read
        for (int p0 = 0; p0 < np; p0 += kRound) {
          const int pg = p0 + grp * kMergeBatch;
          const int pn = min(kMergeBatch, np - pg);
          for (int k = 0; k < pn; ++k) {
            const int64_t r = prow(pg + k, g);
            __stcg(reinterpret_cast<uint4*>(a.ws_acc + r * D) + d4, make_uint4(0u, 0u, 0u, 0u));
            if (d4 == 0) __stcg(reinterpret_cast<uint2*>(a.ws_ml + r * 2), make_uint2(0u, 0u));
          }
        }
      }
    }
    PA_TRACE_ONLY(if (tid == 0 && blockIdx.x < 16384) {
      g_pa_trace_merge[blockIdx.x * 4 + 2] = pa_now();
      g_pa_trace_merge[blockIdx.x * 4 + 3] = np + 1000ull * tr_waits;
    });
  }
  if (blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1 && tid == 0) griddep_wait();
  // device-side handshake: the last merge CTA to finish, once the attention
  // grid has completed (its own outputs written and visible), signals the
  // step done; it does so even after a wait gave up, so that a copy waiting
  // on the signal never waits forever (the status word carries the failure).
  // Every reader of the signal and of the output (the stream waiting on it,
  // the copy engine after it, later kernels) is on this GPU: gpu scope.
  if (a.done != nullptr) {
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      if (atomicAdd(a.done_count, 1u) == gridDim.x * gridDim.y - 1) {
        griddep_wait();
        *a.done_count = 0u;
        __threadfence();
        st_release_gpu_b32(a.done, a.done_value);
      }
    }
  }
}

// The merge launch, allowed to be scheduled while the attention grid runs
// (programmatic stream serialization).
// ROWS: the partials' rows per piece (a.rows; 8 per tile of query columns
// the attention launch held).
template <int D, bool BF16, int ROWS>
cudaError_t launch_merge(const DecodeArgs& args, cudaStream_t s) {
  DecodeArgs a = args;
  cudaLaunchConfig_t cfg = {};
  // D/4 threads per query row and group, at most kMergeThreads per CTA; the
  // live rows spread evenly over the CTAs of a (sequence, kv head) (grid y).
  // Groups: for partials of 8 rows, the most (2 or 1) that keep the grid
  // within kMergeCtasPerSm CTAs per SM; more CTAs than the SMs take in as
  // attention CTAs leave would hold back the next launch's start.
  constexpr int COLS = D / 4;
  const int live = a.n_q * a.group;
  const int64_t pairs = static_cast<int64_t>(a.B) * a.Hkv;
  auto chunks_for = [&](int groups) {
    const int rpc = kMergeThreads / (groups * COLS);
    return (live + rpc - 1) / rpc;
  };
  int groups = ROWS <= 8 ? kMergeMaxGroups : 1;
  const int64_t budget = static_cast<int64_t>(device_sm_count()) * kMergeCtasPerSm;
  while (groups > 1 && pairs * chunks_for(groups) > budget) groups /= 2;
  const int chunks = chunks_for(groups);
  const int rows = (live + chunks - 1) / chunks;
  a.merge_groups = groups;
  cfg.gridDim = dim3(static_cast<unsigned>(pairs), static_cast<unsigned>(chunks));
  // whole warps (the length scan shuffles over full warps)
  cfg.blockDim = dim3(static_cast<unsigned>((rows * groups * COLS + 31) & ~31));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel<D, BF16, ROWS>, a);
}

// cuTensorMapEncodeTiled, from the driver (no link against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// The tensor map of a 16-bit pool [tiles][16 rows][D], seen as a 3-D tensor
// (D elements, 16 rows, tiles; innermost first) and copied in boxes of 64
// elements x 16 rows x 1 tile with the 128-byte swizzle.  Encoding is host
// work only; the last few maps are kept per thread, keyed by pool and shape,
// since a serving loop passes the same pools call after call.
cudaError_t tile_tensor_map(CUtensorMap* m, const void* pool, int D, int64_t tiles) {
  struct Entry {
    const void* pool;
    int64_t tiles;
    int D;
    CUtensorMap map;
  };
  constexpr int kEntries = 40;
  static thread_local Entry cache[kEntries] = {};
  static thread_local int next = 0;
  for (const Entry& e : cache)
    if (e.pool == pool && e.tiles == tiles && e.D == D) {
      *m = e.map;
      return cudaSuccess;
    }
  const auto enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  if (tiles <= 0 || tiles > INT_MAX) return cudaErrorInvalidValue;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), 16, static_cast<cuuint64_t>(tiles)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(2 * D), static_cast<cuuint64_t>(32 * D)};
  const cuuint32_t box[3] = {64, 16, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r =
      enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(pool), dims, strides, box, elem,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  cache[next] = Entry{pool, tiles, D, *m};
  next = (next + 1) % kEntries;
  return cudaSuccess;
}

template <int D, bool FP8, bool BF16, int STAGES, bool APPEND, bool GENERAL, int CTAS, int NT>
cudaError_t launch_one(const DecodeArgs& args, cudaStream_t s) {
  using TL = Tile<D, FP8, STAGES>;
  constexpr int QBUFS = NT > 1 ? kWarps * 8 * NT * D * 2 : 0;   // the warps' query buffers
  DecodeArgs a = args;
  if constexpr (TL::SWZ) {
    const int64_t tiles = static_cast<int64_t>(a.num_blocks) * a.Hkv;
    cudaError_t e = tile_tensor_map(&a.tm_k, a.k_cache, D, tiles);
    if (e == cudaSuccess) e = tile_tensor_map(&a.tm_v, a.v_cache, D, tiles);
    if (e != cudaSuccess) return e;
  }
  const Layout lay = make_layout(TL::RING + TL::PAD + QBUFS, STAGES, a.B);
  auto* kern = decode_kernel<D, FP8, BF16, STAGES, APPEND, GENERAL, CTAS, NT>;
  // The dynamic shared-memory limit is an attribute of the function shared
  // by every host thread: it is raised once per device, under a lock, to the
  // layout of the largest batch a launch takes, so no thread ever lowers it
  // below what another thread's launch asks for.
  {
    static std::mutex mu;
    static bool raised[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!raised[dev]) {
      const int most = make_layout(TL::RING + TL::PAD + QBUFS, STAGES, kMaxBatchPerLaunch).total;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
      if (e != cudaSuccess) return e;
      raised[dev] = true;
    }
  }
  cudaError_t e = cudaSuccess;
  if (a.early) {
    // a programmatic dependent launch: the prologue may overlap the previous
    // kernel on the stream, the rest waits for it (griddepcontrol.wait)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.split_ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(lay.total);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
  } else {
    kern<<<static_cast<unsigned>(a.split_ctas), kThreads, lay.total, s>>>(a);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  if (a.ws_acc == nullptr) return cudaSuccess;
  return launch_merge<D, BF16, 8 * NT>(a, s);
}

// Shared memory and registers per CTA are traded against resident CTAs per
// SM.  16-bit pools: 96 KB of rings per CTA (3 slots of 8 KB per warp at
// D=128), two CTAs per SM.  E4M3 pools move half the bytes per token, so the
// same in-flight bytes take twice the tokens' worth of dequantisation and
// MMA work; there a third CTA per SM (64 KB of rings each, registers capped
// so that 3 x 128 threads fit) hides more of that latency than deeper rings
// would.
#ifndef PA_RING_KB_F16
#define PA_RING_KB_F16 96
#endif
#ifndef PA_CTAS_F16
#define PA_CTAS_F16 2
#endif
#ifndef PA_RING_KB_FP8
#define PA_RING_KB_FP8 64
#endif
#ifndef PA_CTAS_FP8
#define PA_CTAS_FP8 3
#endif
constexpr int ring_kb(bool fp8) { return fp8 ? PA_RING_KB_FP8 : PA_RING_KB_F16; }
constexpr int ctas_per_sm(bool fp8) { return fp8 ? PA_CTAS_FP8 : PA_CTAS_F16; }

// With NT > 1 tiles of query columns per warp (more than 8 query rows per
// (sequence, kv head)) the accumulators take NT times the registers, so both
// pool types run two CTAs per SM, and each warp's query buffer (8 NT rows of
// head_dim 16-bit values) comes out of the 96 KB a CTA has for its rings.
template <int D, bool FP8, bool BF16, int NT>
cudaError_t launch_dtype(const DecodeArgs& a, cudaStream_t s) {
  constexpr int SLOT = 2 * 16 * (FP8 ? D : 2 * D);    // one K and one V tile
  constexpr int QBUF_KB = NT > 1 ? kWarps * 8 * NT * D * 2 / 1024 : 0;
  constexpr int RING_KB = NT > 1 ? 96 - QBUF_KB : ring_kb(FP8);
  constexpr int STAGES_R = RING_KB * 1024 / (kWarps * SLOT);
  constexpr int STAGES = STAGES_R < 2 ? 2 : STAGES_R;
  constexpr int CTAS = NT > 1 ? 2 : ctas_per_sm(FP8);
  const bool general = a.window > 0 || a.n_q > 1;   // a later pass of 1 token is plain
  if (a.k_new != nullptr)
    return general ? launch_one<D, FP8, BF16, STAGES, true, true, CTAS, NT>(a, s)
                   : launch_one<D, FP8, BF16, STAGES, true, false, CTAS, NT>(a, s);
  return general ? launch_one<D, FP8, BF16, STAGES, false, true, CTAS, NT>(a, s)
                 : launch_one<D, FP8, BF16, STAGES, false, false, CTAS, NT>(a, s);
}

template <int NT>
cudaError_t launch_nt(const DecodeArgs& a, bool fp8, bool bf16, cudaStream_t s) {
  if (fp8 && bf16)
    return a.D == 128 ? launch_dtype<128, true, true, NT>(a, s)
                      : launch_dtype<64, true, true, NT>(a, s);
  if (fp8)
    return a.D == 128 ? launch_dtype<128, true, false, NT>(a, s)
                      : launch_dtype<64, true, false, NT>(a, s);
  if (bf16)
    return a.D == 128 ? launch_dtype<128, false, true, NT>(a, s)
                      : launch_dtype<64, false, true, NT>(a, s);
  return a.D == 128 ? launch_dtype<128, false, false, NT>(a, s)
                    : launch_dtype<64, false, false, NT>(a, s);
}

}  // namespace
}  // namespace pa
