// decode_tc.cu -- the decode launch for 17 to 32 query rows per (sequence,
// kv head) over 16-bit pools at head_dim 128, on the fifth-generation tensor
// cores: tcgen05.mma with its accumulators in tensor memory.
//
// It computes what decode_kernel (decode_kernels.cuh) computes -- paged
// attention with block-table indirection and an online softmax ("rvLLM:
// High-performance LLM inference in Rust", CUDA Kernels table, "PagedAttention
// V2"), each kv head serving its group of query heads ("LLM Serving Kernels",
// Projects row 04: GQA/MQA) and, with several query tokens per sequence, the
// causal mask among them (speculative decoding) -- for the query groups that
// need more than one 8-column tile of that kernel's mma.sync, where its warps
// become bound by MMA issue rather than by HBM.
//
// Design (sm_103a, one GB300):
//  * One worker per CTA and one CTA per SM (persistent).  The workers share
//    the batch's stream of (sequence, kv head, 16-token block) units as
//    decode_kernel's warps do, except that each segment also counts
//    kTcSegCost units of fixed cost (DecodeArgs::seg_cost), so that workers
//    with many short pieces get fewer blocks.  Split segments are merged by
//    the same merge launch (DecodeArgs::workers, ::seg_cost tell it the split).
//  * A worker walks its share in chunks of up to 8 blocks (128 tokens) of one
//    piece.  Per chunk, with R = 32 query rows (17 to 32 in use):
//      S^T[128 tokens][R] = K_chunk . Q^T       (M = 128 tokens, K = head_dim)
//      O^T[128 d][R]     += V_chunk^T . P^T     (M = head_dim,   K = 128 tokens)
//    on the tensor cores (kind::f16, fp32 accumulators in tensor memory).
//    The operands sit in shared memory with the 128-byte swizzle: a chunk's
//    K and V as [2 halves of head_dim][128 token rows][128 B] (one TMA box of
//    64 elements x 16 rows per block and half, straight from the pool), the
//    query rows as [2][R][128 B] (two TMA boxes of a 3-D map over q), P as
//    [2 halves of the chunk][R][128 B] (tokens contiguous: K-major).
//  * Roles.  Warp 8 issues the copies: rings of 3 K and 3 V slots (32 KB
//    each); a K slot is refilled once its chunk's scores are computed, a V
//    slot once its PV product is done; block ids are read one 32-block range
//    ahead and the next pieces' query rows are asked of L2 early.  Warp 9
//    issues the MMAs (one thread), each as soon as its inputs are ready: a
//    chunk's scores into one of three S buffers, a PV product once P is
//    written.  Warps 0-7 run the softmax in two warpgroups, each on 16 of the
//    query rows, thread t of a group on tensor-memory lane t: token t of the
//    chunk for S, head_dim element t for O.  They read S^T with tcgen05.ld,
//    mask it, exponentiate, write P and keep per-thread row sums.  At a
//    piece's last chunk they reduce the row sums; its O^T is read and stored
//    (the output, or the split piece's partial) in the next chunk, once the
//    piece's last PV product is done, which that chunk waits for anyway.
//  * With an early prologue, the TMA warp asks L2 for its first 16 K/V tiles
//    and first query rows while the kernel before ends.
//  * The softmax offset of a query row moves only when a score of the chunk
//    exceeds it by more than kTcSlack (log2 units).  Then the group's four
//    warps reduce the exact running maximum, scale the row sums and O^T (in
//    tensor memory) down to it; otherwise the chunk's weights use the
//    standing offset.  Any offset that is the maximum of some scores already
//    seen gives the same softmax (the common factor cancels between O and
//    the sum), keeps every weight at most 2^kTcSlack (in range for f16 and
//    bf16 P) and keeps the sum at least 1, so the merge's check and
//    arithmetic hold unchanged.
//  * Tokens without data (past the context, blocks missing from a short
//    chunk, blocks with an invalid id) get weight 0, and their V rows in
//    shared memory are zeroed before the PV product, so whatever those rows
//    held (NaN included) never reaches O.
//
// Every wait is bounded in time (DecodeArgs::wait_limit_ns).  A wait that
// gives up sets kStatusTimeout and a CTA-wide flag; every role then leaves its
// loop at its next wait, a warpgroup's four warps together (they decide at a
// barrier they all reach), the copies and MMAs still in flight are waited for
// (bounded), and tensor memory is freed before the CTA exits.
#include "decode_kernels.cuh"
#include "pa_tc.cuh"

namespace pa {
namespace {

// Slots of a chunk's K (scores) and of its V (PV product), 32 KB each, 192
// KB in all.  A K slot is free once the chunk's scores are computed; a V
// slot is held longer (until the chunk's P is written and its PV product
// done), so V gets more of them.
#ifndef PA_TC_KSTAGES
#define PA_TC_KSTAGES 3
#endif
#ifndef PA_TC_VSTAGES
#define PA_TC_VSTAGES 3
#endif
constexpr int kTcKStages = PA_TC_KSTAGES;
constexpr int kTcVStages = PA_TC_VSTAGES;
static_assert(kTcKStages >= 2 && kTcVStages >= 2 && kTcKStages + kTcVStages <= 6,
              "the slots fit 192 KB");
constexpr int kTcBlocks = 8;             // blocks per chunk: 128 tokens, the MMA's M
constexpr int kTcGroups = 2;             // softmax warpgroups, each on half of the query rows
constexpr int kTcThreads = 320;          // warps 0-7 softmax, 8 copies, 9 MMA
constexpr int kTcCopyWarp = 8, kTcMmaWarp = 9;
constexpr int kTcHalf = 128 * 128;       // one half (64 of head_dim) of one chunk tensor: 16 KB
constexpr int kTcSlot = 2 * kTcHalf;     // K or V of one chunk: 32 KB
constexpr int kTcVRing = kTcKStages * kTcSlot;   // the V slots follow the K slots
constexpr float kTcSlack = 8.f;          // log2 units
constexpr int kTcSBufs = 3;              // S buffers in tensor memory
constexpr uint32_t kTcCols = 128;        // tensor-memory columns: S x 3, O (R x 4 <= 128)
// A piece's fixed cost (its result, the next piece's first chunk, a part-full
// last chunk), in blocks' worth of streaming time: the units each segment
// adds to the work split.
constexpr int kTcSegCost = 10;

// mbarriers
enum : int {
  kBarKFull = 0,                         // [K] a slot's K copies landed
  kBarKEmpty = kBarKFull + kTcKStages,   // [K] its scores are computed: the K slot is free
  kBarVFull = kBarKEmpty + kTcKStages,   // [V] a slot's V copies landed
  kBarVEmpty = kBarVFull + kTcVStages,   // [V] its PV product is done: the V slot is free
  kBarQFull = kBarVEmpty + kTcVStages,   // [2] a query buffer's copies landed
  kBarQEmpty = kBarQFull + 2,            // [2] a query buffer's last MMA is done
  kBarSFull = kBarQEmpty + 2,            // [3] an S buffer holds a chunk's scores (and
                                         //     its mask is in wmeta): 2 arrivals
  kBarSFree = kBarSFull + kTcSBufs,      // [3] the softmax warps have read it (8 arrivals)
  kBarPFull = kBarSFree + kTcSBufs,      // P written (8 arrivals)
  kBarODone = kBarPFull + 1,             // a PV product is done
  kBarFin = kBarODone + 1,               // every MMA issued is done (teardown)
  kBarCount = kBarFin + 1
};

// Dynamic shared memory, from a 1024-byte aligned base: the ring, two query
// buffers and P (swizzled operands), then the small state.  The host sizes
// the launch with the same function (plus 1024 bytes to align the base).
struct TcLayout {
  int q, p, bars, meta, flags, red, red2, mcol, colf, einv, rowoff, misc, pf, len, total;
};
template <int R>
__host__ __device__ inline TcLayout tc_layout(int B) {
  TcLayout l{};
  int o = (kTcKStages + kTcVStages) * kTcSlot;
  l.q = o;     o += 2 * R * 256;
  l.p = o;     o += R * 256;
  l.bars = o;  o += round16(kBarCount * 8);
  l.meta = o;  o += round16((kTcKStages + kTcSBufs) * 8);
  l.flags = o; o += kTcGroups * 2 * 4 * 4;
  l.red = o;   o += 4 * R * 4;
  l.red2 = o;  o += 4 * R * 4;
  l.mcol = o;  o += R * 4;
  l.colf = o;  o += R * 4;
  l.einv = o;  o += R * 4;
  l.rowoff = o; o += R * 4;
  l.misc = o;  o += 16;
  l.pf = o;    o += round16((B + 1) * 4);
  l.len = o;   o += round16(B * 4);
  l.total = o;
  return l;
}

// Launch arguments: the decode's, plus the tensor map of q as a 3-D tensor
// (head_dim, Hq heads, B * q_tokens tokens) with boxes of 64 elements x G
// heads x n_q tokens: one box is half of the query rows of a (sequence, kv
// head), row i * G + g for query token i and head g of the group.
struct TcArgs {
  DecodeArgs a;
  CUtensorMap tm_q;
};

// A thread's bounded wait for an mbarrier phase.  False when the CTA's dead
// flag is set, or when limit_ns passes (then this thread sets the flag and
// the timeout status bit).
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int* dead,
                                        const DecodeArgs& a) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*dead) return false;
    if (global_ns() - t0 > a.wait_limit_ns) {
      *dead = 1;
      atomicOr(a.status, kStatusTimeout);
      return false;
    }
  }
}
// The same, decided for the whole warp.
__device__ __forceinline__ bool tc_wait_warp(uint32_t bar, uint32_t parity, volatile int* dead,
                                             const DecodeArgs& a) {
  return __all_sync(0xffffffffu, tc_wait(bar, parity, dead, a));
}

// Reduction of N per-lane columns over the warp's 32 lanes (max or sum): the
// result for column lane % N ends in this lane.  Each step halves the columns
// a lane carries, exchanging the half it gives up with the partner lane (N-1
// shuffles), then lanes that hold the same column combine.  v is consumed.
template <int N, bool MAX>
__device__ __forceinline__ float warp_columns(float (&v)[N], int lane) {
#pragma unroll
  for (int n = N / 2; n >= 1; n >>= 1) {
    const bool up = (lane & n) != 0;
#pragma unroll
    for (int j = 0; j < n; ++j) {
      const float give = up ? v[j] : v[j + n];
      const float keep = up ? v[j + n] : v[j];
      const float got = __shfl_xor_sync(0xffffffffu, give, n);
      v[j] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = N; o < 32; o <<= 1) {
    const float got = __shfl_xor_sync(0xffffffffu, r, o);
    r = MAX ? fmaxf(r, got) : r + got;
  }
  return r;
}

// ------------------------------------------------------------ work split
// The stream the workers share holds, per segment (sequence b, kv head h),
// C = seg_cost units of the segment's fixed cost, then its blocks: segment
// (b, h) starts at pf[b] + h * u_b (u_b = C + blocks) and its blocks at C
// after that.  Worker w takes units [w U / N, (w+1) U / N) as the merge
// launch assumes; its pieces are the segments' blocks inside its range (a
// range may hold a segment's fixed-cost units and none of its blocks).
// Chunks are walked as first_chunk / next_chunk walk the plain block stream.
__device__ __forceinline__ int seg_nblk(const int* pf, int b, int Hkv, int C) {
  const int u = (pf[b + 1] - pf[b]) / Hkv;
  return u > 0 ? u - C : 0;
}
// The first unit of segment (b, h)'s blocks.
__device__ __forceinline__ int64_t seg_block0(const int* pf, int b, int h, int Hkv, int C) {
  return pf[b] + static_cast<int64_t>(h) * ((pf[b + 1] - pf[b]) / Hkv) + C;
}
// The first chunk of the segment after (b, h) whose blocks start before hi.
template <int CH>
__device__ __forceinline__ Chunk tc_next_segment(int b, int h, int64_t hi, const int* pf, int B,
                                                 int Hkv, int C) {
  ++h;
  if (h == Hkv) {
    h = 0;
    ++b;
    while (b < B && pf[b + 1] == pf[b]) ++b;
  }
  if (b >= B) return Chunk{0, 0, 0, 0};
  const int64_t sb = seg_block0(pf, b, h, Hkv, C);
  if (sb >= hi) return Chunk{0, 0, 0, 0};
  const int pend = static_cast<int>(min(hi - sb, static_cast<int64_t>(seg_nblk(pf, b, Hkv, C))));
  return Chunk{b, h, 0, min(CH, pend)};
}
template <int CH>
__device__ __forceinline__ Chunk tc_first(int64_t lo, int64_t hi, const int* pf, int B, int Hkv,
                                          int C) {
  if (lo >= hi) return Chunk{0, 0, 0, 0};
  int l = 0, r = B;                        // pf[l] <= lo < pf[r]
  while (r - l > 1) {
    const int mid = (l + r) >> 1;
    if (pf[mid] <= lo) l = mid;
    else r = mid;
  }
  const int u = (pf[l + 1] - pf[l]) / Hkv;
  const int h = static_cast<int>((lo - pf[l]) / u);
  const int64_t sb = seg_block0(pf, l, h, Hkv, C);
  const int c0 = lo > sb ? static_cast<int>(lo - sb) : 0;
  const int pend = static_cast<int>(min(hi - sb, static_cast<int64_t>(u - C)));
  if (c0 < pend) return Chunk{l, h, c0, min(CH, pend - c0)};
  return tc_next_segment<CH>(l, h, hi, pf, B, Hkv, C);
}
template <int CH>
__device__ __forceinline__ Chunk tc_next(const Chunk& x, int64_t hi, const int* pf, int B, int Hkv,
                                         int C) {
  if (x.nb == 0) return Chunk{0, 0, 0, 0};
  const int64_t sb = seg_block0(pf, x.b, x.h, Hkv, C);
  const int pend =
      static_cast<int>(min(hi - sb, static_cast<int64_t>(seg_nblk(pf, x.b, Hkv, C))));
  const int n0 = x.cb0 + x.nb;
  if (n0 < pend) return Chunk{x.b, x.h, n0, min(CH, pend - n0)};
  return tc_next_segment<CH>(x.b, x.h, hi, pf, B, Hkv, C);
}

template <bool BF16>
__device__ __forceinline__ uint16_t to16(float x) {
  if constexpr (BF16) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<const uint16_t*>(&h);
  } else {
    const __half h = __float2half_rn(x);
    return *reinterpret_cast<const uint16_t*>(&h);
  }
}

__device__ __forceinline__ void st_relaxed_b32(void* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <bool BF16, int R>
__global__ void __launch_bounds__(kTcThreads, 1)
decode_tc_kernel(const __grid_constant__ TcArgs ta) {
  const DecodeArgs& a = ta.a;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const TcLayout lay = tc_layout<R>(a.B);
  const uint32_t base = smem_u32(smem);
  const uint32_t ring = base, qbuf0 = base + lay.q, pbuf = base + lay.p;
  auto bar = [&](int i) { return base + lay.bars + 8u * static_cast<uint32_t>(i); };
  int2* meta = reinterpret_cast<int2*>(smem + lay.meta);   // per K slot: valid blocks, last id
  int2* wmeta = meta + kTcKStages;                         // per S buffer: the same, for the softmax
  int* flags = reinterpret_cast<int*>(smem + lay.flags);   // [group][2][4] per-chunk votes
  float* red = reinterpret_cast<float*>(smem + lay.red);   // [group][4][R/2] column maxima
  float* red2 = reinterpret_cast<float*>(smem + lay.red2); // [group][4][R/2] column sums
  float* mcol = reinterpret_cast<float*>(smem + lay.mcol); // [R] running max per row (log2 units)
  float* colf = reinterpret_cast<float*>(smem + lay.colf); // [R] per-row factor
  float* einv = reinterpret_cast<float*>(smem + lay.einv); // [R] a finished piece's 1 / sum
  int* rowoff = reinterpret_cast<int*>(smem + lay.rowoff); // [R] output row offsets
  int* misc = reinterpret_cast<int*>(smem + lay.misc);     // [0] tmem base [1] dead [2] ready ok
  int* pf = reinterpret_cast<int*>(smem + lay.pf);
  int* len = reinterpret_cast<int*>(smem + lay.len);
  volatile int* dead = misc + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.B, Hkv = a.Hkv, Hq = a.Hq, G = a.group;
  const int live = a.n_q * G;            // query rows in use (<= R)

  // ---- 0. device-side handshake (see decode_kernel)
  if (tid == 0) misc[1] = 0;
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
      misc[2] = ok;
      if (!ok) atomicOr(a.status, kStatusTimeout);
    }
    __syncthreads();
    if (!misc[2]) return;
  }
  // ---- 1. blocks per sequence and their prefix sum (as decode_kernel)
  {
    const int per = (B + kTcThreads - 1) / kTcThreads;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) {
      const int L = launch_len(a, a.context_lens[b]);
      len[b] = L;
      sum += stream_units(a, L) * Hkv;
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane == 31) flags[warp] = inc;   // (flags: free until the loops start)
    __syncthreads();
    int ex = inc - sum;
    for (int w = 0; w < warp; ++w) ex += flags[w];
    for (int b = b0; b < b1; ++b) {
      pf[b] = ex;
      ex += stream_units(a, len[b]) * Hkv;
    }
    if (tid == kTcThreads - 1) pf[B] = ex;
    __syncthreads();
  }
  const int64_t W = pf[B];
  const int cta = blockIdx.x;
  const int C = a.seg_cost;
  const int64_t NW = min(static_cast<int64_t>(gridDim.x), W);   // never more workers than units
  const int64_t lo = worker_lo(cta, W, NW), hi = worker_lo(cta + 1, W, NW);
  auto first_block = [&](int b) {   // the segment's first block in the sequence
    return a.window > 0 ? window_first_block(len[b], a.window, a.n_q) : 0;
  };
  griddep_launch_dependents();
  if (a.early) {
    // With an early prologue, while the kernel before ends: ask L2 for this
    // worker's first 16 K/V tiles and its first piece's query rows (a
    // prefetch reads nothing into the SM, so what that kernel writes before
    // it completes is still what the copies read; the block ids come from
    // the tables, which that kernel does not write).
    if (warp == kTcCopyWarp && cta < NW) {
      const Chunk c = tc_first<kChunk>(lo, hi, pf, B, Hkv, C);
      if (c.nb > 0) {
        const int id = load_chunk_id(a, c, first_block(c.b), lane);
        if (lane < min(c.nb, 16) && id >= 0 && id < a.num_blocks) {
          const int64_t tile = static_cast<int64_t>(id) * Hkv + c.h;
          prefetch_l2(static_cast<const uint8_t*>(a.k_cache) + tile * 4096, 4096);
          prefetch_l2(static_cast<const uint8_t*>(a.v_cache) + tile * 4096, 4096);
        }
        prefetch_query_l2<128>(a, c.b, c.h, lane);
      }
    }
    griddep_wait();
  }
  // sequences with nothing to attend: a zero output (the softmax warps)
  if (warp < 4 * kTcGroups) {
    for (int b = cta * 4 * kTcGroups + warp; b < B;
         b += static_cast<int>(gridDim.x) * 4 * kTcGroups) {
      const int L = len[b];
      if (L > 0) continue;
      if (L < 0 && lane == 0) atomicOr(a.status, kStatusBadLen);
      uint16_t* o = static_cast<uint16_t*>(a.out) +
                    (static_cast<int64_t>(b) * a.q_tokens + a.q_first) * Hq * 128;
      for (int i = lane; i < a.n_q * Hq * 128; i += 32) o[i] = 0;
    }
  }
  // ---- 2. this CTA's share of the stream
  if (cta >= NW) return;

  if (tid == 0) {
    for (int i = 0; i < kBarCount; ++i) {
      const bool many = (i >= kBarSFree && i < kBarSFree + kTcSBufs) || i == kBarPFull;
      const bool two = i >= kBarSFull && i < kBarSFull + kTcSBufs;
      mbar_init(bar(i), many ? 4u * kTcGroups : two ? 2u : 1u);
    }
    mbar_init_fence();
  }
  if (warp == kTcMmaWarp) tmem_alloc(base + lay.misc, kTcCols);   // misc[0]
  // query rows past the live ones stay zero (their columns score 0, harmlessly)
  for (int j = tid; j < 2 * R * 256 / 16; j += kTcThreads)
    sts128(qbuf0 + 16 * j, make_uint4(0u, 0u, 0u, 0u));
  if (tid < R) {
    mcol[tid] = -INFINITY;
    // output offset of query row tid (token tid / G, head tid % G of the group)
    const int qi = tid / G;
    rowoff[tid] = (qi * Hq + (tid - qi * G)) * 128;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);

  // the piece a chunk belongs to -- s0: the first unit of its segment's
  // blocks, nbk: the segment's blocks, pend: where the piece ends, in blocks
  // from the segment's first; whole: the segment's blocks all lie in this
  // worker's range
  struct Where {
    int nbk, pend;
    int64_t s0;
    bool whole;
  };
  auto where = [&](const Chunk& x) {
    Where w;
    w.nbk = seg_nblk(pf, x.b, Hkv, C);
    w.s0 = seg_block0(pf, x.b, x.h, Hkv, C);
    w.pend = static_cast<int>(min(hi, w.s0 + w.nbk) - w.s0);
    w.whole = w.s0 >= lo && w.s0 + w.nbk <= hi;
    return w;
  };

  if (warp == kTcCopyWarp) {
    // ================================================== copies (TMA)
    // K and V of a chunk go to separate rings (slot s of each = stage s):
    // a K slot is free once the chunk's scores are computed, a V slot once
    // its PV product is done, so K copies run a chunk further ahead.  The V
    // copies of chunk i-1 are issued after the K copies of chunk i.
    const uint64_t pol = l2_policy_evict_first();
    Chunk c32 = tc_first<kChunk>(lo, hi, pf, B, Hkv, C);
    Chunk n32 = tc_next<kChunk>(c32, hi, pf, B, Hkv, C);
    int id = c32.nb > 0 ? load_chunk_id(a, c32, first_block(c32.b), lane) : -1;
    int idn = n32.nb > 0 ? load_chunk_id(a, n32, first_block(n32.b), lane) : -1;
    if (n32.nb > 0 && n32.cb0 == 0) prefetch_query_l2<128>(a, n32.b, n32.h, lane);
    int i = 0, piece = 0, v_done = 0;     // K fills issued, query loads, V fills issued
    int v_tile = -1;                      // lane j < 8: tile of block j of the pending V fill
    unsigned v_valid = 0;
    bool ok = true;
    auto issue_v = [&]() {                // V copies of chunk v_done (< i)
      const int vs = v_done % kTcVStages;
      if (v_done >= kTcVStages &&
          !tc_wait_warp(bar(kBarVEmpty + vs), (v_done / kTcVStages - 1) & 1, dead, a))
        return false;
      if (lane == 0)
        mbar_arrive_expect_tx(bar(kBarVFull + vs), static_cast<uint32_t>(__popc(v_valid)) * 4096u);
      __syncwarp();
      if (v_tile >= 0) {
        const uint32_t vd = ring + kTcVRing + vs * kTcSlot + lane * 2048;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb)
          tensor3_g2s(vd + hb * kTcHalf, &a.tm_v, 64 * hb, 0, v_tile, bar(kBarVFull + vs), pol);
      }
      ++v_done;
      return true;
    };
    while (ok && c32.nb > 0) {
      for (int k = 0; k < c32.nb; k += kTcBlocks) {
        const int nb = min(kTcBlocks, c32.nb - k);
        const int s = i % kTcKStages;
        if (i >= kTcKStages &&
            !tc_wait_warp(bar(kBarKEmpty + s), (i / kTcKStages - 1) & 1, dead, a)) {
          ok = false;
          break;
        }
        if (i == 0 || c32.cb0 + k == 0) {   // a piece starts: its query rows
          const int j = piece & 1;
          if (piece >= 2 && !tc_wait_warp(bar(kBarQEmpty + j), ((piece >> 1) - 1) & 1, dead, a)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(kBarQFull + j), 2u * 128u * static_cast<uint32_t>(live));
            const int tok = c32.b * a.q_tokens + a.q_first;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb)
              tensor3_g2s(qbuf0 + j * (R * 256) + hb * (R * 128), &ta.tm_q, 64 * hb, c32.h * G,
                          tok, bar(kBarQFull + j), pol);
          }
          ++piece;
        }
        // lane j < nb: block j of the chunk
        const int bid = __shfl_sync(0xffffffffu, id, k + (lane & 7));
        const bool mine = lane < nb;
        const bool okid = mine && bid >= 0 && bid < a.num_blocks;
        if (mine && !okid) atomicOr(a.status, kStatusBadBlock);
        const unsigned valid = __ballot_sync(0xffffffffu, okid) & 0xFFu;
        const int last_id = __shfl_sync(0xffffffffu, bid, nb - 1);
        const int tile = okid ? bid * Hkv + c32.h : -1;
        if (lane == 0) {
          meta[s] = make_int2(static_cast<int>(valid), last_id);
          mbar_arrive_expect_tx(bar(kBarKFull + s), static_cast<uint32_t>(__popc(valid)) * 4096u);
        }
        __syncwarp();
        if (okid) {
          const uint32_t kd = ring + s * kTcSlot + lane * 2048;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb)
            tensor3_g2s(kd + hb * kTcHalf, &a.tm_k, 64 * hb, 0, tile, bar(kBarKFull + s), pol);
        }
        ++i;
        if (v_done < i - 1 && !issue_v()) {
          ok = false;
          break;
        }
        v_tile = tile;
        v_valid = valid;
      }
      c32 = n32;
      id = idn;
      n32 = tc_next<kChunk>(n32, hi, pf, B, Hkv, C);
      idn = n32.nb > 0 ? load_chunk_id(a, n32, first_block(n32.b), lane) : -1;
      if (n32.nb > 0 && n32.cb0 == 0) prefetch_query_l2<128>(a, n32.b, n32.h, lane);
    }
    if (ok && v_done < i) issue_v();      // the last chunk's V
    // no copy outlives the CTA: wait (bounded, never shorter than the
    // default limit, whatever a test set) for each buffer's last fill
    const uint64_t t0 = global_ns();
    const uint64_t drain = a.wait_limit_ns > kWaitLimitNs ? a.wait_limit_ns : kWaitLimitNs;
    auto settle = [&](uint32_t b, int fills) {
      if (fills <= 0) return;
      while (!mbar_try_wait(b, (fills - 1) & 1) && global_ns() - t0 < drain) {
      }
    };
    if (lane == 0) {
      for (int st = 0; st < kTcKStages; ++st)
        settle(bar(kBarKFull + st), (i - st + kTcKStages - 1) / kTcKStages);
      for (int st = 0; st < kTcVStages; ++st)
        settle(bar(kBarVFull + st), (v_done - st + kTcVStages - 1) / kTcVStages);
      for (int j = 0; j < 2; ++j) settle(bar(kBarQFull + j), (piece - j + 1) / 2);
    }
    __syncwarp();
  } else if (warp == kTcMmaWarp) {
    // ================================================== MMA issue
    // Two cursors: the next chunk to score (qi) and the next chunk whose PV
    // product to issue (pi < qi).  Each is issued as soon as its inputs are
    // ready -- a chunk's scores once its K tile has landed and an S buffer is
    // free (three buffers), a PV product once P is written and the V tile
    // has landed -- the PV product first when both are.  So K slots free up
    // as soon as their scores are computed, and no result waits for the next
    // chunk's data.
    constexpr uint32_t kIdQK = umma_idesc_f16<BF16>(128, R, false);
    constexpr uint32_t kIdPV = umma_idesc_f16<BF16>(128, R, true);
    const uint32_t tmem_o = tmem + kTcSBufs * R;
    // operand descriptors of stage 0, query buffer 0 and P; a stage, buffer or
    // K step moves the start address (field bits 0-13, address / 16) only
    const uint64_t dk0 = umma_desc_sw128(ring, 16, 1024);
    const uint64_t dv0 = umma_desc_sw128(ring + kTcVRing, kTcHalf, 1024);
    const uint64_t dq0 = umma_desc_sw128(qbuf0, 16, 1024);
    const uint64_t dp = umma_desc_sw128(pbuf, 16, 1024);
    auto ready = [&](int b, int parity) {   // a phase complete (decided by lane 0)
      uint32_t v = 0;
      if (lane == 0) {
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(v)
            : "r"(bar(b)), "r"(parity & 1)
            : "memory");
      }
      return __shfl_sync(0xffffffffu, v, 0) != 0u;
    };
    Chunk x = tc_first<kTcBlocks>(lo, hi, pf, B, Hkv, C);
    int qi = 0, pi = 0, piece = -1;
    // per scored chunk (qi & 3) until its PV product: whether it starts a
    // piece, and the fused append's V row for its tile (-1: none).  A ring
    // of 4, so chunk qi is scored only once chunk qi-4's PV product is
    // issued (its S buffer alone would allow it earlier: that needs only the
    // PV product of chunk qi-5 done, while chunk qi-4's V tile may not have
    // landed).
    unsigned firsts = 0u;
    int vrows[4] = {-1, -1, -1, -1};
    uint2 vvals[4];
    bool ok = true, issued = false;
    uint64_t idle_since = 0;
    for (;;) {
      bool did = false;
      if (pi < qi && ready(kBarPFull, pi) && ready(kBarVFull + pi % kTcVStages, pi / kTcVStages)) {
        const int ps = pi % kTcVStages;
        if (vrows[pi & 3] >= 0) {           // fused append: the new V row into the tile
          *reinterpret_cast<uint2*>(smem + kTcVRing + ps * kTcSlot + vrows[pi & 3]) =
              vvals[pi & 3];
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        if (lane == 0) {
          const uint64_t dv = dv0 + static_cast<uint64_t>(ps * (kTcSlot >> 4));
          const bool first = (firsts >> (pi & 3)) & 1u;
#pragma unroll
          for (int k = 0; k < 8; ++k)   // 16 tokens a step
            umma_f16(tmem_o, dv + static_cast<uint64_t>(k * (2048 >> 4)),
                     dp + static_cast<uint64_t>(((k >> 2) * (R * 128) + (k & 3) * 32) >> 4), kIdPV,
                     !(first && k == 0));
          umma_commit(bar(kBarVEmpty + ps));
          umma_commit(bar(kBarODone));
        }
        __syncwarp();
        ++pi;
        did = true;
      } else if (x.nb > 0 && qi - pi < 4) {
        const int s = qi % kTcKStages, sbuf = qi % kTcSBufs;
        const bool pfirst = qi == 0 || x.cb0 == 0;
        const int np = pfirst ? piece + 1 : piece;
        if (ready(kBarKFull + s, qi / kTcKStages) &&
            (qi < kTcSBufs || ready(kBarSFree + sbuf, qi / kTcSBufs - 1)) &&
            (!pfirst || ready(kBarQFull + (np & 1), np >> 1))) {
          piece = np;
          const Where wh = where(x);
          const bool plast = x.cb0 + x.nb == wh.pend;
          int vrow = -1;
          if (a.k_new != nullptr && x.cb0 + x.nb == wh.nbk) {
            // Fused append: this step's token of the sequence lands in its
            // last block, the chunk's block nb-1, at row (L-1) % 16: written
            // to the pool and into the tiles just fetched (which may predate
            // the write; the V row once the V tile has landed).
            const int2 mt = meta[s];
            const int L = len[x.b];
            const int row = (L - 1) & 15;
            const int64_t slot = __ldg(a.slots + x.b);
            if (((mt.x >> (x.nb - 1)) & 1) && slot >= 0) {
              if (slot != static_cast<int64_t>(mt.y) * 16 + row) {
                if (lane == 0) atomicOr(a.status, kStatusBadSlot);   // not a decode-step slot
              } else {
                const int64_t src = (static_cast<int64_t>(x.b) * Hkv + x.h) * 128 + 4 * lane;
                const uint2 kv =
                    *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.k_new) + src);
                vvals[qi & 3] =
                    *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.v_new) + src);
                const int64_t prow = (static_cast<int64_t>(mt.y) * Hkv + x.h) * 16 + row;
                *reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.k_pool_w) + prow * 256 +
                                          8 * lane) = kv;
                *reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.v_pool_w) + prow * 256 +
                                          8 * lane) = vvals[qi & 3];
                // elements 4 lane .. 4 lane + 3: half lane / 16, 16-byte
                // chunk (lane % 16) / 2, its 8-byte half lane % 2
                const int tok = (x.nb - 1) * 16 + row;
                const int c = (lane & 15) >> 1;
                vrow = (lane >> 4) * kTcHalf + tok * 128 + ((c ^ (tok & 7)) << 4) + (lane & 1) * 8;
                *reinterpret_cast<uint2*>(smem + s * kTcSlot + vrow) = kv;
                fence_proxy_async_smem();
              }
            }
            __syncwarp();
          }
          vrows[qi & 3] = vrow;
          firsts = (firsts & ~(1u << (qi & 3))) | (pfirst ? 1u << (qi & 3) : 0u);
          if (lane == 0) {   // the chunk's mask for the softmax warps, with its scores
            wmeta[sbuf] = meta[s];
            mbar_arrive(bar(kBarSFull + sbuf));
          }
          tc_fence_after();
          if (lane == 0) {
            const uint64_t dk = dk0 + static_cast<uint64_t>(s * (kTcSlot >> 4));
            const uint64_t dq = dq0 + static_cast<uint64_t>((piece & 1) * (R * 256 >> 4));
#pragma unroll
            for (int k = 0; k < 8; ++k)   // 16 of head_dim a step
              umma_f16(tmem + sbuf * R,
                       dk + static_cast<uint64_t>(((k >> 2) * kTcHalf + (k & 3) * 32) >> 4),
                       dq + static_cast<uint64_t>(((k >> 2) * (R * 128) + (k & 3) * 32) >> 4),
                       kIdQK, k > 0);
            umma_commit(bar(kBarSFull + sbuf));
            umma_commit(bar(kBarKEmpty + s));
            if (plast) umma_commit(bar(kBarQEmpty + (piece & 1)));
          }
          issued = true;
          __syncwarp();
          x = tc_next<kTcBlocks>(x, hi, pf, B, Hkv, C);
          ++qi;
          did = true;
        }
      }
      if (did) {
        idle_since = 0;
        continue;
      }
      if (x.nb == 0 && pi == qi) break;
      // nothing ready: wait a little, give up after the time limit
      if (*dead) {
        ok = false;
        break;
      }
      const uint64_t now = global_ns();
      if (idle_since == 0) {
        idle_since = now;
      } else if (now - idle_since > a.wait_limit_ns) {
        if (lane == 0) {
          *dead = 1;
          atomicOr(a.status, kStatusTimeout);
        }
        ok = false;
        break;
      }
      __nanosleep(32);
    }
    (void)ok;
    // no MMA outlives the CTA: wait (bounded, never shorter than the
    // default limit) for all of them
    if (issued) {
      if (lane == 0) {
        umma_commit(bar(kBarFin));
        const uint64_t t0 = global_ns();
        const uint64_t drain = a.wait_limit_ns > kWaitLimitNs ? a.wait_limit_ns : kWaitLimitNs;
        while (!mbar_try_wait(bar(kBarFin), 0) && global_ns() - t0 < drain) {
        }
      }
      __syncwarp();
    }
  } else {
    // ================================================== softmax (warps 0-7)
    // Warpgroup g (warps 4g .. 4g+3) owns query rows c0 .. c0+RH-1, thread
    // t of the group tensor-memory lane t: token t of the chunk for S, head_dim
    // element t for O.  Per row r every thread holds: mo[r], the offset its
    // weights are taken from (log2 units; 0 before the row has seen a score);
    // thr[r], the raw score above which that offset must move (offset +
    // kTcSlack, over the scale; -inf before any score); l[r], its share of
    // the row sum.  The exact running maximum per row lives in shared memory
    // (mcol), kept by the thread that owns the row (t = r - c0).
    constexpr int RH = R / kTcGroups;
    const int g = warp >> 2, wq = warp & 3;
    const int t = tid & 127;
    const int c0 = g * RH;
    const uint32_t bar_id = 1 + g;
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);   // this warp's lanes
    const float sl2 = a.scale_log2, isl2 = 1.f / a.scale_log2;
    int* gflags = flags + g * 8;
    float* gred = red + g * 4 * RH;
    float* gred2 = red2 + g * 4 * RH;
    float mo[RH], thr[RH], l[RH];
    auto reset_rows = [&]() {
#pragma unroll
      for (int r = 0; r < RH; ++r) {
        mo[r] = 0.f;
        thr[r] = -INFINITY;
        l[r] = 0.f;
      }
    };
    reset_rows();
    // this thread's P column: row r's 16-bit element at pb + r * 128 + sw[r % 8]
    const uint32_t pb = pbuf + (t >> 6) * (R * 128) + (t & 7) * 2;
    uint32_t sw[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) sw[j] = static_cast<uint32_t>(((((t >> 3) & 7) ^ j)) << 4);
    bool bad = false;                     // this warp saw a wait give up
    // a finished piece whose O^T is still to be read and stored
    struct Epilogue {
      int b, h, slot, chunk;
      bool whole, pending;
    } epi{0, 0, 0, 0, false, false};
    // O^T of the finished piece, once its last PV product is done: the
    // group's rows, as outputs (times the owner's 1 / sum) or as partials
    auto store_piece = [&]() {
      epi.pending = false;
      const int q_end = min(c0 + RH, live);
      if (bad || c0 >= q_end) return;
      tc_fence_after();
      uint16_t* out = static_cast<uint16_t*>(a.out) +
                      (static_cast<int64_t>(epi.b) * a.q_tokens + a.q_first) * Hq * 128 +
                      static_cast<int64_t>(epi.h) * G * 128 + t;
      float* ws = a.ws_acc + piece_row(cta, epi.slot, 0, R) * 128 + t;
      float o[RH];
      tmem_ld<RH>(tl + kTcSBufs * R + c0, o);
      tmem_wait_ld();
#pragma unroll
      for (int r = 0; r < RH; ++r) {
        const int q = c0 + r;
        if (q >= q_end) break;
        if (epi.whole)
          out[rowoff[q]] = static_cast<uint16_t>(pack2<BF16>(o[r] * einv[q], 0.f) & 0xFFFFu);
        else
          st_relaxed_b32(ws + q * 128, ws_enc(o[r]));
      }
      tc_fence_before();
    };
    Chunk x = tc_first<kTcBlocks>(lo, hi, pf, B, Hkv, C);
    int i = 0, piece_no = 0;
    while (x.nb > 0) {
      const int vs = i % kTcVStages;       // the chunk's V slot
      const int sb = i % kTcSBufs;
      bad |= !tc_wait_warp(bar(kBarSFull + sb), (i / kTcSBufs) & 1, dead, a);
      const Where wh = where(x);
      const bool pfirst = i == 0 || x.cb0 == 0;
      const bool plast = x.cb0 + x.nb == wh.pend;
      const int L = len[x.b];
      const unsigned valid = static_cast<unsigned>(wmeta[sb].x);
      float v[RH];
      if (!bad) {
        tc_fence_after();
        tmem_ld<RH>(tl + sb * R + c0, v);
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && !bad) mbar_arrive(bar(kBarSFree + sb));
      // Masks: token t has data when its block is in the chunk, has a valid
      // id and the position is inside the context; query row r = i_r G + g
      // (token i_r of n_q) sees relative position rel = pos - (L - n_q) when
      // rel <= i_r and, with a window, rel > i_r - window: r in [rlo, rhi).
      // A warp whose tokens are all seen by every live row skips the masks
      // (rows past the live ones score 0 against zero query rows).
      const int pos = (first_block(x.b) + x.cb0) * 16 + t;
      const bool data = t < x.nb * 16 && ((valid >> (t >> 4)) & 1u) && pos < L;
      const int rel = pos - (L - a.n_q);
      const int rlo = max(rel, 0) * G;
      int rhi = live;
      if (a.window > 0) rhi = min(rhi, max(rel + a.window, 0) * G);
      if (!data) rhi = 0;
      if (!__all_sync(0xffffffffu, rlo == 0 && rhi == live)) {
#pragma unroll
        for (int r = 0; r < RH; ++r) v[r] = c0 + r >= rlo && c0 + r < rhi ? v[r] : -INFINITY;
      }
      bool need = false;
#pragma unroll
      for (int r = 0; r < RH; ++r) need |= v[r] > thr[r];
      // one vote per warp: some score passes its row's threshold (or a wait
      // gave up); the group's four warps read the same votes
      const unsigned vote = __ballot_sync(0xffffffffu, need) != 0u ? 1u : 0u;
      if (lane == 0) gflags[(i & 1) * 4 + wq] = static_cast<int>(vote | (bad || *dead ? 2u : 0u));
      named_bar_sync(bar_id, 128);
      const int f = gflags[(i & 1) * 4] | gflags[(i & 1) * 4 + 1] | gflags[(i & 1) * 4 + 2] |
                    gflags[(i & 1) * 4 + 3];
      if (f & 2) break;                   // (uniform over the group's warps)
      bool o_ready = false;               // the previous PV product is done
      if (f & 1) {
        // new offsets: the exact running maxima, reduced over the chunk's
        // tokens and set by each row's owner; the factor from the old offset
        // (colf) scales the sums here and O^T below
        float c[RH];
#pragma unroll
        for (int r = 0; r < RH; ++r) c[r] = v[r];
        const float cm = warp_columns<RH, true>(c, lane);
        if (lane < RH) gred[wq * RH + lane] = cm;
        named_bar_sync(bar_id, 128);
        if (t < RH) {
          const float mold = mcol[c0 + t];
          const float mx = fmaxf(fmaxf(gred[t], gred[RH + t]), fmaxf(gred[2 * RH + t], gred[3 * RH + t]));
          const float mn = fmaxf(mold, mx * sl2);
          colf[c0 + t] = mn == -INFINITY ? 1.f : fast_exp2(mold - mn);
          mcol[c0 + t] = mn;
        }
        named_bar_sync(bar_id, 128);
#pragma unroll
        for (int r = 0; r < RH; ++r) {
          const float mn = mcol[c0 + r];
          l[r] *= colf[c0 + r];
          mo[r] = mn == -INFINITY ? 0.f : mn;
          thr[r] = mn == -INFINITY ? -INFINITY : (mn + kTcSlack) * isl2;
        }
        if (!pfirst) {
          // O^T columns scaled in tensor memory, once the previous PV is done
          bad |= !tc_wait_warp(bar(kBarODone), (i - 1) & 1, dead, a);
          o_ready = true;
          if (!bad) {
            tc_fence_after();
            float o[RH];
            tmem_ld<RH>(tl + kTcSBufs * R + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int r = 0; r < RH; ++r) o[r] *= colf[c0 + r];
            tmem_st<RH>(tl + kTcSBufs * R + c0, o);
            tmem_wait_st();
          }
        }
      }
      // P (single buffer): the previous PV product must be done reading it
      if (i > 0 && !o_ready) bad |= !tc_wait_warp(bar(kBarODone), (i - 1) & 1, dead, a);
      // the previous piece's O^T (before this chunk's PV product replaces it)
      if (epi.pending) store_piece();
#pragma unroll
      for (int r = 0; r < RH; r += 2) {
        const float p0 = fast_exp2(fmaf(v[r], sl2, -mo[r]));
        const float p1 = fast_exp2(fmaf(v[r + 1], sl2, -mo[r + 1]));
        l[r] += p0;
        l[r + 1] += p1;
        const uint32_t h2 = pack2<BF16>(p0, p1);
        const int rg = c0 + r;
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(pb + rg * 128 + sw[rg & 7]),
                     "h"(static_cast<uint16_t>(h2 & 0xFFFFu))
                     : "memory");
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(pb + (rg + 1) * 128 + sw[(rg + 1) & 7]),
                     "h"(static_cast<uint16_t>(h2 >> 16))
                     : "memory");
      }
      if (g == 0 && __any_sync(0xffffffffu, !data)) {
        // a token without data: its V row (either half) to zero, once the
        // chunk's V copies have landed
        bad |= !tc_wait_warp(bar(kBarVFull + vs), (i / kTcVStages) & 1, dead, a);
        if (!data && !bad) {
          const uint32_t vrow = ring + kTcVRing + vs * kTcSlot + t * 128;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              sts128(vrow + hb * kTcHalf + c * 16, make_uint4(0u, 0u, 0u, 0u));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull));

      if (plast) {
        // ---- the piece's result for the group's rows, first half: row
        // sums (each warp's, then the row owner's total: its reciprocal, or
        // the partial's max and sum).  O^T is read in the next chunk, once
        // the piece's last PV product is done (it is waited for there
        // anyway), so the warps never wait for it here.
        float c[RH];
#pragma unroll
        for (int r = 0; r < RH; ++r) c[r] = l[r];
        const float cs = warp_columns<RH, false>(c, lane);
        if (lane < RH) gred2[wq * RH + lane] = cs;
        named_bar_sync(bar_id, 128);
        epi.b = x.b;
        epi.h = x.h;
        epi.whole = wh.whole;
        epi.slot = piece_no == 0 ? 0 : 1;
        epi.chunk = i;
        epi.pending = true;
        if (!epi.whole && a.ws_acc == nullptr) {
          if (t == 0) atomicOr(a.status, kStatusNoWorkspace);
          epi.pending = false;
        }
        const int q_end = min(c0 + RH, live);
        if (t < RH && c0 + t < q_end && epi.pending) {
          const int q = c0 + t;
          const float sum = (gred2[t] + gred2[RH + t]) + (gred2[2 * RH + t] + gred2[3 * RH + t]);
          if (epi.whole) {
            einv[q] = sum > 0.f ? __frcp_rn(sum) : 0.f;
          } else if (!bad) {
            // a split segment: the merge launch combines its pieces
            st_relaxed_v2(a.ws_ml + piece_row(cta, epi.slot, q, R) * 2, ws_enc(mcol[q]),
                          ws_enc(sum));
          }
        }
        ++piece_no;
        reset_rows();
        if (t < RH) mcol[c0 + t] = -INFINITY;
      }
      x = tc_next<kTcBlocks>(x, hi, pf, B, Hkv, C);
      ++i;
    }
    if (epi.pending) {                    // the last piece: its O^T once its PV is done
      bad |= !tc_wait_warp(bar(kBarODone), epi.chunk & 1, dead, a);
      named_bar_sync(bar_id, 128);        // the owners' reciprocals are visible
      store_piece();
    }
  }
  // ---- teardown: every role has left its loop with nothing in flight
  tc_fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcCols);
  }
}

// The tensor map of q (see TcArgs); the last few are kept per thread, keyed
// by pointer and shape.
cudaError_t q_tensor_map(CUtensorMap* m, const void* q, int Hq, int64_t tokens, int G, int n_q) {
  struct Entry {
    const void* q;
    int64_t tokens;
    int Hq, G, n_q;
    CUtensorMap map;
  };
  constexpr int kEntries = 16;
  static thread_local Entry cache[kEntries] = {};
  static thread_local int next = 0;
  for (const Entry& e : cache)
    if (e.q == q && e.tokens == tokens && e.Hq == Hq && e.G == G && e.n_q == n_q) {
      *m = e.map;
      return cudaSuccess;
    }
  const auto enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  if (tokens <= 0 || tokens > INT_MAX) return cudaErrorInvalidValue;
  const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(tokens)};
  const cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(Hq) * 256};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(n_q)};
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r =
      enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(q), dims, strides, box, elem,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  cache[next] = Entry{q, tokens, Hq, G, n_q, *m};
  next = (next + 1) % kEntries;
  return cudaSuccess;
}

template <bool BF16, int R>
cudaError_t launch_tc(const DecodeArgs& args, cudaStream_t s) {
  TcArgs t{};
  t.a = args;
  DecodeArgs& a = t.a;
  const int64_t tiles = static_cast<int64_t>(a.num_blocks) * a.Hkv;
  cudaError_t e = tile_tensor_map(&a.tm_k, a.k_cache, 128, tiles);
  if (e == cudaSuccess) e = tile_tensor_map(&a.tm_v, a.v_cache, 128, tiles);
  if (e == cudaSuccess)
    e = q_tensor_map(&t.tm_q, a.q, a.Hq, static_cast<int64_t>(a.B) * a.q_tokens, a.group, a.n_q);
  if (e != cudaSuccess) return e;
  // one worker per SM, never more than the workspace holds partials for
  const int sms = device_sm_count();
  const int cap = a.split_ctas * kWarps;
  const int grid = sms < cap ? sms : cap;
  if (grid <= 0) return cudaErrorInvalidValue;
  a.workers = grid;
  a.seg_cost = kTcSegCost;
  auto* kern = decode_tc_kernel<BF16, R>;
  {
    static std::mutex mu;
    static bool raised[kMaxDevices] = {};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!raised[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               tc_layout<R>(kMaxBatchPerLaunch).total + 1024);
      if (e != cudaSuccess) return e;
      raised[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(tc_layout<R>(a.B).total + 1024);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.early ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, t);
  if (e != cudaSuccess) return e;
  if (a.ws_acc == nullptr) return cudaSuccess;
  return launch_merge<128, BF16, R>(a, s);
}

}  // namespace

// 17 to 32 query rows per (sequence, kv head): there, decode_kernel's warps
// hold four tiles of the MMA's 8 columns and are bound by mma.sync issue
// (measured on the Qwen2.5-7B batch: 4 query tokens of 7 heads 103.8 us
// against 107.7, 32 heads on one kv head 36.0 us against 49.9).  With 9 to
// 16 rows decode_kernel stays faster (2 tokens of 7 heads: 76.0 us against
// 95.7), so the kernel above is instantiated for R = 32 only.
bool decode_tc_eligible(const DecodeArgs& a, bool fp8) {
  return !fp8 && a.D == 128 && a.rows == 32 && a.n_q * a.group > 16 &&
         a.n_q * a.group <= 32 && (reinterpret_cast<uintptr_t>(a.q) & 15u) == 0 &&
         a.scale_log2 > 0.f;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, bool bf16, cudaStream_t s) {
  if (a.rows != 32) return cudaErrorInvalidValue;
  return bf16 ? launch_tc<true, 32>(a, s) : launch_tc<false, 32>(a, s);
}

}  // namespace pa
