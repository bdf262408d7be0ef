/*
 * pa.h -- C ABI of libpa: the decode-step hot path of a paged KV cache on
 * one GB300 (sm_103a).
 *
 * Two operations make up one decode step of a vLLM-style serving engine:
 *
 *   1. append: scatter each sequence's new K/V token into a pool of
 *      fixed-size blocks through a slot mapping
 *      ("rvLLM: High-performance LLM inference in Rust", CUDA Kernels table,
 *      "Reshape and Cache"; "rvllm - A Small LLM Inference Engine in Rust",
 *      How it's put together: write positions computed from the block table);
 *   2. decode attention: one query token per sequence attends, with grouped-
 *      query heads, over the blocks its block table lists, with an online
 *      softmax over context partitions merged by log-sum-exp
 *      (rvLLM, CUDA Kernels table, "PagedAttention V2"; "LLM Serving Kernels",
 *      Projects table, row 04 "Paged decode attention").
 *
 * An FP8 variant stores the pool as E4M3 codes with one fp32 scale per
 * (physical block, kv head) and dequantises inside the attention loop (rvLLM,
 * CUDA Kernels table, "FP8 KV Cache"; feature list "FP8 KV cache (E4M3
 * quantization with per-head scaling)"; "LLM Serving Kernels", row 05
 * "E4M3 storage, page scales, fused dequantization").
 *
 * Conventions for every entry point
 *   - A call with zero tokens or zero sequences returns PA_OK at once,
 *     whatever its pointers (empty tensors may have NULL data).
 *   - Pointers named *_cache, q, out, k_new, v_new, slot_mapping,
 *     block_tables, context_lens, *_scale and workspace are DEVICE pointers
 *     owned by the caller; they must be 16-byte aligned.  The library
 *     allocates nothing and keeps no per-call state.
 *   - Layouts are dense row-major:
 *       16-bit pools   [num_blocks][num_kv_heads][block_size][head_dim]
 *       E4M3 pools     same shape, one byte per element
 *       page scales    fp32 [num_blocks][num_kv_heads]
 *       q, out         [num_seqs][num_q_heads][head_dim]
 *       k_new, v_new   [num_tokens][num_kv_heads][head_dim]
 *       block_tables   int32 [num_seqs][max_blocks_per_seq]
 *       context_lens   int32 [num_seqs]  (tokens attended, the new one included)
 *       slot_mapping   int64 [num_tokens] (slot = block * block_size + row;
 *                      a negative slot marks a padding token and is skipped)
 *   - q head hq reads kv head hq / (num_q_heads / num_kv_heads).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on it and never synchronise, except
 *     pa_get_status.
 *   - Argument errors are returned before anything is launched.  Index
 *     errors that only the device can see (a block id outside the pool, a
 *     context length above its bound, a slot outside the pool) are never
 *     dereferenced: the kernel skips the access and sets a bit in the
 *     library's device status word, which pa_get_status reads.
 *   - Supported now: head_dim 64 or 128, block_size 16, num_q_heads /
 *     num_kv_heads from 1 to 32 (multi-query attention included).  Other
 *     shapes return PA_ERR_UNSUPPORTED.
 *   - Host state: for 16-bit pools the decode entry points encode TMA
 *     tensor maps of k_cache and v_cache (host memory, passed by value with
 *     the launch) and keep the last 40 per host thread, keyed by pool
 *     address, tile count and head_dim; the library allocates no device
 *     memory for them.  An encode failure returns PA_ERR_CUDA.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of activations and pools (PA_E4M3: pools only, for
 * pa_decode_default_splits and pa_copy_blocks). */
enum { PA_F16 = 0, PA_BF16 = 1, PA_E4M3 = 2 };

/* Return codes. */
enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, Hq % Hkv != 0 */
    PA_ERR_UNSUPPORTED = 2,  /* head_dim, block_size or group size not supported */
    PA_ERR_WORKSPACE = 3,    /* workspace missing, too small or misaligned */
    PA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    PA_ERR_BOUNDS = 5,       /* pa_get_status: a kernel skipped an out-of-range index */
    PA_ERR_TIMEOUT = 6,      /* pa_get_status: a kernel's bounded wait gave up */
    PA_ERR_SCRATCH_LIMIT = 7 /* pa_decode_noalloc: sizes need more than its static scratch */
};

/* Bits of the device status word (pa_get_status). */
#define PA_STATUS_BAD_BLOCK 1u   /* block table entry outside [0, num_blocks) */
#define PA_STATUS_BAD_LEN 2u     /* context_len < 0, > max_context_len or > max_blocks_per_seq*block_size */
#define PA_STATUS_BAD_SLOT 4u    /* slot >= num_blocks * block_size */
#define PA_STATUS_TIMEOUT 8u     /* a wait (for a copy, or for partial results) reached its time limit */
#define PA_STATUS_NO_WORKSPACE 16u /* a split partition had no workspace (never written) */
#define PA_STATUS_WS_DIRTY 32u   /* a decode read a partial result no decode writes: its workspace
                                    was not zero-filled (or a call that timed out left it so) and
                                    results may be wrong; detected on a best-effort basis */

/* Decode flags (the flags argument of the decode entry points). */
#define PA_DECODE_EARLY_PROLOGUE 1u   /* the prologue may overlap the previous kernel: see pa_decode */
#define PA_DECODE_EARLY_COPIES 2u     /* with EARLY_PROLOGUE: first K/V copies before the wait, see pa_decode */

/*
 * Append: for each token i with s = slot_mapping[i] >= 0 and each kv head h,
 * copy k_new[i][h][:] to k_cache[s / block_size][h][s % block_size][:] and
 * the same for V.  A byte copy: results are bit-exact and no other byte of
 * the pools changes.  Two tokens with the same slot race.
 * dtype: PA_F16 or PA_BF16 (only the element size matters).
 * Source: rvLLM, CUDA Kernels table, "Reshape and Cache"; rvllm (small
 * engine), How it's put together, write_positions.
 */
int pa_cache_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                    const int64_t *slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                    int block_size, int num_blocks, int dtype, void *stream);

/*
 * FP8 append: like pa_cache_append, but each row (dtype PA_F16 or PA_BF16)
 * is written as E4M3 codes, with one fp32 scale per (page, kv head) in
 * k_scale / v_scale [num_blocks][num_kv_heads], for K and V separately:
 *   - a page that receives its first token (slot % block_size == 0) gets
 *     scale = amax(|row|) / 448 (1.0 when amax is 0);
 *   - a later token is encoded with the stored scale s when
 *     fl32(amax(|row|) / s) <= 448, so that no element saturates;
 *   - otherwise the page is re-scaled first: s' = amax(|row|) / 448 is
 *     stored and every code c of the page's rows before the new one becomes
 *     E4M3(fl32(fl32(e4m3(c) * s) / s')).
 * Codes are E4M3(x / scale) with the quotient rounded in fp32 and the code
 * rounded to nearest even.  Within one call, tokens of the same page race:
 * give them in separate calls (one token per sequence per decode step).
 * Source: rvLLM, CUDA Kernels table, "FP8 KV Cache"; LLM Serving Kernels,
 * Projects table, row 05 (E4M3 storage, page scales).
 */
int pa_cache_append_fp8(const void *k_new, const void *v_new, uint8_t *k_cache, uint8_t *v_cache,
                        float *k_scale, float *v_scale, const int64_t *slot_mapping,
                        int num_tokens, int num_kv_heads, int head_dim, int block_size,
                        int num_blocks, int dtype, void *stream);

/*
 * Bulk page quantisation of two fp16 pools (K and V) into E4M3 pools: for
 * every (block, kv head) tile, amax = max |x| over its block_size x head_dim
 * values, scale = amax / 448 in fp32 (1.0 when amax is 0), code =
 * E4M3_RNE_saturating(x / scale) with the quotient rounded in fp32.
 * k_src may equal NULL to quantise V only, and v_src NULL for K only.
 * Source: rvLLM, CUDA Kernels table, "FP8 KV Cache"; LLM Serving Kernels,
 * Projects table, row 05 ("page scales").
 */
int pa_quantize_fp8(const void *k_src, const void *v_src, uint8_t *k_cache, uint8_t *v_cache,
                    float *k_scale, float *v_scale, int num_blocks, int num_kv_heads,
                    int head_dim, int block_size, void *stream);

/*
 * Block copy inside the pools: for each pair i, with src = block_mapping[2i]
 * and dst = block_mapping[2i+1], copy physical block src of k_cache to
 * physical block dst (all num_kv_heads x block_size rows of head_dim
 * elements), the same for v_cache and, for PA_E4M3 pools, the block's
 * num_kv_heads K and V scales.  A byte copy: bit-exact, and no other byte
 * changes.  The copy that forks a block for its new owner (beam search,
 * parallel sampling, copy-on-write of a shared prefix).
 *   pool_type: PA_F16 / PA_BF16 (2-byte elements; scales must be NULL) or
 *   PA_E4M3 (1-byte codes; k_scale and v_scale [num_blocks][num_kv_heads]
 *   required).  block_mapping: int64 [num_pairs][2] on the device.
 * A pair with src == dst is a no-op; a pair with src or dst outside
 * [0, num_blocks) is skipped and sets PA_STATUS_BAD_BLOCK.  Destinations
 * must be distinct and must not be the source of another pair in the same
 * call (those copies race).
 * Source: rvLLM, CUDA Kernels table, "Block Copy"; Architecture,
 * rvllm-block-manager (copy-on-write, prefix sharing).
 */
int pa_copy_blocks(void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                   const int64_t *block_mapping, int num_pairs, int num_kv_heads, int head_dim,
                   int block_size, int num_blocks, int pool_type, void *stream);

/*
 * The E4M3 encoder on its own: codes[i] = E4M3_RNE_saturating(x[i]) for n
 * fp32 values (NaN gives a NaN code).  Exposed so the codec can be checked
 * exhaustively; the quantisers use the same instruction.
 */
int pa_e4m3_encode(const float *x, uint8_t *codes, int64_t n, void *stream);

/*
 * Number of CTAs a decode divides a batch among when split_ctas is 0, on the
 * current device, for pools of type pool_type (PA_F16 or PA_BF16: two per
 * SM; PA_E4M3: three per SM; each the count that is resident at once).
 * Returns 0 for another pool_type.
 */
int pa_decode_default_splits(int pool_type);

/*
 * Bytes of device workspace pa_decode / pa_decode_fp8 need: room for the
 * partial results of the context partitions that cross worker boundaries
 * (a worker is one warp; four per CTA; at most two partials each), which
 * the merge launch reads.  split_ctas 0 means the largest
 * pa_decode_default_splits() over pool types on the current device, so the
 * result serves a default call of any type.  Every call needs one.
 *
 * The caller allocates the workspace and zero-fills it once before its
 * first use (cudaMemsetAsync).  The merge launch tells a written partial
 * from an empty one by its bits and zeroes each partial it has read, so
 * every call leaves the workspace zero-filled and the same workspace then
 * serves call after call, whatever their sizes, without clearing.  After a
 * call whose status shows PA_STATUS_TIMEOUT or PA_STATUS_WS_DIRTY, zero-fill
 * it again.  Calls that share a workspace must not overlap on the device.
 *
 * The size serves calls with up to 8 query rows per (sequence, kv head):
 * queries_per_seq * (num_q_heads / num_kv_heads) <= 8.  Calls with more
 * rows (query groups above 8, or several query tokens) hold 16 or 32 rows
 * per partial and need pa_decode_workspace_size_rows.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int head_dim, int split_ctas);

/*
 * Bytes of decode workspace for calls with up to query_rows =
 * queries_per_seq * (num_q_heads / num_kv_heads) query rows per (sequence,
 * kv head): a launch holds 8, 16 or 32 rows per partial (the widest of its
 * passes: at most 32 rows).  pa_decode_workspace_size(...) equals this with
 * query_rows 8.  Otherwise as pa_decode_workspace_size.
 */
size_t pa_decode_workspace_size_rows(int num_seqs, int num_q_heads, int head_dim, int split_ctas,
                                     int query_rows);

/*
 * Paged GQA decode over a 16-bit pool.  For every sequence b and q head hq,
 *   out[b][hq][:] = sum_t softmax_t(scale * q[b][hq] . K_t) * V_t
 * over the context_lens[b] tokens of b, token t read from physical block
 * block_tables[b][t / block_size], row t % block_size, kv head
 * hq / (num_q_heads / num_kv_heads).  out is rounded to dtype (round to
 * nearest even); a sequence with context_len 0 gets a zero output.
 *
 * The batch's (sequence, kv head, block) units are divided evenly among the
 * 4 * split_ctas warps of split_ctas CTAs (0: pa_decode_default_splits(dtype)).
 * A warp's share of one sequence is a context partition, reduced with an
 * online softmax in fp32.  A sequence split across warps has its partitions
 * merged by log-sum-exp in a second launch on the same stream, a
 * programmatic dependent launch that runs beside the first: it merges a
 * sequence as soon as all its partitions are written, and completes after
 * the first launch has.
 * Results do not depend on split_ctas beyond fp32 rounding, and a given
 * split_ctas is deterministic.
 *   max_context_len: host-side upper bound of context_lens (no device read);
 *   window_size: 0 attends the whole context; W > 0 attends only the last W
 *   positions (L-W .. L-1; the blocks wholly before them are not read);
 *   queries_per_seq: n_q >= 1 query tokens per sequence (speculative or
 *   chunked decoding): q and out are [num_seqs][n_q][num_q_heads][head_dim],
 *   query i sits at position L - n_q + i (its own token and those before it
 *   are in the cache) and attends causally, positions up to its own (within
 *   its window); a query before position 0 gets a zero output.  With
 *   n_q * (num_q_heads / num_kv_heads) <= 32 query rows per (sequence, kv
 *   head) the K/V is read once for all of them; larger n_q (at most 1024)
 *   run as consecutive passes of 32 / group tokens, each reading the K/V
 *   again (pa_decode_noalloc rejects more than 8 rows with
 *   PA_ERR_UNSUPPORTED).  Launches with more than 8 rows hold two CTAs per
 *   SM whatever the pool type (split_ctas 0 then means two per SM).  Over
 *   16-bit pools at head_dim 128, a launch with 17 to 32 rows runs its
 *   products on the fifth-generation tensor cores instead (tcgen05, one CTA
 *   of ten warps per SM): the batch is then divided among min(SMs,
 *   4 * split_ctas) CTAs, with the same workspace and merge;
 *   workspace: at least pa_decode_workspace_size_rows(..., query_rows) bytes
 *   (pa_decode_workspace_size(...) when query_rows <= 8), 256-byte aligned;
 *   flags: 0, or PA_DECODE_EARLY_PROLOGUE: the attention launch becomes a
 *   programmatic dependent launch.  Its prologue (reading context_lens and
 *   block_tables, dividing the batch among the warps, reading each warp's
 *   first block ids) may then run while the kernel before it on the stream
 *   is still finishing; everything else (q, the pools and scales, the new
 *   rows, out, the workspace) waits until that kernel has completed, except
 *   that the prologue asks L2 to prefetch each warp's first K/V tiles (a
 *   hint that reads nothing into the SMs; L2 is coherent, so writes that
 *   kernel makes to the pools are still seen).  Set it
 *   only when the kernel just before the call on the stream does not write
 *   context_lens or block_tables (for example, when they are uploaded by a
 *   copy before the forward pass).  Results are the same either way.
 *   PA_DECODE_EARLY_COPIES (only together with PA_DECODE_EARLY_PROLOGUE;
 *   alone: PA_ERR_INVALID_ARG) lets the prologue go further on the mma.sync
 *   launch (up to 16 query rows per kv head): before waiting, each warp
 *   copies into shared memory its first K/V tiles that lie wholly before its
 *   sequence's last two blocks.  Set it only when, besides the above, the
 *   kernels before the call on the stream write nothing in the pools this
 *   call reads except in each sequence's last two blocks -- as the previous
 *   decode step of the same batch does (its append, E4M3 re-scales
 *   included), or an append of up to 17 draft tokens -- and write no page
 *   scale of another block.  Results are the same either way.
 * Source: rvLLM, CUDA Kernels table, "PagedAttention V2" (block-table
 * indirection, online softmax); LLM Serving Kernels, Projects table, row 04;
 * rvllm (small engine), How it's put together (GQA, read_blocks).
 */
int pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
              int max_context_len, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
              int block_size, int num_blocks, float scale, int window_size, int queries_per_seq,
              int dtype, int split_ctas,
              void *workspace, size_t workspace_bytes, unsigned flags, void *stream);

/*
 * Paged GQA decode over an E4M3 pool: as pa_decode (q and out of dtype
 * PA_F16 or PA_BF16), K_t = e4m3(k_code) * k_scale[block][kv head] and V_t
 * likewise, dequantised in registers inside the attention loop.  A bf16 q
 * enters the fp16 tensor-core products scaled by a power of two per
 * (sequence, kv head), so that its largest element lies in [2^14, 2^15);
 * the scale is taken out of the scores.
 * Source: rvLLM, CUDA Kernels table, "FP8 KV Cache" and "PagedAttention V2";
 * LLM Serving Kernels, Projects table, row 05 ("fused dequantization").
 */
int pa_decode_fp8(void *out, const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                  const float *k_scale, const float *v_scale, const int32_t *block_tables,
                  int max_blocks_per_seq, const int32_t *context_lens, int max_context_len,
                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                  int num_blocks, float scale, int window_size, int queries_per_seq,
                  int dtype, int split_ctas, void *workspace,
                  size_t workspace_bytes, unsigned flags, void *stream);

/*
 * One whole decode step in one attention launch (plus pa_decode's merge
 * launch): append this step's K/V token of every sequence, then attend over
 * the sequence's context including it, as
 * pa_cache_append followed by pa_decode would, with the same results (the
 * pools bit-identical, out within fp32 rounding).
 *   k_new, v_new: [num_seqs][num_kv_heads][head_dim], the dtype of q;
 *   slot_mapping: [num_seqs], the slot of position context_lens[b] - 1 of
 *   sequence b (a decode step's slot), or negative for a padding sequence
 *   that appends nothing.  Any other slot is not written and sets
 *   PA_STATUS_BAD_SLOT.  A sequence with context_len 0 appends nothing.
 * The warp that attends a sequence's last block writes the new row to the
 * pool and into its copy of that block, so no launch-wide ordering is
 * needed.  Other arguments as pa_decode.
 * Source: rvLLM, CUDA Kernels table, "Reshape and Cache" and "PagedAttention
 * V2"; rvLLM, Completed Optimizations (fused kernels, fewer launches); rvllm
 * (small engine), How it's put together (write_positions then read_blocks in
 * one forward).
 */
int pa_decode_step(void *out, const void *q, const void *k_new, const void *v_new,
                   void *k_cache, void *v_cache, const int64_t *slot_mapping,
                   const int32_t *block_tables, int max_blocks_per_seq,
                   const int32_t *context_lens, int max_context_len, int num_seqs,
                   int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                   int num_blocks, float scale, int window_size, int dtype, int split_ctas,
                   void *workspace, size_t workspace_bytes, unsigned flags, void *stream);

/*
 * pa_decode_step over E4M3 pools: q, k_new, v_new and out of dtype PA_F16 or
 * PA_BF16; the new row is encoded as pa_cache_append_fp8 does (a page's first
 * row sets its K and V scales, a later row that would saturate re-scales the
 * page) and attended as pa_decode_fp8 does.
 * Source: as pa_decode_step, and rvLLM, CUDA Kernels table, "FP8 KV Cache".
 */
int pa_decode_step_fp8(void *out, const void *q, const void *k_new, const void *v_new,
                       uint8_t *k_cache, uint8_t *v_cache, float *k_scale, float *v_scale,
                       const int64_t *slot_mapping, const int32_t *block_tables,
                       int max_blocks_per_seq, const int32_t *context_lens, int max_context_len,
                       int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int num_blocks, float scale, int window_size, int dtype,
                       int split_ctas, void *workspace, size_t workspace_bytes, unsigned flags,
                       void *stream);

/*
 * Device-side ordering of a decode step against copies made on other
 * streams, for serving loops that upload each step's inputs (q, new rows,
 * slots, block tables, context lengths) and read its output back while the
 * previous step still runs.  Ordering those copies with stream events puts
 * waits and records between the kernels of consecutive steps on the compute
 * stream, which keeps the next step's launch from overlapping the end of
 * the previous one (PA_DECODE_EARLY_PROLOGUE); with this handshake the
 * compute stream holds nothing but the steps' kernels:
 *   - the copy stream uploads the step's inputs, then writes ready_value to
 *     *ready with pa_stream_write_value (ordered after the upload);
 *   - the step's attention launch waits, bounded by 2 s, until
 *     (int32_t)(*ready - ready_value) >= 0 before it reads any input; a CTA
 *     that gives up sets PA_STATUS_TIMEOUT and returns;
 *   - once its output is complete, the step stores done_value to *done
 *     (the merge launch's CTAs count themselves on *done_count, which must
 *     be zero before the first step that uses it and is zero again after
 *     each); a step that hit a timeout still stores it, so a stream waiting
 *     on *done never waits forever (its pa_get_status shows the failure);
 *   - the read-back stream waits with pa_stream_wait_value(..., done,
 *     done_value) and copies the output; an upload that reuses the step's
 *     input buffers waits on *done likewise.
 * ready, done and done_count are device words, 4-byte aligned, owned by the
 * caller; give each in-flight step its own (a ring of slots), with values
 * that grow from step to step.
 * No counterpart in the pages: host-device plumbing of a serving loop.
 */
typedef struct pa_step_sync {
    const uint32_t *ready;
    uint32_t *done;
    uint32_t *done_count;
    uint32_t ready_value;
    uint32_t done_value;
} pa_step_sync;

/* pa_decode_step / pa_decode_step_fp8 with the handshake above (sync must
 * not be NULL).  Results are those of the plain calls. */
int pa_decode_step_synced(void *out, const void *q, const void *k_new, const void *v_new,
                          void *k_cache, void *v_cache, const int64_t *slot_mapping,
                          const int32_t *block_tables, int max_blocks_per_seq,
                          const int32_t *context_lens, int max_context_len, int num_seqs,
                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          int num_blocks, float scale, int window_size, int dtype,
                          int split_ctas, void *workspace, size_t workspace_bytes,
                          unsigned flags, const pa_step_sync *sync, void *stream);
int pa_decode_step_fp8_synced(void *out, const void *q, const void *k_new, const void *v_new,
                              uint8_t *k_cache, uint8_t *v_cache, float *k_scale,
                              float *v_scale, const int64_t *slot_mapping,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, int max_context_len, int num_seqs,
                              int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                              int num_blocks, float scale, int window_size, int dtype,
                              int split_ctas, void *workspace, size_t workspace_bytes,
                              unsigned flags, const pa_step_sync *sync, void *stream);

/*
 * One whole pipelined step of a serving loop in one call: the step's packed
 * inputs uploaded from pinned host memory on copy_stream, the handshake's
 * ready word written after them, the step (as pa_decode_step_synced /
 * pa_decode_step_fp8_synced) launched on `stream`, and on back_stream a wait
 * for the step's done word, the output copied to pinned host memory and
 * `reuse_event` recorded.  When slot_reused is set, the upload first waits
 * for `reuse_event` (the previous read-back of this slot, recorded by the
 * call that used the slot before), so that neither the slot's inputs nor its
 * output are overwritten while still in use.  The decode arguments (q,
 * k_new, v_new, slot_mapping, block_tables, context_lens) point into the
 * device buffer the upload fills.  Streams are cudaStream_t and the event a
 * cudaEvent_t, passed as void*; all are the caller's.  If the step cannot
 * be launched the call returns its error after the upload and before any
 * wait on the done word (so nothing waits for a step that never ran).
 * No counterpart in the pages: host-device plumbing of a serving loop, one
 * library call per step instead of a dozen runtime calls.
 */
typedef struct pa_step_copies {
    const void *host_in;     /* pinned host: the step's inputs, in_bytes */
    void *dev_in;            /* device: where they are uploaded */
    size_t in_bytes;
    const void *dev_out;     /* device: the step's output, out_bytes */
    void *host_out;          /* pinned host: where it is read back */
    size_t out_bytes;
    void *copy_stream;
    void *back_stream;
    void *reuse_event;
    int slot_reused;
} pa_step_copies;

int pa_decode_step_pipelined(void *out, const void *q, const void *k_new, const void *v_new,
                             void *k_cache, void *v_cache, const int64_t *slot_mapping,
                             const int32_t *block_tables, int max_blocks_per_seq,
                             const int32_t *context_lens, int max_context_len, int num_seqs,
                             int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                             int num_blocks, float scale, int window_size, int dtype,
                             int split_ctas, void *workspace, size_t workspace_bytes,
                             unsigned flags, const pa_step_sync *sync,
                             const pa_step_copies *io, void *stream);
int pa_decode_step_fp8_pipelined(void *out, const void *q, const void *k_new, const void *v_new,
                                 uint8_t *k_cache, uint8_t *v_cache, float *k_scale,
                                 float *v_scale, const int64_t *slot_mapping,
                                 const int32_t *block_tables, int max_blocks_per_seq,
                                 const int32_t *context_lens, int max_context_len,
                                 int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int num_blocks, float scale, int window_size,
                                 int dtype, int split_ctas, void *workspace,
                                 size_t workspace_bytes, unsigned flags,
                                 const pa_step_sync *sync, const pa_step_copies *io,
                                 void *stream);

/*
 * Stream-ordered 32-bit device-word operations (the driver's stream memory
 * operations): pa_stream_write_value stores value to *addr once the work
 * before it on stream has completed (its writes visible first);
 * pa_stream_wait_value holds the work after it on stream until
 * (int32_t)(*addr - value) >= 0.  addr is a 4-byte aligned device pointer.
 * PA_ERR_UNSUPPORTED when the driver or device does not offer them.  Such a
 * wait has no time limit of its own: wait only on words a step of this
 * library (or the caller) is certain to write.
 */
int pa_stream_write_value(void *stream, uint32_t *addr, uint32_t value);
int pa_stream_wait_value(void *stream, const uint32_t *addr, uint32_t value);

/*
 * pa_decode without a caller-provided workspace, for callers that cannot
 * allocate device memory: code inside a host framework that owns all device
 * memory and forbids raw allocations, latency-critical loops where
 * cudaMalloc would synchronise the device, plain C callers without a device
 * allocator.  The paper has no counterpart; it exists for those callers.
 *
 * Arguments and results are those of pa_decode (16-bit pools); the scratch
 * lives in a static array of PA_NOALLOC_SCRATCH_BYTES inside the library,
 * held by every GPU that loads it until the process exits.  Sizes whose
 * scratch would exceed it return PA_ERR_SCRATCH_LIMIT (the default split at
 * head_dim 128 needs about 10 MB on a 152-SM GPU).  The call allocates
 * nothing and frees nothing.  The first call on a device looks up the
 * array's device address (make it before any stream capture).  All calls on
 * a device share the array: calls that overlap on the GPU race.  The array
 * starts zero-filled and every call leaves it so; after a pa_get_status
 * that shows PA_STATUS_TIMEOUT or PA_STATUS_WS_DIRTY, the next call on that
 * device zeroes it first (a stream-ordered memset).  That clearing is made
 * by the host call, so a CUDA graph that captured pa_decode_noalloc before
 * such a status never makes it: its replays would merge partials the
 * failed call left behind.  Re-capture such graphs after a direct call
 * (the direct call clears the scratch).
 */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)
int pa_decode_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, int max_context_len, int num_seqs,
                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      int num_blocks, float scale, int window_size, int queries_per_seq,
                      int dtype, int split_ctas, unsigned flags, void *stream);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word.  Returns PA_OK when it was clear, PA_ERR_TIMEOUT when a wait gave
 * up, PA_ERR_WORKSPACE when a decode found its workspace dirty,
 * PA_ERR_BOUNDS for index errors, PA_ERR_CUDA when CUDA failed; the raw
 * bits go to *bits when bits is not NULL.
 */
int pa_get_status(void *stream, unsigned *bits);

/*
 * Failure-path tests of the kernels' bounded waits.  Every wait a kernel of
 * this library makes (an mbarrier wait for an asynchronous copy, the merge
 * launch's poll for partial results another grid writes) gives up after a
 * time limit (2 s in the entry points above), sets PA_STATUS_TIMEOUT and
 * lets the kernel return, so a lost copy or a missing partial never hangs the
 * GPU.  These two calls make such a wait run out on purpose, with a short
 * limit, so that a test can check the status and that the context stays
 * usable.  Neither faults, traps or spins without bound.
 *
 * pa_test_wait_timeout: one warp waits, with the attention loop's bounded
 * wait, on an mbarrier that nothing completes; after limit_ns (1 .. 2e9) it
 * sets PA_STATUS_TIMEOUT.
 *
 * pa_test_merge_timeout: the merge launch of a pa_decode with these sizes,
 * run alone, so no attention launch ever writes the partials it polls for;
 * with a zero-filled workspace every CTA of a split sequence gives up after
 * limit_ns and sets PA_STATUS_TIMEOUT, writing neither out nor the
 * workspace.  context_lens is a device array as for pa_decode; at most 512
 * sequences; n_q = 1, no window.
 * Neither has a counterpart in the pages: they exist to test the library.
 */
int pa_test_wait_timeout(uint64_t limit_ns, void *stream);
int pa_test_merge_timeout(void *out, const int32_t *context_lens, int max_context_len,
                          int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                          int dtype, int split_ctas, void *workspace, size_t workspace_bytes,
                          uint64_t limit_ns, void *stream);

/* A static string naming a return code. */
const char *pa_status_string(int code);

/* ABI version: major * 100 + minor. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
