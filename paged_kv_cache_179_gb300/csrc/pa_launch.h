// pa_launch.h -- kernel launchers shared between the translation units of
// libpa.  The C ABI (abi.cu) validates arguments and then calls these.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {

// Sequences per decode launch: each CTA keeps per-sequence prefix sums of
// the batch in shared memory; the host splits larger batches.
constexpr int kMaxBatchPerLaunch = 512;

// Devices the library keeps per-device state for (ordinals 0 .. 63).
constexpr int kMaxDevices = 64;

// Default time limit of every wait a kernel makes: an mbarrier wait for an
// asynchronous copy, or the merge launch's poll for another grid's partial
// results.  A wait that ends normally takes microseconds; one that reaches
// the limit gives up, and the kernel sets kStatusTimeout and returns instead
// of hanging.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// All pointers are device pointers; sizes were validated by the caller.
struct DecodeArgs {
  // 16-bit pools: tensor maps of k_cache and v_cache that copy one
  // (block, kv head) tile with the 128-byte swizzle (set by the launcher)
  CUtensorMap tm_k, tm_v;
  void* out;                    // [B][Hq][D] f16/bf16
  const void* q;                // [B][Hq][D] f16/bf16
  const void* k_cache;          // [NB][Hkv][16][D] f16/bf16 or e4m3
  const void* v_cache;
  const float* k_scale;         // [NB][Hkv] (E4M3 pools only)
  const float* v_scale;
  const int32_t* block_tables;  // [B][mbs]
  const int32_t* context_lens;  // [B]
  float* ws_acc;                // [split_ctas*4][2][rows][D] partial sums (unnormalised), and
  float* ws_ml;                 // [split_ctas*4][2][rows][2] partial (max, sum) in log2 units;
                                // both bit-inverted, zero when not written
  unsigned* status;             // device status word
  // fused append (pa_decode_step*): this step's new rows and where they go;
  // null for a plain decode
  const void* k_new;            // [B][Hkv][D] f16/bf16 (fp16 for E4M3 pools)
  const void* v_new;
  const int64_t* slots;         // [B], slot of position context_lens[b] - 1
  void* k_pool_w;               // the pools and scales the new rows are written to
  void* v_pool_w;
  float* k_scale_w;
  float* v_scale_w;
  int mbs;                      // max blocks per sequence (block table row stride)
  int B, Hq, Hkv, group, D;
  int num_blocks;
  int max_context_len;
  int split_ctas;               // CTAs the batch's blocks are divided among
  int workers;                  // workers they are divided among (0: split_ctas x 4 warps)
  int seg_cost;                 // units each non-empty segment adds before its blocks in the
                                // stream the workers share (0: the stream is blocks alone)
  int window;                   // sliding window in tokens (0: the whole context)
  int n_q;                      // query tokens this launch serves (n_q * group <= rows)
  int rows;                     // query rows per (sequence, kv head) a launch holds: 8, 16 or 32
  int merge_groups;             // piece groups per merge CTA (set by the merge launch)
  int q_tokens;                 // query tokens per sequence in q and out
  int q_first;                  // the first of them this launch serves
  int early;                    // programmatic dependent launch: prologue before griddepcontrol.wait
  int early_copies;             // with early: first K/V copies (not of the last two blocks) before it
  float scale_log2;             // softmax scale * log2(e)
  uint64_t wait_limit_ns;       // time limit of every wait (kWaitLimitNs unless a test shortens it)
  // device-side ordering against copies on other streams (null: none).  The
  // attention launch waits (bounded) until *ready reaches ready_value before
  // it reads anything; the merge launch's CTAs count themselves on
  // *done_count and the last one, once the attention grid has completed,
  // resets the count and stores done_value to *done.
  const uint32_t* ready;
  uint32_t* done;
  uint32_t* done_count;
  uint32_t ready_value;
  uint32_t done_value;
};

// Largest query rows per (sequence, kv head) one launch serves: four tiles of
// the MMA's 8 columns.
constexpr int kMaxRowsPerLaunch = 32;
// CTAs a default launch uses for this pool type and query rows per
// (sequence, kv head)
int decode_default_ctas(bool fp8, int rows = 1);
int decode_max_default_ctas();       // the largest of those over pool types
// Rows per piece a launch serving `query_rows` rows holds: 8, 16 or 32.
int decode_rows(int query_rows);
// Workspace bytes for launches of up to `rows` query rows per (sequence, kv head).
size_t decode_workspace_bytes(int B, int Hq, int D, int split_ctas, int rows);
// Points a's workspace fields into ws, for a's sizes (a.split_ctas, a.D, a.rows).
void decode_workspace_split(DecodeArgs& a, void* ws);

cudaError_t launch_decode(const DecodeArgs& a, bool fp8, bool bf16, cudaStream_t s);
// The launches with two and four tiles of query columns per warp (a.rows 16
// and 32), each in a translation unit of its own.
cudaError_t launch_decode_tiles2(const DecodeArgs& a, bool fp8, bool bf16, cudaStream_t s);
cudaError_t launch_decode_tiles4_16bit(const DecodeArgs& a, bool bf16, cudaStream_t s);
cudaError_t launch_decode_tiles4_e4m3(const DecodeArgs& a, bool bf16, cudaStream_t s);
// The launch on the fifth-generation tensor cores (decode_tc.cu) for 17 to
// 32 query rows per (sequence, kv head) over 16-bit pools at head_dim 128;
// launch_decode takes it whenever decode_tc_eligible holds.
bool decode_tc_eligible(const DecodeArgs& a, bool fp8);
cudaError_t launch_decode_tc(const DecodeArgs& a, bool bf16, cudaStream_t s);
// The merge launch alone (no attention launch writes its partials): the
// failure-path test of its bounded poll.
cudaError_t launch_merge_only(const DecodeArgs& a, bool bf16, cudaStream_t s);
// Stores value to *done (release, gpu scope): the handshake's done signal
// of a step that launches nothing else.
cudaError_t launch_signal_done(uint32_t* done, uint32_t value, cudaStream_t s);
// One warp waiting on an mbarrier that nothing completes, with the decode's
// bounded wait: the failure-path test of that wait.
cudaError_t launch_wait_probe(unsigned* status, uint64_t limit_ns, cudaStream_t s);

cudaError_t launch_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                          const int64_t* slots, int T, int Hkv, int row_bytes, int block_size,
                          int64_t num_blocks, unsigned* status, cudaStream_t s);

cudaError_t launch_append_fp8(const void* k_new, const void* v_new, uint8_t* k_cache,
                              uint8_t* v_cache, float* k_scale, float* v_scale,
                              const int64_t* slots, int T, int Hkv, int D, int block_size,
                              int64_t num_blocks, bool bf16, unsigned* status, cudaStream_t s);

cudaError_t launch_quantize_fp8(const void* src, uint8_t* codes, float* scales,
                                int64_t num_tiles, int tile_elems, cudaStream_t s);

cudaError_t launch_e4m3_encode(const float* x, uint8_t* codes, int64_t n, cudaStream_t s);
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                               const int64_t* pairs, int num_pairs, int Hkv, int row_bytes,
                               int block_size, int64_t num_blocks, unsigned* status,
                               cudaStream_t s);

int device_sm_count();
// Address of the current device's status word (set up on first use).
int device_status_word(unsigned** out);
// Called when a status read shows a wait that gave up or a dirty workspace
// on the current device: the no-alloc scratch's flags are cleared before
// its next use.
void noalloc_scratch_suspect();

}  // namespace pa
