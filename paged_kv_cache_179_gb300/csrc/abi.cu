// abi.cu -- the extern "C" entry points declared in include/pa.h.
//
// Each entry point checks its arguments on the host (returning an error code
// before anything is launched), then launches the kernels of append.cu,
// quantize.cu and decode.cu on the caller's stream.  The only state the
// library keeps is one device status word per device (index errors and wait
// timeouts seen by kernels) and a per-device cache of its address and SM
// count.
#include <climits>
#include <cmath>
#include <mutex>

#include <cudaTypedefs.h>

#include "pa.h"
#include "pa_launch.h"

__device__ unsigned int g_pa_status_word;

namespace pa {
namespace {

struct DeviceState {
  bool ready = false;
  unsigned* status = nullptr;
  int sm_count = 0;
};
std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

// Status word address and SM count of the current device (set up once).
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& d = g_devices[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_status_word) != cudaSuccess) return PA_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PA_ERR_CUDA;
    d.status = static_cast<unsigned*>(p);
    d.sm_count = sms;
    d.ready = true;
  }
  *out = &d;
  return PA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

struct DecodeShape {
  int B, Hq, Hkv, D, bs, NB, mbs, max_ctx, splits, window;
  int nq = 1;   // query tokens per sequence
  unsigned flags = 0;   // PA_DECODE_* flags
};

int check_decode_shape(const DecodeShape& s, float scale) {
  if (s.B < 0 || s.Hq <= 0 || s.Hkv <= 0 || s.Hq % s.Hkv != 0) return PA_ERR_INVALID_ARG;
  if (s.NB <= 0 || s.mbs <= 0 || s.max_ctx < 0) return PA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(s.max_ctx) > static_cast<int64_t>(s.mbs) * s.bs) return PA_ERR_INVALID_ARG;
  if (s.splits < 0 || s.window < 0) return PA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (s.D != 64 && s.D != 128) return PA_ERR_UNSUPPORTED;
  if (s.bs != 16) return PA_ERR_UNSUPPORTED;
  if (s.nq < 1 || s.nq > 1024) return PA_ERR_INVALID_ARG;
  if (s.Hq / s.Hkv > kMaxRowsPerLaunch) return PA_ERR_UNSUPPORTED;
  if (s.flags & ~(PA_DECODE_EARLY_PROLOGUE | PA_DECODE_EARLY_COPIES)) return PA_ERR_INVALID_ARG;
  if ((s.flags & PA_DECODE_EARLY_COPIES) && !(s.flags & PA_DECODE_EARLY_PROLOGUE))
    return PA_ERR_INVALID_ARG;
  if (s.B > 65535 || s.Hkv > 65535) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

// The fused step's extra inputs (all null for a plain decode).
struct AppendArgs {
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  const int64_t* slots = nullptr;
  void* k_pool = nullptr;
  void* v_pool = nullptr;
  float* k_scale = nullptr;
  float* v_scale = nullptr;
};

// Query tokens one launch pair serves: all n_q when their n_q * G rows fit
// kMaxRowsPerLaunch (the K/V is then read once for all of them), else as many
// as fit, in consecutive passes.
int tokens_per_pass(int nq, int group) {
  return nq * group <= kMaxRowsPerLaunch ? nq : kMaxRowsPerLaunch / group;
}

int run_decode(DecodeShape s, void* out, const void* q, const void* k, const void* v,
               const float* ks, const float* vs, const int32_t* bt, const int32_t* cl,
               float scale, bool fp8, bool bf16, void* ws, size_t ws_bytes, void* stream,
               const AppendArgs& ap = AppendArgs(), const pa_step_sync* sync = nullptr) {
  if (s.B == 0) return PA_OK;
  const int group = s.Hq / s.Hkv;
  const int per_pass = tokens_per_pass(s.nq, group);
  const int rows = per_pass * group;   // query rows per (sequence, kv head) of the widest pass
  auto ws_ok = [&]() {   // every split needs one: its four warps divide the batch
    const size_t need = decode_workspace_bytes(s.B, s.Hq, s.D, s.splits, rows);
    return ws != nullptr && ws_bytes >= need && aligned(ws, 256);
  };
  if (s.splits > 0 && !ws_ok()) return PA_ERR_WORKSPACE;   // checked before touching CUDA
  DeviceState* dev = nullptr;
  if (int rc = device_state(&dev)) return rc;
  if (s.splits == 0) {
    s.splits = decode_default_ctas(fp8, rows);
    if (!ws_ok()) return PA_ERR_WORKSPACE;
  }
  DecodeArgs a{};
  a.k_cache = k;
  a.v_cache = v;
  a.k_scale = ks;
  a.v_scale = vs;
  a.status = dev->status;
  a.mbs = s.mbs;
  a.Hq = s.Hq;
  a.Hkv = s.Hkv;
  a.group = group;
  a.D = s.D;
  a.num_blocks = s.NB;
  a.max_context_len = s.max_ctx;
  a.split_ctas = s.splits;
  a.window = s.window;
  a.n_q = s.nq;
  a.q_tokens = s.nq;
  a.q_first = 0;
  a.early = (s.flags & PA_DECODE_EARLY_PROLOGUE) ? 1 : 0;
  a.early_copies = (s.flags & PA_DECODE_EARLY_COPIES) ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit_ns = kWaitLimitNs;
  a.k_pool_w = ap.k_pool;
  a.v_pool_w = ap.v_pool;
  a.k_scale_w = ap.k_scale;
  a.v_scale_w = ap.v_scale;
  // Batches above kMaxBatchPerLaunch run as consecutive launch pairs
  // (attention, merge) on the stream, each reusing the workspace.
  const size_t out_row = static_cast<size_t>(s.nq) * s.Hq * s.D * 2;   // q, out: 16-bit
  for (int b0 = 0; b0 < s.B; b0 += kMaxBatchPerLaunch) {
    DecodeArgs c = a;
    c.B = s.B - b0 < kMaxBatchPerLaunch ? s.B - b0 : kMaxBatchPerLaunch;
    c.out = static_cast<uint8_t*>(out) + b0 * out_row;
    c.q = static_cast<const uint8_t*>(q) + b0 * out_row;
    c.block_tables = bt + static_cast<int64_t>(b0) * s.mbs;
    c.context_lens = cl + b0;
    if (ap.k_new != nullptr) {
      const size_t new_row = static_cast<size_t>(s.Hkv) * s.D * 2;   // new rows are 16-bit
      c.k_new = static_cast<const uint8_t*>(ap.k_new) + b0 * new_row;
      c.v_new = static_cast<const uint8_t*>(ap.v_new) + b0 * new_row;
      c.slots = ap.slots + b0;
    }
    // One launch pair serves up to 32 query rows per (sequence, kv head)
    // (the warps hold 1, 2 or 4 tiles of the MMA's 8 columns): n_q tokens of
    // a group of G heads fit when n_q * G <= 32, and the K/V is read once for
    // all of them; more tokens run as consecutive passes of 32 / G tokens,
    // every pass reading the K/V again.
    for (int t0 = 0; t0 < s.nq; t0 += per_pass) {
      c.q_first = t0;
      c.n_q = s.nq - t0 < per_pass ? s.nq - t0 : per_pass;
      c.rows = decode_rows(c.n_q * group);
      decode_workspace_split(c, ws);
      // device-side handshake: the first attention launch waits for the
      // upload, the last merge launch signals the call done
      const bool first = b0 == 0 && t0 == 0;
      const bool last = b0 + kMaxBatchPerLaunch >= s.B && t0 + per_pass >= s.nq;
      c.ready = sync != nullptr && first ? sync->ready : nullptr;
      c.ready_value = sync != nullptr ? sync->ready_value : 0u;
      c.done = sync != nullptr && last ? sync->done : nullptr;
      c.done_count = sync != nullptr && last ? sync->done_count : nullptr;
      c.done_value = sync != nullptr ? sync->done_value : 0u;
      if (cudaError_t e = launch_decode(c, fp8, bf16, static_cast<cudaStream_t>(stream)))
        return cuda_status(e);
    }
  }
  return PA_OK;
}

bool sync_ok(const pa_step_sync* sync) {
  if (sync == nullptr) return true;
  return sync->ready != nullptr && sync->done != nullptr && sync->done_count != nullptr &&
         aligned(sync->ready, 4) && aligned(sync->done, 4) && aligned(sync->done_count, 4);
}

// cuStreamWriteValue32 / cuStreamWaitValue32, from the driver (no link against libcuda).
struct StreamMemOps {
  PFN_cuStreamWriteValue32_v11070 write = nullptr;
  PFN_cuStreamWaitValue32_v11070 wait = nullptr;
};
const StreamMemOps& stream_mem_ops() {
  static const StreamMemOps ops = [] {
    StreamMemOps o;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &f, 11070, cudaEnableDefault,
                                         &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
      o.write = reinterpret_cast<PFN_cuStreamWriteValue32_v11070>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &f, 11070, cudaEnableDefault,
                                         &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
      o.wait = reinterpret_cast<PFN_cuStreamWaitValue32_v11070>(f);
    return o;
  }();
  return ops;
}

int cu_status(CUresult r) {
  if (r == CUDA_SUCCESS) return PA_OK;
  return r == CUDA_ERROR_NOT_SUPPORTED ? PA_ERR_UNSUPPORTED : PA_ERR_CUDA;
}

}  // namespace

int device_sm_count() {
  DeviceState* d = nullptr;
  return device_state(&d) == PA_OK ? d->sm_count : 148;
}

int device_status_word(unsigned** out) {
  DeviceState* d = nullptr;
  if (int rc = device_state(&d)) return rc;
  *out = d->status;
  return PA_OK;
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_version(void) { return 101; }

const char* pa_status_string(int code) {
  switch (code) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape";
    case PA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_BOUNDS: return "a kernel skipped an out-of-range index";
    case PA_ERR_TIMEOUT: return "a kernel's bounded wait gave up";
    case PA_ERR_SCRATCH_LIMIT: return "request exceeds the library's static scratch array";
    default: return "unknown status";
  }
}

int pa_cache_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                    const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                    int block_size, int num_blocks, int dtype, void* stream) {
  if (num_tokens == 0) return PA_OK;   // nothing to move (empty tensors may have null data)
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
  if (head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;   // rows move as 16-byte chunks
  for (const void* p : {k_new, v_new, static_cast<const void*>(k_cache),
                        static_cast<const void*>(v_cache)})
    if (!aligned(p, 16)) return PA_ERR_INVALID_ARG;
  if (!aligned(slot_mapping, 8)) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (static_cast<int64_t>(num_tokens) * num_kv_heads * (head_dim / 8) > (INT64_C(1) << 40))
    return PA_ERR_UNSUPPORTED;
  DeviceState* dev = nullptr;
  if (int rc = device_state(&dev)) return rc;
  return cuda_status(launch_append(k_new, v_new, k_cache, v_cache, slot_mapping, num_tokens,
                                   num_kv_heads, head_dim * 2, block_size, num_blocks,
                                   dev->status, static_cast<cudaStream_t>(stream)));
}

int pa_cache_append_fp8(const void* k_new, const void* v_new, uint8_t* k_cache, uint8_t* v_cache,
                        float* k_scale, float* v_scale, const int64_t* slot_mapping,
                        int num_tokens, int num_kv_heads, int head_dim, int block_size,
                        int num_blocks, int dtype, void* stream) {
  if (num_tokens == 0) return PA_OK;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
  if (!k_new || !v_new || !k_cache || !v_cache || !k_scale || !v_scale || !slot_mapping)
    return PA_ERR_INVALID_ARG;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  for (const void* p : {k_new, v_new, static_cast<const void*>(k_cache),
                        static_cast<const void*>(v_cache)})
    if (!aligned(p, 16)) return PA_ERR_INVALID_ARG;
  if (!aligned(k_scale, 4) || !aligned(v_scale, 4) || !aligned(slot_mapping, 8))
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  DeviceState* dev = nullptr;
  if (int rc = device_state(&dev)) return rc;
  return cuda_status(launch_append_fp8(k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                                       slot_mapping, num_tokens, num_kv_heads, head_dim,
                                       block_size, num_blocks, dtype == PA_BF16, dev->status,
                                       static_cast<cudaStream_t>(stream)));
}

int pa_quantize_fp8(const void* k_src, const void* v_src, uint8_t* k_cache, uint8_t* v_cache,
                    float* k_scale, float* v_scale, int num_blocks, int num_kv_heads,
                    int head_dim, int block_size, void* stream) {
  if (!k_src && !v_src) return PA_ERR_INVALID_ARG;
  if (k_src && (!k_cache || !k_scale)) return PA_ERR_INVALID_ARG;
  if (v_src && (!v_cache || !v_scale)) return PA_ERR_INVALID_ARG;
  if (num_blocks < 0 || num_kv_heads <= 0) return PA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (block_size != 16) return PA_ERR_UNSUPPORTED;
  for (const void* p : {k_src, v_src, static_cast<const void*>(k_cache),
                        static_cast<const void*>(v_cache)})
    if (p && !aligned(p, 16)) return PA_ERR_INVALID_ARG;
  if ((k_scale && !aligned(k_scale, 4)) || (v_scale && !aligned(v_scale, 4)))
    return PA_ERR_INVALID_ARG;
  const int64_t tiles = static_cast<int64_t>(num_blocks) * num_kv_heads;
  if (tiles == 0) return PA_OK;
  DeviceState* dev = nullptr;
  if (int rc = device_state(&dev)) return rc;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int tile_elems = block_size * head_dim;
  if (k_src)
    if (cudaError_t e = launch_quantize_fp8(k_src, k_cache, k_scale, tiles, tile_elems, s))
      return cuda_status(e);
  if (v_src)
    if (cudaError_t e = launch_quantize_fp8(v_src, v_cache, v_scale, tiles, tile_elems, s))
      return cuda_status(e);
  return PA_OK;
}

int pa_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                   const int64_t* block_mapping, int num_pairs, int num_kv_heads, int head_dim,
                   int block_size, int num_blocks, int pool_type, void* stream) {
  if (num_pairs < 0 || num_kv_heads <= 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
  if (pool_type != PA_F16 && pool_type != PA_BF16 && pool_type != PA_E4M3)
    return PA_ERR_INVALID_ARG;
  const bool fp8 = pool_type == PA_E4M3;
  if (fp8 != (k_scale != nullptr) || fp8 != (v_scale != nullptr)) return PA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (block_size != 16) return PA_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !block_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_mapping, 8))
    return PA_ERR_INVALID_ARG;
  if ((k_scale && !aligned(k_scale, 4)) || (v_scale && !aligned(v_scale, 4)))
    return PA_ERR_INVALID_ARG;
  DeviceState* dev = nullptr;
  if (int rc = device_state(&dev)) return rc;
  return cuda_status(launch_copy_blocks(k_cache, v_cache, k_scale, v_scale, block_mapping,
                                        num_pairs, num_kv_heads, head_dim * (fp8 ? 1 : 2),
                                        block_size, num_blocks, dev->status,
                                        static_cast<cudaStream_t>(stream)));
}

int pa_e4m3_encode(const float* x, uint8_t* codes, int64_t n, void* stream) {
  if (!x || !codes || n < 0) return PA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(codes, 16)) return PA_ERR_INVALID_ARG;
  if (n == 0) return PA_OK;
  DeviceState* dev = nullptr;
  if (int rc = device_state(&dev)) return rc;
  return cuda_status(launch_e4m3_encode(x, codes, n, static_cast<cudaStream_t>(stream)));
}

size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int head_dim, int split_ctas) {
  return pa_decode_workspace_size_rows(num_seqs, num_q_heads, head_dim, split_ctas, 8);
}

size_t pa_decode_workspace_size_rows(int num_seqs, int num_q_heads, int head_dim, int split_ctas,
                                     int query_rows) {
  if (split_ctas < 0 || query_rows <= 0) return 0;
  if (split_ctas == 0) split_ctas = decode_max_default_ctas();
  // the widest pass: at most kMaxRowsPerLaunch rows
  const int rows = query_rows < kMaxRowsPerLaunch ? query_rows : kMaxRowsPerLaunch;
  return decode_workspace_bytes(num_seqs, num_q_heads, head_dim, split_ctas, rows);
}

int pa_decode_default_splits(int pool_type) {
  if (pool_type != PA_F16 && pool_type != PA_BF16 && pool_type != PA_E4M3) return 0;
  return decode_default_ctas(pool_type == PA_E4M3);
}

int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
              int max_context_len, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
              int block_size, int num_blocks, float scale, int window_size, int queries_per_seq,
              int dtype, int split_ctas,
              void* workspace, size_t workspace_bytes, unsigned flags, void* stream) {
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return PA_ERR_INVALID_ARG;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
  DecodeShape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                      num_blocks, max_blocks_per_seq, max_context_len, split_ctas, window_size};
  s.nq = queries_per_seq;
  s.flags = flags;
  if (int rc = check_decode_shape(s, scale)) return rc;
  for (const void* p : {static_cast<const void*>(out), q, k_cache, v_cache})
    if (!aligned(p, 16)) return PA_ERR_INVALID_ARG;
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4)) return PA_ERR_INVALID_ARG;
  return run_decode(s, out, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens,
                    scale, false, dtype == PA_BF16, workspace, workspace_bytes, stream);
}

int pa_decode_fp8(void* out, const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                  const float* k_scale, const float* v_scale, const int32_t* block_tables,
                  int max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                  int num_blocks, float scale, int window_size, int queries_per_seq,
                  int dtype, int split_ctas, void* workspace,
                  size_t workspace_bytes, unsigned flags, void* stream) {
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !k_scale || !v_scale || !block_tables ||
      !context_lens)
    return PA_ERR_INVALID_ARG;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
  DecodeShape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                      num_blocks, max_blocks_per_seq, max_context_len, split_ctas, window_size};
  s.nq = queries_per_seq;
  s.flags = flags;
  if (int rc = check_decode_shape(s, scale)) return rc;
  for (const void* p : {static_cast<const void*>(out), q, static_cast<const void*>(k_cache),
                        static_cast<const void*>(v_cache)})
    if (!aligned(p, 16)) return PA_ERR_INVALID_ARG;
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(k_scale, 4) ||
      !aligned(v_scale, 4))
    return PA_ERR_INVALID_ARG;
  return run_decode(s, out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                    scale, true, dtype == PA_BF16, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

int decode_step_16(void* out, const void* q, const void* k_new, const void* v_new, void* k_cache,
                   void* v_cache, const int64_t* slot_mapping, const int32_t* block_tables,
                   int max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                   int num_blocks, float scale, int window_size, int dtype, int split_ctas,
                   void* workspace, size_t workspace_bytes, unsigned flags,
                   const pa_step_sync* sync, void* stream) {
  if (num_seqs == 0) {   // nothing to attend; a handshake still gets its done signal
    if (sync == nullptr) return PA_OK;
    if (!sync_ok(sync)) return PA_ERR_INVALID_ARG;
    return cuda_status(launch_signal_done(sync->done, sync->done_value,
                                          static_cast<cudaStream_t>(stream)));
  }
  if (!out || !q || !k_new || !v_new || !k_cache || !v_cache || !slot_mapping ||
      !block_tables || !context_lens)
    return PA_ERR_INVALID_ARG;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
  if (!sync_ok(sync)) return PA_ERR_INVALID_ARG;
  DecodeShape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                num_blocks, max_blocks_per_seq, max_context_len, split_ctas, window_size};
  s.flags = flags;
  if (int rc = check_decode_shape(s, scale)) return rc;
  for (const void* p : {static_cast<const void*>(out), q, k_new, v_new,
                        static_cast<const void*>(k_cache), static_cast<const void*>(v_cache)})
    if (!aligned(p, 16)) return PA_ERR_INVALID_ARG;
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(slot_mapping, 8))
    return PA_ERR_INVALID_ARG;
  AppendArgs ap;
  ap.k_new = k_new;
  ap.v_new = v_new;
  ap.slots = slot_mapping;
  ap.k_pool = k_cache;
  ap.v_pool = v_cache;
  return run_decode(s, out, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens,
                    scale, false, dtype == PA_BF16, workspace, workspace_bytes, stream, ap, sync);
}

int decode_step_e4m3(void* out, const void* q, const void* k_new, const void* v_new,
                     uint8_t* k_cache, uint8_t* v_cache, float* k_scale, float* v_scale,
                     const int64_t* slot_mapping, const int32_t* block_tables,
                     int max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
                     int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                     int block_size, int num_blocks, float scale, int window_size, int dtype,
                     int split_ctas, void* workspace, size_t workspace_bytes, unsigned flags,
                     const pa_step_sync* sync, void* stream) {
  if (num_seqs == 0) {   // nothing to attend; a handshake still gets its done signal
    if (sync == nullptr) return PA_OK;
    if (!sync_ok(sync)) return PA_ERR_INVALID_ARG;
    return cuda_status(launch_signal_done(sync->done, sync->done_value,
                                          static_cast<cudaStream_t>(stream)));
  }
  if (!out || !q || !k_new || !v_new || !k_cache || !v_cache || !k_scale || !v_scale ||
      !slot_mapping || !block_tables || !context_lens)
    return PA_ERR_INVALID_ARG;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
  if (!sync_ok(sync)) return PA_ERR_INVALID_ARG;
  DecodeShape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                num_blocks, max_blocks_per_seq, max_context_len, split_ctas, window_size};
  s.flags = flags;
  if (int rc = check_decode_shape(s, scale)) return rc;
  for (const void* p : {static_cast<const void*>(out), q, k_new, v_new,
                        static_cast<const void*>(k_cache), static_cast<const void*>(v_cache)})
    if (!aligned(p, 16)) return PA_ERR_INVALID_ARG;
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(k_scale, 4) ||
      !aligned(v_scale, 4) || !aligned(slot_mapping, 8))
    return PA_ERR_INVALID_ARG;
  AppendArgs ap;
  ap.k_new = k_new;
  ap.v_new = v_new;
  ap.slots = slot_mapping;
  ap.k_pool = k_cache;
  ap.v_pool = v_cache;
  ap.k_scale = k_scale;
  ap.v_scale = v_scale;
  return run_decode(s, out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                    scale, true, dtype == PA_BF16, workspace, workspace_bytes, stream, ap, sync);
}

}  // namespace

extern "C" {

int pa_decode_step(void* out, const void* q, const void* k_new, const void* v_new,
                   void* k_cache, void* v_cache, const int64_t* slot_mapping,
                   const int32_t* block_tables, int max_blocks_per_seq,
                   const int32_t* context_lens, int max_context_len, int num_seqs,
                   int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                   int num_blocks, float scale, int window_size, int dtype, int split_ctas,
                   void* workspace, size_t workspace_bytes, unsigned flags, void* stream) {
  return decode_step_16(out, q, k_new, v_new, k_cache, v_cache, slot_mapping, block_tables,
                        max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                        num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                        window_size, dtype, split_ctas, workspace, workspace_bytes, flags,
                        nullptr, stream);
}

int pa_decode_step_synced(void* out, const void* q, const void* k_new, const void* v_new,
                          void* k_cache, void* v_cache, const int64_t* slot_mapping,
                          const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* context_lens, int max_context_len, int num_seqs,
                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          int num_blocks, float scale, int window_size, int dtype,
                          int split_ctas, void* workspace, size_t workspace_bytes,
                          unsigned flags, const pa_step_sync* sync, void* stream) {
  if (sync == nullptr) return PA_ERR_INVALID_ARG;
  return decode_step_16(out, q, k_new, v_new, k_cache, v_cache, slot_mapping, block_tables,
                        max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                        num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                        window_size, dtype, split_ctas, workspace, workspace_bytes, flags, sync,
                        stream);
}

int pa_decode_step_fp8(void* out, const void* q, const void* k_new, const void* v_new,
                       uint8_t* k_cache, uint8_t* v_cache, float* k_scale, float* v_scale,
                       const int64_t* slot_mapping, const int32_t* block_tables,
                       int max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
                       int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int num_blocks, float scale, int window_size, int dtype,
                       int split_ctas, void* workspace, size_t workspace_bytes, unsigned flags,
                       void* stream) {
  return decode_step_e4m3(out, q, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                          slot_mapping, block_tables, max_blocks_per_seq, context_lens,
                          max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                          block_size, num_blocks, scale, window_size, dtype, split_ctas,
                          workspace, workspace_bytes, flags, nullptr, stream);
}

int pa_decode_step_fp8_synced(void* out, const void* q, const void* k_new, const void* v_new,
                              uint8_t* k_cache, uint8_t* v_cache, float* k_scale,
                              float* v_scale, const int64_t* slot_mapping,
                              const int32_t* block_tables, int max_blocks_per_seq,
                              const int32_t* context_lens, int max_context_len, int num_seqs,
                              int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                              int num_blocks, float scale, int window_size, int dtype,
                              int split_ctas, void* workspace, size_t workspace_bytes,
                              unsigned flags, const pa_step_sync* sync, void* stream) {
  if (sync == nullptr) return PA_ERR_INVALID_ARG;
  return decode_step_e4m3(out, q, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                          slot_mapping, block_tables, max_blocks_per_seq, context_lens,
                          max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                          block_size, num_blocks, scale, window_size, dtype, split_ctas,
                          workspace, workspace_bytes, flags, sync, stream);
}

}  // extern "C"

namespace {

bool copies_ok(const pa_step_copies* io) {
  return io != nullptr && io->host_in != nullptr && io->dev_in != nullptr &&
         io->dev_out != nullptr && io->host_out != nullptr && io->reuse_event != nullptr &&
         io->in_bytes > 0 && io->out_bytes > 0;
}

// The copies before a pipelined step: wait for the slot's last read-back
// (when reused), upload, then the ready word.
int upload_and_signal(const pa_step_copies* io, const pa_step_sync* sync) {
  const cudaStream_t cs = static_cast<cudaStream_t>(io->copy_stream);
  if (io->slot_reused &&
      cudaStreamWaitEvent(cs, static_cast<cudaEvent_t>(io->reuse_event), 0) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaMemcpyAsync(io->dev_in, io->host_in, io->in_bytes, cudaMemcpyHostToDevice, cs) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  const StreamMemOps& ops = stream_mem_ops();
  if (ops.write == nullptr) return PA_ERR_UNSUPPORTED;
  return cu_status(ops.write(static_cast<CUstream>(cs),
                             reinterpret_cast<CUdeviceptr>(sync->ready), sync->ready_value,
                             CU_STREAM_WRITE_VALUE_DEFAULT));
}

// The copies after a launched step: wait for its done word, read the output
// back, record the slot's event.
int wait_and_read_back(const pa_step_copies* io, const pa_step_sync* sync) {
  const cudaStream_t bs = static_cast<cudaStream_t>(io->back_stream);
  const StreamMemOps& ops = stream_mem_ops();
  if (ops.wait == nullptr) return PA_ERR_UNSUPPORTED;
  if (int rc = cu_status(ops.wait(static_cast<CUstream>(bs),
                                  reinterpret_cast<CUdeviceptr>(sync->done), sync->done_value,
                                  CU_STREAM_WAIT_VALUE_GEQ)))
    return rc;
  if (cudaMemcpyAsync(io->host_out, io->dev_out, io->out_bytes, cudaMemcpyDeviceToHost, bs) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return cuda_status(cudaEventRecord(static_cast<cudaEvent_t>(io->reuse_event), bs));
}

}  // namespace

extern "C" {

int pa_decode_step_pipelined(void* out, const void* q, const void* k_new, const void* v_new,
                             void* k_cache, void* v_cache, const int64_t* slot_mapping,
                             const int32_t* block_tables, int max_blocks_per_seq,
                             const int32_t* context_lens, int max_context_len, int num_seqs,
                             int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                             int num_blocks, float scale, int window_size, int dtype,
                             int split_ctas, void* workspace, size_t workspace_bytes,
                             unsigned flags, const pa_step_sync* sync,
                             const pa_step_copies* io, void* stream) {
  if (sync == nullptr || !sync_ok(sync) || !copies_ok(io)) return PA_ERR_INVALID_ARG;
  if (int rc = upload_and_signal(io, sync)) return rc;
  if (int rc = decode_step_16(out, q, k_new, v_new, k_cache, v_cache, slot_mapping,
                              block_tables, max_blocks_per_seq, context_lens, max_context_len,
                              num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                              num_blocks, scale, window_size, dtype, split_ctas, workspace,
                              workspace_bytes, flags, sync, stream))
    return rc;
  return wait_and_read_back(io, sync);
}

int pa_decode_step_fp8_pipelined(void* out, const void* q, const void* k_new, const void* v_new,
                                 uint8_t* k_cache, uint8_t* v_cache, float* k_scale,
                                 float* v_scale, const int64_t* slot_mapping,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int max_context_len,
                                 int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int num_blocks, float scale, int window_size,
                                 int dtype, int split_ctas, void* workspace,
                                 size_t workspace_bytes, unsigned flags,
                                 const pa_step_sync* sync, const pa_step_copies* io,
                                 void* stream) {
  if (sync == nullptr || !sync_ok(sync) || !copies_ok(io)) return PA_ERR_INVALID_ARG;
  if (int rc = upload_and_signal(io, sync)) return rc;
  if (int rc = decode_step_e4m3(out, q, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                                slot_mapping, block_tables, max_blocks_per_seq, context_lens,
                                max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                block_size, num_blocks, scale, window_size, dtype, split_ctas,
                                workspace, workspace_bytes, flags, sync, stream))
    return rc;
  return wait_and_read_back(io, sync);
}

int pa_stream_write_value(void* stream, uint32_t* addr, uint32_t value) {
  if (addr == nullptr || !aligned(addr, 4)) return PA_ERR_INVALID_ARG;
  const StreamMemOps& ops = stream_mem_ops();
  if (ops.write == nullptr) return PA_ERR_UNSUPPORTED;
  return cu_status(ops.write(static_cast<CUstream>(stream), reinterpret_cast<CUdeviceptr>(addr),
                             value, CU_STREAM_WRITE_VALUE_DEFAULT));
}

int pa_stream_wait_value(void* stream, const uint32_t* addr, uint32_t value) {
  if (addr == nullptr || !aligned(addr, 4)) return PA_ERR_INVALID_ARG;
  const StreamMemOps& ops = stream_mem_ops();
  if (ops.wait == nullptr) return PA_ERR_UNSUPPORTED;
  return cu_status(ops.wait(static_cast<CUstream>(stream), reinterpret_cast<CUdeviceptr>(addr),
                            value, CU_STREAM_WAIT_VALUE_GEQ));
}

int pa_test_wait_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > kWaitLimitNs) return PA_ERR_INVALID_ARG;
  DeviceState* dev = nullptr;
  if (int rc = device_state(&dev)) return rc;
  return cuda_status(launch_wait_probe(dev->status, limit_ns, static_cast<cudaStream_t>(stream)));
}

int pa_test_merge_timeout(void* out, const int32_t* context_lens, int max_context_len,
                          int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                          int dtype, int split_ctas, void* workspace, size_t workspace_bytes,
                          uint64_t limit_ns, void* stream) {
  if (!out || !context_lens || !workspace) return PA_ERR_INVALID_ARG;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
  if (limit_ns == 0 || limit_ns > kWaitLimitNs) return PA_ERR_INVALID_ARG;
  if (num_seqs <= 0 || num_seqs > kMaxBatchPerLaunch || split_ctas <= 0 || max_context_len < 0)
    return PA_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return PA_ERR_INVALID_ARG;
  if (num_q_heads / num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (!aligned(out, 16) || !aligned(context_lens, 4) || !aligned(workspace, 256))
    return PA_ERR_INVALID_ARG;
  if (workspace_bytes < decode_workspace_bytes(num_seqs, num_q_heads, head_dim, split_ctas, 8))
    return PA_ERR_WORKSPACE;
  DeviceState* dev = nullptr;
  if (int rc = device_state(&dev)) return rc;
  DecodeArgs a{};
  a.out = out;
  a.context_lens = context_lens;
  a.status = dev->status;
  a.mbs = (max_context_len + 15) / 16 > 0 ? (max_context_len + 15) / 16 : 1;
  a.B = num_seqs;
  a.Hq = num_q_heads;
  a.Hkv = num_kv_heads;
  a.group = num_q_heads / num_kv_heads;
  a.D = head_dim;
  a.max_context_len = max_context_len;
  a.split_ctas = split_ctas;
  a.n_q = 1;
  a.q_tokens = 1;
  a.rows = 8;
  a.wait_limit_ns = limit_ns;
  decode_workspace_split(a, workspace);
  return cuda_status(launch_merge_only(a, dtype == PA_BF16, static_cast<cudaStream_t>(stream)));
}

int pa_get_status(void* stream, unsigned* bits) {
  DeviceState* dev = nullptr;
  if (int rc = device_state(&dev)) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ERR_CUDA;
  unsigned v = 0, zero = 0;
  if (cudaMemcpy(&v, dev->status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaMemcpy(dev->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return PA_ERR_CUDA;
  if (bits) *bits = v;
  if (v & (PA_STATUS_TIMEOUT | PA_STATUS_WS_DIRTY)) noalloc_scratch_suspect();
  if (v & PA_STATUS_TIMEOUT) return PA_ERR_TIMEOUT;
  if (v & PA_STATUS_WS_DIRTY) return PA_ERR_WORKSPACE;
  if (v) return PA_ERR_BOUNDS;
  return PA_OK;
}

}  // extern "C"
