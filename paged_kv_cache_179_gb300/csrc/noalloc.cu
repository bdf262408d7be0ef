// noalloc.cu -- pa_decode_noalloc: paged GQA decode for callers that cannot
// allocate device memory.
//
// pa_decode needs a caller-allocated workspace (the partial results of
// context partitions split across warps, which the merge launch reads).  Some callers cannot provide one: code running inside
// a host framework that owns every byte of device memory and forbids raw
// allocations, latency-critical serving loops where cudaMalloc would
// synchronise the device, and plain C callers with no device allocator of
// their own.  This entry point runs the same kernel with its scratch in a
// fixed array compiled into the library, so it allocates nothing.
//
// The array is PA_NOALLOC_SCRATCH_BYTES (16 MiB); every GPU that loads the
// library holds it until the process exits.  All calls on a device share it.
// It starts zero-filled, as every static device array does, and each call
// leaves it zero-filled again, so it never needs clearing; after a status
// read that shows a wait that gave up or a dirty workspace, the next call
// zeroes it first.  Calls that overlap on the GPU (different streams, or
// different host threads) race on the array and must not be issued.
#include <climits>
#include <cmath>
#include <mutex>

#include "pa.h"
#include "pa_launch.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

using pa::kMaxDevices;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};
bool g_scratch_suspect[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device with that device current, and cached.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return PA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PA_OK;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

void pa::noalloc_scratch_suspect() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  g_scratch_suspect[dev] = true;
}

extern "C" int pa_decode_noalloc(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_tables,
                                 int max_blocks_per_seq, const int32_t* context_lens,
                                 int max_context_len, int num_seqs, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                 float scale, int window_size, int queries_per_seq,
                                 int dtype, int split_ctas, unsigned flags, void* stream) {
  using namespace pa;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return PA_ERR_INVALID_ARG;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return PA_ERR_INVALID_ARG;
  if (num_blocks <= 0 || max_blocks_per_seq <= 0 || max_context_len < 0 || split_ctas < 0 ||
      window_size < 0 || queries_per_seq < 1 ||
      (flags & ~(PA_DECODE_EARLY_PROLOGUE | PA_DECODE_EARLY_COPIES)) != 0 ||
      ((flags & PA_DECODE_EARLY_COPIES) && !(flags & PA_DECODE_EARLY_PROLOGUE)))
    return PA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_context_len) >
      static_cast<int64_t>(max_blocks_per_seq) * block_size)
    return PA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (block_size != 16) return PA_ERR_UNSUPPORTED;
  if (num_q_heads / num_kv_heads * queries_per_seq > 8) return PA_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  for (const void* p : {static_cast<const void*>(out), q, k_cache, v_cache})
    if (!aligned_to(p, 16)) return PA_ERR_INVALID_ARG;
  if (!aligned_to(block_tables, 4) || !aligned_to(context_lens, 4)) return PA_ERR_INVALID_ARG;

  // set-up on the first call on this device: the scratch array's address
  void* ws = nullptr;
  if (int rc = scratch_address(&ws)) return rc;
  unsigned* status = nullptr;
  if (int rc = device_status_word(&status)) return rc;
  const int splits = split_ctas == 0 ? decode_default_ctas(false) : split_ctas;
  const size_t need = decode_workspace_bytes(num_seqs, num_q_heads, head_dim, splits, 8);
  if (need == 0 || need > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_SCRATCH_LIMIT;

  DecodeArgs a{};
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.status = status;
  a.mbs = max_blocks_per_seq;
  a.Hq = num_q_heads;
  a.Hkv = num_kv_heads;
  a.group = num_q_heads / num_kv_heads;
  a.D = head_dim;
  a.num_blocks = num_blocks;
  a.max_context_len = max_context_len;
  a.split_ctas = splits;
  a.window = window_size;
  a.n_q = queries_per_seq;
  a.q_tokens = queries_per_seq;
  a.q_first = 0;
  a.rows = 8;
  a.early = (flags & PA_DECODE_EARLY_PROLOGUE) ? 1 : 0;
  a.early_copies = (flags & PA_DECODE_EARLY_COPIES) ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit_ns = kWaitLimitNs;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    // a status read saw a wait give up or a dirty workspace: partials may be
    // left in the scratch, so zero it (stream-ordered) before this call
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_suspect[dev]) {
      if (cudaMemsetAsync(ws, 0, PA_NOALLOC_SCRATCH_BYTES, s) != cudaSuccess)
        return PA_ERR_CUDA;
      g_scratch_suspect[dev] = false;
    }
  }
  const size_t row = static_cast<size_t>(queries_per_seq) * num_q_heads * head_dim * 2;
  for (int b0 = 0; b0 < num_seqs; b0 += kMaxBatchPerLaunch) {
    DecodeArgs c = a;
    c.B = num_seqs - b0 < kMaxBatchPerLaunch ? num_seqs - b0 : kMaxBatchPerLaunch;
    c.out = static_cast<uint8_t*>(out) + b0 * row;
    c.q = static_cast<const uint8_t*>(q) + b0 * row;
    c.block_tables = block_tables + static_cast<int64_t>(b0) * max_blocks_per_seq;
    c.context_lens = context_lens + b0;
    decode_workspace_split(c, ws);
    if (launch_decode(c, false, dtype == PA_BF16, s) != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}
