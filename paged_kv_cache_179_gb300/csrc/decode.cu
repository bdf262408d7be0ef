// decode.cu -- the decode launches with one tile of 8 query columns per warp
// (up to 8 query rows per (sequence, kv head)), the dispatch to the two- and
// four-tile launches of decode_t2.cu and decode_t4_*.cu, the decode
// workspace layout, and the failure-path probes of the bounded waits.  The
// kernels themselves are in decode_kernels.cuh.
#include "decode_kernels.cuh"

namespace pa {
namespace {

// One warp: lane 0 sets up an mbarrier that nothing ever completes and waits
// on it as the attention loop waits for its tiles (bounded by limit_ns), then
// reports the timeout.  Used only to test that failure path.
__global__ void wait_probe_kernel(unsigned* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    mbar_init_fence();
  }
  __syncwarp();
  if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar), 0, limit_ns)) && threadIdx.x == 0)
    atomicOr(status, kStatusTimeout);
}

}  // namespace

int decode_default_ctas(bool fp8, int rows) {
  return device_sm_count() * (rows > 8 ? 2 : ctas_per_sm(fp8));
}

int decode_max_default_ctas() {
  return device_sm_count() * (PA_CTAS_F16 > PA_CTAS_FP8 ? PA_CTAS_F16 : PA_CTAS_FP8);
}

namespace {
// Workspace: partial rows (acc, then (max, sum)) of two pieces per worker,
// each part 256-byte aligned.  Zero-filled between calls.
struct WsLayout {
  size_t acc, ml, total;
};
WsLayout ws_layout(int D, int split_ctas, int rows_per_piece) {
  const int64_t rows = static_cast<int64_t>(split_ctas) * kWarps * 2 * rows_per_piece;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  WsLayout l{};
  l.acc = 0;
  l.ml = up(static_cast<size_t>(rows) * D * 4);
  l.total = l.ml + up(static_cast<size_t>(rows) * 2 * 4);
  return l;
}
}  // namespace

cudaError_t launch_merge_only(const DecodeArgs& a, bool bf16, cudaStream_t s) {
  if (a.rows != 8) return cudaErrorInvalidValue;
  if (a.D == 128) return bf16 ? launch_merge<128, true, 8>(a, s) : launch_merge<128, false, 8>(a, s);
  return bf16 ? launch_merge<64, true, 8>(a, s) : launch_merge<64, false, 8>(a, s);
}

// A step with nothing to attend still signals its handshake's done word.
__global__ void signal_done_kernel(uint32_t* done, uint32_t value) {
  st_release_gpu_b32(done, value);
}

cudaError_t launch_signal_done(uint32_t* done, uint32_t value, cudaStream_t s) {
  signal_done_kernel<<<1, 1, 0, s>>>(done, value);
  return cudaGetLastError();
}

cudaError_t launch_wait_probe(unsigned* status, uint64_t limit_ns, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

int decode_rows(int query_rows) {
  return query_rows <= kGroupMax ? kGroupMax : query_rows <= 2 * kGroupMax ? 2 * kGroupMax
                                                                          : 4 * kGroupMax;
}

size_t decode_workspace_bytes(int B, int Hq, int D, int split_ctas, int rows) {
  if (B <= 0 || Hq <= 0 || D <= 0 || split_ctas <= 0 || rows <= 0) return 0;
  return ws_layout(D, split_ctas, decode_rows(rows)).total;
}

void decode_workspace_split(DecodeArgs& a, void* ws) {
  const WsLayout l = ws_layout(a.D, a.split_ctas, a.rows);
  uint8_t* base = static_cast<uint8_t*>(ws);
  a.ws_acc = reinterpret_cast<float*>(base + l.acc);
  a.ws_ml = reinterpret_cast<float*>(base + l.ml);
}

cudaError_t launch_decode(const DecodeArgs& a, bool fp8, bool bf16, cudaStream_t s) {
  if (a.rows == 8) return launch_nt<1>(a, fp8, bf16, s);
  if (decode_tc_eligible(a, fp8)) return launch_decode_tc(a, bf16, s);
  if (a.rows == 16) return launch_decode_tiles2(a, fp8, bf16, s);
  if (a.rows == 32)
    return fp8 ? launch_decode_tiles4_e4m3(a, bf16, s) : launch_decode_tiles4_16bit(a, bf16, s);
  return cudaErrorInvalidValue;
}

}  // namespace pa
