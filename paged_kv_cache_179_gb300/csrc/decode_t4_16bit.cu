// decode_t4_16bit.cu -- decode launches over 16-bit pools with four tiles of 8
// query columns per warp (17 to 32 query rows per (sequence, kv head)),
// instantiated apart so the library's translation units compile in parallel.
#undef PA_TRACE
#include "decode_kernels.cuh"

namespace pa {

cudaError_t launch_decode_tiles4_16bit(const DecodeArgs& a, bool bf16, cudaStream_t s) {
  if (bf16)
    return a.D == 128 ? launch_dtype<128, false, true, 4>(a, s) : launch_dtype<64, false, true, 4>(a, s);
  return a.D == 128 ? launch_dtype<128, false, false, 4>(a, s) : launch_dtype<64, false, false, 4>(a, s);
}

}  // namespace pa
