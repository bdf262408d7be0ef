// decode_t2.cu -- decode launches with two tiles of 8 query columns per warp
// (9 to 16 query rows per (sequence, kv head): query groups of 9 to 16, or
// several query tokens), instantiated apart so the library's translation
// units compile in parallel.
#undef PA_TRACE
#include "decode_kernels.cuh"

namespace pa {

cudaError_t launch_decode_tiles2(const DecodeArgs& a, bool fp8, bool bf16, cudaStream_t s) {
  return launch_nt<2>(a, fp8, bf16, s);
}

}  // namespace pa
