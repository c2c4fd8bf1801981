// head_dim = 64 instantiations of the decode kernel (decode_kernel.cuh).
#include "decode_kernel.cuh"

namespace fia {

cudaError_t launch_decode_d64(const DecodeParams& p, bool bf16, cudaStream_t s) {
  return bf16 ? launch_decode_group<64, true>(p, s) : launch_decode_group<64, false>(p, s);
}

}  // namespace fia
