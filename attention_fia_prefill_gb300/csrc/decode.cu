// Decode launcher and the head_dim = 128 instantiations of the decode kernel
// (the kernel itself is in decode_kernel.cuh; head_dim = 64 is compiled in
// decode_d64.cu so the two build in parallel).  Units of at most 16 rows with
// head_dim 128 go to the warp-level kernel of decode_gqa.cu.
#include "decode_kernel.cuh"

namespace fia {

cudaError_t launch_decode_d64(const DecodeParams& p, bool bf16, cudaStream_t s);
cudaError_t launch_decode_gqa(const DecodeParams& p, bool bf16, cudaStream_t s);

cudaError_t launch_decode(const DecodeParams& p, int head_dim, bool bf16, cudaStream_t s) {
  if (head_dim == 128 && p.rows <= 16 && p.force_tc == 0) return launch_decode_gqa(p, bf16, s);
  if (head_dim == 128) return bf16 ? launch_decode_group<128, true>(p, s) : launch_decode_group<128, false>(p, s);
  if (head_dim == 64) return launch_decode_d64(p, bf16, s);
  return cudaErrorInvalidValue;
}

}  // namespace fia
