// paged_decode_bf16.cu -- instantiates the paged decode kernels for bf16 storage.
#include "paged_decode.cuh"

namespace photon {
cudaError_t launch_paged_decode_bf16(const DecodeArgs& a, cudaStream_t stream) {
  return launch_decode_t<__nv_bfloat16>(a, stream);
}
}  // namespace photon
