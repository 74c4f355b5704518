// paged_decode_f32.cu -- instantiates the paged decode kernels for f32 storage.
#include "paged_decode.cuh"

namespace photon {
cudaError_t launch_paged_decode_f32(const DecodeArgs& a, cudaStream_t stream) {
  return launch_decode_t<float>(a, stream);
}
}  // namespace photon
