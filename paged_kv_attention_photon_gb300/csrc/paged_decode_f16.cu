// paged_decode_f16.cu -- instantiates the paged decode kernels for f16 storage.
#include "paged_decode.cuh"

namespace photon {
cudaError_t launch_paged_decode_f16(const DecodeArgs& a, cudaStream_t stream) {
  return launch_decode_t<__half>(a, stream);
}
cudaError_t launch_paged_decode_fp8(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.D) {
    case 64: return launch_decode_fp8_d<64>(a, stream);
    case 128: return launch_decode_fp8_d<128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace photon

#ifdef PHOTON_PROBE
// Tuning builds only: copy the per-CTA timeline of the last fp16 decode.
extern "C" int photon_probe_read(void* dst, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(dst, photon::g_probe, bytes);
}
extern "C" int photon_probe_merge_read(void* dst, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(dst, photon::g_probe_merge, bytes);
}
extern "C" int photon_probe_stamp(void* stream, int big) {
  if (big > 0) {
    cudaFuncSetAttribute(photon::probe_stamp_big_kernel,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    photon::probe_stamp_big_kernel<<<152, 32, 200 * 1024, static_cast<cudaStream_t>(stream)>>>();
  } else {
    photon::probe_stamp_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(big < 0 ? 1 : 0);
  }
  return (int)cudaGetLastError();
}
extern "C" int photon_probe_stamp_read(void* dst) {
  return (int)cudaMemcpyFromSymbol(dst, photon::g_probe_stamp, 16);
}
#endif
