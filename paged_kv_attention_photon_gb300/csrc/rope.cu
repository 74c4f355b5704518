// rope.cu -- cos/sin table of the rotary position embedding.
//
// PhotonInfer README, "Key features / GPU-optimized kernels": batched RoPE is
// one of the fused operations.  The rotation is the rotate-half form: for
// k < d/2 the pair (x[k], x[k + d/2]) turns by theta = pos * base^(-2k/d).
// The table holds (cos theta, sin theta) for every position and pair, computed
// in double and stored as fp32, so the decode step only loads it: the angles
// reach several thousand radians, where an fp32 product pos * base^(-2k/d)
// alone would already be off by ~1e-3.
#include "photon_common.cuh"

namespace photon {
namespace {

__global__ void __launch_bounds__(256) rope_table_kernel(double log2_base, int max_pos, int d,
                                                         float2* table) {
  const int half = d / 2;
  const long long total = (long long)max_pos * half;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int pos = (int)(i / half), k = (int)(i % half);
    const double inv_freq = exp2(-2.0 * (double)k / (double)d * log2_base);
    double s, c;
    sincos((double)pos * inv_freq, &s, &c);
    table[i] = make_float2((float)c, (float)s);
  }
}

}  // namespace

cudaError_t launch_rope_table(double base, int max_pos, int d, float2* table,
                              cudaStream_t stream) {
  const long long total = (long long)max_pos * (d / 2);
  long long grid = (total + 255) / 256;
  if (grid > 152 * 16) grid = 152 * 16;
  if (grid < 1) grid = 1;
  rope_table_kernel<<<(int)grid, 256, 0, stream>>>(log2(base), max_pos, d, table);
  return cudaGetLastError();
}

}  // namespace photon
