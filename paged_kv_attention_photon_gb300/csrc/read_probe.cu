// read_probe.cu -- the decode's K/V read pattern with no arithmetic: a
// measuring aid for the decode kernel's roofline.
//
// Each chunk named by an offset is one (block, KV head) run of the K pool and
// the same run of the V pool -- 16 rows of head_dim elements, the unit the
// decode kernel copies.  A persistent grid (two CTAs per SM) takes runs of
// consecutive chunks round robin; in each CTA one warp streams the chunks of
// its runs into a ring of shared-memory stages with 1-D bulk copies, exactly
// as the decode's producer warp does, and nothing reads them.  The time of a
// call is therefore the practical ceiling of the decode's own data movement:
// random 4 KB chunks (at head_dim 128, fp16) in the decode's order, through
// the same copy engine, at the same bytes in flight per SM.
#include "photon_common.cuh"

namespace photon {
namespace {

constexpr int kProbeStages = 12;
constexpr int kProbeMaxChunk = 4096;                 // bytes of one K (or V) chunk
constexpr int kProbeSmem = kProbeStages * 2 * kProbeMaxChunk;

__global__ void __launch_bounds__(32) read_probe_kernel(const unsigned char* __restrict__ k,
                                                        const unsigned char* __restrict__ v,
                                                        const int64_t* __restrict__ offs,
                                                        int64_t n, uint32_t chunk_bytes,
                                                        int run, uint64_t pool_bytes,
                                                        uint32_t* err) {
  extern __shared__ __align__(128) unsigned char probe_smem[];
  __shared__ __align__(8) uint64_t full[kProbeStages];
  const int lane = threadIdx.x;
  if (lane == 0) {
    for (int s = 0; s < kProbeStages; ++s) mbar_init(&full[s], 1);
    mbar_init_fence();
  }
  __syncwarp();
  const int64_t runs = (n + run - 1) / run;
  uint32_t st = 0;
  bool ok = true;
  for (int64_t r = blockIdx.x; r < runs && ok; r += gridDim.x) {
    const int64_t c_end = min(n, (r + 1) * run);
    for (int64_t c0 = r * run; c0 < c_end && ok; c0 += 32) {
      // lane j holds the offset of chunk c0 + j: one coalesced load per 32 chunks
      const int64_t mine = c0 + lane < c_end ? __ldg(offs + c0 + lane) : -1;
      const int cnt = c_end - c0 < 32 ? (int)(c_end - c0) : 32;
      for (int i = 0; i < cnt; ++i) {
        const int64_t off = __shfl_sync(0xffffffffu, mine, i);
        if (lane == 0) {
          const int slot = st % kProbeStages;
          if (st >= (uint32_t)kProbeStages &&
              !mbar_wait_bounded(&full[slot], ((st / kProbeStages) - 1) & 1u)) {
            ok = false;
          } else {
            const bool valid = off >= 0 && (off & 15) == 0 &&
                               (uint64_t)off + chunk_bytes <= pool_bytes;
            if (!valid) raise_error(err, kErrBlock);
            mbar_arrive_expect_tx(&full[slot], valid ? 2u * chunk_bytes : 0u);
            if (valid) {
              unsigned char* dst = probe_smem + slot * 2 * kProbeMaxChunk;
              bulk_copy_g2s(dst, k + off, chunk_bytes, &full[slot]);
              bulk_copy_g2s(dst + kProbeMaxChunk, v + off, chunk_bytes, &full[slot]);
            }
            ++st;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
    }
  }
  if (lane == 0) {
    if (!ok) raise_error(err, kErrTimeout);
    // every copy issued lands before the CTA retires
    const uint32_t first = st > (uint32_t)kProbeStages ? st - kProbeStages : 0u;
    for (uint32_t s = first; s < st; ++s)
      if (!mbar_wait_bounded(&full[s % kProbeStages], (s / kProbeStages) & 1u)) {
        raise_error(err, kErrTimeout);
        break;
      }
  }
}

}  // namespace

cudaError_t launch_read_probe(const void* k, const void* v, const int64_t* offs, int64_t n,
                              uint32_t chunk_bytes, int run, uint64_t pool_bytes, int num_sms,
                              uint32_t* err, cudaStream_t stream) {
  if (chunk_bytes == 0 || chunk_bytes > (uint32_t)kProbeMaxChunk || chunk_bytes % 16 || run < 1)
    return cudaErrorInvalidValue;
  static bool configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(read_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kProbeSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  read_probe_kernel<<<2 * num_sms, 32, kProbeSmem, stream>>>(
      static_cast<const unsigned char*>(k), static_cast<const unsigned char*>(v), offs, n,
      chunk_bytes, run, pool_bytes, err);
  return cudaGetLastError();
}

}  // namespace photon
