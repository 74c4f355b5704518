// cache_write.cu -- batched KV cache-write scatter and the diagnostic
// block-table gather.
//
// PhotonInfer README, "Technical details / Paged attention": the K/V rows of
// many sequences are written into the block-wise cache by one kernel, each row
// going to the slot its sequence's cache offset names.  The row move is a bit
// copy done in 16-byte chunks (README "Key features": vectorised 128-bit
// access), one chunk per thread, chunks of a row on neighbouring threads so
// both the read of the new rows and the write into the pool coalesce.
#include <cuda_fp8.h>

#include "photon_common.cuh"

namespace photon {
namespace {

__global__ void __launch_bounds__(256) cache_write_kernel(CacheWriteArgs a) {
  pdl_launch_dependents();  // a PDL-launched successor may start its prologue
  pdl_wait_primary();       // inputs may come from the previous kernel in the stream
  const int cpr = a.row_bytes >> 4;                    // 16-byte chunks per row
  const int64_t total = (int64_t)a.T * a.Hkv * 2 * cpr;
  const int64_t nslots = (int64_t)a.NB * a.block_size;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx % cpr);
    int64_t r = idx / cpr;
    const int which = (int)(r & 1);                    // 0 = K, 1 = V
    r >>= 1;
    const int h = (int)(r % a.Hkv);
    const int64_t t = r / a.Hkv;
    const int64_t slot = a.slot_mapping[t];
    if (slot < 0) continue;                            // padding row
    if (slot >= nslots) {
      if (c == 0 && which == 0 && h == 0) raise_error(a.err, kErrSlot);
      continue;
    }
    const int64_t blk = slot / a.block_size, off = slot % a.block_size;
    const char* src = static_cast<const char*>(which ? a.v : a.k) +
                      ((t * a.Hkv + h) * (int64_t)a.row_bytes) + 16 * c;
    char* dst = static_cast<char*>(which ? a.v_cache : a.k_cache) +
                (((blk * a.Hkv + h) * a.block_size + off) * (int64_t)a.row_bytes) + 16 * c;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
}

// Quantising write into an e4m3 cache: one thread per 8 elements of a row (a
// 16-byte fp16 load, an 8-byte code store); x * inv_scale in fp32, then the
// round-to-nearest-even, finite-saturating conversion.
__global__ void __launch_bounds__(256) cache_write_fp8_kernel(CacheWriteFp8Args a) {
  pdl_launch_dependents();
  pdl_wait_primary();
  const int cpr = a.D / 8;                             // 8-element pieces per row
  const int64_t total = (int64_t)a.T * a.Hkv * 2 * cpr;
  const int64_t nslots = (int64_t)a.NB * a.block_size;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx % cpr);
    int64_t r = idx / cpr;
    const int which = (int)(r & 1);                    // 0 = K, 1 = V
    r >>= 1;
    const int h = (int)(r % a.Hkv);
    const int64_t t = r / a.Hkv;
    const int64_t slot = a.slot_mapping[t];
    if (slot < 0) continue;                            // padding row
    if (slot >= nslots) {
      if (c == 0 && which == 0 && h == 0) raise_error(a.err, kErrSlot);
      continue;
    }
    const int64_t blk = slot / a.block_size, off = slot % a.block_size;
    const uint4 raw = *reinterpret_cast<const uint4*>(
        static_cast<const __half*>(which ? a.v : a.k) + (t * a.Hkv + h) * (int64_t)a.D + 8 * c);
    const __half2* hp = reinterpret_cast<const __half2*>(&raw);
    const float inv = which ? a.v_inv : a.k_inv;
    uint32_t word[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(hp[i]);
      const uint32_t c0 = __nv_cvt_float_to_fp8(f.x * inv, __NV_SATFINITE, __NV_E4M3);
      const uint32_t c1 = __nv_cvt_float_to_fp8(f.y * inv, __NV_SATFINITE, __NV_E4M3);
      word[i >> 1] |= (c0 | (c1 << 8)) << (16 * (i & 1));
    }
    unsigned char* dst = static_cast<unsigned char*>(which ? a.v_cache : a.k_cache) +
                         ((blk * a.Hkv + h) * a.block_size + off) * (int64_t)a.D + 8 * c;
    *reinterpret_cast<uint2*>(dst) = make_uint2(word[0], word[1]);
  }
}

__global__ void __launch_bounds__(256) gather_kernel(GatherArgs a) {
  const int cpr = a.row_bytes >> 4;
  const int64_t span = (int64_t)a.MBS * a.block_size;
  const int64_t total = (int64_t)a.B * a.Hkv * span * cpr;
  const int64_t span_max = span;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx % cpr);
    int64_t r = idx / cpr;
    const int64_t j = r % span;
    r /= span;
    const int h = (int)(r % a.Hkv);
    const int b = (int)(r / a.Hkv);
    const int64_t doff = (((int64_t)b * a.Hkv + h) * span + j) * a.row_bytes + 16 * c;
    uint4 kval = make_uint4(0, 0, 0, 0), vval = make_uint4(0, 0, 0, 0);
    const int ctx = a.context_lens[b];
    if (ctx < 0 || ctx > span_max) {
      if (j == 0 && c == 0 && h == 0) raise_error(a.err, kErrContext);
    } else if (j < ctx) {
      const int blk = a.block_tables[(int64_t)b * a.MBS + j / a.block_size];
      if (blk < 0 || blk >= a.NB) {
        if (c == 0) raise_error(a.err, kErrBlock);
      } else {
        const int64_t soff =
            (((int64_t)blk * a.Hkv + h) * a.block_size + j % a.block_size) * a.row_bytes + 16 * c;
        kval = *reinterpret_cast<const uint4*>(static_cast<const char*>(a.k_cache) + soff);
        vval = *reinterpret_cast<const uint4*>(static_cast<const char*>(a.v_cache) + soff);
      }
    }
    *reinterpret_cast<uint4*>(static_cast<char*>(a.k_dense) + doff) = kval;
    *reinterpret_cast<uint4*>(static_cast<char*>(a.v_dense) + doff) = vval;
  }
}

int grid_for(int64_t total, int threads) {
  int64_t g = (total + threads - 1) / threads;
  const int64_t cap = 152 * 32;  // grid-stride beyond this
  return (int)(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace

cudaError_t launch_cache_write(const CacheWriteArgs& a, cudaStream_t stream) {
  const int64_t total = (int64_t)a.T * a.Hkv * 2 * (a.row_bytes >> 4);
  if (total == 0) return cudaSuccess;
  return launch_pdl(cache_write_kernel, dim3(grid_for(total, 256)), dim3(256), 0, stream, a);
}

cudaError_t launch_cache_write_fp8(const CacheWriteFp8Args& a, cudaStream_t stream) {
  const int64_t total = (int64_t)a.T * a.Hkv * 2 * (a.D / 8);
  if (total == 0) return cudaSuccess;
  return launch_pdl(cache_write_fp8_kernel, dim3(grid_for(total, 256)), dim3(256), 0, stream, a);
}

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t stream) {
  const int64_t total = (int64_t)a.B * a.Hkv * a.MBS * a.block_size * (a.row_bytes >> 4);
  if (total == 0) return cudaSuccess;
  gather_kernel<<<grid_for(total, 256), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace photon
