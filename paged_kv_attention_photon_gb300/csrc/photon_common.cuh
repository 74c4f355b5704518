// photon_common.cuh -- internal declarations shared by the CUDA translation
// units of libphoton_paged.so (not part of the public ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace photon {

// Bits of the sticky device error word (see photon_get_last_device_error).
enum : uint32_t { kErrBlock = 1u, kErrSlot = 2u, kErrContext = 4u };

__device__ __forceinline__ void raise_error(uint32_t* word, uint32_t bit) {
  atomicOr(word, bit);
}

// Storage element traits: how one 16-byte chunk widens to fp32 and how fp32
// narrows back for the output row.
template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kPerChunk = 4;
  __device__ __forceinline__ static void widen(const uint4& c, float* f) {
    f[0] = __uint_as_float(c.x);
    f[1] = __uint_as_float(c.y);
    f[2] = __uint_as_float(c.z);
    f[3] = __uint_as_float(c.w);
  }
  __device__ __forceinline__ static float narrow(float x) { return x; }
};

template <>
struct Elem<__half> {
  static constexpr int kPerChunk = 8;
  __device__ __forceinline__ static void widen(const uint4& c, float* f) {
    const __half2* h = reinterpret_cast<const __half2*>(&c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __half22float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ __forceinline__ static __half narrow(float x) { return __float2half_rn(x); }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kPerChunk = 8;
  __device__ __forceinline__ static void widen(const uint4& c, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ __forceinline__ static __nv_bfloat16 narrow(float x) { return __float2bfloat16_rn(x); }
};

// Streaming 16-byte global load that bypasses L1 allocation: every K/V byte
// of a decode step is read exactly once.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ------------------------------------------------------------------ launches
struct DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* out;
  float* ws_m;      // [B][Hq][pmax]   running max (log2 domain) per partition
  float* ws_l;      // [B][Hq][pmax]   sum of weights per partition
  float* ws_o;      // [B][Hq][pmax][D] unnormalised weighted V sum per partition
  uint32_t* err;    // sticky device error word
  float qscale;     // scale * log2(e): scores are kept in the log2 domain
  int B, Hq, Hkv, D, NB, MBS, part, pmax;
  cudaEvent_t ev_start, ev_stop;  // optional timing hook around the split kernel
};

struct CacheWriteArgs {
  const void* k;
  const void* v;
  const int64_t* slot_mapping;
  void* k_cache;
  void* v_cache;
  uint32_t* err;
  int T, Hkv, row_bytes, block_size, NB;
};

struct GatherArgs {
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* k_dense;
  void* v_dense;
  uint32_t* err;
  int B, Hkv, row_bytes, block_size, NB, MBS;
};

cudaError_t launch_cache_write(const CacheWriteArgs& a, cudaStream_t stream);
cudaError_t launch_gather(const GatherArgs& a, cudaStream_t stream);

// One entry per storage dtype; each returns cudaErrorInvalidValue for a
// (head_dim, group) pair that is not instantiated.
cudaError_t launch_paged_decode_f32(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_paged_decode_f16(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_paged_decode_bf16(const DecodeArgs& a, cudaStream_t stream);

// Block size, partition bounds and threads per CTA of the decode kernels.
constexpr int kBlockSize = 16;
constexpr int kDecodeWarps = 4;
constexpr int kMergeWarps = 4;

}  // namespace photon
