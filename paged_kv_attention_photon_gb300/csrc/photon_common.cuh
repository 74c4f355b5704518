// photon_common.cuh -- internal declarations shared by the CUDA translation
// units of libphoton_paged.so (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace photon {

// Bits of the sticky device error word (see photon_get_last_device_error).
enum : uint32_t {
  kErrBlock = 1u, kErrSlot = 2u, kErrContext = 4u, kErrPosition = 16u, kErrQuery = 32u
};

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
  __device__ __forceinline__ static float to_f32(float x) { return x; }
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
  __device__ __forceinline__ static float to_f32(__half x) { return __half2float(x); }
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
  __device__ __forceinline__ static float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
};

// PHOTON_FAST_EXP selects the PTX ex2.approx.ftz instruction (relative error
// about 2^-22; results below 2^-126 flush to zero) for the softmax weights
// instead of the exp2f library call.
#ifndef PHOTON_FAST_EXP
#define PHOTON_FAST_EXP 1
#endif

__device__ __forceinline__ float softmax_exp2(float x) {
#if PHOTON_FAST_EXP
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
#else
  return exp2f(x);
#endif
}

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
// One partition p of sequence b (the KV head is added by the kernel):
// tokens [tok_begin, tok_end); nparts is the number of partitions of the
// sequence.
struct WorkItem {
  int b, p, tok_begin, tok_end, nparts, ctx;
  int q0, nq;  // few-token multi-query mode: the sequence's first query row and count
};

struct DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* out;
  float* ws_m;        // [B][Hq][pmax]    running max (log2 domain) per partition
  float* ws_l;        // [B][Hq][pmax]    sum of weights per partition
  float* ws_o;        // [B][Hq][pmax][D] unnormalised weighted V sum per partition
  unsigned long long* ws_ctrl;  // work-queue control: [0] guard word, [1] queue counter
  // Fused step only (all null otherwise): row b of k_new / v_new is sequence
  // b's new token at position ctx_b - 1; the attention kernel attends over it
  // and writes it to its cache slot.
  const void* k_new;
  const void* v_new;
  const int64_t* slot_mapping;
  void* k_cache_w;
  void* v_cache_w;
  // Fused step with RoPE only (null otherwise): (cos, sin) per position and
  // pair, [rope_max_pos][D/2]; q rows and the new K rows turn by ctx - 1.
  const float2* rope_cs;
  int rope_max_pos;
  // Few-token multi-query mode only (null otherwise): sequence b's query
  // tokens are rows query_start[b] .. query_start[b+1]-1 of q and out, the
  // last ones of its context (token i at position ctx - n + i, attending to
  // keys 0 .. that position); max_q bounds their count, max_q * G <= 8; the
  // workspace partials are per (token row, q head, partition).
  const int32_t* query_start;
  int max_q, num_tokens;
  uint32_t* err;      // sticky device error word
  float qscale;       // scale * log2(e): scores are kept in the log2 domain
  float v_scale;      // e4m3 cache only: the V scale (applied in each item's combine)
  int B, Hq, Hkv, D, NB, MBS, part, pmax;
  int num_sms;        // SMs of the current device
  cudaEvent_t ev_start, ev_stop;  // optional timing hook around the decode kernels
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

// Quantising cache write into an e4m3 cache: row t of k / v (fp16) is stored
// at slot_mapping[t] as the codes of x * inv_scale (fp32 product, round to
// nearest even, saturating at +-448).
struct CacheWriteFp8Args {
  const void* k;
  const void* v;
  const int64_t* slot_mapping;
  void* k_cache;
  void* v_cache;
  uint32_t* err;
  float k_inv, v_inv;
  int T, Hkv, D, block_size, NB;
};
cudaError_t launch_cache_write_fp8(const CacheWriteFp8Args& a, cudaStream_t stream);

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
cudaError_t launch_rope_table(double base, int max_pos, int d, float2* table,
                              cudaStream_t stream);
cudaError_t launch_gather(const GatherArgs& a, cudaStream_t stream);

// One entry per storage dtype; each returns cudaErrorInvalidValue for a
// (head_dim, group) pair that is not instantiated.
// Decode consumer selection (photon_debug_set_decode_consumer): 0 by group
// size, 1 CUDA-core consumer, 2 tensor-core consumer (16-bit storage only).
extern std::atomic<int> g_decode_consumer;

cudaError_t launch_paged_decode_f32(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_paged_decode_f16(const DecodeArgs& a, cudaStream_t stream);
// e4m3 K/V cache, fp16 q and out (photon_paged_decode_fp8): a.qscale holds
// scale * k_scale * log2(e), a.v_scale the V scale.
cudaError_t launch_paged_decode_fp8(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_paged_decode_bf16(const DecodeArgs& a, cudaStream_t stream);

// Multi-query (causal) paged attention: query_start[b] .. query_start[b+1]-1
// are sequence b's new query tokens, the last ones of its context.
struct MultiQueryArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;
  void* out;
  uint32_t* err;
  float qscale;       // scale * log2(e)
  int B, Hq, Hkv, D, NB, MBS, max_query_len;
  int num_tokens;     // rows of q and out
  int dtype;          // 1 = fp16, 2 = bf16
  // split-KV: each tile's keys are cut into partitions of `part` keys (a
  // multiple of 64); pmax partitions per row at most.  pmax == 1: no split,
  // no workspace.  Otherwise partials [num_tokens][Hq][pmax] (m, l) and
  // [...][D] (o), merged by a second kernel.
  int part, pmax;
  float* ws_m;
  float* ws_l;
  float* ws_o;
};
cudaError_t launch_multi_query(const MultiQueryArgs& a, cudaStream_t stream);
// The same operation on tcgen05 / TMEM tiles of 128 rows (no key split).
cudaError_t launch_multi_query_tc(const MultiQueryArgs& a, cudaStream_t stream);


// Launch with programmatic stream serialization: the kernel may be scheduled
// while its predecessor in the stream finishes and must call
// pdl_wait_primary() before touching memory the predecessor writes.
template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kBlockSize = 16;
// Guard value the merge kernel leaves in ws_ctrl[0] after resetting the
// queue counter; any other value (a fresh workspace) makes the attention
// kernel hand items out statically for that call.
constexpr unsigned long long kQueueReady = 0x70686f746f6e5131ull;

}  // namespace photon

// ------------------------------------------------------------------ PTX helpers
namespace photon {

enum : uint32_t { kErrTimeout = 8u };
// A bounded wait gives up after this long (ns of %globaltimer), flags
// kErrTimeout and lets the kernel unwind instead of hanging.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t tx_bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(tx_bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete; false after
// kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`
// (both addresses 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// L2 policy for data read exactly once (the K/V stream of a decode): evict
// first, so that it does not push out what is read again soon (the split-KV
// partials the merge reads).  A hint only: no effect on values.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk copy with an L2 cache policy (see bulk_copy_g2s).
__device__ __forceinline__ void bulk_copy_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                                   uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Hint: bring a line into L2 (no architectural effect on values).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Programmatic dependent launch controls (no-ops without the launch attribute).
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ tensor copies and warp MMA
// Tensor map over a K or V pool seen as rows of head_dim elements:
// (num_blocks x Hkv x 16) rows; dtype 1 = fp16, 2 = bf16: box 16 rows x 64
// elements, 128-byte swizzle; dtype 3 = e4m3 codes: box 16 rows x head_dim
// codes, 128-byte swizzle at head_dim 128, 64-byte at 64.  Defined in
// multi_query_tc.cu.
cudaError_t make_pool_map(CUtensorMap* map, const void* pool, int dtype, int NB, int Hkv, int D);

// 2-D tiled bulk tensor copy of one box into this CTA's shared memory,
// completing on `bar`.
__device__ __forceinline__ void tma_load_box(uint32_t dst, const CUtensorMap* map, int x, int y,
                                             uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// tma_load_box with an L2 cache policy.
__device__ __forceinline__ void tma_load_box_hint(uint32_t dst, const CUtensorMap* map, int x,
                                                  int y, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Brings a tensor map (a __grid_constant__ kernel parameter) into the copy
// unit's descriptor cache ahead of its first use.  A hint only.
__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Warp-level tensor-core product D += A B (m16n8k16, fp32 accumulate) and the
// packing of two fp32 values into one operand register of the storage type.
template <typename T>
struct Mma;

template <>
struct Mma<__half> {
  __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  // the two halves of a packed register back in fp32
  __device__ __forceinline__ static float2 unpack(uint32_t v) {
    return __half22float2(*reinterpret_cast<const __half2*>(&v));
  }
};

template <>
struct Mma<__nv_bfloat16> {
  __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static float2 unpack(uint32_t v) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
  }
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Transpose of an 8x8 matrix of 16-bit elements held in the warp's fragment
// layout (lane l: row l/4, columns 2(l%4) and 2(l%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

}  // namespace photon
