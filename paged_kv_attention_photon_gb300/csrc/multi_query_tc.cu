// multi_query_tc.cu -- the multi-query causal paged attention on the fifth-
// generation tensor cores: tcgen05.mma with operands in shared memory and the
// accumulators in tensor memory (TMEM).  Same operation and arguments as the
// warp-level kernel in multi_query.cu; used for query batches large enough
// to fill the device without a key split (chunked prefill).
//
// PhotonInfer README: "Technical details / Paged attention" (block-wise KV
// cache, per-sequence offsets) and "Roadmap" (FlashAttention-2 style IO-aware
// attention for long sequences).
//
// A CTA owns 256 query rows of one (sequence, KV head) as two tiles of 128
// and runs 14 warps in fixed roles: 8 softmax warps (4 per tile), a K copy
// warp, a V copy warp, and per tile an S-issuing and a P V-issuing MMA warp.
// Row r of a tile is (token r / G, head r % G of the KV head's group) and
// lives in TMEM lane r, so thread r of the tile's softmax warps owns row r
// from the scores to the output: the softmax needs no shuffles.  Per chunk of
// kTcKeys keys:
//   K, V     2-D tensor-map copies (boxes of 16 rows x 64 elements, 128-byte
//            swizzle) straight from the paged pool through the block table,
//            into a K ring and a V ring
//   S = Q K^T    D/16 MMAs per tile (M=128, N=kTcKeys, K=16), fp32 in TMEM,
//                128 / kTcKeys S buffers per tile
//   softmax  each thread loads its scores (tcgen05.ld), masks the keys after
//            its position, updates (m, l), and writes its weights P as
//            fp16/bf16 pairs back over the first half of the same S buffer
//            (tcgen05.st)
//   O += P V     kTcKeys/16 MMAs per tile (M=128, N=D, K=16) with A (= P)
//                read from TMEM, accumulating in TMEM; V is an MN-major
//                operand read from the same swizzled rows as K
// The running maximum only moves when a new score exceeds it by more than
// 2^8 (log2 domain), and only then is the TMEM accumulator rescaled: between
// rescales the weights use a stale maximum, which the final O / l cancels
// exactly, and a weight stays below 2^8, far inside fp16/bf16 range.
//
// Operands are K-major with the 128-byte swizzle: a tile of R rows and 64
// 16-bit elements per row is R/8 atoms of 8 rows x 128 bytes, 16-byte chunk c
// of row r stored at chunk c ^ (r % 8); rows past 64 elements continue in the
// next 64-element block of R x 128 bytes.  The Q tiles are loaded once per
// CTA with cp.async into the same layout.
//
// CTAs start in the order of their linear index, which is mapped onto the
// (sequence, KV head, tile) items sorted by the length of their causal key
// range, longest first (tc_item_of).
#include <cuda.h>

#include <type_traits>

#include "photon_common.cuh"

namespace photon {
namespace {

constexpr int kTcRows = 128;    // query rows per CTA = TMEM lanes
constexpr int kTcThreads = 128;
// Keys per chunk (tuning knob: 64 or 32).  A tile's S buffers fill columns
// [0, 128) of its TMEM, so there are 128 / kTcKeys of them.
#ifndef PHOTON_TC_KEYS
#define PHOTON_TC_KEYS 64
#endif
constexpr int kTcKeys = PHOTON_TC_KEYS;
static_assert(kTcKeys == 32 || kTcKeys == 64, "chunks of 32 or 64 keys");
constexpr int kNumS = 128 / kTcKeys;   // S buffers per tile; chunk c uses buffer c % kNumS
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemS = 0;     // S buffers: columns [0, 128)
constexpr uint32_t kTmemO = 128;   // O: columns [128, 128 + D)
constexpr float kRescaleLog2 = 8.f;

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);  // start address
  d |= (uint64_t)1 << 16;                  // leading byte offset (unused when swizzled)
  d |= (uint64_t)(1024 >> 4) << 32;        // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                  // descriptor version
  d |= (uint64_t)2 << 61;                  // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: fp32 accumulate, A and B of type T, both
// K-major, M x N.
template <typename T>
__device__ __forceinline__ uint32_t f16_idesc(int M, int N) {
  constexpr uint32_t fmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// One tcgen05.mma (D += A B, kind::f16, A and B from shared-memory
// descriptors, accumulate unless `accumulate` is 0), executed by the whole
// (converged) warp with the product issued only where `issue` is nonzero:
// the operand descriptors stay warp-uniform, and no branch separates the
// issuing lane from the rest of the warp.
__device__ __forceinline__ void tc_mma_warp(uint32_t d_tmem, uint64_t a, uint64_t b,
                                            uint32_t idesc, uint32_t accumulate, uint32_t issue) {
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.b32 p, %4, 0;\nsetp.ne.b32 q, %5, 0;\n"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(issue));
}
// The same with A in tensor memory (a_tmem: lane 0 of the operand's 128
// rows, first column; 16-bit elements packed two per column, the lower k in
// the low half).
__device__ __forceinline__ void tc_mma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                               uint32_t idesc, uint32_t accumulate,
                                               uint32_t issue) {
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.b32 p, %4, 0;\nsetp.ne.b32 q, %5, 0;\n"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate), "r"(issue));
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane.  The wait sits in
// the same asm statement as the load, so no use of the registers can be
// scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 64 consecutive columns: two loads in flight, one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr), "r"(taddr + 32)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Softmax arithmetic on Blackwell's paired fp32 instructions (tuning knobs):
// PHOTON_TC_PACKED: the exponent arguments and the row sum two lanes per
// instruction (fma/add .f32x2, each lane rounded as the scalar form);
// PHOTON_TC_FMAX3: the row maximum with three-input max.
#ifndef PHOTON_TC_PACKED
#define PHOTON_TC_PACKED 1
#endif
#ifndef PHOTON_TC_FMAX3
#define PHOTON_TC_FMAX3 1
#endif
// (d0, d1) = (a0 * b + c, a1 * b + c), one rounding per lane
__device__ __forceinline__ void fma_f32x2(float& d0, float& d1, float a0, float a1, float b,
                                          float c) {
  asm("{\n.reg .b64 ra, rb, rc, rd;\nmov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %4};\n"
      "mov.b64 rc, {%5, %5};\nfma.rn.f32x2 rd, ra, rb, rc;\nmov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// (d0, d1) += (a0, a1)
__device__ __forceinline__ void add_f32x2(float& d0, float& d1, float a0, float a1) {
  asm("{\n.reg .b64 ra, rb, rd;\nmov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %5};\n"
      "add.rn.f32x2 rd, ra, rb;\nmov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(d0), "f"(d1), "f"(a0), "f"(a1));
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// The weights of one row's chunk against the maximum m (log2 domain):
// p_j = 2^(s_j * qmul - m), packed as 16-bit pairs into w (key 2j in the low
// half of w[j]); returns their fp32 sum.
template <typename T>
__device__ __forceinline__ float tc_weights(const float (&s)[kTcKeys], float qmul, float m,
                                            float (&w)[kTcKeys / 2]) {
  float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kTcKeys / 2; ++j) {
    float x0, x1;
#if PHOTON_TC_PACKED
    fma_f32x2(x0, x1, s[2 * j], s[2 * j + 1], qmul, -m);
#else
    x0 = fmaf(s[2 * j], qmul, -m);
    x1 = fmaf(s[2 * j + 1], qmul, -m);
#endif
    const float p0 = softmax_exp2(x0), p1 = softmax_exp2(x1);
#if PHOTON_TC_PACKED
    add_f32x2(sum4[(j & 1) * 2], sum4[(j & 1) * 2 + 1], p0, p1);
#else
    sum4[j & 3] += p0 + p1;
#endif
    uint32_t bits;
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
      __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
      bits = *reinterpret_cast<uint32_t*>(&h);
    } else {
      __half2 h = __floats2half2_rn(p0, p1);
      bits = *reinterpret_cast<uint32_t*>(&h);
    }
    w[j] = __uint_as_float(bits);
  }
  return (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
}

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Byte offset of 16-byte chunk c (of the row's D/8) of row r in a K-major
// 128-byte-swizzled tile of R rows.
template <int R>
__device__ __forceinline__ uint32_t sw_chunk(int r, int c) {
  return (uint32_t)((c >> 3) * (R * 128) + (r >> 3) * 1024 + (r & 7) * 128 +
                    (((c & 7) ^ (r & 7)) << 4));
}

// Shared-memory plan of the warp-specialised kernel: two Q tiles of 128 rows,
// then a K ring and a V ring of chunks (filled by the tensor memory
// accelerator).  Ring depths are tuning knobs; measured on the 16 x 1024
// prefill while P still went through shared memory: 3 + 3 stages 0.392 ms,
// 4 K + 2 V 0.394 ms, 5 K + 1 V 0.595 ms.
#ifndef PHOTON_TC_KSTAGES
#define PHOTON_TC_KSTAGES (PHOTON_TC_KEYS == 64 ? 3 : 6)
#endif
#ifndef PHOTON_TC_VSTAGES
#define PHOTON_TC_VSTAGES (PHOTON_TC_KEYS == 64 ? 3 : 6)
#endif
template <typename T, int D>
struct TcCfg {
  static constexpr int kTiles = 2;
  static constexpr int kKStages = PHOTON_TC_KSTAGES;   // K ring: a stage is free once S of its chunk is done
  static constexpr int kVStages = PHOTON_TC_VSTAGES;   // V ring: free once the P V product of its chunk is done
  static constexpr int kQBytes = kTcRows * D * 2;     // one Q tile
  static constexpr int kKBytes = kTcKeys * D * 2;     // one K chunk
  static constexpr int kVBytes = kTcKeys * D * 2;     // one V chunk

  static constexpr int kOffQ = 0;                               // [kTiles]
  static constexpr int kOffK = kOffQ + kTiles * kQBytes;        // [kKStages]
  static constexpr int kOffV = kOffK + kKStages * kKBytes;      // [kVStages]
  static constexpr int kUsed = kOffV + kVStages * kVBytes;
  static constexpr int kSmem = kUsed + 1024;   // + alignment of the base to a swizzle atom
  // softmax warps, then the K copy warp, the V copy warp, and per tile an
  // S-issuing and a P V-issuing warp
  static constexpr int kThreads = kTiles * kTcThreads + 64 + kTiles * 64;
};

// MN-major (V) operand: the same 128-byte-swizzled rows of 64 elements as the
// K-major tiles, but the MMA walks N along a row: 64-element blocks of N are
// 64 keys x 128 B = 8 KB apart (leading byte offset), groups of 8 keys 1 KB
// apart (stride byte offset).
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((kTcKeys * 128) >> 4) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar) { mbar_arrive(bar); }

// Work class of the CTA of (sequence b, tile): 1 + floor(log2(key chunks))
// for a CTA with rows, 0 for one without (or one whose arguments the kernel
// rejects, which only writes zero rows).
template <int kSuperRows>
__device__ __forceinline__ int tc_work_class(const MultiQueryArgs& a, int b, int tile, int G) {
  const int q0 = __ldg(a.query_start + b);
  const int n = __ldg(a.query_start + b + 1) - q0;
  const int ctx = __ldg(a.context_lens + b);
  if (n <= 0 || q0 < 0 || q0 + n > a.num_tokens || n > a.max_query_len || ctx < n ||
      ctx > a.MBS * kBlockSize)
    return 0;
  const int row0 = tile * kSuperRows;
  const int rows = min(kSuperRows, n * G - row0);
  if (rows <= 0) return 0;
  const int kend = ctx - n + (row0 + rows - 1) / G + 1;
  const int chunks = (kend + kTcKeys - 1) / kTcKeys;
  return 32 - __clz(chunks);
}

// The (sequence, KV head, tile) of this CTA.  CTAs are started in the order
// of their linear index, so the index is mapped onto the items sorted by
// work class, largest first (the longest causal key ranges start first and
// the short ones fill in behind them); inside a class the natural order
// (sequence, KV head, tile) keeps the tiles of one sequence's KV head
// together, so its K/V rows are read from HBM once and then hit L2.  Every
// thread of the CTA takes part; the scratch is shared memory.
template <int kSuperRows>
__device__ __forceinline__ void tc_item_of(const MultiQueryArgs& a, int G, int& b_out,
                                           int& kvh_out, int& tile_out, int* hist, int* wsum,
                                           int* sel) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x, nwarps = (nthr + 31) / 32;
  const int T = gridDim.x, B = a.B, H = a.Hkv;
  const int L = (int)((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x);
  for (int i = tid; i < 33; i += nthr) hist[i] = 0;
  __syncthreads();
  for (int p = tid; p < B * T; p += nthr)
    atomicAdd(&hist[tc_work_class<kSuperRows>(a, p / T, p % T, G)], 1);
  __syncthreads();
  if (tid == 0) {
    int acc = 0, C = 0, j = 0;
    for (int c = 32; c >= 0; --c) {
      const int items = hist[c] * H;
      if (L < acc + items) {
        C = c;
        j = L - acc;
        break;
      }
      acc += items;
    }
    sel[0] = C;
    sel[1] = j;
  }
  __syncthreads();
  const int C = sel[0], j = sel[1];
  // items of class C in natural order: find the sequence by a running
  // (chunked) block scan of its item count
  int carry = 0;
  for (int base = 0; base < B; base += nthr) {
    const int b = base + tid;
    int cnt = 0;
    if (b < B)
      for (int t = 0; t < T; ++t) cnt += tc_work_class<kSuperRows>(a, b, t, G) == C ? 1 : 0;
    const int items = cnt * H;
    int v = items;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int w = lane < nwarps ? wsum[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < nwarps) wsum[32 + lane] = w;   // inclusive over warps
    }
    __syncthreads();
    const int excl = carry + (warp > 0 ? wsum[32 + warp - 1] : 0) + v - items;
    if (items > 0 && j >= excl && j < excl + items) {
      const int r = j - excl;
      int k = r % cnt;
      int tile = 0;
      for (int t = 0; t < T; ++t) {
        if (tc_work_class<kSuperRows>(a, b, t, G) != C) continue;
        if (k-- == 0) {
          tile = t;
          break;
        }
      }
      sel[2] = b;
      sel[3] = r / cnt;
      sel[4] = tile;
    }
    carry += wsum[32 + nwarps - 1];
    __syncthreads();
  }
  b_out = sel[2];
  kvh_out = sel[3];
  tile_out = sel[4];
}

#ifdef PHOTON_PROBE
// Tuning builds only (never compiled into the library by default): the
// per-chunk timeline of one CTA (the last tile of KV head 0 of the last
// sequence) and the start and end of every CTA.
constexpr int kTcProbeChunks = 160;
static __device__ unsigned long long g_tc_probe[kTcProbeChunks][20];
static __device__ unsigned long long g_tc_cta[4096][2];
#define TC_PROBE(c, i)                                                                \
  do {                                                                               \
    if (probe_cta && (c) < kTcProbeChunks) g_tc_probe[c][i] = global_timer_ns();      \
  } while (0)
#else
#define TC_PROBE(c, i) do { } while (0)
#endif

// Warp roles: a CTA owns 256 query rows of one (sequence, KV head) as two
// tiles of 128.  Warps 0-3 own tile 0 and warps 4-7 tile 1 (thread r of a
// tile: TMEM lane r of that tile's columns): softmax, O rescale, epilogue.
// Warp 8 copies K and warp 9 copies V: each one's lane 0 issues the bulk
// tensor copies of a chunk as soon as a stage of its ring is free.  The two
// rings are separate because their stages are held for different spans: a
// K chunk only until S of its chunk is computed, a V chunk until the P V
// product, after the softmax; with one ring for both, the copy latency of
// every chunk sat on the chain through the softmax.  Warps 10 and 11 issue
// the S products of tiles 0 and 1, warps 12 and 13 their P V products (lane
// 0 of each), so four instruction streams feed the tensor cores (one thread
// issuing every MMA took about twice the tensor cores' execution time per
// chunk); warp 12's lanes also zero the V rows that lie past the last key.
// Both tiles use every K/V chunk, so each chunk is fetched once for 256 rows.
// TMEM: tile t owns columns [256 t, 256 t + 256): the S buffers in [0, 128),
// then O.  P of a chunk overwrites the first half of its own S buffer, so S
// of chunk c + kNumS, which reuses the buffer, waits for the P V product of
// chunk c.
// Barriers (each completes once per use; a use's parity is its index & 1):
//   k_full[s], v_full[s]  K (V) of a chunk landed in stage s (copy transaction bytes)
//   k_free[s]      the S products reading K stage s finished (one commit per MMA warp)
//   v_free[s]      the P V products reading V stage s finished (one commit per MMA warp)
//   v_zeroed[s]    warp 12 zeroed the V rows of stage s past the last key
//   s_full[t][b]   S of a chunk is in tile t's TMEM buffer b (MMA commit)
//   p_full[t][b]   tile t's P of that chunk is in buffer b (4 softmax warp arrivals)
//   p_done[t][b]   the P V product reading buffer b finished (MMA commit)
// The b-indexed barriers serve chunks b, b + kNumS, ...: chunk c's use of one
// has parity (c / kNumS) & 1.
template <typename T, int D>
__global__ void __launch_bounds__(TcCfg<T, D>::kThreads)
    paged_multi_query_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                                const __grid_constant__ CUtensorMap tm_v, const MultiQueryArgs a) {
  using C = TcCfg<T, D>;
  constexpr int SK = C::kKStages, SV = C::kVStages;
  constexpr int NT = C::kTiles;
  constexpr int kSuper = NT * kTcRows;
  extern __shared__ unsigned char tc_smem_raw[];
  __shared__ __align__(8) uint64_t k_full[SK], k_free[SK], v_full[SV], v_free[SV],
      s_full[NT][kNumS], p_full[NT][kNumS], p_done[NT][kNumS], v_zeroed[SV];
  __shared__ uint32_t tmem_slot;
  __shared__ int tail_rows[SV];   // per V stage: first V row to zero (kTcKeys = none)
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t sQ = sbase + C::kOffQ, sK = sbase + C::kOffK, sV = sbase + C::kOffV;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.Hq / a.Hkv;
#ifdef PHOTON_PROBE
  const int cta_lin = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
  if (tid == 0 && cta_lin < 4096) g_tc_cta[cta_lin][0] = global_timer_ns();
#endif
  __shared__ int ord_hist[33], ord_wsum[64], ord_sel[5];
  int b, kvh, tile;
  tc_item_of<kSuper>(a, G, b, kvh, tile, ord_hist, ord_wsum, ord_sel);
#ifdef PHOTON_PROBE
  const bool probe_cta = cta_lin == 0;   // the first CTA started: the largest class
#endif
  const int q0 = __ldg(a.query_start + b);
  const int n = __ldg(a.query_start + b + 1) - q0;
  const int ctx = __ldg(a.context_lens + b);
  const int row0 = tile * kSuper;
  const T* qg = static_cast<const T*>(a.q);
  T* outg = static_cast<T*>(a.out);

  if (n <= 0 || q0 < 0 || q0 + n > a.num_tokens) {
    if ((n < 0 || q0 < 0 || q0 + n > a.num_tokens) && tile == 0 && kvh == 0 && tid == 0)
      raise_error(a.err, kErrQuery);
    return;
  }
  if (n > a.max_query_len || ctx < n || ctx > a.MBS * kBlockSize) {
    if (tile == 0 && kvh == 0 && tid == 0)
      raise_error(a.err, n > a.max_query_len ? kErrQuery : kErrContext);
    const int rows = min(kSuper, max(0, min(n, a.max_query_len) * G - row0));
    for (int p = tid; p < rows * (D / 8); p += C::kThreads) {
      const int r = row0 + p / (D / 8), ch = p % (D / 8);
      T* dst = outg + ((size_t)(q0 + r / G) * a.Hq + kvh * G + r % G) * D + ch * 8;
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const int rows_here = min(kSuper, n * G - row0);   // rows of the CTA, tile 0 first
  if (rows_here <= 0) return;
  const int ntiles = (rows_here + kTcRows - 1) / kTcRows;   // tiles with rows: 1 or 2
  const int first_pos = ctx - n;
  const int kend = first_pos + (row0 + rows_here - 1) / G + 1;   // keys [0, kend)
  const int nchunks = (kend + kTcKeys - 1) / kTcKeys;

  // ---- setup: barriers, TMEM, the Q tiles (rows past the CTA's rows zero)
  if (tid == 0) {
    for (int i = 0; i < SK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_free[i], NT);   // one commit per tile's MMA warp
    }
    for (int i = 0; i < SV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_free[i], NT);
      mbar_init(&v_zeroed[i], 1);
    }
    for (int t = 0; t < NT; ++t) {
      for (int i = 0; i < kNumS; ++i) {
        mbar_init(&s_full[t][i], 1);
        mbar_init(&p_full[t][i], 4);   // one arrival per softmax warp of the tile
        mbar_init(&p_done[t][i], 1);
      }
    }
    mbar_init_fence();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_slot)),
                 "r"(NT * kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  for (int p = tid; p < kSuper * (D / 8); p += C::kThreads) {
    const int r = p / (D / 8), ch = p % (D / 8);
    const bool valid = r < rows_here;
    const int rr = row0 + r;
    const T* src = valid ? qg + ((size_t)(q0 + rr / G) * a.Hq + kvh * G + rr % G) * D + ch * 8 : qg;
    cp_async16_zfill(sQ + (r / kTcRows) * C::kQBytes + sw_chunk<kTcRows>(r % kTcRows, ch), src,
                     valid);
  }
  cp_async_wait_all();
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;

  auto lane0_ok = [&](bool v) { return __shfl_sync(0xffffffffu, v ? 1 : 0, 0) != 0; };
  if (warp == NT * 4 || warp == NT * 4 + 1) {
    // ================================================================ copies
    // warp NT*4: K chunks into the K ring; warp NT*4 + 1: V chunks into the V ring
    const bool is_v = warp == NT * 4 + 1;
    const int nst = is_v ? SV : SK;
    uint64_t* full = is_v ? v_full : k_full;
    uint64_t* freed = is_v ? v_free : k_free;
    const CUtensorMap* map = is_v ? &tm_v : &tm_k;
    const uint32_t ring = is_v ? sV : sK;
    const int32_t* table = a.block_tables + (size_t)b * a.MBS;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int st = c % nst;
      if (c >= nst) {   // the stage's previous chunk, c - nst, has been consumed
        ok = lane0_ok(mbar_wait_bounded(&freed[st], ((c / nst) - 1) & 1));
        if (!ok) break;
      }
      if (lane != 0) continue;
      uint32_t bytes = 0;
      int tail = kTcKeys;
      constexpr int kBlocks = kTcKeys / kBlockSize;   // pool blocks per chunk
      int phys[kBlocks];
#pragma unroll
      for (int i = 0; i < kBlocks; ++i) {
        const int kb = c * kBlocks + i;   // 16-key block of the sequence
        phys[i] = -1;
        if (kb * kBlockSize < kend) {
          const int p = __ldg(table + kb);
          if (p >= 0 && p < a.NB) {
            phys[i] = p;
            bytes += kBlockSize * D * 2u;
          } else if (!is_v) {
            raise_error(a.err, kErrBlock);
          }
        }
        // rows to zero: past kend, or a whole skipped block
        const int valid_rows = phys[i] < 0 ? 0 : min(kBlockSize, kend - kb * kBlockSize);
        if (valid_rows < kBlockSize && tail == kTcKeys) tail = i * kBlockSize + valid_rows;
      }
      if (is_v) tail_rows[st] = tail;   // published by the barrier's arrive below
      if (!is_v) TC_PROBE(c, 6);
      mbar_arrive_expect_tx(&full[st], bytes);
#pragma unroll
      for (int i = 0; i < kBlocks; ++i) {
        if (phys[i] < 0) continue;
        const int y = (phys[i] * a.Hkv + kvh) * kBlockSize;
#pragma unroll
        for (int h = 0; h < D / 64; ++h)
          tma_load_box(ring + st * C::kKBytes + h * (kTcKeys * 128) + i * 2048, map, h * 64, y,
                       &full[st]);
      }
    }
    if (!ok && lane == 0) raise_error(a.err, kErrTimeout);
  } else if (warp >= NT * 4 + 2) {
    // ================================================================ MMAs
    // per tile one warp issues the S products and one the P V products (lane
    // 0 issues): the four streams go out in parallel, and each waits only for
    // what its own products need
    const int t = (warp - (NT * 4 + 2)) & (NT - 1);
    const bool issues_s = warp - (NT * 4 + 2) < NT;
    const bool tile_used = t < ntiles;
    const uint32_t id_s = f16_idesc<T>(kTcRows, kTcKeys);
    const uint32_t id_o = f16_idesc<T>(kTcRows, D) | (1u << 16);   // B (V) MN-major
    // Operand descriptors, built once: a descriptor's start-address field
    // holds address >> 4 in its low 14 bits, and every operand here lies
    // below 256 KB of the shared window, so the descriptor of base + off is
    // the base's descriptor plus off >> 4 (no carry leaves the field).  Each
    // MMA then costs one add per operand instead of a rebuilt descriptor.
    const uint64_t qa = sw128_desc(sQ) + (uint64_t)((t * C::kQBytes) >> 4);
    const uint64_t k_desc = sw128_desc(sK), v_desc = sw128_mn_desc(sV);
    uint32_t zero_phase = 0;   // bit s: parity of V stage s's next zeroing (both P V warps alike)
    for (int c = 0; c <= nchunks && ok; ++c) {
      if (issues_s && c < nchunks) {
        const int st = c % SK;
        ok = lane0_ok(mbar_wait_bounded(&k_full[st], (c / SK) & 1));
        if (!ok) break;
        if (lane == 0 && t == 0) TC_PROBE(c, 7);
        if (tile_used) {
          if (c >= kNumS) {
            // buffer c % kNumS holds P of chunk c - kNumS until its P V product is done
            ok = lane0_ok(mbar_wait_bounded(&p_done[t][c % kNumS], ((c - kNumS) / kNumS) & 1));
            if (!ok) break;
          }
          if (lane == 0 && t == 0) TC_PROBE(c, 4);
          tc_fence_after();
          const uint64_t kb = k_desc + (uint64_t)((st * C::kKBytes) >> 4);
          const uint32_t dst = tmem + t * kTmemCols + kTmemS + (c % kNumS) * kTcKeys;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk & 3) * 32;
            tc_mma_warp(dst, qa + (uint64_t)(((kk >> 2) * (kTcRows * 128) + koff) >> 4),
                        kb + (uint64_t)(((kk >> 2) * (kTcKeys * 128) + koff) >> 4), id_s, kk > 0,
                        lane == 0);
          }
          if (lane == 0) {
            tc_commit(&s_full[t][c % kNumS]);
            TC_PROBE(c, 8 + t);
          }
        }
        if (lane == 0) tc_commit(&k_free[st]);   // this tile's S of the K stage are done
      }
      if (!issues_s && c >= 1) {
        // P V of the previous chunk, once its V landed and its weights are written
        const int pc = c - 1, pst = pc % SV, pb = pc % kNumS;
        if (lane == 0 && t == 0) TC_PROBE(pc, 10);
        ok = lane0_ok(mbar_wait_bounded(&v_full[pst], (pc / SV) & 1));
        if (!ok) break;
        if (lane == 0 && t == 0) TC_PROBE(pc, 11);
        // zero the V rows past the last key (a partial or missing block):
        // they are multiplied by zero weights, and 0 x NaN would not vanish.
        // Tile 0's P V warp writes the zeros and signals v_zeroed; tile 1's
        // waits for it before its products read the stage.
        const int tail = tail_rows[pst];
        if (tail < kTcKeys) {
          if (t == 0) {
            unsigned char* vt = smem + C::kOffV + pst * C::kVBytes;
            for (int p = lane; p < (kTcKeys - tail) * (D / 8); p += 32) {
              const int r = tail + p / (D / 8), ch = p % (D / 8);
              *reinterpret_cast<uint4*>(vt + sw_chunk<kTcKeys>(r, ch)) = make_uint4(0, 0, 0, 0);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&v_zeroed[pst]);
          } else {
            ok = lane0_ok(mbar_wait_bounded(&v_zeroed[pst], (zero_phase >> pst) & 1u));
            if (!ok) break;
          }
          zero_phase ^= 1u << pst;
        }
        __syncwarp();
        if (tile_used) {
          ok = lane0_ok(mbar_wait_bounded(&p_full[t][pb], (pc / kNumS) & 1));
          if (!ok) break;
          if (lane == 0 && t == 0) TC_PROBE(pc, 5);
          tc_fence_after();
          // P of chunk pc: 16-bit pairs in the first 32 columns of S buffer pb
          const uint32_t pa = tmem + t * kTmemCols + kTmemS + pb * kTcKeys;
          const uint64_t vb = v_desc + (uint64_t)((pst * C::kVBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kTcKeys / 16; ++kk)
            tc_mma_ts_warp(tmem + t * kTmemCols + kTmemO, pa + kk * 8,
                           vb + (uint64_t)((kk * 2048) >> 4), id_o, (pc > 0 || kk > 0) ? 1u : 0u,
                           lane == 0);
          if (lane == 0) {
            tc_commit(&p_done[t][pb]);
            TC_PROBE(pc, 12 + t);
          }
        }
        if (lane == 0) tc_commit(&v_free[pst]);
      }
    }
    if (!ok && lane == 0) raise_error(a.err, kErrTimeout);
  } else {
    // ================================================================ softmax rows
    const int t = warp >> 2;                    // tile of this warp
    const int trow = (warp & 3) * 32 + lane;    // row inside the tile = TMEM lane
    const int crow = t * kTcRows + trow;        // row inside the CTA
    const bool tile_used = t < ntiles;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tbase = tmem + t * kTmemCols;
    const int my_row = min(crow, rows_here - 1);
    const int my_pos = first_pos + (row0 + my_row) / G;
    const int pos_min = first_pos + (row0 + min(t * kTcRows + (warp & 3) * 32, rows_here - 1)) / G;
    float m_run = -INFINITY, l_run = 0.f;
    const float qscale = a.qscale;
    const float qmul = qscale > 0.f ? qscale : 1.f;   // multiplier left for the exponent
    for (int c = 0; c < nchunks && tile_used; ++c) {
      ok = mbar_wait_bounded(&s_full[t][c % kNumS], (c / kNumS) & 1);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      if (lane == 0 && (warp == 0 || warp == 4)) TC_PROBE(c, warp == 0 ? 0 : 3);
      tc_fence_after();
      // the chunk's scores (tcgen05.ld), masked where they reach past the
      // row's position.  With a positive scale the maximum is taken on the
      // raw scores and the scale is folded into the exponent's fused
      // multiply-add; otherwise the scores are scaled here and the
      // multiplier is 1.
      const int key0 = c * kTcKeys;
      float s[kTcKeys];
      if constexpr (kTcKeys == 64)
        tmem_ld64(tbase + lane_base + kTmemS + (c % kNumS) * kTcKeys, s);
      else
        tmem_ld32(tbase + lane_base + kTmemS + (c % kNumS) * kTcKeys, s);
      if (key0 + kTcKeys - 1 > pos_min) {
#pragma unroll
        for (int j = 0; j < kTcKeys; ++j)
          if (key0 + j > my_pos) s[j] = -INFINITY;
      }
      if (!(qscale > 0.f)) {
#pragma unroll
        for (int j = 0; j < kTcKeys; ++j) s[j] *= qscale;
      }
      if (lane == 0 && warp == 0) TC_PROBE(c, 1);
      // the row maximum as 8 independent chains; the running maximum only
      // moves when a score passes it by more than 2^8, and then what is
      // accumulated so far is rescaled (warp-wide TMEM access: a warp
      // rescales if any of its rows must, the others by 1)
      float m8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) m8[k] = s[k];
#if PHOTON_TC_FMAX3
#pragma unroll
      for (int j = 8; j + 16 <= kTcKeys; j += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = fmax3(m8[k], s[j + k], s[j + 8 + k]);
      if ((kTcKeys - 8) % 16) {
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = fmaxf(m8[k], s[kTcKeys - 8 + k]);
      }
#else
#pragma unroll
      for (int j = 8; j < kTcKeys; ++j) m8[j & 7] = fmaxf(m8[j & 7], s[j]);
#endif
      const float mx = qmul * fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                    fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      const bool moved = mx > m_run + kRescaleLog2;
      const float corr = moved ? softmax_exp2(m_run - mx) : 1.f;   // 0 on the first chunk
      l_run *= corr;
      if (moved) m_run = mx;
      if (lane == 0 && warp == 0) TC_PROBE(c, 15);
      // the product of chunk c - 1 updates O, so a rescale waits for it
      if (c > 0 && __any_sync(0xffffffffu, moved)) {
        ok = mbar_wait_bounded(&p_done[t][(c - 1) % kNumS], ((c - 1) / kNumS) & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int col = 0; col < D; col += 32) {
          float o[32];
          tmem_ld32(tbase + lane_base + kTmemO + col, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= corr;
          tmem_st32(tbase + lane_base + kTmemO + col, o);
        }
        tc_fence_before();
      }
      // P as 16-bit pairs over the first kTcKeys / 2 columns of this chunk's
      // S buffer, whose scores are all read
      float w[kTcKeys / 2];
      const float lsum = tc_weights<T>(s, qmul, m_run, w);
      if (lane == 0 && warp == 0) TC_PROBE(c, 16);
      if constexpr (kTcKeys == 64)
        tmem_st32(tbase + lane_base + kTmemS + (c % kNumS) * kTcKeys, w);   // waits for the store
      else
        tmem_st16(tbase + lane_base + kTmemS + (c % kNumS) * kTcKeys, w);
      l_run += lsum;
      if (lane == 0 && (warp == 0 || warp == 4)) TC_PROBE(c, warp == 0 ? 2 : 14);
      // the tensor-memory stores are ordered before the P V product, then
      // one arrival per warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cnt(&p_full[t][c % kNumS]);
    }
    // ---- the last product, then O / l
    if (tile_used) {
      if (ok) {
        ok = mbar_wait_bounded(&p_done[t][(nchunks - 1) % kNumS], ((nchunks - 1) / kNumS) & 1);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (!ok) {
        if (lane == 0) raise_error(a.err, kErrTimeout);
      } else {
        tc_fence_after();
        const bool store = crow < rows_here;
        const int rr = row0 + my_row;
        T* dst = outg + ((size_t)(q0 + rr / G) * a.Hq + kvh * G + rr % G) * D;
        const float inv = 1.f / l_run;
#pragma unroll 1
        for (int col = 0; col < D; col += 32) {
          float o[32];
          tmem_ld32(tbase + lane_base + kTmemO + col, o);   // warp-wide: every lane
          if (!store) continue;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float x0 = o[ch * 8 + 2 * e] * inv, x1 = o[ch * 8 + 2 * e + 1] * inv;
              if constexpr (std::is_same<T, __nv_bfloat16>::value) {
                __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
                w[e] = *reinterpret_cast<uint32_t*>(&h);
              } else {
                __half2 h = __floats2half2_rn(x0, x1);
                w[e] = *reinterpret_cast<uint32_t*>(&h);
              }
            }
            *reinterpret_cast<uint4*>(dst + col + ch * 8) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(NT * kTmemCols)
                 : "memory");
#ifdef PHOTON_PROBE
  if (tid == 0 && cta_lin < 4096) g_tc_cta[cta_lin][1] = global_timer_ns();
#endif
}

}  // namespace

cudaError_t make_pool_map(CUtensorMap* map, const void* pool, int dtype, int NB, int Hkv, int D) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<EncodeFn>(fn);
  }
  // 16-bit pools: boxes of 64 elements (128 bytes) per row, 128-byte swizzle.
  // e4m3 pools (dtype 3): one box per block row of D codes, the 128-byte
  // swizzle at D = 128 and the 64-byte one at D = 64 (a row is the swizzle
  // span either way).
  const bool codes = dtype == 3;
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)NB * Hkv * kBlockSize};
  const cuuint64_t strides[1] = {(cuuint64_t)D * (codes ? 1 : 2)};
  const cuuint32_t box[2] = {codes ? (cuuint32_t)D : 64u, (cuuint32_t)kBlockSize};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType type = codes        ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : dtype == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapSwizzle swz =
      codes && D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  const CUresult r = encode(map, type, 2, const_cast<void*>(pool), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

template <typename T, int D>
cudaError_t launch_tc(const MultiQueryArgs& a, cudaStream_t stream) {
  using C = TcCfg<T, D>;
  auto kern = paged_multi_query_tc_kernel<T, D>;
  static bool configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  CUtensorMap tk, tv;
  if ((e = make_pool_map(&tk, a.k_cache, a.dtype, a.NB, a.Hkv, a.D)) != cudaSuccess) return e;
  if ((e = make_pool_map(&tv, a.v_cache, a.dtype, a.NB, a.Hkv, a.D)) != cudaSuccess) return e;
  const int G = a.Hq / a.Hkv;
  const int rows = C::kTiles * kTcRows;
  const int tiles = (a.max_query_len * G + rows - 1) / rows;
  kern<<<dim3(tiles, a.Hkv, a.B), C::kThreads, C::kSmem, stream>>>(tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

#ifdef PHOTON_PROBE
// Tuning builds only: the timeline of the last tcgen05 multi-query call.
extern "C" int photon_tc_probe_read(void* chunks, size_t chunk_bytes, void* ctas,
                                    size_t cta_bytes) {
  cudaError_t e = cudaMemcpyFromSymbol(chunks, g_tc_probe, chunk_bytes);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(ctas, g_tc_cta, cta_bytes);
  return (int)e;
}
#endif

cudaError_t launch_multi_query_tc(const MultiQueryArgs& a, cudaStream_t stream) {
  if (!a.q || !a.k_cache || !a.v_cache || !a.block_tables || !a.context_lens || !a.query_start ||
      !a.out || !a.err)
    return cudaErrorInvalidValue;
  if (a.dtype == 1) {
    if (a.D == 64) return launch_tc<__half, 64>(a, stream);
    if (a.D == 128) return launch_tc<__half, 128>(a, stream);
  } else if (a.dtype == 2) {
    if (a.D == 64) return launch_tc<__nv_bfloat16, 64>(a, stream);
    if (a.D == 128) return launch_tc<__nv_bfloat16, 128>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace photon
