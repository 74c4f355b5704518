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
// A CTA is (128-row query tile, KV head, sequence), 4 warps.  Row r of the
// tile is (token r / G, head r % G of the KV head's group) and lives in TMEM
// lane r, so thread r owns row r from the scores to the output: the softmax
// needs no shuffles.  Per chunk of 64 keys:
//   S = Q K^T    one thread issues D/16 MMAs (M=128, N=64, K=16) into TMEM
//   softmax      each thread loads its 64 scores (tcgen05.ld), masks the keys
//                after its position, updates (m, l), writes its 64 weights
//                P as fp16/bf16 into a swizzled shared tile
//   O += P V     4 MMAs (M=128, N=D, K=16) accumulate in TMEM
// The running maximum only moves when a new score exceeds it by more than
// 2^8 (log2 domain), and only then is the TMEM accumulator rescaled: between
// rescales the weights use a stale maximum, which the final O / l cancels
// exactly, and a weight stays below 2^8, far inside fp16/bf16 range.
//
// Operands are K-major with the 128-byte swizzle: a tile of R rows and 64
// 16-bit elements per row is R/8 atoms of 8 rows x 128 bytes, 16-byte chunk c
// of row r stored at chunk c ^ (r % 8); rows past 64 elements continue in the
// next 64-element block of R x 128 bytes.  K rows arrive with cp.async; V is
// needed transposed (d rows, key columns), so each thread loads 16-byte V
// pieces into registers one chunk ahead and scatters them as 2-byte stores.
#include <type_traits>

#include "photon_common.cuh"

namespace photon {
namespace {

constexpr int kTcRows = 128;    // query rows per CTA = TMEM lanes
constexpr int kTcThreads = 128;
constexpr int kTcKeys = 64;     // keys per chunk
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemS = 0;     // S: two buffers, columns [0, 64) and [64, 128)
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

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
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
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
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

template <typename T, int D>
struct TcCfg {
  static constexpr int kQBytes = kTcRows * D * 2;     // Q tile
  static constexpr int kKBytes = kTcKeys * D * 2;     // one K chunk
  static constexpr int kVBytes = kTcKeys * D * 2;     // one V chunk
  static constexpr int kPBytes = kTcRows * kTcKeys * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;       // [2]
  static constexpr int kOffV = kOffK + 2 * kKBytes;   // [2]
  static constexpr int kOffP = kOffV + 2 * kVBytes;
  static constexpr int kUsed = kOffP + kPBytes;
  // at least ~100 KB so that no more than two CTAs (2 x 256 TMEM columns)
  // share an SM, plus 1 KB to align the base to a swizzle atom
  static constexpr int kSmem = (kUsed > 100 * 1024 ? kUsed : 100 * 1024) + 1024;
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

template <typename T, int D>
__global__ void __launch_bounds__(kTcThreads) paged_multi_query_tc_kernel(const MultiQueryArgs a) {
  using C = TcCfg<T, D>;
  extern __shared__ unsigned char tc_smem_raw[];
  __shared__ __align__(8) uint64_t bar_s[2];   // S(c) completes on bar_s[c & 1]
  __shared__ __align__(8) uint64_t bar_o;      // each P V product
  __shared__ uint32_t tmem_slot;
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t sQ = sbase + C::kOffQ, sK = sbase + C::kOffK, sV = sbase + C::kOffV,
                 sP = sbase + C::kOffP;

  const int b = blockIdx.z, kvh = blockIdx.y, tile = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int G = a.Hq / a.Hkv;
  const int q0 = __ldg(a.query_start + b);
  const int n = __ldg(a.query_start + b + 1) - q0;
  const int ctx = __ldg(a.context_lens + b);
  const int row0 = tile * kTcRows;
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
    const int rows = min(kTcRows, max(0, min(n, a.max_query_len) * G - row0));
    for (int p = tid; p < rows * (D / 8); p += kTcThreads) {
      const int r = row0 + p / (D / 8), ch = p % (D / 8);
      T* dst = outg + ((size_t)(q0 + r / G) * a.Hq + kvh * G + r % G) * D + ch * 8;
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const int rows_here = min(kTcRows, n * G - row0);
  if (rows_here <= 0) return;
  const int first_pos = ctx - n;
  const int kend = first_pos + (row0 + rows_here - 1) / G + 1;   // keys [0, kend)
  const int nchunks = (kend + kTcKeys - 1) / kTcKeys;
  const int my_row = min(tid, rows_here - 1);
  const int my_pos = first_pos + (row0 + my_row) / G;
  const int pos_min = first_pos + (row0 + min(warp * 32, rows_here - 1)) / G;

  // ---- barriers, TMEM
  if (tid == 0) {
    mbar_init(&bar_s[0], 1);
    mbar_init(&bar_s[1], 1);
    mbar_init(&bar_o, 1);
    mbar_init_fence();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }

  // ---- loads: Q tile (rows past the tile zero); K and V chunks keep their
  // rows of 16-byte chunks, swizzled (K read K-major, V read MN-major)
  for (int p = tid; p < kTcRows * (D / 8); p += kTcThreads) {
    const int r = p / (D / 8), ch = p % (D / 8);
    const bool valid = r < rows_here;
    const int rr = row0 + r;
    const T* src = valid ? qg + ((size_t)(q0 + rr / G) * a.Hq + kvh * G + rr % G) * D + ch * 8 : qg;
    cp_async16_zfill(sQ + sw_chunk<kTcRows>(r, ch), src, valid);
  }
  const T* kg = static_cast<const T*>(a.k_cache);
  const T* vg = static_cast<const T*>(a.v_cache);
  const int32_t* table = a.block_tables + (size_t)b * a.MBS;
  // 64 keys of chunk c (zero past kend or for a bad block) into a tile
  auto load_chunk = [&](const T* pool, uint32_t dst, int c) {
    for (int p = tid; p < kTcKeys * (D / 8); p += kTcThreads) {
      const int r = p / (D / 8), ch = p % (D / 8);
      const int j = c * kTcKeys + r;
      long long off = -1;
      if (j < kend) {
        const int blk = __ldg(table + j / kBlockSize);
        if (blk >= 0 && blk < a.NB)
          off = (((long long)blk * a.Hkv + kvh) * kBlockSize + j % kBlockSize) * D + ch * 8;
        else
          raise_error(a.err, kErrBlock);
      }
      cp_async16_zfill(dst + sw_chunk<kTcKeys>(r, ch), off >= 0 ? pool + off : pool, off >= 0);
    }
  };
  auto commit_group = [] { asm volatile("cp.async.commit_group;" ::: "memory"); };
  load_chunk(kg, sK, 0);
  load_chunk(vg, sV, 0);
  commit_group();
  if (nchunks > 1) load_chunk(kg, sK + C::kKBytes, 1);
  commit_group();
  cp_async_wait_all();
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t id_s = f16_idesc<T>(kTcRows, kTcKeys);
  const uint32_t id_o = f16_idesc<T>(kTcRows, D) | (1u << 16);   // B (V) MN-major

  auto issue_s = [&](int c) {   // S(c) = Q K(c)^T into S buffer c & 1
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t koff = (kk & 3) * 32;   // 16 elements inside a 64-element block
      tc_mma(tmem + kTmemS + (c & 1) * kTcKeys,
             sw128_desc(sQ + (kk >> 2) * (kTcRows * 128) + koff),
             sw128_desc(sK + (c & 1) * C::kKBytes + (kk >> 2) * (kTcKeys * 128) + koff), id_s,
             kk > 0);
    }
    tc_commit(&bar_s[c & 1]);
  };
  if (tid == 0) issue_s(0);

  // Per chunk c:  wait S(c) | load K(c+2), issue S(c+1) | softmax(c) |
  // wait PV(c-1), rescale O, load V(c+1) | P(c) to shared | sync | PV(c).
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;
  for (int c = 0; c < nchunks; ++c) {
    ok = __syncthreads_and(mbar_wait_bounded(&bar_s[c & 1], (c >> 1) & 1) ? 1 : 0) != 0;
    if (!ok) break;
    tc_fence_after();
    if (c + 2 < nchunks) load_chunk(kg, sK + (c & 1) * C::kKBytes, c + 2);
    commit_group();
    if (c + 1 < nchunks && tid == 0) issue_s(c + 1);

    float s[kTcKeys];
    tmem_ld32(tmem + lane_base + kTmemS + (c & 1) * kTcKeys, s);
    tmem_ld32(tmem + lane_base + kTmemS + (c & 1) * kTcKeys + 32, s + 32);
    const int key0 = c * kTcKeys;
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < kTcKeys; ++j) {
      float v = s[j] * a.qscale;
      if (key0 + kTcKeys - 1 > pos_min && key0 + j > my_pos) v = -INFINITY;
      s[j] = v;
      mx = fmaxf(mx, v);
    }
    // the maximum moves only when a score passes it by more than 2^8; then
    // what is accumulated so far is rescaled (TMEM loads and stores are
    // warp-wide: a warp rescales if any of its rows must, the others by 1)
    const bool moved = mx > m_run + kRescaleLog2;
    const float corr = moved ? softmax_exp2(m_run - mx) : 1.f;   // 0 on the first chunk
    l_run *= corr;
    if (moved) m_run = mx;
    if (c > 0) {
      ok = __syncthreads_and(mbar_wait_bounded(&bar_o, (c - 1) & 1) ? 1 : 0) != 0;
      if (!ok) break;
      tc_fence_after();
      if (__any_sync(0xffffffffu, moved)) {
#pragma unroll 1
        for (int col = 0; col < D; col += 32) {
          float o[32];
          tmem_ld32(tmem + lane_base + kTmemO + col, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= corr;
          tmem_st32(tmem + lane_base + kTmemO + col, o);
        }
      }
    }
    if (c + 1 < nchunks) load_chunk(vg, sV + ((c + 1) & 1) * C::kVBytes, c + 1);
    commit_group();
    float sum = 0.f;
    unsigned char* prow = smem + C::kOffP;
#pragma unroll
    for (int ch = 0; ch < kTcKeys / 8; ++ch) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p0 = softmax_exp2(s[ch * 8 + 2 * e] - m_run);
        const float p1 = softmax_exp2(s[ch * 8 + 2 * e + 1] - m_run);
        sum += p0 + p1;
        if constexpr (std::is_same<T, __nv_bfloat16>::value) {
          __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
          w[e] = *reinterpret_cast<uint32_t*>(&h);
        } else {
          __half2 h = __floats2half2_rn(p0, p1);
          w[e] = *reinterpret_cast<uint32_t*>(&h);
        }
      }
      *reinterpret_cast<uint4*>(prow + sw_chunk<kTcRows>(tid, ch)) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
    l_run += sum;
    // everything but V(c+1) has landed: K(c+2) for the next S, V(c) for this PV
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kTcKeys / 16; ++kk)
        tc_mma(tmem + kTmemO, sw128_desc(sP + kk * 32),
               sw128_mn_desc(sV + (c & 1) * C::kVBytes + kk * 2048), id_o,
               (c > 0 || kk > 0) ? 1u : 0u);
      tc_commit(&bar_o);
    }
  }
  // ---- the last product, then O / l
  if (ok) ok = __syncthreads_and(mbar_wait_bounded(&bar_o, (nchunks - 1) & 1) ? 1 : 0) != 0;
  if (!ok && tid == 0) raise_error(a.err, kErrTimeout);
  tc_fence_after();
  if (ok) {
    const bool store = tid < rows_here;
    const int rr = row0 + my_row;
    T* dst = outg + ((size_t)(q0 + rr / G) * a.Hq + kvh * G + rr % G) * D;
    const float inv = 1.f / l_run;
#pragma unroll 1
    for (int col = 0; col < D; col += 32) {
      float o[32];
      tmem_ld32(tmem + lane_base + kTmemO + col, o);   // warp-wide: every lane
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
  } else {
    // a timed-out tile leaves its rows unwritten (the error word says so);
    // let any product still in flight land before TMEM is released
    if (tid == 0) raise_error(a.err, kErrTimeout);
    mbar_wait_bounded(&bar_o, (nchunks - 1) & 1);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
}

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
  const int G = a.Hq / a.Hkv;
  const int tiles = (a.max_query_len * G + kTcRows - 1) / kTcRows;
  kern<<<dim3(tiles, a.Hkv, a.B), kTcThreads, C::kSmem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

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
