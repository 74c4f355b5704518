// multi_query.cu -- multi-query causal attention over the block-paged KV
// cache: several new query tokens per sequence (a chunk of a prompt, or the
// draft tokens of a speculative step), each attending to every cached key at
// or before its own position.
//
// PhotonInfer README: "Technical details / Paged attention" (block-wise KV
// cache, per-sequence offsets) and "Roadmap" (FlashAttention-2 style IO-aware
// attention for long sequences).  With several query rows per KV head the
// score and value products are dense contractions, so they run on the tensor
// cores (warp-level mma.sync m16n8k16, fp16/bf16 in, fp32 accumulate) in the
// FlashAttention-2 arrangement: a CTA keeps a 64-row query tile in registers
// and streams the keys of its sequence through shared memory 64 at a time,
// with an online (max, sum) softmax per row.
//
// A CTA is (query tile, KV head, sequence); its 64 rows are the pairs
// (token i, head g of the KV head's group), row = i * G + g, so the G query
// heads that share a KV head share every K/V tile.  Keys arrive through the
// block table with 16-byte cp.async copies into XOR-swizzled tiles (row r's
// 16-byte chunk c sits at chunk c ^ (r & 7)), which keeps every ldmatrix of
// the K, V and Q tiles free of bank conflicts; keys past the tile's last
// position are zero-filled and masked.
#include "photon_common.cuh"

namespace photon {
namespace {

constexpr int kMqRows = 64;     // query rows per CTA: 4 warps x 16
constexpr int kMqThreads = 128;
constexpr int kMqKeys = 64;     // keys per stage (4 blocks of 16)
constexpr int kMqStages = 2;

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

// 16-byte global -> shared copy; src_bytes = 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a swizzled tile of
// D-element rows.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * (D * 2) + ((chunk ^ (row & 7)) << 4));
}

template <typename T, int D>
struct MqCfg {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kChunks = D / 8;                    // 16-byte chunks per row
  static constexpr int kQBytes = kMqRows * kRowBytes;
  static constexpr int kTileBytes = kMqKeys * kRowBytes;   // one K or V stage
  static constexpr int kSmem = kQBytes + 2 * kMqStages * kTileBytes;
};

template <typename T, int D>
__global__ void __launch_bounds__(kMqThreads) paged_multi_query_kernel(const MultiQueryArgs a) {
  using C = MqCfg<T, D>;
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t sQ = smem_addr(smem);
  const uint32_t sK = sQ + C::kQBytes;
  const uint32_t sV = sK + kMqStages * C::kTileBytes;

  const int b = blockIdx.z, kvh = blockIdx.y;
  const int tile = blockIdx.x / a.pmax, part_idx = blockIdx.x % a.pmax;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.Hq / a.Hkv;
  const int q0 = __ldg(a.query_start + b);
  const int n = __ldg(a.query_start + b + 1) - q0;
  const int ctx = __ldg(a.context_lens + b);
  const int row0 = tile * kMqRows;
  const T* qg = static_cast<const T*>(a.q);
  T* outg = static_cast<T*>(a.out);

  if (n <= 0 || q0 < 0 || q0 + n > a.num_tokens) {
    // no query rows, or rows outside q / out: nothing to touch
    if ((n < 0 || q0 < 0 || q0 + n > a.num_tokens) && tile == 0 && kvh == 0 && tid == 0)
      raise_error(a.err, kErrQuery);
    return;
  }
  if (n > a.max_query_len || ctx < n || ctx > a.MBS * kBlockSize) {
    // inconsistent lengths: flag once, zero the rows this tile owns
    if (part_idx != 0) return;
    if (tile == 0 && kvh == 0 && tid == 0)
      raise_error(a.err, n > a.max_query_len ? kErrQuery : kErrContext);
    const int rows = min(kMqRows, max(0, min(n, a.max_query_len) * G - row0));
    for (int p = tid; p < rows * C::kChunks; p += kMqThreads) {
      const int r = row0 + p / C::kChunks, ch = p % C::kChunks;
      T* dst = outg + ((size_t)(q0 + r / G) * a.Hq + kvh * G + r % G) * D + ch * 8;
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const int rows_here = min(kMqRows, n * G - row0);
  if (rows_here <= 0) return;
  const int first_pos = ctx - n;                        // position of query token 0
  const int tok_last = (row0 + rows_here - 1) / G;      // last token of this tile
  const int kend = first_pos + tok_last + 1;            // keys [0, kend) are needed
  // this CTA's partition of them: [kb, ke), a multiple of 64 keys long
  const int kb = part_idx * a.part;
  if (kb >= kend) return;
  const int ke = min(kb + a.part, kend);
  const int nparts = (kend + a.part - 1) / a.part;       // partitions of this tile

  // ---- query tile into shared memory; rows past the tile are zero
  for (int p = tid; p < kMqRows * C::kChunks; p += kMqThreads) {
    const int r = p / C::kChunks, ch = p % C::kChunks;
    const bool valid = r < rows_here;
    const int rr = row0 + r;
    const T* src = valid ? qg + ((size_t)(q0 + rr / G) * a.Hq + kvh * G + rr % G) * D + ch * 8 : qg;
    cp_async16(sQ + swz<D>(r, ch), src, valid);
  }
  const T* kg = static_cast<const T*>(a.k_cache);
  const T* vg = static_cast<const T*>(a.v_cache);
  const int32_t* table = a.block_tables + (size_t)b * a.MBS;
  auto load_stage = [&](int c, int buf) {
    const int key0 = kb + c * kMqKeys;
    for (int p = tid; p < kMqKeys * C::kChunks; p += kMqThreads) {
      const int r = p / C::kChunks, ch = p % C::kChunks;
      const int j = key0 + r;
      bool valid = j < ke;
      size_t off = 0;
      if (valid) {
        const int blk = __ldg(table + j / kBlockSize);
        if (blk < 0 || blk >= a.NB) {
          valid = false;
          raise_error(a.err, kErrBlock);
        } else {
          off = (((size_t)blk * a.Hkv + kvh) * kBlockSize + j % kBlockSize) * D + ch * 8;
        }
      }
      cp_async16(sK + buf * C::kTileBytes + swz<D>(r, ch), kg + off, valid);
      cp_async16(sV + buf * C::kTileBytes + swz<D>(r, ch), vg + off, valid);
    }
  };
  const int nchunks = (ke - kb + kMqKeys - 1) / kMqKeys;
  load_stage(0, 0);
  cp_async_commit();

  // ---- per-thread state: rows lo = warp*16 + lane/4 and hi = lo + 8
  const bool active = warp * 16 < rows_here;
  int pos[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = min(warp * 16 + (lane >> 2) + 8 * h, rows_here - 1);
    pos[h] = first_pos + (row0 + r) / G;
  }
  const int pos_min = first_pos + (row0 + min(warp * 16, rows_here - 1)) / G;
  uint32_t qa[D / 16][4];
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};

  for (int c = 0; c < nchunks; ++c) {
    if (c + 1 < nchunks) load_stage(c + 1, (c + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (active) {
      if (c == 0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ldsm_x4(sQ + swz<D>(warp * 16 + (lane & 15), kk * 2 + (lane >> 4)), qa[kk][0],
                  qa[kk][1], qa[kk][2], qa[kk][3]);
      }
      const uint32_t kbuf = sK + (c & 1) * C::kTileBytes;
      const uint32_t vbuf = sV + (c & 1) * C::kTileBytes;
      // S = Q K^T for 16 rows x 64 keys
      float s[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbuf + swz<D>(np * 16 + ((lane >> 4) << 3) + (lane & 7),
                              kk * 2 + ((lane >> 3) & 1)),
                  b0, b1, b2, b3);
          Mma<T>::run(s[2 * np], qa[kk], b0, b1);
          Mma<T>::run(s[2 * np + 1], qa[kk], b2, b3);
        }
      }
      // scale into the log2 domain; mask keys after each row's position
      // keys past ke only occur when ke == kend, and those lie past every
      // row's position: the causal mask covers them
      const int key0 = kb + c * kMqKeys;
      const bool mask = key0 + kMqKeys - 1 > pos_min;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = s[i][e] * a.qscale;
          if (mask && key0 + i * 8 + 2 * (lane & 3) + (e & 1) > pos[e >> 1]) v = -INFINITY;
          s[i][e] = v;
        }
      // online softmax per row (a row's 64 scores sit in the 4 lanes of a quad)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fmaxf(s[i][2 * h], s[i][2 * h + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_r[h], mx);
        // a row with every key so far masked (possible in a later partition)
        // keeps m = -inf: exponents then use 0, giving weights 0, not NaN
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float corr = softmax_exp2(m_r[h] - m_use);
        m_r[h] = m_new;
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          s[i][2 * h] = softmax_exp2(s[i][2 * h] - m_use);
          s[i][2 * h + 1] = softmax_exp2(s[i][2 * h + 1] - m_use);
          sum += s[i][2 * h] + s[i][2 * h + 1];
        }
        l_r[h] = l_r[h] * corr + sum;
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
          o[i][2 * h] *= corr;
          o[i][2 * h + 1] *= corr;
        }
      }
      // O += P V: P (16 x 64) from the score registers, V through ldmatrix.trans
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t pa[4];
        pa[0] = Mma<T>::pack(s[2 * ks][0], s[2 * ks][1]);
        pa[1] = Mma<T>::pack(s[2 * ks][2], s[2 * ks][3]);
        pa[2] = Mma<T>::pack(s[2 * ks + 1][0], s[2 * ks + 1][1]);
        pa[3] = Mma<T>::pack(s[2 * ks + 1][2], s[2 * ks + 1][3]);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_trans(vbuf + swz<D>(ks * 16 + (((lane >> 3) & 1) << 3) + (lane & 7),
                                    dp * 2 + (lane >> 4)),
                        b0, b1, b2, b3);
          Mma<T>::run(o[2 * dp], pa, b0, b1);
          Mma<T>::run(o[2 * dp + 1], pa, b2, b3);
        }
      }
    }
    __syncthreads();  // this stage's buffer is refilled two iterations on
  }

  // ---- one partition: normalise and store the tile's valid rows; several:
  // leave (m, l, unnormalised o) for the merge kernel
  if (!active) return;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float l = l_r[h];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const int r = warp * 16 + (lane >> 2) + 8 * h;
    if (r >= rows_here) continue;
    const int rr = row0 + r;
    if (nparts > 1) {
      const size_t prow = ((size_t)(q0 + rr / G) * a.Hq + kvh * G + rr % G) * a.pmax + part_idx;
      if ((lane & 3) == 0) {
        a.ws_m[prow] = m_r[h];
        a.ws_l[prow] = l;
      }
      float* po = a.ws_o + prow * D + 2 * (lane & 3);
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
        *reinterpret_cast<float2*>(po + i * 8) = make_float2(o[i][2 * h], o[i][2 * h + 1]);
      continue;
    }
    const float inv = 1.f / l;
    T* dst = outg + ((size_t)(q0 + rr / G) * a.Hq + kvh * G + rr % G) * D + 2 * (lane & 3);
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
      *reinterpret_cast<uint32_t*>(dst + i * 8) = Mma<T>::pack(o[i][2 * h] * inv,
                                                                o[i][2 * h + 1] * inv);
  }
}

// Combines the partitions of the rows whose tile was split: one warp per
// (query token, q head) row of sequence blockIdx.y.  Partition p of a row at
// position pos holds keys [p*part, (p+1)*part) up to pos; the ones past pos
// were fully masked and are skipped.
template <typename T, int D>
__global__ void __launch_bounds__(128) multi_query_merge_kernel(const MultiQueryArgs a) {
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = __ldg(a.query_start + b);
  const int n = __ldg(a.query_start + b + 1) - q0;
  const int ctx = __ldg(a.context_lens + b);
  if (n <= 0 || q0 < 0 || q0 + n > a.num_tokens || n > a.max_query_len || ctx < n ||
      ctx > a.MBS * kBlockSize)
    return;  // flagged (and zeroed where possible) by the attention kernel
  const int row = blockIdx.x * 4 + warp;  // (token i, head h) of this sequence
  if (row >= n * a.Hq) return;
  const int i = row / a.Hq, h = row % a.Hq;
  const int G = a.Hq / a.Hkv;
  const int r = i * G + h % G;            // row inside its KV head's tiles
  const int tile = r / kMqRows;
  const int rows_here = min(kMqRows, n * G - tile * kMqRows);
  const int tok_last = (tile * kMqRows + rows_here - 1) / G;
  const int kend = ctx - n + tok_last + 1;
  if (kend <= a.part) return;             // single partition: written directly
  const int pos = ctx - n + i;
  const int np = pos / a.part + 1;        // partitions that hold keys <= pos
  const size_t base = ((size_t)(q0 + i) * a.Hq + h) * a.pmax;
  float mx = -INFINITY;
  for (int p = 0; p < np; ++p) mx = fmaxf(mx, a.ws_m[base + p]);
  float den = 0.f;
  constexpr int kPer = D / 32;
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  for (int p = 0; p < np; ++p) {
    const float w = softmax_exp2(a.ws_m[base + p] - mx);
    den += w * a.ws_l[base + p];
    const float* po = a.ws_o + (base + p) * D + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] += w * po[e];
  }
  const float inv = 1.f / den;
  T* dst = static_cast<T*>(a.out) + ((size_t)(q0 + i) * a.Hq + h) * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; ++e) dst[e] = Elem<T>::narrow(acc[e] * inv);
}

template <typename T, int D>
cudaError_t launch_mq(const MultiQueryArgs& a, cudaStream_t stream) {
  using C = MqCfg<T, D>;
  auto kern = paged_multi_query_kernel<T, D>;
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
  const int tiles = (a.max_query_len * G + kMqRows - 1) / kMqRows;
  dim3 grid(tiles * a.pmax, a.Hkv, a.B);
  kern<<<grid, kMqThreads, C::kSmem, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.pmax == 1) return e;
  dim3 mgrid((a.max_query_len * a.Hq + 3) / 4, a.B);
  multi_query_merge_kernel<T, D><<<mgrid, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_multi_query(const MultiQueryArgs& a, cudaStream_t stream) {
  if (!a.q || !a.k_cache || !a.v_cache || !a.block_tables || !a.context_lens || !a.query_start ||
      !a.out || !a.err || a.pmax < 1 || a.part < kMqKeys || a.part % kMqKeys != 0)
    return cudaErrorInvalidValue;
  if (a.pmax > 1 && (!a.ws_m || !a.ws_l || !a.ws_o)) return cudaErrorInvalidValue;
  if (a.dtype == 1) {
    if (a.D == 64) return launch_mq<__half, 64>(a, stream);
    if (a.D == 128) return launch_mq<__half, 128>(a, stream);
  } else if (a.dtype == 2) {
    if (a.D == 64) return launch_mq<__nv_bfloat16, 64>(a, stream);
    if (a.D == 128) return launch_mq<__nv_bfloat16, 128>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace photon
