// multi_query.cu -- multi-query causal attention over the block-paged KV
// cache: several new query tokens per sequence (a chunk of a prompt, or the
// draft tokens of a speculative step), each attending to every cached key at
// or before its own position.
//
// PhotonInfer README: "Technical details / Paged attention" (block-wise KV
// cache, per-sequence offsets) and "Roadmap" (FlashAttention-2 style IO-aware
// attention for long sequences).  This is the kernel for few query rows per
// sequence (speculative verification), which cannot fill the device by query
// tiles alone: each tile's keys are also split into partitions that run in
// parallel and are merged by their log-sum-exp weights.  The score and value
// products run on warp-level tensor-core instructions (mma.sync m16n8k16,
// fp16/bf16 in, fp32 accumulate) in the FlashAttention-2 arrangement: a CTA
// keeps a 64-row query tile in registers and streams its partition's keys
// through shared memory 64 at a time, with an online (max, sum) softmax per
// row.
//
// A CTA is (query tile, key partition, KV head, sequence); its 64 rows are the
// pairs (token i, head g of the KV head's group), row = i * G + g, so the G
// query heads that share a KV head share every K/V tile.  K and V arrive as
// tensor-map copies (boxes of 16 rows x 64 elements with the 128-byte
// swizzle, straight from the pool through the block table) issued by a copy
// warp into a 3-stage ring; the swizzle keeps every ldmatrix of the tiles free
// of bank conflicts.  Keys past the partition's end are masked and their V
// rows zeroed.
#include <cuda.h>

#include "photon_common.cuh"

namespace photon {
namespace {

constexpr int kMqRows = 64;     // query rows per CTA: 4 warps x 16
constexpr int kMqThreads = 128;
constexpr int kMqKeys = 64;     // keys per stage (4 blocks of 16)

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
#ifndef PHOTON_MQ_STAGES
#define PHOTON_MQ_STAGES 2
#endif
  static constexpr int kStages = PHOTON_MQ_STAGES;
  static constexpr int kRowBytes = D * 2;
  static constexpr int kChunks = D / 8;                    // 16-byte chunks per row
  static constexpr int kQBytes = kMqRows * kRowBytes;
  static constexpr int kKVBytes = kMqKeys * kRowBytes;     // one K or V chunk
  static constexpr int kOffQ = 0;
  // the Q tile's space also holds the key-split combine: 64 rows of 64 fp32,
  // padded to 72 so that neighbouring rows fall in other banks
  static constexpr int kCombStride = 72;
  static constexpr int kQSpace = kQBytes > 64 * kCombStride * 4 ? kQBytes : 64 * kCombStride * 4;
  static constexpr int kOffK = kQSpace;                    // [kStages]
  static constexpr int kOffV = kOffK + kStages * kKVBytes; // [kStages]
  static constexpr int kUsed = kOffV + kStages * kKVBytes;
  static constexpr int kSmem = kUsed + 1024;               // + alignment to a swizzle atom
  static constexpr int kThreads = kMqThreads + 32;         // 4 MMA warps + 1 copy warp
};

// Byte offset of 16-byte chunk c of row r in a tile of 64 rows laid out as the
// tensor-map copies write it: 64-element column blocks of 64 rows x 128 B, the
// 128-byte swizzle inside each 8-row atom.
__device__ __forceinline__ uint32_t tma_chunk(int r, int c) {
  return (uint32_t)((c >> 3) * (kMqKeys * 128) + (r >> 3) * 1024 + (r & 7) * 128 +
                    (((c & 7) ^ (r & 7)) << 4));
}

// One 64-key chunk for one warp's 16 query rows, over NP groups of 16 keys
// starting at group g0 of the chunk: S = Q K^T on the tensor cores, mask,
// online softmax update, O += P V.  State (o, m, l) stays in registers.
template <typename T, int D, int NP>
__device__ __forceinline__ void mq_chunk(uint32_t kbuf, uint32_t vbuf, int g0, int key0,
                                         const uint32_t (&qa)[D / 16][4], float (&o)[D / 8][4],
                                         float (&m_r)[2], float (&l_r)[2], const int (&pos)[2],
                                         int pos_min, float qscale, int lane) {
  float s[2 * NP][4];
#pragma unroll
  for (int i = 0; i < 2 * NP; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
    for (int g = 0; g < NP; ++g) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kbuf + tma_chunk((g0 + g) * 16 + ((lane >> 4) << 3) + (lane & 7),
                               kk * 2 + ((lane >> 3) & 1)),
              b0, b1, b2, b3);
      Mma<T>::run(s[2 * g], qa[kk], b0, b1);
      Mma<T>::run(s[2 * g + 1], qa[kk], b2, b3);
    }
  }
  // scale into the log2 domain; mask keys after each row's position (keys past
  // the partition's end only occur when it ends the tile, past every row)
  const int kbase = key0 + g0 * 16;
  const bool mask = kbase + 16 * NP - 1 > pos_min;
#pragma unroll
  for (int i = 0; i < 2 * NP; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = s[i][e] * qscale;
      if (mask && kbase + i * 8 + 2 * (lane & 3) + (e & 1) > pos[e >> 1]) v = -INFINITY;
      s[i][e] = v;
    }
  // online softmax per row (a row's scores sit in the 4 lanes of a quad)
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 2 * NP; ++i) mx = fmaxf(mx, fmaxf(s[i][2 * h], s[i][2 * h + 1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_r[h], mx);
    // a row whose keys so far are all masked keeps m = -inf: its exponents
    // use 0, giving weights 0, not NaN
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float corr = softmax_exp2(m_r[h] - m_use);
    m_r[h] = m_new;
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 2 * NP; ++i) {
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
  // O += P V: P from the score registers, V through ldmatrix.trans
#pragma unroll
  for (int g = 0; g < NP; ++g) {
    uint32_t pa[4];
    pa[0] = Mma<T>::pack(s[2 * g][0], s[2 * g][1]);
    pa[1] = Mma<T>::pack(s[2 * g][2], s[2 * g][3]);
    pa[2] = Mma<T>::pack(s[2 * g + 1][0], s[2 * g + 1][1]);
    pa[3] = Mma<T>::pack(s[2 * g + 1][2], s[2 * g + 1][3]);
#pragma unroll
    for (int dp = 0; dp < D / 16; ++dp) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_trans(vbuf + tma_chunk((g0 + g) * 16 + (((lane >> 3) & 1) << 3) + (lane & 7),
                                     dp * 2 + (lane >> 4)),
                    b0, b1, b2, b3);
      Mma<T>::run(o[2 * dp], pa, b0, b1);
      Mma<T>::run(o[2 * dp + 1], pa, b2, b3);
    }
  }
}

// Work item of the persistent kernel: (sequence, query tile, key partition,
// KV head).  Items are numbered sequence by sequence, then tile, partition and
// KV head; a CTA takes items blockIdx.x, blockIdx.x + gridDim.x, ... and both
// of its roles walk the numbering with the same cursor, so they agree on every
// item without talking.
struct MqItem {
  int b, kvh, tile, part_idx;
  int q0, n, ctx;
  bool bad;            // inconsistent lengths: the item zero-fills its rows
};

struct MqCursor {
  int b = -1;          // sequence whose items are [base, base + cnt)
  long long base = 0;
  int cnt = 0;
};

// Items of sequence b (0 for an empty or out-of-range one).
__device__ __forceinline__ int mq_seq_items(const MultiQueryArgs& a, int b, int G) {
  const int q0 = __ldg(a.query_start + b);
  const int n = __ldg(a.query_start + b + 1) - q0;
  if (n <= 0 || q0 < 0 || q0 + n > a.num_tokens) return 0;
  const int ctx = __ldg(a.context_lens + b);
  const int tiles = (min(n, a.max_query_len) * G + kMqRows - 1) / kMqRows;
  if (n > a.max_query_len || ctx < n || ctx > a.MBS * kBlockSize) return tiles * a.Hkv;
  int parts = 0;
  for (int t = 0; t < tiles; ++t) {
    const int rows = min(kMqRows, n * G - t * kMqRows);
    const int kend = ctx - n + (t * kMqRows + rows - 1) / G + 1;
    parts += (kend + a.part - 1) / a.part;
  }
  return parts * a.Hkv;
}

// Locates item `item` (items asked for in increasing order); false past the end.
__device__ __forceinline__ bool mq_locate(const MultiQueryArgs& a, int G, MqCursor& cur,
                                          long long item, MqItem& it) {
  while (item >= cur.base + cur.cnt) {
    cur.base += cur.cnt;
    if (++cur.b >= a.B) return false;
    cur.cnt = mq_seq_items(a, cur.b, G);
    if (cur.cnt == 0 && threadIdx.x == 0 && blockIdx.x == 0) {
      // no items: an empty sequence, or query rows outside q / out (flagged)
      const int q0 = __ldg(a.query_start + cur.b);
      const int n = __ldg(a.query_start + cur.b + 1) - q0;
      if (n < 0 || q0 < 0 || q0 + n > a.num_tokens) raise_error(a.err, kErrQuery);
    }
  }
  const int b = cur.b;
  int j = (int)(item - cur.base);
  it.b = b;
  it.kvh = j % a.Hkv;
  j /= a.Hkv;
  it.q0 = __ldg(a.query_start + b);
  it.n = __ldg(a.query_start + b + 1) - it.q0;
  it.ctx = __ldg(a.context_lens + b);
  it.bad = it.n > a.max_query_len || it.ctx < it.n || it.ctx > a.MBS * kBlockSize;
  if (it.bad) {
    it.tile = j;
    it.part_idx = 0;
    return true;
  }
  const int tiles = (it.n * G + kMqRows - 1) / kMqRows;
  for (int t = 0; t < tiles; ++t) {
    const int rows = min(kMqRows, it.n * G - t * kMqRows);
    const int kend = it.ctx - it.n + (t * kMqRows + rows - 1) / G + 1;
    const int parts = (kend + a.part - 1) / a.part;
    if (j < parts) {
      it.tile = t;
      it.part_idx = j;
      return true;
    }
    j -= parts;
  }
  return false;   // not reached for consistent counts
}

// Barrier of the 4 MMA warps (named barrier 1, 128 threads) that also tells
// whether every one of them got through its waits.
__device__ __forceinline__ bool mma_warps_all(bool ok) {
  int n;
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.s32 p, %1, 0;\n bar.red.popc.u32 %0, 1, 128, p;\n}"
      : "=r"(n)
      : "r"(ok ? 1 : 0)
      : "memory");
  return n == 128;
}
__device__ __forceinline__ void mma_warps_sync() {
  asm volatile("bar.sync 2, 128;" ::: "memory");
}

// Persistent CTAs (2 per SM).  Roles: warps 0-3 compute (warp-level
// mma.sync); warp 4 copies: its lane 0 issues, per 64-key chunk of each item,
// one tensor-map box (16 rows x 64 elements, 128-byte swizzle) per pool block
// and 64-column half for K and for V into a ring of kStages stages, as soon as
// the 4 compute warps have released the stage; the ring runs on across items.
template <typename T, int D>
__global__ void __launch_bounds__(MqCfg<T, D>::kThreads, 2)
    paged_multi_query_kernel(const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v, const MultiQueryArgs a) {
  using C = MqCfg<T, D>;
  constexpr int S = C::kStages;
  extern __shared__ unsigned char mq_smem_raw[];
  __shared__ __align__(8) uint64_t full[S], empty[S];
  __shared__ float comb_m[4 * 32], comb_l[4 * 32];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(mq_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_addr(smem) + C::kOffQ;
  const uint32_t sK = smem_addr(smem) + C::kOffK;
  const uint32_t sV = smem_addr(smem) + C::kOffV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.Hq / a.Hkv;
  const T* qg = static_cast<const T*>(a.q);
  T* outg = static_cast<T*>(a.out);

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == 4) {
    // ================================================================ copies
    MqCursor cur;
    MqItem it;
    int g = 0;   // chunks issued so far (ring position)
    for (long long item = blockIdx.x; mq_locate(a, G, cur, item, it); item += gridDim.x) {
      if (it.bad) continue;
      const int row0 = it.tile * kMqRows;
      const int rows_here = min(kMqRows, it.n * G - row0);
      const int kend = it.ctx - it.n + (row0 + rows_here - 1) / G + 1;
      const int kb = it.part_idx * a.part;
      const int ke = min(kb + a.part, kend);
      const int nchunks = (ke - kb + kMqKeys - 1) / kMqKeys;
      // the partition's block ids, a window of 256 at a time (lane j: blocks
      // w + j, w + j + 32, ...); one window covers a 4096-key partition, a
      // longer (unsplit) one reloads it every 64 chunks
      const int32_t* table = a.block_tables + (size_t)it.b * a.MBS + kb / kBlockSize;
      const int nblk = (ke - kb + kBlockSize - 1) / kBlockSize;
      constexpr int kTblPerLane = 4096 / kBlockSize / 32;
      constexpr int kWindow = kTblPerLane * 32;              // blocks per window
      int tbl[kTblPerLane];
      auto load_window = [&](int w) {
#pragma unroll
        for (int k = 0; k < kTblPerLane; ++k) {
          const int j = w + k * 32 + lane;
          tbl[k] = j < nblk ? __ldg(table + j) : -1;
        }
      };
      load_window(0);
      bool ok = true;
      for (int c = 0; c < nchunks; ++c, ++g) {
        if (c > 0 && (4 * c) % kWindow == 0) load_window(4 * c);
        const int st = g % S;
        if (g >= S) {   // the 4 compute warps are done with the stage's previous chunk
          ok = __shfl_sync(0xffffffffu, mbar_wait_bounded(&empty[st], ((g / S) - 1) & 1) ? 1 : 0,
                           0) != 0;
          if (!ok) break;
        }
        int phys[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j = c * 4 + i;   // block of the partition
          const int jw = j % kWindow;  // its place in the current window
          int v = -1;
#pragma unroll
          for (int k = 0; k < kTblPerLane; ++k) {
            const int t = __shfl_sync(0xffffffffu, tbl[k], jw & 31);
            if ((jw >> 5) == k) v = t;
          }
          phys[i] = j < nblk ? v : -2;   // -2: past the partition (nothing to load)
        }
        if (lane == 0) {
          uint32_t bytes = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (phys[i] == -2) continue;
            if (phys[i] >= 0 && phys[i] < a.NB) {
              bytes += 2u * kBlockSize * D * 2u;
            } else {
              raise_error(a.err, kErrBlock);
              phys[i] = -1;
            }
          }
          mbar_arrive_expect_tx(&full[st], bytes);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (phys[i] < 0) continue;
            const int y = (phys[i] * a.Hkv + it.kvh) * kBlockSize;
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
              tma_load_box(sK + st * C::kKVBytes + h * (kMqKeys * 128) + i * 2048, &tm_k,
                           h * 64, y, &full[st]);
              tma_load_box(sV + st * C::kKVBytes + h * (kMqKeys * 128) + i * 2048, &tm_v,
                           h * 64, y, &full[st]);
            }
          }
        }
        __syncwarp();
      }
      if (!ok) {
        if (lane == 0) raise_error(a.err, kErrTimeout);
        break;
      }
    }
    return;
  }

  // ================================================================ compute warps
  MqCursor cur;
  MqItem it;
  int g = 0;   // chunks consumed so far (ring position)
  bool ok = true;
  for (long long item = blockIdx.x; ok && mq_locate(a, G, cur, item, it); item += gridDim.x) {
    const int row0 = it.tile * kMqRows;
    if (it.bad) {
      // inconsistent lengths: flag once, zero the rows this tile owns
      if (it.tile == 0 && it.kvh == 0 && tid == 0)
        raise_error(a.err, it.n > a.max_query_len ? kErrQuery : kErrContext);
      const int rows = min(kMqRows, max(0, min(it.n, a.max_query_len) * G - row0));
      for (int p = tid; p < rows * C::kChunks; p += kMqThreads) {
        const int r = row0 + p / C::kChunks, ch = p % C::kChunks;
        T* dst = outg + ((size_t)(it.q0 + r / G) * a.Hq + it.kvh * G + r % G) * D + ch * 8;
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    const int q0 = it.q0, kvh = it.kvh, part_idx = it.part_idx;
    const int rows_here = min(kMqRows, it.n * G - row0);
    const int first_pos = it.ctx - it.n;                  // position of query token 0
    const int kend = first_pos + (row0 + rows_here - 1) / G + 1;
    const int kb = part_idx * a.part;
    const int ke = min(kb + a.part, kend);
    const int nparts = (kend + a.part - 1) / a.part;
    const int nchunks = (ke - kb + kMqKeys - 1) / kMqKeys;

    // ---- query tile into shared memory (rows past the tile zero)
    for (int p = tid; p < kMqRows * C::kChunks; p += kMqThreads) {
      const int r = p / C::kChunks, ch = p % C::kChunks;
      const bool valid = r < rows_here;
      const int rr = row0 + r;
      const T* src =
          valid ? qg + ((size_t)(q0 + rr / G) * a.Hq + kvh * G + rr % G) * D + ch * 8 : qg;
      cp_async16(sQ + swz<D>(r, ch), src, valid);
    }
    cp_async_commit();
    cp_async_wait<0>();
    mma_warps_sync();

    // The tile's rows form RG groups of 16 (RG = 1 .. 4).  With fewer than
    // four groups the spare warps split the keys instead: KS = 4 / RG warps
    // share a row group, warp w taking row group w % RG and the keys
    // 64/KS * (w / RG) .. of every chunk; their partial states are combined
    // at the end.  A few draft tokens (at most 16 rows) keep all four warps busy.
    const int RG = min(4, (rows_here + 15) / 16);
    const int KS = RG == 1 ? 4 : (RG == 2 ? 2 : 1);
    const int rg = warp % RG, ks = warp / RG;
    const bool active = ks < KS;          // (RG = 3 leaves warp 3 idle)
    const int rbase = rg * 16;
    const int NP = 4 / KS;                // 16-key groups per warp and chunk
    int pos[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = min(rbase + (lane >> 2) + 8 * h, rows_here - 1);
      pos[h] = first_pos + (row0 + r) / G;
    }
    const int pos_min = first_pos + (row0 + min(rbase, rows_here - 1)) / G;
    uint32_t qa[D / 16][4];
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
    if (active) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        ldsm_x4(sQ + swz<D>(rbase + (lane & 15), kk * 2 + (lane >> 4)), qa[kk][0], qa[kk][1],
                qa[kk][2], qa[kk][3]);
    }

    for (int c = 0; c < nchunks; ++c, ++g) {
      const int st = g % S;
      // the verdict of the wait is shared by the 4 compute warps, so that they
      // all leave together and no one is left at a named barrier
      ok = mma_warps_all(mbar_wait_bounded(&full[st], (g / S) & 1));
      if (!ok) {
        if (tid == 0) raise_error(a.err, kErrTimeout);
        break;
      }
      const int key0 = kb + c * kMqKeys;
      const uint32_t kbuf = sK + st * C::kKVBytes;
      const uint32_t vbuf = sV + st * C::kKVBytes;
      // V rows past the partition's last key hold other blocks' data (maybe
      // NaN): they meet zero weights, and 0 x NaN would not vanish -> zero them
      const int valid_keys = ke - key0;
      if (valid_keys < kMqKeys) {
        unsigned char* vt = smem + C::kOffV + st * C::kKVBytes;
        for (int p = tid; p < (kMqKeys - valid_keys) * C::kChunks; p += kMqThreads) {
          const int r = valid_keys + p / C::kChunks, ch = p % C::kChunks;
          *reinterpret_cast<uint4*>(vt + tma_chunk(r, ch)) = make_uint4(0, 0, 0, 0);
        }
        mma_warps_sync();
      }
      if (active) {
        if (NP == 1)
          mq_chunk<T, D, 1>(kbuf, vbuf, ks, key0, qa, o, m_r, l_r, pos, pos_min, a.qscale, lane);
        else if (NP == 2)
          mq_chunk<T, D, 2>(kbuf, vbuf, 2 * ks, key0, qa, o, m_r, l_r, pos, pos_min, a.qscale,
                            lane);
        else
          mq_chunk<T, D, 4>(kbuf, vbuf, 0, key0, qa, o, m_r, l_r, pos, pos_min, a.qscale, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (!ok) break;

    // quad-reduced row sums
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 1);
      l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 2);
    }

    if (KS > 1) {
      // ---- combine the KS warps' states of each row group through shared
      // memory: (m, l) in a small array, o in the Q tile's space (free now),
      // 64 columns at a time
      const int nrows = RG * 16;   // 16 or 32
      if (active && (lane & 3) == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = rbase + (lane >> 2) + 8 * h;
          comb_m[ks * nrows + r] = m_r[h];
          comb_l[ks * nrows + r] = l_r[h];
        }
      }
      constexpr int CS = C::kCombStride;
      float* co = reinterpret_cast<float*>(smem + C::kOffQ);   // [KS][nrows][CS]
      const int tpr = kMqThreads / nrows;                      // threads per row: 8 or 4
      const int cols = 64 / tpr;
      // thread: row tid / tpr, columns k, k + tpr, k + 2 tpr, ... (k = tid % tpr)
      const int r = tid / tpr, k0 = tid % tpr;
      for (int half = 0; half < D / 64; ++half) {
        mma_warps_sync();   // (the Q tile is no longer read; the previous half is done)
        if (active) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int rr = rbase + (lane >> 2) + 8 * h;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<float2*>(co + (ks * nrows + rr) * CS + i * 8 + 2 * (lane & 3)) =
                  make_float2(o[half * 8 + i][2 * h], o[half * 8 + i][2 * h + 1]);
          }
        }
        mma_warps_sync();
        if (r < rows_here) {
          float M = -INFINITY;
          for (int w = 0; w < KS; ++w) M = fmaxf(M, comb_m[w * nrows + r]);
          const float Mu = M == -INFINITY ? 0.f : M;
          float wgt[4] = {0.f, 0.f, 0.f, 0.f}, L = 0.f;
          for (int w = 0; w < KS; ++w) {
            wgt[w] = softmax_exp2(comb_m[w * nrows + r] - Mu);
            L += wgt[w] * comb_l[w * nrows + r];
          }
          const int rr = row0 + r;
          const size_t orow = (size_t)(q0 + rr / G) * a.Hq + kvh * G + rr % G;
          if (nparts > 1) {
            const size_t prow = orow * a.pmax + part_idx;
            if (half == 0 && tid % tpr == 0) {
              a.ws_m[prow] = M;
              a.ws_l[prow] = L;
            }
            float* po = a.ws_o + prow * D + half * 64;
            for (int e = 0; e < cols; ++e) {
              const int col = k0 + e * tpr;
              float acc = 0.f;
              for (int w = 0; w < KS; ++w) acc += wgt[w] * co[(w * nrows + r) * CS + col];
              po[col] = acc;
            }
          } else {
            const float inv = 1.f / L;
            T* dst = outg + orow * D + half * 64;
            for (int e = 0; e < cols; ++e) {
              const int col = k0 + e * tpr;
              float acc = 0.f;
              for (int w = 0; w < KS; ++w) acc += wgt[w] * co[(w * nrows + r) * CS + col];
              dst[col] = Elem<T>::narrow(acc * inv);
            }
          }
        }
      }
      mma_warps_sync();   // the Q tile's space is free for the next item
      continue;
    }

    // ---- one warp per row group.  One partition: normalise and store the
    // tile's valid rows; several: leave (m, l, unnormalised o) for the merge
    if (active) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float l = l_r[h];
        const int r = rbase + (lane >> 2) + 8 * h;
        if (r >= rows_here) continue;
        const int rr = row0 + r;
        if (nparts > 1) {
          const size_t prow =
              ((size_t)(q0 + rr / G) * a.Hq + kvh * G + rr % G) * a.pmax + part_idx;
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
          *reinterpret_cast<uint32_t*>(dst + i * 8) =
              Mma<T>::pack(o[i][2 * h] * inv, o[i][2 * h + 1] * inv);
      }
    }
    mma_warps_sync();   // every warp has read the Q tile before the next item loads it
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
  CUtensorMap tk, tv;
  if ((e = make_pool_map(&tk, a.k_cache, a.dtype, a.NB, a.Hkv, a.D)) != cudaSuccess) return e;
  if ((e = make_pool_map(&tv, a.v_cache, a.dtype, a.NB, a.Hkv, a.D)) != cudaSuccess) return e;
  int sms = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  kern<<<2 * sms, C::kThreads, C::kSmem, stream>>>(tk, tv, a);   // persistent: 2 per SM
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
