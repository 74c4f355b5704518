// paged_decode.cuh -- split-KV paged decode attention and its partition merge.
//
// PhotonInfer README, "Key features / GPU-optimized kernels": batched paged
// attention over a block-wise KV cache, softmax computed in a numerically
// stable way, 128-bit vectorised loads; "Technical details / Paged attention":
// per-sequence cache offsets (here: block tables).
//
// Two launches per call, chained with programmatic dependent launch so each
// one's start-up overlaps its predecessor:
//   1. attention: a persistent grid that fills every SM.  Work items are
//      (sequence, partition, KV head); split-KV partitioning cuts each context
//      into ceil(ctx / part) partitions, so long sequences give many items and
//      short ones few.  In each CTA one producer warp derives its items from
//      context_lens and streams the K and V chunks of
//      the blocks they name from the pool into a ring of shared-memory stages
//      with 1-D bulk copies (cp.async.bulk, completion on an mbarrier); the
//      consumer warps compute scores, an online softmax and the weighted V sum
//      from shared memory.  A block's rows for one KV head are one contiguous
//      chunk of the pool ([num_blocks][Hkv][16][d]), so every copy is a single
//      16-byte-aligned run of 16*d elements.  A sequence with one partition
//      writes its output row directly; a longer one leaves (m, l, o) per
//      partition in the workspace;
//   2. merge: out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p with
//      M = max_p m_p, for every (sequence, q head) with two or more partitions,
//      and the zero rows of empty sequences.
//      (Merging inside the attention kernel, by the CTA that finishes a
//      sequence's last partition, needs a device-scope fence per partition;
//      under a full HBM stream those fences and the serialised merges cost far
//      more than this short kernel.)
//
// Consumer arithmetic.  Each consumer warp takes one 16-token block of a
// stage, in one of two forms (photon_debug_set_decode_consumer):
//  * tensor cores (the default for fp16/bf16 storage and G >= 2 query heads
//    per KV head): the producer brings the blocks as tensor-map copies with
//    the 128-byte swizzle, and the warp computes S^T = K Q^T (16 keys x the G
//    heads, padded to 8) and O^T += V^T P^T with mma.sync m16n8k16 from
//    conflict-free ldmatrix reads; P is fed as its storage-type rounding plus
//    the residual, so the weights keep ~2^-17 relative precision;
//  * CUDA cores (fp32 storage, G = 1): eight lanes cover one token row with
//    16-byte shared-memory loads (a quarter warp reads 128 contiguous bytes:
//    no bank conflicts), four rows per load step, four steps per block.  A
//    lane keeps its slice of the G query rows in registers, pre-multiplied by
//    scale*log2(e), so every loaded K/V element serves all G heads; scores are
//    summed over the eight lanes of a row with three xor-shuffles.
// Either way the softmax is the online form in the log2 domain: per block the
// warp takes the block maximum, rescales its running (l, o) by
// 2^(m_old - m_new) and accumulates 2^(s - m_new) and 2^(s - m_new) * V.  At
// the end of an item the warps' states are combined through shared memory by
// the same log-sum-exp rule.
#pragma once

#include <float.h>
#include <math.h>
#include <string.h>

#include <type_traits>

#include "photon_common.cuh"

namespace photon {

template <typename T, int D, int G>
struct DecodeCfg {
  static constexpr int kChunk = Elem<T>::kPerChunk;          // elements per 16 bytes
  static constexpr int kRowChunks = D * (int)sizeof(T) / 16;  // 16-byte chunks per row
  static constexpr int kLanesPerRow = 8;
  static constexpr int kPPL = kRowChunks / kLanesPerRow;      // chunks per lane per row
  static constexpr int kEPL = kPPL * kChunk;                  // elements per lane
  static constexpr int kRowsPerStep = 32 / kLanesPerRow;      // rows per warp load step
  static constexpr int kSteps = kBlockSize / kRowsPerStep;    // load steps per block
  static_assert(kRowChunks % kLanesPerRow == 0, "row must split over 8 lanes");
};

// Stage header written by the producer, read by the consumers after the
// stage's full barrier completes.
struct StageHdr {
  int b, kvh, p, nparts;
  int tok_end, blk0;   // exclusive token end of the item; first logical block of the stage
  int nblk;            // blocks carried by this stage (<= consumer warps)
  int flags;           // kFirst | kLast | kDone, valid-block mask << 8
  // fused step: the stage block (new_warp) whose row new_row is this
  // sequence's new token, to be stored at physical block new_phys; -1 if none
  int new_warp, new_phys, new_row;
  int pos;             // the sequence's new-token position, ctx - 1 (RoPE angle, causal limit)
  int q0, nq;          // query rows of the item's sequence (decode: b and 1)
};
enum : int { kFirst = 1, kLast = 2, kDone = 4 };

// Split-KV partitions of a context of ctx tokens with partition size part:
// nfull = ctx / part full partitions, then the remainder.  When there are two
// or more full ones the last of them is cut in two halves (of part / 32 * 16
// tokens and the rest), so that the work list can end with small items:
// partitions 0 .. nfull - 2 full, nfull - 1 and nfull the halves, nfull + 1
// the remainder.
__host__ __device__ __forceinline__ int partition_split(int ctx, int part) {
  return ctx / part >= 2 && part >= 32 ? 1 : 0;
}
__host__ __device__ __forceinline__ int partitions_of(int ctx, int part) {
  return ctx / part + partition_split(ctx, part) + (ctx % part != 0 ? 1 : 0);
}
__device__ __forceinline__ void partition_range(int ctx, int part, int p, int& begin, int& end) {
  const int nfull = ctx / part;
  if (!partition_split(ctx, part) || p < nfull - 1) {
    begin = p * part;
    end = min(begin + part, ctx);
    return;
  }
  const int last = (nfull - 1) * part, half = part / 32 * 16;
  begin = p == nfull - 1 ? last : p == nfull ? last + half : nfull * part;
  end = p == nfull - 1 ? last + half : p == nfull ? nfull * part : ctx;
}

// Runs of the work list: partition 0 of every sequence, the further full
// partitions, the halves of the last full ones, then up to log2(4096/16) + 1
// = 9 classes of tail partitions.
constexpr int kMaxRuns = 12;

// Persistent-kernel geometry: NC consumer warps, 1 producer warp, S ring stages.
// M: the tensor-core consumer, whose blocks arrive as swizzled tensor-map
// copies: every block starts on a 1024-byte swizzle atom (the dynamic
// shared-memory base is aligned up at run time, hence kAlignPad), and the
// fused step's new K/V row lands in a side slot of its stage.
// X: few-token multi-query mode (tensor-core consumer only): up to 8 query
// slots (token, head) per item instead of the G heads of one token.
// F: the cache holds e4m3 codes (one byte per element; q and out stay fp16):
// the stages carry the code blocks as tensor-map copies in the swizzled
// layout of code_chunk, and the tensor-core math widens the codes to fp16 in
// registers as it loads its fragments.
#ifndef PHOTON_FP8_BPW
#define PHOTON_FP8_BPW 2
#endif
template <typename T, int D, int G, int NC, int S, bool R = false, bool M = false, bool X = false,
          bool F = false>
struct PersistCfg {
  using C = DecodeCfg<T, D, G>;
  static constexpr int kThreads = (NC + 1) * 32;
  static constexpr int kBlockElems = kBlockSize * D;
  static constexpr int kElemBytes = F ? 1 : (int)sizeof(T);       // one cache element
  static constexpr int kBlockBytes = kBlockElems * kElemBytes;    // one cache block (a stage slot)
  static constexpr int kSlots = X ? 8 : G;                      // query rows per item
  static constexpr int kQBytes = kSlots * D * (int)sizeof(T);
  // with RoPE the item's (cos, sin) row, D/2 float pairs, follows its q rows
  static constexpr int kCsBytes = R ? 4 * D : 0;
  static constexpr int kQStride = (kQBytes + kCsBytes + 127) / 128 * 128;
  // blocks per warp and stage (PHOTON_FP8_BPW, e4m3 cache only; 2 by
  // default): each consumer warp takes two consecutive blocks of a stage,
  // which spreads the stage protocol over twice the bytes and gives the warp
  // two blocks of independent work; the larger stages leave room for two
  // CTAs per SM instead of three.  qwen_b64 fp8 decode: 56.9 us with two,
  // 60.0 us with one block per warp (three CTAs per SM)
  static constexpr int kBPW = F ? PHOTON_FP8_BPW : 1;
  static constexpr int kStageBlocks = NC * kBPW;
  static constexpr int kStageBytes = 2 * kStageBlocks * kBlockBytes;  // K blocks, then V blocks
  static constexpr int kOffFull = 0;
  static constexpr int kOffEmpty = kOffFull + 8 * S;
  static constexpr int kOffSync = kOffEmpty + 8 * S;
  static constexpr int kOffAbort = kOffSync + 8;
  static constexpr int kOffRuns = kOffAbort + 4;                        // int[kMaxRuns + 1]
  static constexpr int kOffHdr = (kOffRuns + 4 * (kMaxRuns + 1) + 15) / 16 * 16;
  static constexpr int kOffQ = (kOffHdr + (int)sizeof(StageHdr) * S + 127) / 128 * 128;
  static constexpr int kKVAlign = M ? 1024 : 128;
  static constexpr int kOffKV = (kOffQ + kQStride * S + kKVAlign - 1) / kKVAlign * kKVAlign;
  // M only: the new token's K row then V row, per stage
  static constexpr int kSideBytes = M && !F ? 2 * D * (int)sizeof(T) : 0;
  static constexpr int kOffSide = kOffKV + kStageBytes * S;
  // Per-warp (m, l) at an item's end, double-buffered by item parity.  The
  // warps' o rows (kSlots x D fp32 each) go to their own K (then V) block
  // areas of the item's last stage, which is released only after the combine.
  static constexpr int kOffPm = kOffSide + kSideBytes * S;
  static constexpr int kOffPl = kOffPm + 4 * 2 * NC * kSlots;   // float[2][NC][kSlots]
  static constexpr int kAlignPad = M ? 1024 : 0;
  static constexpr int kSmemBytes = kOffPl + 4 * 2 * NC * kSlots + kAlignPad;
  static constexpr int kPoRowsPerBlock = kBlockBytes / (D * 4);  // o rows in one block area
  static_assert(kSlots <= 2 * kPoRowsPerBlock, "a warp's o rows must fit its K and V block areas");
  // the producer's 32-entry block-table slices must split into whole stages
  static_assert(NC >= 1 && NC <= 32 && 32 % kStageBlocks == 0 && kStageBlocks <= 8,
                "blocks per stage must divide 32 and fit the stage header's mask");
  static_assert(!X || (M && !R), "the few-token mode runs on the tensor-core consumer, no RoPE");
  static_assert(!M || (kBlockBytes % 1024 == 0 && sizeof(T) == 2), "swizzled blocks");
  static_assert(!F || (M && !R && !X && std::is_same<T, __half>::value),
                "the fp8 cache: plain decode on the tensor-core consumer, fp16 q and out");
};

// ------------------------------------------------------------------ consumer math
// Process one 16-token block held in shared memory (ks: K rows, vs: V rows,
// row-major [16][D]); rows >= n_valid are masked.
template <typename T, int D, int G>
__device__ __forceinline__ void attend_block(const T* __restrict__ ks, const T* __restrict__ vs,
                                             int n_valid, const float (&qf)[G][DecodeCfg<T, D, G>::kEPL],
                                             float (&m)[G], float (&l)[G],
                                             float (&o)[G][DecodeCfg<T, D, G>::kEPL], int lane) {
  using C = DecodeCfg<T, D, G>;
  const int c = lane & 7, tg = lane >> 3;
  float sc[C::kSteps][G];
  {
    uint4 kr[C::kSteps][C::kPPL];
#pragma unroll
    for (int s = 0; s < C::kSteps; ++s) {
      const int row = s * C::kRowsPerStep + tg;
#pragma unroll
      for (int i = 0; i < C::kPPL; ++i)
        kr[s][i] = row < n_valid
                       ? *reinterpret_cast<const uint4*>(ks + row * D + (c + 8 * i) * C::kChunk)
                       : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int s = 0; s < C::kSteps; ++s) {
      float kf[C::kEPL];
#pragma unroll
      for (int i = 0; i < C::kPPL; ++i) Elem<T>::widen(kr[s][i], kf + i * C::kChunk);
      const int row = s * C::kRowsPerStep + tg;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < C::kEPL; ++e) acc = fmaf(qf[g][e], kf[e], acc);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        sc[s][g] = row < n_valid ? acc : -INFINITY;
      }
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float mx = sc[0][g];
#pragma unroll
    for (int s = 1; s < C::kSteps; ++s) mx = fmaxf(mx, sc[s][g]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    if (mx > m[g]) {  // warp-uniform: m and mx agree on all lanes
      const float corr = softmax_exp2(m[g] - mx);
      l[g] *= corr;
#pragma unroll
      for (int e = 0; e < C::kEPL; ++e) o[g][e] *= corr;
      m[g] = mx;
    }
  }
  uint4 vr[C::kSteps][C::kPPL];
#pragma unroll
  for (int s = 0; s < C::kSteps; ++s) {
    const int row = s * C::kRowsPerStep + tg;
#pragma unroll
    for (int i = 0; i < C::kPPL; ++i)
      vr[s][i] = row < n_valid
                     ? *reinterpret_cast<const uint4*>(vs + row * D + (c + 8 * i) * C::kChunk)
                     : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int s = 0; s < C::kSteps; ++s) {
    float vf[C::kEPL];
#pragma unroll
    for (int i = 0; i < C::kPPL; ++i) Elem<T>::widen(vr[s][i], vf + i * C::kChunk);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float pw = softmax_exp2(sc[s][g] - m[g]);   // 0 for masked rows
      l[g] += pw;
#pragma unroll
      for (int e = 0; e < C::kEPL; ++e) o[g][e] = fmaf(pw, vf[e], o[g][e]);
    }
  }
}

// ------------------------------------------------------------------ tensor-core consumer math
// Byte offset of 16-byte chunk `chunk` (0 .. D/8 - 1) of row `row` of a block
// as the tensor-map copies lay it out: D/64 column halves of 16 rows x 128 B,
// the 128-byte swizzle inside each 8-row atom.
__device__ __forceinline__ uint32_t blk_chunk(int row, int chunk) {
  return (uint32_t)((chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// One 16-token block for one warp on mma.sync m16n8k16 (fp32 accumulate).
// The G query rows of the KV head's group are the n = 8 columns (slots >= G
// hold zero rows), so the block's keys and the head dimension are the m side:
//   S^T (16 keys x 8)  = K (16 x D) * Q^T (D x 8),       D/16 products;
//   O^T (D x 8)       += V^T (D x 16 keys) * P^T (16 x 8), D/16 products per
//                        half of P (below).
// Lane l holds query slots 2(l%4) and 2(l%4)+1: their scores for keys l/4 and
// l/4 + 8, their running max m and a partial sum l over the keys this lane
// sees, and their O^T accumulators for dims 16i + l/4 and 16i + l/4 + 8.
// P^T, the B operand of the second product, is the score fragment packed and
// transposed 8x8 at a time (movmatrix).  P is split into a rounded part and
// its rounding residual, two products, so the weights enter the sum with
// about 2^-17 relative error instead of one storage-type rounding; the sums l
// take the fp32 weights.  Scores are the fp32 products times qscale.
// kQLo: q is an fp32 value (rotated by RoPE) given as bq + bql, its rounding
// to the storage type and the residual, so S^T takes two products per step.
// Rows >= n_valid: their scores are set to -inf and their V rows must be
// zero (0 * NaN would otherwise reach the accumulators).
// kCausal (few-token multi-query mode): the lane's two slots see keys up to
// positions lim[0], lim[1] (key0 = position of the block's row 0); a slot can
// then have no key in a block, or in a whole item, so the max and rescale
// steps guard against -inf - -inf.
//
// kCodes (e4m3 cache, fp16 q): kblk / vblk hold the blocks' codes, one byte per
// element, rows of D codes in the tensor copies' swizzled layout (code_chunk),
// and the fragments are widened from the codes in registers: ldmatrix moves
// code pairs as 16-bit elements, cvt turns each pair into an fp16 pair.  The
// head dimension is walked in a permuted order that keeps every widened pair
// where its fragment wants it:
//   S^T: k-step kk covers code chunk kk (dims 16kk .. 16kk+15); the MMA's k
//        index 2t+j is dim 16kk + 4t + j, 2t+8+j is dim 16kk + 4t + 2 + j
//        (t = lane % 4), so bq must hold q's dims in that order;
//   O^T: tile i covers dims 16i .. 16i+15 with MMA row r as dim 16i + 2r and
//        row r + 8 as dim 16i + 2r + 1 (the caller stores o in that order).
template <int D>
__device__ __forceinline__ uint32_t code_chunk(int row, int chunk) {
  if constexpr (D == 128) return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
  else return (uint32_t)(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}
__device__ __forceinline__ void widen_e4m3x4(uint32_t codes, uint32_t& lo, uint32_t& hi);
template <typename T, int D, bool kQLo, bool kCausal, bool kCodes = false>
__device__ __forceinline__ void attend_block_mma(uint32_t kblk, uint32_t vblk, int n_valid,
                                                 float qscale, const uint32_t (&bq)[D / 16][2],
                                                 const uint32_t (&bql)[D / 16][2],
                                                 float (&m)[2], float (&l)[2],
                                                 float (&o)[D / 16][4], int lane, int key0,
                                                 const int (&lim)[2]) {
  const int r = lane >> 2;
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (kCodes) {
    // ldmatrix row addresses: matrices (keys 0-7 | 8-15) x (code chunks 2j | 2j+1);
    // two independent accumulator chains (even and odd chunks)
    const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int khi = lane >> 4;
    float s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
      uint32_t c0, c1, c2, c3;
      ldsm_x4(kblk + code_chunk<D>(krow, 2 * j + khi), c0, c1, c2, c3);
      uint32_t a[4];
      widen_e4m3x4(c0, a[0], a[2]);
      widen_e4m3x4(c1, a[1], a[3]);
      Mma<T>::run(s, a, bq[2 * j][0], bq[2 * j][1]);
      widen_e4m3x4(c2, a[0], a[2]);
      widen_e4m3x4(c3, a[1], a[3]);
      Mma<T>::run(s2, a, bq[2 * j + 1][0], bq[2 * j + 1][1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) s[i] += s2[i];
  } else {
    // ldmatrix row addresses: matrices (keys 0-7 | 8-15) x (dims lo | hi of the k-step)
    const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int khi = lane >> 4;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a[4];
      ldsm_x4(kblk + blk_chunk(krow, 2 * kk + khi), a[0], a[1], a[2], a[3]);
      Mma<T>::run(s, a, bq[kk][0], bq[kk][1]);
      if constexpr (kQLo) Mma<T>::run(s, a, bql[kk][0], bql[kk][1]);
    }
  }
  const bool v0 = r < n_valid, v1 = r + 8 < n_valid;
  bool ok[4] = {v0, v0, v1, v1};
  if constexpr (kCausal) {
    ok[0] = ok[0] && key0 + r <= lim[0];
    ok[1] = ok[1] && key0 + r <= lim[1];
    ok[2] = ok[2] && key0 + r + 8 <= lim[0];
    ok[3] = ok[3] && key0 + r + 8 <= lim[1];
  }
  const float x0 = ok[0] ? s[0] * qscale : -INFINITY;   // key r,     slot 2t
  const float x1 = ok[1] ? s[1] * qscale : -INFINITY;   // key r,     slot 2t + 1
  const float x2 = ok[2] ? s[2] * qscale : -INFINITY;   // key r + 8, slot 2t
  const float x3 = ok[3] ? s[3] * qscale : -INFINITY;   // key r + 8, slot 2t + 1
  float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
  }
  // decode: key 0 is always valid, so the block maxima are finite
  const float n0 = fmaxf(m[0], mx0), n1 = fmaxf(m[1], mx1);
  if (__any_sync(0xffffffffu, n0 > m[0] || n1 > m[1])) {
    float c0 = softmax_exp2(m[0] - n0), c1 = softmax_exp2(m[1] - n1);
    if constexpr (kCausal) {
      c0 = n0 > m[0] ? c0 : 1.f;   // also covers m = n = -inf
      c1 = n1 > m[1] ? c1 : 1.f;
    }
    l[0] *= c0;
    l[1] *= c1;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      o[i][0] *= c0;
      o[i][1] *= c1;
      o[i][2] *= c0;
      o[i][3] *= c1;
    }
    m[0] = n0;
    m[1] = n1;
  }
  // a slot with no key so far has m = -inf and only -inf scores: weights 0
  const float mr0 = kCausal && m[0] == -INFINITY ? 0.f : m[0];
  const float mr1 = kCausal && m[1] == -INFINITY ? 0.f : m[1];
  const float p0 = softmax_exp2(x0 - mr0), p1 = softmax_exp2(x1 - mr1);
  const float p2 = softmax_exp2(x2 - mr0), p3 = softmax_exp2(x3 - mr1);
  l[0] += p0 + p2;
  l[1] += p1 + p3;
  const uint32_t h01 = Mma<T>::pack(p0, p1), h23 = Mma<T>::pack(p2, p3);
  const float2 r01 = Mma<T>::unpack(h01), r23 = Mma<T>::unpack(h23);
  const uint32_t b0 = movmatrix_trans(h01), b1 = movmatrix_trans(h23);
  const uint32_t e0 = movmatrix_trans(Mma<T>::pack(p0 - r01.x, p1 - r01.y));
  const uint32_t e1 = movmatrix_trans(Mma<T>::pack(p2 - r23.x, p3 - r23.y));
  if constexpr (kCodes) {
    // ldmatrix.trans over code pairs: matrices (keys 0-7 | 8-15) x (code
    // chunks 2j | 2j+1).  Lane (r, t) receives, per matrix, codes 2r and
    // 2r+1 of keys 2t and 2t+1; a byte permute pairs them by dim (keys 2t,
    // 2t+1 at dim 2r, then at dim 2r+1) and cvt widens each pair.
    const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int vhi = lane >> 4;
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
      uint32_t c[4];
      ldsm_x4_trans(vblk + code_chunk<D>(vrow, 2 * j + vhi), c[0], c[1], c[2], c[3]);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t w0 = __byte_perm(c[2 * h], 0u, 0x3120);
        const uint32_t w1 = __byte_perm(c[2 * h + 1], 0u, 0x3120);
        uint32_t a[4];
        widen_e4m3x4(w0, a[0], a[1]);
        widen_e4m3x4(w1, a[2], a[3]);
        Mma<T>::run(o[2 * j + h], a, b0, b1);
        Mma<T>::run(o[2 * j + h], a, e0, e1);
      }
    }
  } else {
    // ldmatrix.trans row addresses: matrices (keys 0-7 | 8-15) x (dims lo | hi of the tile)
    const int vrow = (lane & 7) + (lane >> 4) * 8;
    const int vhi = (lane >> 3) & 1;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      uint32_t a[4];
      ldsm_x4_trans(vblk + blk_chunk(vrow, 2 * i + vhi), a[0], a[1], a[2], a[3]);
      Mma<T>::run(o[i], a, b0, b1);
      Mma<T>::run(o[i], a, e0, e1);
    }
  }
}

// Four e4m3 codes (bytes 0..3 of `codes`) widened exactly to two fp16
// pairs: bytes 0, 1 into lo, bytes 2, 3 into hi (the lower byte's value in
// the low half).  Every e4m3 value is an fp16 value.  The 16-bit halves are
// handed to the conversions as register halves, so no shift separates them.
__device__ __forceinline__ void widen_e4m3x4(uint32_t codes, uint32_t& lo, uint32_t& hi) {
  asm("{\n.reg .b16 l, h;\nmov.b32 {l, h}, %2;\ncvt.rn.f16x2.e4m3x2 %0, l;\n"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(codes));
}

// ------------------------------------------------------------------ RoPE
// Rotate-half rotary embedding: for k < D/2 the pair (x[k], x[k + D/2]) turns
// by the table's (cos, sin) for (pos, k).  Positions outside the table are
// flagged and left unrotated.
//
// The item's (cos, sin) row for its position sits in shared memory next to
// its q rows (the producer copies it with them).
//
// q rows, in the lane's registers: lane c of a row group holds chunks
// c, c + 8, ... of each row; a pair's partner sits in the same lane when the
// chunk distance D/2/kChunk is a multiple of 8, otherwise (16-bit D = 64) in
// lane c ^ 4 of the same row group.
template <typename T, int D, int G>
__device__ __forceinline__ void rope_q(float (&qf)[G][DecodeCfg<T, D, G>::kEPL],
                                       const float2* __restrict__ cs, int max_pos, int pos,
                                       int c, uint32_t* err, int ctid) {
  using C = DecodeCfg<T, D, G>;
  constexpr int kHalfChunks = (D / 2) / C::kChunk;
  constexpr bool kInLane = kHalfChunks % 8 == 0;
  constexpr int kSlotShift = kInLane ? (kHalfChunks / 8) * C::kChunk : 0;
  if (pos < 0 || pos >= max_pos) {
    if (ctid == 0) raise_error(err, kErrPosition);
    return;
  }
  const float2* row = cs;
  if constexpr (kInLane) {
    // slots of the lower half are the first kEPL/2; each one's partner is
    // kSlotShift further on in the same lane
#pragma unroll
    for (int s = 0; s < C::kEPL / 2; ++s) {
      const int e = (c + 8 * (s / C::kChunk)) * C::kChunk + s % C::kChunk;
      const float2 t = row[e];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float x0 = qf[g][s], x1 = qf[g][s + kSlotShift];
        qf[g][s] = x0 * t.x - x1 * t.y;
        qf[g][s + kSlotShift] = x1 * t.x + x0 * t.y;
      }
    }
  } else {
    const bool lower = c < 4;
#pragma unroll
    for (int s = 0; s < C::kEPL; ++s) {
      const int e = (c + 8 * (s / C::kChunk)) * C::kChunk + s % C::kChunk;
      const float2 t = row[lower ? e : e - D / 2];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float x = qf[g][s];
        const float partner = __shfl_xor_sync(0xffffffffu, x, 4);
        qf[g][s] = lower ? x * t.x - partner * t.y : x * t.x + partner * t.y;
      }
    }
  }
}

// Pairs k = lane, lane + 32, ... of the item's (cos, sin) row, kept in
// registers for the new K row (the shared copy is recycled with its stage).
template <int D>
struct RopeLaneCs {
  float2 w[(D / 2 + 31) / 32];
};

// One row of D elements in shared memory, rotated in place by a warp and
// rounded back to the storage type.
template <typename T, int D>
__device__ __forceinline__ void rope_row(T* row, const RopeLaneCs<D>& cs, int max_pos, int pos,
                                         int lane) {
  if (pos < 0 || pos >= max_pos) return;  // flagged by rope_q of the same item
#pragma unroll
  for (int i = 0; i < (D / 2 + 31) / 32; ++i) {
    const int k = lane + 32 * i;
    if (k >= D / 2) break;
    const float2 w = cs.w[i];
    const float x0 = Elem<T>::to_f32(row[k]), x1 = Elem<T>::to_f32(row[k + D / 2]);
    row[k] = Elem<T>::narrow(x0 * w.x - x1 * w.y);
    row[k + D / 2] = Elem<T>::narrow(x1 * w.x + x0 * w.y);
  }
}

// Arrive-and-wait of the NC consumer warps on `bar` (bounded).
__device__ __forceinline__ bool consumer_sync(uint64_t* bar, uint32_t& phase, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = mbar_wait_bounded(bar, phase);
  phase ^= 1u;
  return ok;
}

#ifdef PHOTON_PROBE
// Per-CTA timeline for tuning builds only (never compiled into the library by
// default): [0] start, [1] first stage issued, [2] producer done, [3] first
// stage consumed, [4] consumers done, [7] items.
constexpr int kProbeCtas = 1024;
constexpr int kProbeSlots = 48;  // [8 + 2k]: item k's first copy issued, [9 + 2k]: item k combined
static __device__ unsigned long long g_probe[kProbeCtas][kProbeSlots];
// merge kernel CTAs: [0] entry, [1] past the dependency wait, [2] done
static __device__ unsigned long long g_probe_merge[4096][4];
// a one-thread kernel's time stamp, launched by the tuning harness just
// before a call (the gap to the attention kernel's entry is its launch)
static __device__ unsigned long long g_probe_stamp[2];
static __global__ void probe_stamp_kernel(int slot) { g_probe_stamp[slot] = global_timer_ns(); }
// the same with a large shared-memory request (the carveout of the attention
// kernel), to tell a launch's own cost from a carveout change
static __global__ void probe_stamp_big_kernel() {
  extern __shared__ unsigned char stamp_smem[];
  stamp_smem[threadIdx.x] = 0;
  g_probe_stamp[0] = global_timer_ns();
}
#define PROBE_SET(i, v) \
  do { if (blockIdx.x < kProbeCtas && (i) < kProbeSlots) g_probe[blockIdx.x][i] = (v); } while (0)
#else
#define PROBE_SET(i, v) do { } while (0)
#endif

// ------------------------------------------------------------------ attention kernel
// kRope: the fused step with the rotary embedding (q rows and the new K row
// turn by the token's position); a separate instantiation, so the plain path
// carries none of it.
// kMma: the tensor-core consumer (attend_block_mma); its K/V blocks arrive as
// tensor-map copies (tmk, tmv: the pools as rows of D elements, boxes of 16
// rows x 64 elements, 128-byte swizzle).  The other instantiations take the
// maps but never read them.
// kMulti: the few-token multi-query mode (photon_paged_multi_query with
// max_query_len * G <= 8): an item's query slots are the (token, head) pairs
// of its sequence's n query tokens, each with its causal limit.
// kFp8: the e4m3 cache (photon_paged_decode_fp8): K/V blocks arrive as
// swizzled tensor-map boxes of codes, and the block math widens the codes it
// needs in registers; the K scale is folded into qscale, the V scale into
// the item's combine.  Two CTAs share an SM with two blocks per warp, three
// with one (PHOTON_FP8_CTAS, a tuning knob for the register cap).
#ifndef PHOTON_FP8_CTAS
#define PHOTON_FP8_CTAS (PHOTON_FP8_BPW > 1 ? 2 : 3)
#endif
template <typename T, int D, int G, int NC, int S, bool kRope, bool kMma, bool kMulti,
          bool kFp8 = false>
__global__ void __launch_bounds__((NC + 1) * 32, kFp8 && NC <= 4 ? PHOTON_FP8_CTAS : 1)
    paged_decode_attention_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                                  const __grid_constant__ CUtensorMap tmv) {
  using PC = PersistCfg<T, D, G, NC, S, kRope, kMma, kMulti, kFp8>;
  using C = DecodeCfg<T, D, G>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // swizzled tensor copies want their 1024-byte atoms aligned in the shared window
  unsigned char* const smem =
      kMma ? smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u) : smem_raw;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + PC::kOffFull);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + PC::kOffEmpty);
  uint64_t* sync = reinterpret_cast<uint64_t*>(smem + PC::kOffSync);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + PC::kOffAbort);
  StageHdr* hdr = reinterpret_cast<StageHdr*>(smem + PC::kOffHdr);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) PROBE_SET(5, global_timer_ns());
  // the producer's first tensor copies need the maps' descriptors
  if (kMma && threadIdx.x == NC * 32) {
    prefetch_tensor_map(&tmk);
    prefetch_tensor_map(&tmv);
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NC);
    }
    mbar_init(sync, NC);
    *abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  // Warm L2 with the context lengths and block tables while the previous
  // kernel finishes (a hint only: the values are read after the wait).
  {
    const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t nthr = (size_t)gridDim.x * blockDim.x;
    const size_t tbytes = (size_t)a.B * a.MBS * sizeof(int32_t);
    for (size_t off = tid * 128; off < tbytes; off += nthr * 128)
      prefetch_l2(reinterpret_cast<const char*>(a.block_tables) + off);
    for (size_t off = tid * 128; off < (size_t)a.B * sizeof(int32_t); off += nthr * 128)
      prefetch_l2(reinterpret_cast<const char*>(a.context_lens) + off);
  }
  // Everything below may read what the previous kernel in the stream wrote
  // (the cache write's rows, context lengths, block tables, q).
  pdl_wait_primary();
  // The merge kernel may be scheduled as CTAs retire; it waits for this grid.
  pdl_launch_dependents();

  const int span = a.MBS * kBlockSize;
  auto ctx_of = [&](int b) -> int {
    const int c = b < a.B ? __ldg(a.context_lens + b) : 0;
    if constexpr (kMulti) {
      // sequences without query tokens, or whose rows or lengths the merge
      // kernel rejects, get no items
      if (b >= a.B) return 0;
      const int q0 = __ldg(a.query_start + b), n = __ldg(a.query_start + b + 1) - q0;
      if (n <= 0 || n > a.max_q || q0 < 0 || q0 > a.num_tokens - n || c < n || c > span) return 0;
      return c;
    }
    return (c < 0 || c > span) ? 0 : c;  // rejected lengths count as empty
  };
  auto fail = [&](void) {
    if (lane == 0) {
      raise_error(a.err, kErrTimeout);
      *abort_flag = 1;
    }
  };

  if (warp == NC) {
    // ================================================================ producer
    // Work list, derived here from context_lens with no planning kernel.  The
    // (sequence, partition) pairs come in runs: first partition 0 of every
    // sequence (sequence order: pair q is sequence q, located without any
    // count, so a CTA's first item and its block-table slice load together
    // with the context lengths), then every further full partition (sequence
    // order, then partition order), then the partial tail partitions, class
    // by class from the longest to the shortest -- so the items handed out
    // last are the smallest (longest-processing-time first, without a sort).
    // Each pair is expanded over the KV heads (item = pair * Hkv + kvh); an
    // empty sequence's partition 0 is an item with no blocks and is skipped.
    // For the runs after the first the warp keeps a window of 32 sequences
    // (lane j: sequence wb + j's context length, its pair count in the
    // current run and the pairs before it) and slides it forward as its
    // items advance, with the next window's lengths already loaded.  A
    // software pipeline keeps every round trip off the copy stream: while
    // item i's stages are issued, the block-table slice of item i+1 is in
    // flight and the index of item i+2 is taken (then located).
    PROBE_SET(0, global_timer_ns());
    // Run sizes of the work list, counted by this warp: run 0 holds partition
    // 0 of each sequence, run 1 the full partitions after it, run 2 the two
    // halves of each sequence's last full partition (partition_split), run
    // 3 + k the tail partitions of class k (of sequences with a full
    // partition before them), where a tail of nb blocks (of P16 = part / 16
    // per partition) has class floor(log2(floor(P16 / nb))): halves of the
    // partition size, largest first.  Only this warp needs them, so the
    // consumers never wait for it.
    const int P16 = a.part / kBlockSize;
    auto tail_class = [&](int ctxv) -> int {
      const int tail = ctxv % a.part;
      if (!tail || ctxv < a.part) return -1;
      const int nb = (tail + kBlockSize - 1) / kBlockSize;
      return 31 - __clz(P16 / nb);
    };
    int* run_start = reinterpret_cast<int*>(smem + PC::kOffRuns);  // pairs before run r
    const int N = gridDim.x;
    // This CTA's first item (g0): partition 0 of sequence g0 / Hkv when there
    // is one; its context length, table slice and new-row slot are loaded
    // now, beside the windows of context lengths below.
    const int b_first = blockIdx.x / a.Hkv;
    const bool first_in_run0 = b_first < a.B;
    const int ctx_first = first_in_run0 ? ctx_of(b_first) : 0;
    const int tb_first =
        first_in_run0 && lane < min(32, a.MBS) ? __ldg(a.block_tables + (size_t)b_first * a.MBS + lane)
                                              : -1;
    const bool fused = a.k_new != nullptr;
    const long long sl_first = fused && first_in_run0 ? (long long)__ldg(a.slot_mapping + b_first) : -1ll;
    // The first two windows of context lengths are loaded once, up front, and
    // serve both this count and the walk below (a batch of up to 64 sequences
    // needs no other load).
    const int ctx_w0 = ctx_of(lane), ctx_w1 = ctx_of(32 + lane);
    const bool dynamic =
        __shfl_sync(0xffffffffu, lane == 0 && a.ws_ctrl[0] == kQueueReady ? 1 : 0, 0) != 0;
    // The run sizes (the second item on needs them).  When the first item is
    // partition 0 of a sequence, they are counted right after its first
    // stage is issued, so the counting stays off the path to the first copy.
    auto count_runs = [&]() {
      int cnt[kMaxRuns];
#pragma unroll
      for (int r = 0; r < kMaxRuns; ++r) cnt[r] = 0;
      auto count = [&](int c) {
        const int split = partition_split(c, a.part);
        cnt[1] += c >= a.part ? c / a.part - 1 - split : 0;
        cnt[2] += 2 * split;
        const int k = tail_class(c);
#pragma unroll
        for (int r = 3; r < kMaxRuns; ++r) cnt[r] += (k == r - 3) ? 1 : 0;
      };
      count(ctx_w0);
      count(ctx_w1);
      for (int b = 64 + lane; b < a.B; b += 32) count(ctx_of(b));
      int acc = 0;
#pragma unroll
      for (int r = 1; r < kMaxRuns; ++r) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cnt[r] += __shfl_xor_sync(0xffffffffu, cnt[r], o);
      }
      cnt[0] = a.B;
#pragma unroll
      for (int r = 0; r < kMaxRuns; ++r) {
        if (lane == 0) run_start[r] = acc;
        acc += cnt[r];
      }
      if (lane == 0) run_start[kMaxRuns] = acc;
      __syncwarp();
      PROBE_SET(6, global_timer_ns());
    };
    // every K/V byte of the call is read once: evict first from L2, so the
    // partials the merge kernel reads back stay there
    const uint64_t kv_policy = l2_evict_first_policy();
    const T* kpool = static_cast<const T*>(a.k_cache);
    const T* vpool = static_cast<const T*>(a.v_cache);
    const T* qbase = static_cast<const T*>(a.q);
    uint32_t st = 0;
    bool aborted = false;
    int items_done = 0;

    // the run the window walk is in: 1 full partitions, 2 halves, 3 + k tails of class k
    int run = 1;
    int wb = 0, wbase = 0, w_ctx = 0, w_np = 0, w_excl = 0, w_tot = 0;
    auto set_window = [&](int ctxv) {
      w_ctx = ctxv;
      const int split = partition_split(ctxv, a.part);
      w_np = run == 1   ? (ctxv >= a.part ? ctxv / a.part - 1 - split : 0)
             : run == 2 ? 2 * split
                        : (tail_class(ctxv) == run - 3 ? 1 : 0);
      int incl = w_np;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      w_excl = incl - w_np;
      w_tot = __shfl_sync(0xffffffffu, incl, 31);
    };
    // The first two windows stay in registers: a batch of up to 64 sequences
    // never reloads context lengths when a new run starts.
    set_window(ctx_w0);
    int pre_ctx = ctx_w1;
    // Partition 0 of sequence b (run 0), from its context length.
    auto first_partition = [&](int b, int ctxb, WorkItem& it) {
      it.b = b;
      it.p = 0;
      it.tok_begin = 0;
      it.tok_end = min(ctxb, a.part);
      it.nparts = partitions_of(ctxb, a.part);
      if constexpr (kRope || kMulti) it.ctx = ctxb;
      if constexpr (kMulti) {
        it.q0 = __ldg(a.query_start + b);
        it.nq = __ldg(a.query_start + b + 1) - it.q0;
      }
    };
    // (sequence, partition) of pair index `pair`; false past the last pair.
    // Pairs after run 0 must be asked for in nondecreasing order.
    auto locate = [&](int pair, WorkItem& it) -> bool {
      if (pair >= run_start[kMaxRuns]) return false;
      if (pair < run_start[1]) {
        // run 0: pair q is sequence q
        const int ctxb = pair < 32   ? __shfl_sync(0xffffffffu, ctx_w0, pair)
                         : pair < 64 ? __shfl_sync(0xffffffffu, ctx_w1, pair - 32)
                                     : ctx_of(pair);
        first_partition(pair, ctxb, it);
        return true;
      }
      if (pair >= run_start[run + 1]) {
        do {
          ++run;
        } while (pair >= run_start[run + 1]);
        wb = 0;
        wbase = 0;
        set_window(ctx_w0);
        pre_ctx = ctx_w1;
      }
      const int q = pair - run_start[run];
      while (q >= wbase + w_tot) {
        if (wb + 32 >= a.B) return false;  // never walks past the batch
        wbase += w_tot;
        wb += 32;
        set_window(pre_ctx);
        pre_ctx = wb + 32 < 64 ? ctx_w1 : ctx_of(wb + 32 + lane);
      }
      const int rel = q - wbase;
      // lanes with excl <= rel form a prefix; the last of them owns the pair
      const int j = 31 - __clz(__ballot_sync(0xffffffffu, w_excl <= rel));
      const int excl = __shfl_sync(0xffffffffu, w_excl, j);
      const int ctxj = __shfl_sync(0xffffffffu, w_ctx, j);
      const int nfull = ctxj / a.part;
      it.b = wb + j;
      it.p = run == 1   ? rel - excl + 1
             : run == 2 ? nfull - 1 + (rel - excl)
                        : nfull + partition_split(ctxj, a.part);
      partition_range(ctxj, a.part, it.p, it.tok_begin, it.tok_end);
      it.nparts = partitions_of(ctxj, a.part);
      if constexpr (kRope || kMulti) it.ctx = ctxj;
      if constexpr (kMulti) {
        // first used two items later: the loads stay off this path
        it.q0 = __ldg(a.query_start + it.b);
        it.nq = __ldg(a.query_start + it.b + 1) - it.q0;
      }
      return true;
    };
    // Lane j holds the physical block of logical block (chunk*32 + j) of the item.
    auto load_table = [&](const WorkItem& it, int chunk) -> int {
      const int blk0 = it.tok_begin / kBlockSize;
      const int nblk = (it.tok_end - it.tok_begin + kBlockSize - 1) / kBlockSize;
      const int j = chunk * 32 + lane;
      return j < nblk ? __ldg(a.block_tables + (size_t)it.b * a.MBS + blk0 + j) : -1;
    };

    // The first two items of every CTA are fixed (c and c + N); after that a
    // clean queue hands out 2N, 2N + 1, ... in the order CTAs ask (so a CTA
    // on a faster path takes more), and a fresh workspace falls back to the
    // fixed stride.  Each CTA's indices increase, as locate() requires.
    unsigned long long* queue = a.ws_ctrl + 1;
    int next_static = blockIdx.x + 2 * N;
    auto grab = [&]() -> int {  // value valid in lane 0 (dynamic) or all lanes (static)
      if (!dynamic) {
        const int v = next_static;
        next_static += N;
        return v;
      }
      return lane == 0 ? 2 * N + (int)atomicAdd(queue, 1ull) : 0;
    };
    auto bcast = [&](int raw) -> int { return dynamic ? __shfl_sync(0xffffffffu, raw, 0) : raw; };
    int g0 = blockIdx.x, g1 = g0 + N;
    WorkItem it0{}, it1{};
    // fused step: slot of the sequence's new row, needed by its last partition
    auto load_slot = [&](const WorkItem& it) -> long long {
      return fused && it.p == it.nparts - 1 ? (long long)__ldg(a.slot_mapping + it.b) : -1ll;
    };
    bool v0;
    int tb0 = -1;
    long long sl0 = -1ll;
    bool counted = false;
    if (first_in_run0 && ctx_first > 0) {
      // the loads issued above: the first copies need nothing else
      first_partition(b_first, ctx_first, it0);
      v0 = true;
      tb0 = tb_first;
      sl0 = it0.nparts == 1 ? sl_first : -1ll;
    } else {
      count_runs();
      counted = true;
      v0 = locate(g0 / a.Hkv, it0);
      tb0 = v0 ? load_table(it0, 0) : -1;
      sl0 = v0 ? load_slot(it0) : -1ll;
    }
    bool v1 = counted && v0 && locate(g1 / a.Hkv, it1);
    while (v0 && !aborted) {
      // The next item's table slice and slot load while this item's stages
      // are issued; the item after it is taken from the queue now and
      // located once they are, so a CTA commits to at most two items ahead.
      // (For the very first item this happens after its first stage.)
      int tb1 = -1, g2raw = 0;
      long long sl1 = -1ll;
      auto prefetch_next = [&]() {
        tb1 = v1 ? load_table(it1, 0) : -1;
        sl1 = v1 ? load_slot(it1) : -1ll;
        g2raw = grab();
      };
      if (counted) prefetch_next();

      const int kvh = g0 % a.Hkv;
      const int tok_begin = it0.tok_begin;
      const int blk0 = tok_begin / kBlockSize;
      const int nblk = (it0.tok_end - tok_begin + kBlockSize - 1) / kBlockSize;
      const size_t head_off = (size_t)kvh * PC::kBlockElems;
      int tb = tb0, chunk = 0;
      for (int k0 = 0; k0 < nblk; k0 += PC::kStageBlocks) {
        if (k0 >= 32 * (chunk + 1)) tb = load_table(it0, ++chunk);
        const int slot = st % S;
        const uint32_t ph = (st / S) & 1u;
        bool ok_wait = true;
        if (lane == 0) ok_wait = mbar_wait_bounded(&empty[slot], ph ^ 1u);
        if (!__shfl_sync(0xffffffffu, ok_wait ? 1 : 0, 0)) {
          fail();
          aborted = true;
          break;
        }
        const int nb = min(PC::kStageBlocks, nblk - k0);
        const int phys = __shfl_sync(0xffffffffu, tb, (k0 + lane) & 31);
        const int tok = (blk0 + k0 + lane) * kBlockSize;
        const int rows = min(kBlockSize, it0.tok_end - tok);
        const bool valid = lane < nb && phys >= 0 && phys < a.NB;
        if (lane < nb && !valid) raise_error(a.err, kErrBlock);
        const unsigned mask = __ballot_sync(0xffffffffu, valid);
        // Fused step: the block holding the sequence's last position takes that
        // row from k_new / v_new, provided its slot is the one the table gives.
        bool new_here = false;
        if (fused && valid && tok + rows == it0.tok_end && it0.p == it0.nparts - 1) {
          const long long table_slot = (long long)phys * kBlockSize + (rows - 1);
          if (sl0 == table_slot) {
            new_here = true;
          } else {
            raise_error(a.err, kErrSlot);
          }
        }
        const unsigned new_mask = __ballot_sync(0xffffffffu, new_here);
        const int new_lane = new_mask ? __ffs(new_mask) - 1 : -1;
        const int new_phys = __shfl_sync(0xffffffffu, phys, new_lane >= 0 ? new_lane : 0);
        const int new_rows = __shfl_sync(0xffffffffu, rows, new_lane >= 0 ? new_lane : 0);
        // tensor-map copies move whole 16-row boxes; the new row rides beside them
        int bytes = valid ? 2 * (kMma ? kBlockSize : rows) * D * PC::kElemBytes : 0;
        if (kMma && new_here) bytes += 2 * D * (int)sizeof(T);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
        const bool first = k0 == 0;
        if (lane == 0) {
          StageHdr h;
          h.b = it0.b;
          h.kvh = kvh;
          h.p = it0.p;
          h.nparts = it0.nparts;
          h.tok_end = it0.tok_end;
          h.blk0 = blk0 + k0;
          h.nblk = nb;
          h.flags = (first ? kFirst : 0) | (k0 + PC::kStageBlocks >= nblk ? kLast : 0) |
                    (int)(mask << 8);
          h.new_warp = new_lane;
          h.new_phys = new_lane >= 0 ? new_phys : -1;
          h.new_row = new_lane >= 0 ? new_rows - 1 : -1;
          h.pos = (kRope || kMulti) ? it0.ctx - 1 : 0;
          h.q0 = kMulti ? it0.q0 : it0.b;
          h.nq = kMulti ? it0.nq : 1;
          hdr[slot] = h;
          const bool cs_copy = kRope && first && h.pos >= 0 && h.pos < a.rope_max_pos;
          const int qbytes = kMulti ? it0.nq * G * D * (int)sizeof(T) : PC::kQBytes;
          mbar_arrive_expect_tx(&full[slot], (uint32_t)(bytes + (first ? qbytes : 0) +
                                                        (cs_copy ? PC::kCsBytes : 0)));
        }
        __syncwarp();
        unsigned char* stage = smem + PC::kOffKV + slot * PC::kStageBytes;
        if (kFp8 && valid) {
          // one box of 16 code rows per K and V, swizzled (code_chunk)
          const int y = (phys * a.Hkv + kvh) * kBlockSize;
          tma_load_box_hint(smem_addr(stage + lane * PC::kBlockBytes), &tmk, 0, y, &full[slot],
                            kv_policy);
          tma_load_box_hint(smem_addr(stage + (PC::kStageBlocks + lane) * PC::kBlockBytes), &tmv, 0, y,
                            &full[slot], kv_policy);
        } else if (kMma && valid) {
          const int y = (phys * a.Hkv + kvh) * kBlockSize;
          const uint32_t kd = smem_addr(stage + lane * PC::kBlockBytes);
          const uint32_t vd = smem_addr(stage + (PC::kStageBlocks + lane) * PC::kBlockBytes);
#pragma unroll
          for (int hx = 0; hx < D / 64; ++hx) {
            tma_load_box_hint(kd + hx * 2048, &tmk, hx * 64, y, &full[slot], kv_policy);
            tma_load_box_hint(vd + hx * 2048, &tmv, hx * 64, y, &full[slot], kv_policy);
          }
          if (new_here) {
            const size_t nsrc = ((size_t)it0.b * a.Hkv + kvh) * D;
            const uint32_t rb = (uint32_t)(D * (int)sizeof(T));
            unsigned char* side = smem + PC::kOffSide + slot * PC::kSideBytes;
            bulk_copy_g2s(side, static_cast<const T*>(a.k_new) + nsrc, rb, &full[slot]);
            bulk_copy_g2s(side + rb, static_cast<const T*>(a.v_new) + nsrc, rb, &full[slot]);
          }
        } else if (valid) {
          const size_t src = (size_t)phys * a.Hkv * PC::kBlockElems + head_off;
          const int cache_rows = new_here ? rows - 1 : rows;
          const uint32_t nbytes = (uint32_t)(cache_rows * D * (int)sizeof(T));
          if (nbytes) {
            bulk_copy_g2s_hint(stage + lane * PC::kBlockBytes, kpool + src, nbytes, &full[slot],
                               kv_policy);
            bulk_copy_g2s_hint(stage + (PC::kStageBlocks + lane) * PC::kBlockBytes, vpool + src, nbytes,
                               &full[slot], kv_policy);
          }
          if (new_here) {
            const size_t nsrc = ((size_t)it0.b * a.Hkv + kvh) * D;
            const uint32_t rb = (uint32_t)(D * (int)sizeof(T));
            bulk_copy_g2s(stage + lane * PC::kBlockBytes + nbytes,
                          static_cast<const T*>(a.k_new) + nsrc, rb, &full[slot]);
            bulk_copy_g2s(stage + (PC::kStageBlocks + lane) * PC::kBlockBytes + nbytes,
                          static_cast<const T*>(a.v_new) + nsrc, rb, &full[slot]);
          }
        }
        if (kMulti) {
          // token i's G q rows, one copy per token
          if (first && lane < it0.nq)
            bulk_copy_g2s(smem + PC::kOffQ + slot * PC::kQStride + lane * G * D * (int)sizeof(T),
                          qbase + ((size_t)(it0.q0 + lane) * a.Hq + (size_t)kvh * G) * D,
                          (uint32_t)(G * D * (int)sizeof(T)), &full[slot]);
        } else if (first && lane == 0) {
          bulk_copy_g2s(smem + PC::kOffQ + slot * PC::kQStride,
                        qbase + ((size_t)it0.b * a.Hq + (size_t)kvh * G) * D, PC::kQBytes,
                        &full[slot]);
        }
        if constexpr (kRope) {
          // the item's (cos, sin) row rides with its q rows
          const int pos = it0.ctx - 1;
          if (first && lane == 0 && pos >= 0 && pos < a.rope_max_pos)
            bulk_copy_g2s(smem + PC::kOffQ + slot * PC::kQStride + PC::kQBytes,
                          a.rope_cs + (size_t)pos * (D / 2), (uint32_t)PC::kCsBytes,
                          &full[slot]);
        }
        if (st == 0) PROBE_SET(1, global_timer_ns());
        if (first && lane == 0) PROBE_SET(8 + 2 * items_done, global_timer_ns());
        ++st;
        if (!counted) {
          count_runs();
          counted = true;
          v1 = locate(g1 / a.Hkv, it1);
          prefetch_next();
        }
      }
      const int g2 = bcast(g2raw);
      WorkItem it2{};
      const bool v2 = v1 && locate(g2 / a.Hkv, it2);
      ++items_done;
      g0 = g1;
      it0 = it1;
      v0 = v1;
      tb0 = tb1;
      sl0 = sl1;
      g1 = g2;
      it1 = it2;
      v1 = v2;
    }
    if (!aborted) {
      // End marker: a stage with no data.
      const int slot = st % S;
      const uint32_t ph = (st / S) & 1u;
      bool ok_wait = true;
      if (lane == 0) ok_wait = mbar_wait_bounded(&empty[slot], ph ^ 1u);
      if (__shfl_sync(0xffffffffu, ok_wait ? 1 : 0, 0)) {
        if (lane == 0) {
          hdr[slot].flags = kDone;
          mbar_arrive(&full[slot]);
        }
      } else {
        fail();
        aborted = true;
      }
    }
    PROBE_SET(2, global_timer_ns());
    PROBE_SET(7, items_done);
    if (aborted && lane == 0) {
      // Let the copies still in flight land before the CTA retires.
      const uint32_t first_st = st > (uint32_t)S ? st - S : 0u;
      for (uint32_t s2 = first_st; s2 < st; ++s2)
        (void)mbar_wait_bounded(&full[s2 % S], (s2 / S) & 1u);
    }
    return;
  }

  // ================================================================== consumers
  float qf[G][C::kEPL];
  float m[G], l[G], o[G][C::kEPL];
  // tensor-core consumer: Q^T operand fragments, (m, l) of slots 2(l%4) and
  // 2(l%4)+1, O^T accumulators
  uint32_t tq[kMma ? D / 16 : 1][2];
  uint32_t tql[kMma && kRope ? D / 16 : 1][2];  // RoPE: residual of the rotated q rows
  float tm[2], tl[2], to[kMma ? D / 16 : 1][4];
  int tlim[2] = {0, 0};  // few-token mode: last key position each of the lane's slots sees
  int nslots = G;        // query slots of the current item
  RopeLaneCs<D> kcs;  // RoPE only: this lane's (cos, sin) pairs of the current item
  float* const pm_buf = reinterpret_cast<float*>(smem + PC::kOffPm);
  float* const pl_buf = reinterpret_cast<float*>(smem + PC::kOffPl);
  int parity = 0;  // which partial buffer this item's end uses
  const int c = lane & 7, tg = lane >> 3;
  const int ctid = threadIdx.x;  // 0 .. NC*32-1
  uint32_t st = 0, sync_phase = 0;
#ifdef PHOTON_PROBE
  int items_seen = 0;
#endif

  while (true) {
    const int slot = st % S;
    const uint32_t ph = (st / S) & 1u;
    if (!mbar_wait_bounded(&full[slot], ph) || *abort_flag) {
      fail();
      return;
    }
    if (st == 0 && ctid == 0) PROBE_SET(3, global_timer_ns());
    const StageHdr h = hdr[slot];
    if (h.flags & kDone) {
      if (ctid == 0) PROBE_SET(4, global_timer_ns());
      return;
    }
    if (kMma && (h.flags & kFirst)) {
      const unsigned char* qarea = smem + PC::kOffQ + slot * PC::kQStride;
      const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qarea);
      const int t2 = 2 * (lane & 3);
      // the lane's slot for the Q^T operand; decode: head g, few-token mode:
      // (token slot / G, head slot % G), rows consecutive in shared memory
      nslots = kMulti ? h.nq * G : G;
      const int slot_g = (lane >> 2) < nslots ? (lane >> 2) : PC::kSlots;
      if constexpr (kMulti) {
        // token i sits at position ctx - nq + i = pos + 1 - nq + i
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tlim[j] = t2 + j < nslots ? h.pos + 1 - h.nq + (t2 + j) / G : -1;
      }
      if constexpr (kRope && kMma) {
        // q rows turned by the token's position in fp32, then split into
        // their storage-type rounding and its residual
        const float2* cs_row = reinterpret_cast<const float2*>(qarea + PC::kQBytes);
        const bool in_table = h.pos >= 0 && h.pos < a.rope_max_pos;
        if (!in_table && ctid == 0) raise_error(a.err, kErrPosition);
        const T* qrow = reinterpret_cast<const T*>(qarea) + (slot_g < G ? slot_g : 0) * D;
        auto turned = [&](int e) -> float {
          const float x = Elem<T>::to_f32(qrow[e]);
          if (!in_table) return x;
          constexpr int kHalf = D / 2;
          const float2 w = cs_row[e < kHalf ? e : e - kHalf];
          const float partner = Elem<T>::to_f32(qrow[e < kHalf ? e + kHalf : e - kHalf]);
          return e < kHalf ? x * w.x - partner * w.y : x * w.x + partner * w.y;
        };
        auto split = [&](int e, uint32_t& hi, uint32_t& lo) {
          const float x0 = turned(e), x1 = turned(e + 1);
          hi = Mma<T>::pack(x0, x1);
          const float2 r = Mma<T>::unpack(hi);
          lo = Mma<T>::pack(x0 - r.x, x1 - r.y);
        };
#pragma unroll
        for (int kk = 0; kk < (kMma ? D / 16 : 1); ++kk) {
          uint32_t h0 = 0u, l0 = 0u, h1 = 0u, l1 = 0u;
          if (slot_g < G) {
            split(16 * kk + t2, h0, l0);
            split(16 * kk + t2 + 8, h1, l1);
          }
          tq[kk][0] = h0;
          tq[kk][1] = h1;
          tql[kk][0] = l0;
          tql[kk][1] = l1;
        }
        if (in_table) {
#pragma unroll
          for (int i = 0; i < (D / 2 + 31) / 32; ++i)
            if (lane + 32 * i < D / 2) kcs.w[i] = cs_row[lane + 32 * i];
        }
      } else {
        // e4m3 cache: the k-steps walk each 16-dim chunk in the order the
        // widened code pairs come in (attend_block_mma, kCodes)
        const int lo = kFp8 ? 2 * t2 : t2, hi = kFp8 ? 2 * t2 + 2 : t2 + 8;
#pragma unroll
        for (int kk = 0; kk < (kMma ? D / 16 : 1); ++kk) {
          tq[kk][0] = slot_g < PC::kSlots ? q32[(slot_g * D + 16 * kk + lo) / 2] : 0u;
          tq[kk][1] = slot_g < PC::kSlots ? q32[(slot_g * D + 16 * kk + hi) / 2] : 0u;
        }
      }
#pragma unroll
      for (int kk = 0; kk < (kMma ? D / 16 : 1); ++kk)
#pragma unroll
        for (int j = 0; j < 4; ++j) to[kk][j] = 0.f;
      tm[0] = tm[1] = -INFINITY;
      tl[0] = tl[1] = 0.f;
    } else if (h.flags & kFirst) {
      const T* qs = reinterpret_cast<const T*>(smem + PC::kOffQ + slot * PC::kQStride);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int i = 0; i < C::kPPL; ++i) {
          const uint4 raw = *reinterpret_cast<const uint4*>(qs + g * D + (c + 8 * i) * C::kChunk);
          float t[C::kChunk];
          Elem<T>::widen(raw, t);
#pragma unroll
          for (int e = 0; e < C::kChunk; ++e) {
            qf[g][i * C::kChunk + e] = kRope ? t[e] : t[e] * a.qscale;
            o[g][i * C::kChunk + e] = 0.f;
          }
        }
      }
      if constexpr (kRope) {
        // turn the raw rows first, then scale them like the plain path
        const float2* cs_row = reinterpret_cast<const float2*>(qs + G * D);
        rope_q<T, D, G>(qf, cs_row, a.rope_max_pos, h.pos, c, a.err, ctid);
        if (h.pos >= 0 && h.pos < a.rope_max_pos) {
#pragma unroll
          for (int i = 0; i < (D / 2 + 31) / 32; ++i)
            if (lane + 32 * i < D / 2) kcs.w[i] = cs_row[lane + 32 * i];
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int e = 0; e < C::kEPL; ++e) qf[g][e] *= a.qscale;
      }
    }
    if (kFp8) {
      // fp8 cache: the warp's K and V code blocks are used as they landed;
      // the V rows past the context (the box brought whatever the pool
      // holds there) are zeroed first, since 0 x NaN would reach the sums
#pragma unroll
      for (int bb = 0; bb < PC::kBPW; ++bb) {
        const int blk = warp * PC::kBPW + bb;
        if (blk >= h.nblk || !((h.flags >> (8 + blk)) & 1)) continue;
        unsigned char* const kb =
            smem + PC::kOffKV + slot * PC::kStageBytes + blk * PC::kBlockBytes;
        unsigned char* const vb = kb + PC::kStageBlocks * PC::kBlockBytes;
        const int n_valid = min(kBlockSize, h.tok_end - (h.blk0 + blk) * kBlockSize);
        if (n_valid < kBlockSize) {
          for (int i = lane; i < (kBlockSize - n_valid) * (D / 16); i += 32)
            *reinterpret_cast<uint4*>(vb + n_valid * D + i * 16) = make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async_smem();  // the stage is refilled by tensor copies later
          __syncwarp();
        }
        if constexpr (kFp8)
          attend_block_mma<T, D, false, false, true>(smem_addr(kb), smem_addr(vb), n_valid,
                                                     a.qscale, tq, tq, tm, tl, to, lane, 0, tlim);
      }
    } else if (kMma && warp < h.nblk && ((h.flags >> (8 + warp)) & 1)) {
      unsigned char* const kb = smem + PC::kOffKV + slot * PC::kStageBytes + warp * PC::kBlockBytes;
      unsigned char* const vb = kb + PC::kStageBlocks * PC::kBlockBytes;
      const int n_valid = min(kBlockSize, h.tok_end - (h.blk0 + warp) * kBlockSize);
      constexpr int kRowChunks = D * (int)sizeof(T) / 16;
      bool wrote = false;
      if (warp == h.new_warp) {
        // fused step: the new token's rows came beside the stage; put them in
        // row new_row of the blocks (the box brought that slot's stale row)
        // and store them to their cache slot
        unsigned char* side = smem + PC::kOffSide + slot * PC::kSideBytes;
        if constexpr (kRope) {
          // with RoPE the new K row turns by its position first
          rope_row<T, D>(reinterpret_cast<T*>(side), kcs, a.rope_max_pos, h.pos, lane);
          __syncwarp();
        }
        const size_t dst = (((size_t)h.new_phys * a.Hkv + h.kvh) * kBlockSize + h.new_row) * D;
        for (int i = lane; i < 2 * kRowChunks; i += 32) {
          const bool is_v = i >= kRowChunks;
          const int ch = is_v ? i - kRowChunks : i;
          const uint4 val = *reinterpret_cast<const uint4*>(side + i * 16);
          *reinterpret_cast<uint4*>((is_v ? vb : kb) + blk_chunk(h.new_row, ch)) = val;
          T* cache = static_cast<T*>(is_v ? a.v_cache_w : a.k_cache_w);
          *reinterpret_cast<uint4*>(cache + dst + ch * (16 / (int)sizeof(T))) = val;
        }
        wrote = true;
      }
      if (n_valid < kBlockSize) {
        // rows past the context carry whatever the pool holds: zero their V
        for (int i = lane; i < (kBlockSize - n_valid) * kRowChunks; i += 32)
          *reinterpret_cast<uint4*>(vb + blk_chunk(n_valid + i / kRowChunks, i % kRowChunks)) =
              make_uint4(0u, 0u, 0u, 0u);
        wrote = true;
      }
      if (wrote) {
        fence_proxy_async_smem();  // the stage is refilled by tensor copies later
        __syncwarp();
      }
      if constexpr (kMma) {
        const int key0 = (h.blk0 + warp) * kBlockSize;
        if constexpr (kRope)
          attend_block_mma<T, D, true, false>(smem_addr(kb), smem_addr(vb), n_valid, a.qscale, tq,
                                              tql, tm, tl, to, lane, key0, tlim);
        else
          attend_block_mma<T, D, false, kMulti>(smem_addr(kb), smem_addr(vb), n_valid, a.qscale,
                                                tq, tq, tm, tl, to, lane, key0, tlim);
      }
    } else if (warp < h.nblk && ((h.flags >> (8 + warp)) & 1)) {
      const T* stage = reinterpret_cast<const T*>(smem + PC::kOffKV + slot * PC::kStageBytes);
      const int n_valid = min(kBlockSize, h.tok_end - (h.blk0 + warp) * kBlockSize);
      if (kRope && warp == h.new_warp) {
        // fused step with RoPE: turn the new K row by its position, in place,
        // before it is attended and stored
        rope_row<T, D>(const_cast<T*>(stage) + warp * PC::kBlockElems + h.new_row * D, kcs,
                       a.rope_max_pos, h.pos, lane);
        fence_proxy_async_smem();  // the stage is refilled by bulk copies later
        __syncwarp();
      }
      attend_block<T, D, G>(stage + warp * PC::kBlockElems,
                            stage + (PC::kStageBlocks + warp) * PC::kBlockElems,
                            n_valid, qf, m, l, o, lane);
      if (warp == h.new_warp) {
        // fused step: this block's row new_row is the new token; store it
        constexpr int kRowChunks = D * (int)sizeof(T) / 16;
        constexpr int kPerChunk = 16 / (int)sizeof(T);
        const size_t dst = (((size_t)h.new_phys * a.Hkv + h.kvh) * kBlockSize + h.new_row) * D;
        const T* krow = stage + warp * PC::kBlockElems + h.new_row * D;
        const T* vrow = stage + (PC::kStageBlocks + warp) * PC::kBlockElems + h.new_row * D;
        for (int i = lane; i < 2 * kRowChunks; i += 32) {
          const bool is_v = i >= kRowChunks;
          const int ch = is_v ? i - kRowChunks : i;
          const uint4 val = *reinterpret_cast<const uint4*>((is_v ? vrow : krow) + ch * kPerChunk);
          T* cache = static_cast<T*>(is_v ? a.v_cache_w : a.k_cache_w);
          *reinterpret_cast<uint4*>(cache + dst + ch * kPerChunk) = val;
        }
      }
    }
    __syncwarp();
    ++st;
    if (!(h.flags & kLast)) {
      if (lane == 0) mbar_arrive(&empty[slot]);
      continue;
    }

    // ---- end of the item: combine the warps' (m, l, o).  (m, l) alternate
    // between two buffers by item, so one barrier per item suffices: a warp
    // can only come back to a buffer after every warp has passed the next
    // item's barrier, i.e. finished reading it here.  Warp w's o rows sit in
    // its K block area of this (last) stage, [slots][D] fp32, and the stage is
    // released once the combine has read them.
    constexpr int kSl = PC::kSlots;
    float* const pm = pm_buf + parity * NC * kSl;
    float* const pl = pl_buf + parity * NC * kSl;
    unsigned char* const last_stage = smem + PC::kOffKV + slot * PC::kStageBytes;
    // o row of slot g of warp w: its K block area holds the first
    // kPoRowsPerBlock rows, its V block area the rest
    auto po_row = [&](int w, int g) -> float* {
      constexpr int kPer = PC::kPoRowsPerBlock;
      // warp w's own (first) block of the stage: it has finished reading it
      const int area = (g < kPer ? 0 : PC::kStageBlocks) + w * PC::kBPW;
      return reinterpret_cast<float*>(last_stage + area * PC::kBlockBytes) + (g % kPer) * D;
    };
    parity ^= 1;
    if constexpr (kMma) {
      // lane partial sums over the 8 key rows; slots >= G are padding
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        tl[0] += __shfl_xor_sync(0xffffffffu, tl[0], off);
        tl[1] += __shfl_xor_sync(0xffffffffu, tl[1], off);
      }
      const int r = lane >> 2;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int g = 2 * (lane & 3) + j;   // the slot
        if (g < nslots) {
#pragma unroll
          for (int i = 0; i < (kMma ? D / 16 : 1); ++i) {
            // accumulator rows r and r + 8 of tile i: dims 16i + r and
            // 16i + r + 8, or 16i + 2r and 16i + 2r + 1 over an e4m3 cache
            po_row(warp, g)[16 * i + (kFp8 ? 2 * r : r)] = to[i][j];
            po_row(warp, g)[16 * i + (kFp8 ? 2 * r + 1 : r + 8)] = to[i][2 + j];
          }
          if (r == 0) {
            pm[warp * kSl + g] = tm[j];
            pl[warp * kSl + g] = tl[j];
          }
        }
      }
    }
#pragma unroll
    for (int g = 0; g < (kMma ? 0 : G); ++g) {
      l[g] += __shfl_xor_sync(0xffffffffu, l[g], 8);
      l[g] += __shfl_xor_sync(0xffffffffu, l[g], 16);
#pragma unroll
      for (int e = 0; e < C::kEPL; ++e) {
        o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], 8);
        o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], 16);
      }
    }
    if (!kMma && tg == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int i = 0; i < C::kPPL; ++i)
#pragma unroll
          for (int e = 0; e < C::kChunk; ++e)
            po_row(warp, g)[(c + 8 * i) * C::kChunk + e] = o[g][i * C::kChunk + e];
        if (c == 0) {
          pm[warp * kSl + g] = m[g];
          pl[warp * kSl + g] = l[g];
        }
      }
    }
    fence_proxy_async_smem();  // o rows written into a stage that copies refill later
    if (!consumer_sync(sync, sync_phase, lane)) {
      fail();
      return;
    }
    // four consecutive elements of one slot's row per thread and pass
    for (int idx = ctid; idx < nslots * (D / 4); idx += NC * 32) {
      const int g = idx / (D / 4), e = (idx % (D / 4)) * 4;   // slot (token g / G, head g % G)
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NC; ++w)
        if (pl[w * kSl + g] > 0.f) M = fmaxf(M, pm[w * kSl + g]);
      float L = 0.f;
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        const float lw = pl[w * kSl + g];
        if (lw > 0.f) {
          const float wt = exp2f(pm[w * kSl + g] - M);
          const float4 v = *reinterpret_cast<const float4*>(po_row(w, g) + e);
          L = fmaf(wt, lw, L);
          O.x = fmaf(wt, v.x, O.x);
          O.y = fmaf(wt, v.y, O.y);
          O.z = fmaf(wt, v.z, O.z);
          O.w = fmaf(wt, v.w, O.w);
        }
      }
      if constexpr (kFp8) {
        // the V scale of the e4m3 cache (the K scale is in qscale)
        O.x *= a.v_scale;
        O.y *= a.v_scale;
        O.z *= a.v_scale;
        O.w *= a.v_scale;
      }
      const int hq = h.kvh * G + g % G;
      const size_t qrow = kMulti ? (size_t)h.q0 + g / G : (size_t)h.b;   // row of q / out
      if (h.nparts == 1) {
        T* out = static_cast<T*>(a.out) + (qrow * a.Hq + hq) * D + e;
        const float4 r = L > 0.f ? make_float4(O.x / L, O.y / L, O.z / L, O.w / L)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (sizeof(T) == 2) {
          uint2 u;
          u.x = Mma<T>::pack(r.x, r.y);
          u.y = Mma<T>::pack(r.z, r.w);
          *reinterpret_cast<uint2*>(out) = u;
        } else {
          *reinterpret_cast<float4*>(out) = r;
        }
      } else {
        const size_t row = (qrow * a.Hq + hq) * a.pmax + h.p;
        *reinterpret_cast<float4*>(a.ws_o + row * D + e) = O;
        if (e == 0) {
          a.ws_m[row] = M;
          a.ws_l[row] = L;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);  // the item's last stage, now read
#ifdef PHOTON_PROBE
    if (ctid == 0) PROBE_SET(9 + 2 * items_seen, global_timer_ns());
    ++items_seen;
#endif
  }
}

// ------------------------------------------------------------------ merge kernel
// One warp per (sequence, q head) -- per (sequence, q head, query token) in
// the few-token mode.  Empty (or rejected) contexts get a zero row;
// sequences with two or more partitions get the merge:
//   M = max_p m_p,  w_p = 2^(m_p - M) (0 for an empty partition),
//   out = sum_p w_p o_p / sum_p w_p l_p.
// Built for latency: a lane owns D/32 consecutive output elements, and the
// partial rows of up to 32 partitions are loaded unconditionally and at once,
// together with the (m, l) pairs (lane p holds those of partition p), so a
// sequence with <= 32 partitions costs one round trip to L2.
// Two warps per CTA: small enough (64 threads) for a merge CTA to be resident
// next to two attention CTAs, so merges start as soon as the attention grid
// completes.
#ifndef PHOTON_MERGE_WARPS
#define PHOTON_MERGE_WARPS 2
#endif
constexpr int kMergeWarps = PHOTON_MERGE_WARPS;
// Partial rows loaded at once per lane: one round trip for up to
// PHOTON_MERGE_ROWS partitions (a tuning knob: fewer rows take fewer
// registers, so more merge warps are resident beside the attention CTAs).
#ifndef PHOTON_MERGE_ROWS
#define PHOTON_MERGE_ROWS 32
#endif
constexpr int kMergeRows = PHOTON_MERGE_ROWS;

template <typename T, int D>
__global__ void __launch_bounds__(kMergeWarps * 32) paged_decode_merge_kernel(const DecodeArgs a) {
  constexpr int EPL = D / 32;
  // This kernel runs only after the attention kernel has passed its own wait
  // for the kernel before it, so the context lengths and query starts (which
  // the attention kernel does not write) can be read before waiting for the
  // attention grid: one round trip off the merge's critical path.  Rows of
  // empty or rejected sequences are not touched by the attention kernel
  // either.
  // item = (b * Hq + h) * max_q + i: sequence b, q head h, its query token
  // i (decode: max_q = 1, one token)
  const int mq = a.query_start ? a.max_q : 1;
  const int item = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const bool live = item < a.B * a.Hq * mq;
  const int bh = item / mq, ti = item % mq;
  const int b = live ? bh / a.Hq : 0, hq = live ? bh % a.Hq : 0;
  const int ctx = live ? __ldg(a.context_lens + b) : 0;
  const int span = a.MBS * kBlockSize;
#ifdef PHOTON_PROBE
  if (threadIdx.x == 0 && blockIdx.x < 4096) g_probe_merge[blockIdx.x][0] = global_timer_ns();
#endif
  // the sequence's output rows: decode, row b; few-token mode, rows q0 .. q0 + n - 1
  int q0 = b, n = 1;
  bool skip = !live;
  if (a.query_start && live) {
    q0 = __ldg(a.query_start + b);
    n = __ldg(a.query_start + b + 1) - q0;
    if (n < 0 || q0 < 0 || q0 > a.num_tokens - n) {
      // rows outside q / out: flagged, nothing written
      if (lane == 0 && hq == 0 && ti == 0) raise_error(a.err, kErrQuery);
      skip = true;
    } else if (n > a.max_q || ctx < n || ctx > span) {
      // inconsistent lengths: flagged, the rows it may own zeroed
      if (lane == 0 && hq == 0 && ti == 0)
        raise_error(a.err, n > a.max_q ? kErrQuery : kErrContext);
      if (ti < n) {
        T* out = static_cast<T*>(a.out) + ((size_t)(q0 + ti) * a.Hq + hq) * D + lane * EPL;
#pragma unroll
        for (int e = 0; e < EPL; ++e) out[e] = Elem<T>::narrow(0.f);
      }
      skip = true;
    } else if (ti >= n) {
      skip = true;   // fewer tokens than max_q
    }
  } else if (live && (ctx <= 0 || ctx > span)) {
    // decode: an empty or rejected context gives a zero row
    if (ctx != 0 && lane == 0 && hq == 0) raise_error(a.err, kErrContext);
    T* out = static_cast<T*>(a.out) + (size_t)item * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[e] = Elem<T>::narrow(0.f);
    skip = true;
  }
  pdl_wait_primary();
#ifdef PHOTON_PROBE
  if (threadIdx.x == 0 && blockIdx.x < 4096) g_probe_merge[blockIdx.x][1] = global_timer_ns();
#endif
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // The attention grid is done handing out items: leave the queue clean for
    // the next call.
    a.ws_ctrl[1] = 0ull;
    a.ws_ctrl[0] = kQueueReady;
  }
  if (skip) return;
  const int nparts = partitions_of(ctx, a.part);
  if (nparts < 2) return;                             // the attention kernel wrote out

  {
    const size_t orow = (size_t)(q0 + ti) * a.Hq + hq;   // row of out
    const size_t row0 = orow * a.pmax;
    T* out = static_cast<T*>(a.out) + orow * D + lane * EPL;
    const float* pm = a.ws_m + row0;
    const float* pl = a.ws_l + row0;
    const float* po = a.ws_o + row0 * D + lane * EPL;

    float O[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) O[e] = 0.f;
    float M = -INFINITY, L = 0.f;
    for (int p0 = 0; p0 < nparts; p0 += 32) {
      const int np = min(32, nparts - p0);
      float v[kMergeRows][EPL];
#pragma unroll
      for (int u = 0; u < kMergeRows; ++u)
#pragma unroll
        for (int e = 0; e < EPL; ++e) v[u][e] = u < np ? po[(size_t)(p0 + u) * D + e] : 0.f;
      const float lp = lane < np ? pl[p0 + lane] : 0.f;
      const float mp = lane < np && lp > 0.f ? pm[p0 + lane] : -INFINITY;
      // running max over the chunks; rescale what was accumulated so far
      float mc = mp;
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, s));
      const float Mn = fmaxf(M, mc);
      if (Mn == -INFINITY) continue;                    // nothing in this chunk or before
      const float scale_old = exp2f(M - Mn);            // 0 when M = -inf
      const float w = lp > 0.f ? exp2f(mp - Mn) : 0.f;
      float lw = w * lp;
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, s);
      L = L * scale_old + lw;
#pragma unroll
      for (int e = 0; e < EPL; ++e) O[e] *= scale_old;
#pragma unroll
      for (int u = 0; u < kMergeRows; ++u) {
        const float wu = __shfl_sync(0xffffffffu, w, u);
#pragma unroll
        for (int e = 0; e < EPL; ++e) O[e] = fmaf(wu, v[u][e], O[e]);
      }
#pragma unroll
      for (int u0 = kMergeRows; u0 < 32; u0 += kMergeRows) {  // rest of the chunk, if any
        if (u0 >= np) break;
#pragma unroll
        for (int u = 0; u < kMergeRows; ++u)
#pragma unroll
          for (int e = 0; e < EPL; ++e)
            v[u][e] = u0 + u < np ? po[(size_t)(p0 + u0 + u) * D + e] : 0.f;
#pragma unroll
        for (int u = 0; u < kMergeRows; ++u) {
          const float wu = __shfl_sync(0xffffffffu, w, u0 + u);
#pragma unroll
          for (int e = 0; e < EPL; ++e) O[e] = fmaf(wu, v[u][e], O[e]);
        }
      }
      M = Mn;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[e] = Elem<T>::narrow(O[e] * inv);
  }
#ifdef PHOTON_PROBE
  if (lane == 0 && blockIdx.x < 4096) g_probe_merge[blockIdx.x][2] = global_timer_ns();
#endif
}

// Resident CTAs per SM of an attention-kernel instantiation (queried once per
// device, after raising its dynamic shared-memory limit).
template <typename T, int D, int G, int NC, int S, bool kRope, bool kMma, bool kMulti,
          bool kFp8 = false>
int attention_ctas_per_sm() {
  using PC = PersistCfg<T, D, G, NC, S, kRope, kMma, kMulti, kFp8>;
  constexpr int kMaxDev = 64;
  static int cache[kMaxDev];  // 0 = not yet queried
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  if (cache[dev] > 0) return cache[dev];
  auto kern = paged_decode_attention_kernel<T, D, G, NC, S, kRope, kMma, kMulti, kFp8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PC::kSmemBytes) !=
      cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, PC::kThreads, PC::kSmemBytes) !=
      cudaSuccess)
    return 0;
  cache[dev] = n;
  return n;
}

// Tuning knobs (compile time): consumer warps per CTA and the shared-memory
// ring budget per CTA.  With the defaults two CTAs share an SM.
#ifndef PHOTON_CONSUMER_WARPS
#define PHOTON_CONSUMER_WARPS 4
#endif
#ifndef PHOTON_RING_KB
#define PHOTON_RING_KB 96
#endif
#ifndef PHOTON_RING_KB_D64
#define PHOTON_RING_KB_D64 64
#endif
// Ring budget of an instantiation.  16-bit blocks of head_dim 64 take a 64 KB
// ring (four 16 KB stages) so that three CTAs share an SM: their consumers
// do half the tensor-core work per byte of the head_dim-128 ones, and the
// third CTA's warps keep more of them busy (batch-256 mix: 208 -> 168 us
// against a 96 KB ring at two CTAs per SM).
template <typename T, int D>
constexpr int ring_bytes() {
  return (D == 64 && sizeof(T) == 2 ? PHOTON_RING_KB_D64 : PHOTON_RING_KB) * 1024;
}

template <typename T, int D>
constexpr int stages_for(int nc) {
  return (ring_bytes<T, D>() / (2 * nc * kBlockSize * D * (int)sizeof(T))) < 2
             ? 2
             : (ring_bytes<T, D>() / (2 * nc * kBlockSize * D * (int)sizeof(T)));
}

// Which consumer a (D, G) instantiation runs by default: the tensor-core one
// for 16-bit storage and groups of PHOTON_MMA_MIN_G or more query heads per KV
// head.  The CUDA-core consumer spends about 33 instructions per K/V element
// pair and query head (widening, G dot products with shuffle reductions, G
// weighted sums); at G = 4, d = 64 that outruns the issue rate (ncu: issue
// slots 57% busy, DRAM 47%), and at G = 2, d = 128 it still costs about 7% of
// the step against the tensor-core consumer.
#ifndef PHOTON_MMA_MIN_G
#define PHOTON_MMA_MIN_G 2
#endif

template <typename T, int D, int G, int NC, int S, bool kRope, bool kMma, bool kMulti = false,
          bool kFp8 = false>
cudaError_t launch_attention(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                             cudaStream_t stream) {
  using PC = PersistCfg<T, D, G, NC, S, kRope, kMma, kMulti, kFp8>;
  const int per_sm = attention_ctas_per_sm<T, D, G, NC, S, kRope, kMma, kMulti, kFp8>();
  if (per_sm <= 0) return cudaErrorInvalidConfiguration;
#ifdef PHOTON_PROBE_NO_PDL
  // tuning builds only: the attention kernel as a plain launch
  paged_decode_attention_kernel<T, D, G, NC, S, kRope, kMma, kMulti, kFp8>
      <<<dim3(per_sm * a.num_sms), dim3(PC::kThreads), PC::kSmemBytes, stream>>>(a, tk, tv);
  return cudaGetLastError();
#else
  return launch_pdl(paged_decode_attention_kernel<T, D, G, NC, S, kRope, kMma, kMulti, kFp8>,
                    dim3(per_sm * a.num_sms), dim3(PC::kThreads), PC::kSmemBytes, stream, a, tk,
                    tv);
#endif
}

template <typename T, int D, int G>
cudaError_t launch_decode_impl(const DecodeArgs& a0, cudaStream_t stream) {
  constexpr int NC = PHOTON_CONSUMER_WARPS;
  constexpr int S = stages_for<T, D>(NC);
  DecodeArgs a = a0;
  // Every buffer the kernels touch must have been carved out by the caller.
  if (!a.q || !a.k_cache || !a.v_cache || !a.block_tables || !a.context_lens || !a.out ||
      !a.ws_m || !a.ws_l || !a.ws_o || !a.ws_ctrl || !a.err)
    return cudaErrorInvalidValue;
  const bool rope = a.rope_cs != nullptr;
  // few-token multi-query mode: tensor-core consumer only, at most 8 slots
  const bool multi = a.query_start != nullptr;
  if (multi && (sizeof(T) != 2 || rope || a.max_q < 1 || a.max_q * G > 8))
    return cudaErrorInvalidValue;
  CUtensorMap tk, tv;
  memset(&tk, 0, sizeof(tk));
  memset(&tv, 0, sizeof(tv));
  bool mma = false;
  if constexpr (sizeof(T) == 2) {
    const int choice = g_decode_consumer.load(std::memory_order_relaxed);  // 0: by group size, 1: CUDA cores, 2: tensor cores
    mma = (multi || choice == 2 || (choice == 0 && G >= PHOTON_MMA_MIN_G)) &&
          (int64_t)a.NB * a.Hkv * kBlockSize <= INT32_MAX;
    if (multi && !mma) return cudaErrorInvalidValue;
    const int dt = std::is_same<T, __half>::value ? 1 : 2;
    if (mma && (make_pool_map(&tk, a.k_cache, dt, a.NB, a.Hkv, D) != cudaSuccess ||
                make_pool_map(&tv, a.v_cache, dt, a.NB, a.Hkv, D) != cudaSuccess))
      return cudaErrorInvalidValue;
  }

  if (a.ev_start) cudaEventRecord(a.ev_start, stream);
  cudaError_t err;
  if (mma) {
    if constexpr (sizeof(T) == 2)
      err = multi  ? launch_attention<T, D, G, NC, S, false, true, true>(a, tk, tv, stream)
            : rope ? launch_attention<T, D, G, NC, S, true, true>(a, tk, tv, stream)
                   : launch_attention<T, D, G, NC, S, false, true>(a, tk, tv, stream);
    else
      err = cudaErrorInvalidValue;
  } else if (rope) {
    err = launch_attention<T, D, G, NC, S, true, false>(a, tk, tv, stream);
  } else {
    err = launch_attention<T, D, G, NC, S, false, false>(a, tk, tv, stream);
  }
  if (err != cudaSuccess) return err;
  const int items = a.B * a.Hq * (multi ? a.max_q : 1);
  err = launch_pdl(paged_decode_merge_kernel<T, D>, dim3((items + kMergeWarps - 1) / kMergeWarps),
                   dim3(kMergeWarps * 32), 0, stream, a);
  if (err != cudaSuccess) return err;
  if (a.ev_stop) cudaEventRecord(a.ev_stop, stream);
  return cudaSuccess;
}

// The e4m3 cache: stages of 4 code blocks per warp-block slot, i.e. 8 blocks
// per K and V with two blocks per warp (32 KB a stage at d = 128), in a 96 KB
// ring, so that two CTAs share an SM (64 KB and three CTAs with one block per
// warp).
#ifndef PHOTON_RING_KB_FP8
#define PHOTON_RING_KB_FP8 (PHOTON_FP8_BPW > 1 ? 96 : 64)
#endif
constexpr int kRingBytesFp8 = PHOTON_RING_KB_FP8 * 1024;

template <int D, int G>
cudaError_t launch_decode_fp8_impl(const DecodeArgs& a, cudaStream_t stream) {
  constexpr int NC = PHOTON_CONSUMER_WARPS;
  constexpr int kStage = 2 * NC * PHOTON_FP8_BPW * kBlockSize * D;
  constexpr int S = kRingBytesFp8 / kStage < 2 ? 2 : kRingBytesFp8 / kStage;
  if (!a.q || !a.k_cache || !a.v_cache || !a.block_tables || !a.context_lens || !a.out ||
      !a.ws_m || !a.ws_l || !a.ws_o || !a.ws_ctrl || !a.err || a.k_new || a.rope_cs ||
      a.query_start)
    return cudaErrorInvalidValue;
  if ((int64_t)a.NB * a.Hkv * kBlockSize > INT32_MAX) return cudaErrorInvalidValue;
  CUtensorMap tk, tv;
  if (make_pool_map(&tk, a.k_cache, 3, a.NB, a.Hkv, D) != cudaSuccess ||
      make_pool_map(&tv, a.v_cache, 3, a.NB, a.Hkv, D) != cudaSuccess)
    return cudaErrorInvalidValue;
  if (a.ev_start) cudaEventRecord(a.ev_start, stream);
  cudaError_t err = launch_attention<__half, D, G, NC, S, false, true, false, true>(
      a, tk, tv, stream);
  if (err != cudaSuccess) return err;
  err = launch_pdl(paged_decode_merge_kernel<__half, D>,
                   dim3((a.B * a.Hq + kMergeWarps - 1) / kMergeWarps), dim3(kMergeWarps * 32), 0,
                   stream, a);
  if (err != cudaSuccess) return err;
  if (a.ev_stop) cudaEventRecord(a.ev_stop, stream);
  return cudaSuccess;
}

template <int D>
cudaError_t launch_decode_fp8_d(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.Hq / a.Hkv) {
    case 1: return launch_decode_fp8_impl<D, 1>(a, stream);
    case 2: return launch_decode_fp8_impl<D, 2>(a, stream);
    case 4: return launch_decode_fp8_impl<D, 4>(a, stream);
    case 8: return launch_decode_fp8_impl<D, 8>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int D>
cudaError_t launch_decode_d(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.Hq / a.Hkv) {
    case 1: return launch_decode_impl<T, D, 1>(a, stream);
    case 2: return launch_decode_impl<T, D, 2>(a, stream);
    case 4: return launch_decode_impl<T, D, 4>(a, stream);
    case 8: return launch_decode_impl<T, D, 8>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.D) {
    case 64: return launch_decode_d<T, 64>(a, stream);
    case 128: return launch_decode_d<T, 128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace photon
