// paged_decode.cuh -- split-KV paged decode attention and its partition merge.
//
// PhotonInfer README, "Key features / GPU-optimized kernels": batched paged
// attention over a block-wise KV cache, softmax computed in a numerically
// stable way, 128-bit vectorised loads; "Technical details / Paged attention":
// per-sequence cache offsets (here: block tables).
//
// Work decomposition.  The context [0, ctx_b) of sequence b is cut into
// partitions of `part` tokens (a multiple of the 16-token block).  One CTA
// owns one (partition, KV head, sequence) and computes, for the G query heads
// that share the KV head (GQA), the running max m, the weight sum l and the
// unnormalised weighted sum of V over its tokens.  A sequence with a single
// partition writes its output row directly; longer ones leave (m, l, o) in
// the workspace and the merge kernel combines them by their log-sum-exp
// weights:  M = max_p m_p,  out = sum_p 2^(m_p-M) o_p / sum_p 2^(m_p-M) l_p.
//
// Inside a CTA each warp takes whole 16-token blocks (blocks w, w+4, ...).
// A block's K (and V) rows for one KV head are one contiguous chunk of the
// pool.  Eight lanes cover one token row with 16-byte loads (a quarter-warp
// reads 128 contiguous bytes), so a warp holds four rows per load step and
// four steps cover the block.  Scores are reduced across the eight lanes of a
// row with three xor-shuffles; each loaded K/V element is reused by all G
// heads from registers.  The softmax is the online form: per block the warp
// takes the block maximum, rescales its running (l, o) by 2^(m_old - m_new)
// and accumulates 2^(s - m_new).  Scores are kept in the log2 domain (q is
// pre-multiplied by scale * log2 e), so exp is one exp2f.
#pragma once

#include <float.h>
#include <math.h>

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

template <typename T, int D, int G>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    paged_decode_split_kernel(const DecodeArgs a) {
  using C = DecodeCfg<T, D, G>;
  constexpr int NW = kDecodeWarps;
  const int p = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = lane & 7, tg = lane >> 3;

  __shared__ float sm_m[NW][G], sm_l[NW][G];
  __shared__ __align__(16) float sm_o[NW][G][D];

  const int ctx = __ldg(a.context_lens + b);
  const int span = a.MBS * kBlockSize;
  const bool bad_ctx = ctx < 0 || ctx > span;
  const int nparts = bad_ctx ? 0 : (ctx + a.part - 1) / a.part;
  if (nparts == 0) {
    // Empty (or rejected) context: the output row is zero.
    if (p == 0) {
      if (bad_ctx && kvh == 0 && threadIdx.x == 0) raise_error(a.err, kErrContext);
      T* out = static_cast<T*>(a.out) + ((size_t)b * a.Hq + (size_t)kvh * G) * D;
      for (int i = threadIdx.x; i < G * D; i += blockDim.x) out[i] = Elem<T>::narrow(0.f);
    }
    return;
  }
  if (p >= nparts) return;

  const int tok_begin = p * a.part;
  const int tok_end = min(ctx, tok_begin + a.part);
  const int blk_begin = tok_begin / kBlockSize;
  const int blk_end = (tok_end + kBlockSize - 1) / kBlockSize;

  // q rows of the G heads of this group; each lane keeps its own elements,
  // pre-scaled into the log2 domain.
  float qf[G][C::kEPL];
  {
    const T* qb = static_cast<const T*>(a.q) + ((size_t)b * a.Hq + (size_t)kvh * G) * D;
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int i = 0; i < C::kPPL; ++i) {
        const uint4 raw =
            *reinterpret_cast<const uint4*>(qb + (size_t)g * D + (c + 8 * i) * C::kChunk);
        float t[C::kChunk];
        Elem<T>::widen(raw, t);
#pragma unroll
        for (int e = 0; e < C::kChunk; ++e) qf[g][i * C::kChunk + e] = t[e] * a.qscale;
      }
    }
  }

  float m[G], l[G], o[G][C::kEPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < C::kEPL; ++e) o[g][e] = 0.f;
  }

  const T* kpool = static_cast<const T*>(a.k_cache);
  const T* vpool = static_cast<const T*>(a.v_cache);
  const int32_t* table = a.block_tables + (size_t)b * a.MBS;

  for (int blk = blk_begin + warp; blk < blk_end; blk += NW) {
    const int phys = __ldg(table + blk);
    if (phys < 0 || phys >= a.NB) {
      if (lane == 0) raise_error(a.err, kErrBlock);
      continue;  // the block's tokens are treated as absent
    }
    const int n_valid = min(kBlockSize, tok_end - blk * kBlockSize);
    const size_t chunk = ((size_t)phys * a.Hkv + kvh) * (size_t)(kBlockSize * D);

    uint4 kr[C::kSteps][C::kPPL], vr[C::kSteps][C::kPPL];
#pragma unroll
    for (int s = 0; s < C::kSteps; ++s) {
      const int row = s * C::kRowsPerStep + tg;
#pragma unroll
      for (int i = 0; i < C::kPPL; ++i) {
        const size_t off = chunk + (size_t)row * D + (c + 8 * i) * C::kChunk;
        if (row < n_valid) {
          kr[s][i] = ld_stream16(kpool + off);
          vr[s][i] = ld_stream16(vpool + off);
        } else {
          kr[s][i] = make_uint4(0, 0, 0, 0);
          vr[s][i] = make_uint4(0, 0, 0, 0);
        }
      }
    }

    float sc[C::kSteps][G];
#pragma unroll
    for (int s = 0; s < C::kSteps; ++s) {
      float kf[C::kEPL];
#pragma unroll
      for (int i = 0; i < C::kPPL; ++i) Elem<T>::widen(kr[s][i], kf + i * C::kChunk);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < C::kEPL; ++e) acc = fmaf(qf[g][e], kf[e], acc);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        const int row = s * C::kRowsPerStep + tg;
        sc[s][g] = row < n_valid ? acc : -INFINITY;
      }
    }

#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mx = sc[0][g];
#pragma unroll
      for (int s = 1; s < C::kSteps; ++s) mx = fmaxf(mx, sc[s][g]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float mnew = fmaxf(m[g], mx);
      if (mnew > m[g]) {  // warp-uniform: m and mx are identical on all lanes
        const float corr = exp2f(m[g] - mnew);
        l[g] *= corr;
#pragma unroll
        for (int e = 0; e < C::kEPL; ++e) o[g][e] *= corr;
        m[g] = mnew;
      }
    }

#pragma unroll
    for (int s = 0; s < C::kSteps; ++s) {
      float vf[C::kEPL];
#pragma unroll
      for (int i = 0; i < C::kPPL; ++i) Elem<T>::widen(vr[s][i], vf + i * C::kChunk);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pw = exp2f(sc[s][g] - m[g]);
        l[g] += pw;
#pragma unroll
        for (int e = 0; e < C::kEPL; ++e) o[g][e] = fmaf(pw, vf[e], o[g][e]);
      }
    }
  }

  // Sum over the four row groups of the warp (lanes with the same c).
#pragma unroll
  for (int g = 0; g < G; ++g) {
    l[g] += __shfl_xor_sync(0xffffffffu, l[g], 8);
    l[g] += __shfl_xor_sync(0xffffffffu, l[g], 16);
#pragma unroll
    for (int e = 0; e < C::kEPL; ++e) {
      o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], 8);
      o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], 16);
    }
  }
  if (tg == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int i = 0; i < C::kPPL; ++i)
#pragma unroll
        for (int e = 0; e < C::kChunk; ++e)
          sm_o[warp][g][(c + 8 * i) * C::kChunk + e] = o[g][i * C::kChunk + e];
      if (c == 0) {
        sm_m[warp][g] = m[g];
        sm_l[warp][g] = l[g];
      }
    }
  }
  __syncthreads();

  // Combine the warps' partial states.
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int g = idx / D, e = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w)
      if (sm_l[w][g] > 0.f) M = fmaxf(M, sm_m[w][g]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      if (sm_l[w][g] > 0.f) {
        const float wt = exp2f(sm_m[w][g] - M);
        L = fmaf(wt, sm_l[w][g], L);
        O = fmaf(wt, sm_o[w][g][e], O);
      }
    }
    const int h = kvh * G + g;
    if (nparts == 1) {
      T* out = static_cast<T*>(a.out) + ((size_t)b * a.Hq + h) * D;
      out[e] = Elem<T>::narrow(L > 0.f ? O / L : 0.f);
    } else {
      const size_t row = ((size_t)b * a.Hq + h) * a.pmax + p;
      a.ws_o[row * D + e] = O;
      if (e == 0) {
        a.ws_m[row] = M;
        a.ws_l[row] = L;
      }
    }
  }
}

// One warp per (sequence, q head): combine the partitions' (m, l, o).
template <typename T, int D>
__global__ void __launch_bounds__(kMergeWarps * 32) paged_decode_merge_kernel(const DecodeArgs a) {
  constexpr int EPL = D / 32;
  const int item = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  if (item >= a.B * a.Hq) return;
  const int lane = threadIdx.x & 31;
  const int b = item / a.Hq, h = item % a.Hq;
  const int ctx = __ldg(a.context_lens + b);
  if (ctx < 0 || ctx > a.MBS * kBlockSize) return;  // split kernel wrote zeros
  const int nparts = (ctx + a.part - 1) / a.part;
  if (nparts < 2) return;                             // split kernel wrote out
  const size_t row0 = ((size_t)b * a.Hq + h) * a.pmax;
  const float* pm = a.ws_m + row0;
  const float* pl = a.ws_l + row0;
  const float* po = a.ws_o + row0 * D + lane * EPL;

  float M = -INFINITY;
  for (int p = lane; p < nparts; p += 32)
    if (pl[p] > 0.f) M = fmaxf(M, pm[p]);
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, s));

  float L = 0.f, O[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) O[e] = 0.f;
  for (int p = 0; p < nparts; ++p) {
    const float lp = pl[p];
    if (!(lp > 0.f)) continue;
    const float wt = exp2f(pm[p] - M);
    L = fmaf(wt, lp, L);
#pragma unroll
    for (int e = 0; e < EPL; ++e) O[e] = fmaf(wt, po[(size_t)p * D + e], O[e]);
  }
  T* out = static_cast<T*>(a.out) + ((size_t)b * a.Hq + h) * D + lane * EPL;
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) out[e] = Elem<T>::narrow(L > 0.f ? O[e] * inv : 0.f);
}

template <typename T, int D, int G>
cudaError_t launch_decode_impl(const DecodeArgs& a, cudaStream_t stream) {
  const dim3 grid(a.pmax, a.Hkv, a.B);
  if (a.ev_start) cudaEventRecord(a.ev_start, stream);
  paged_decode_split_kernel<T, D, G><<<grid, kDecodeWarps * 32, 0, stream>>>(a);
  if (a.ev_stop) cudaEventRecord(a.ev_stop, stream);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || a.pmax < 2) return err;
  const int items = a.B * a.Hq;
  paged_decode_merge_kernel<T, D>
      <<<(items + kMergeWarps - 1) / kMergeWarps, kMergeWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
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
