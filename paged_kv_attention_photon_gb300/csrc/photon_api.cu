// photon_api.cu -- the extern "C" boundary of libphoton_paged.so.
//
// Host-side argument checks, workspace carving, the sticky device error word
// and dispatch to the kernels.  Error handling follows the PhotonInfer
// README's "Modern C++20 architecture" notes (errors propagate as explicit
// Result-style values, buffers are used in place without copies): every call
// returns a status, nothing throws across the boundary, and the library never
// allocates or copies the caller's data.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>

#include "../../include/photon_paged.h"
#include "photon_common.cuh"

namespace photon {
// selftest.cu
cudaError_t launch_wait_probe(unsigned long long limit_ns, uint32_t* err, cudaStream_t stream);
// read_probe.cu
cudaError_t launch_read_probe(const void* k, const void* v, const int64_t* offs, int64_t n,
                              uint32_t chunk_bytes, int run, uint64_t pool_bytes, int num_sms,
                              uint32_t* err, cudaStream_t stream);
std::atomic<int> g_decode_consumer{0};
}  // namespace photon

namespace {

// Sticky device error word, one per device that loads the library.
__device__ uint32_t g_photon_error_word;

constexpr int kMaxDevices = 64;
std::atomic<uint32_t*> g_err_ptr[kMaxDevices];

std::atomic<cudaEvent_t> g_ev_start{nullptr};
// photon_paged_multi_query kernel choice: 0 = by the plan, 1 = warp-level
// mma.sync kernel, 2 = tcgen05 kernel.
std::atomic<int> g_mq_kernel{0};
std::atomic<cudaEvent_t> g_ev_stop{nullptr};

constexpr int kMaxPartition = 4096;
// Default partition: about 192 KB of K+V per (partition, KV head) work item,
// i.e. a few microseconds of one SM's share of HBM bandwidth, so the last
// items of the persistent grid finish close together.
constexpr int kItemBytes = 192 * 1024;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_bytes(int32_t dtype) { return dtype == PHOTON_F32 ? 4u : 2u; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Checks shared by every call.  Launches nothing, touches no CUDA state.
photon_status_t check_shape(const photon_paged_shape_t* s) {
  if (!s) return PHOTON_ERR_INVALID_ARG;
  if (s->num_seqs < 0 || s->num_q_heads <= 0 || s->num_kv_heads <= 0 || s->num_blocks < 0 ||
      s->max_blocks_per_seq <= 0 || s->head_dim <= 0 || s->block_size <= 0)
    return PHOTON_ERR_INVALID_ARG;
  if (s->num_q_heads % s->num_kv_heads != 0) return PHOTON_ERR_INVALID_ARG;
  const int g = s->num_q_heads / s->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return PHOTON_ERR_UNSUPPORTED;
  if (s->head_dim != 64 && s->head_dim != 128) return PHOTON_ERR_UNSUPPORTED;
  if (s->block_size != photon::kBlockSize) return PHOTON_ERR_UNSUPPORTED;
  if (s->dtype != PHOTON_F32 && s->dtype != PHOTON_F16 && s->dtype != PHOTON_BF16)
    return PHOTON_ERR_UNSUPPORTED;
  if (s->partition_size != 0 &&
      (s->partition_size < s->block_size || s->partition_size > kMaxPartition ||
       s->partition_size % s->block_size != 0))
    return PHOTON_ERR_INVALID_ARG;
  // Index arithmetic inside the kernels stays in 32-bit for these.
  if ((int64_t)s->max_blocks_per_seq * s->block_size > INT_MAX / 2) return PHOTON_ERR_UNSUPPORTED;
  if (s->num_seqs > 65535 || s->num_kv_heads > 65535) return PHOTON_ERR_UNSUPPORTED;
  return PHOTON_OK;
}

// kv_bytes: bytes per cached element (0: the shape's dtype; 1: an e4m3 cache)
int partition_of(const photon_paged_shape_t* s, int kv_bytes = 0) {
  if (s->partition_size) return s->partition_size;
  const int eb = kv_bytes > 0 ? kv_bytes : (int)elem_bytes(s->dtype);
  const int per_token = 2 * s->head_dim * eb;  // K + V bytes
  int part = kItemBytes / per_token / s->block_size * s->block_size;
  // A small batch has too few such items to keep the grid busy, and one
  // item's latency then sets the call's time: shrink the partition so that
  // even the largest contexts the shape allows give about two items per
  // resident CTA (2 per SM on 152 SMs), rounded to the nearest whole stage of
  // 64 tokens (one 16-token block per consumer warp: a partial stage costs as
  // much time as a full one).  Against rounding down to a block, the rounding
  // measured 11 % faster on the batch-4 sweep shape and 9 % on batch 16.
  constexpr int64_t kTargetItems = 2 * 2 * 152;
  constexpr int64_t kStageTokens = 64;
  const int64_t span_tokens = (int64_t)s->num_seqs * s->max_blocks_per_seq * s->block_size *
                              s->num_kv_heads;
  int64_t fit = (span_tokens / kTargetItems + kStageTokens / 2) / kStageTokens * kStageTokens;
  if (fit < kStageTokens) fit = kStageTokens;
  if (fit < part) part = (int)fit;
  if (part < s->block_size) part = s->block_size;
  if (part > kMaxPartition) part = kMaxPartition;
  return part;
}

// Partitions of the longest context the shape allows: its full partitions,
// one more when the last full one is cut in halves (two or more full ones,
// partition size >= 32: the attention kernel's partition_split), and the
// remainder.
int max_partitions_of(const photon_paged_shape_t* s, int kv_bytes = 0) {
  const int64_t span = (int64_t)s->max_blocks_per_seq * s->block_size;
  const int part = partition_of(s, kv_bytes);
  const int64_t nfull = span / part;
  return (int)(nfull + (nfull >= 2 && part >= 32 ? 1 : 0) + (span % part != 0 ? 1 : 0));
}

// Workspace: [queue control][m][l][o] (the last three per query row, q head
// and partition; a decode has one query row per sequence, the few-token
// multi-query path one per query token), each section 256-byte aligned.
struct WorkspaceLayout {
  size_t off_ctrl, off_m, off_l, off_o, total;
};

WorkspaceLayout layout_of(const photon_paged_shape_t* s, int64_t query_rows = -1,
                          int kv_bytes = 0) {
  WorkspaceLayout w{};
  if (query_rows < 0) query_rows = s->num_seqs;
  const size_t pairs = (size_t)query_rows * (size_t)max_partitions_of(s, kv_bytes);
  const size_t rows = pairs * s->num_q_heads;
  w.off_ctrl = 0;
  w.off_m = 256;
  w.off_l = round_up(w.off_m + rows * sizeof(float), 256);
  w.off_o = round_up(w.off_l + rows * sizeof(float), 256);
  w.total = round_up(w.off_o + rows * (size_t)s->head_dim * sizeof(float), 256);
  if (rows == 0) w.total = 0;
  return w;
}

// SM count of the current device (cached per device).
std::atomic<int> g_num_sms[kMaxDevices];

photon_status_t num_sms(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PHOTON_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PHOTON_ERR_UNSUPPORTED;
  int n = g_num_sms[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return PHOTON_ERR_CUDA;
    g_num_sms[dev].store(n, std::memory_order_relaxed);
  }
  *out = n;
  return PHOTON_OK;
}

// Device address of the error word for the current device.
photon_status_t error_word(uint32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PHOTON_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PHOTON_ERR_UNSUPPORTED;
  uint32_t* p = g_err_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_photon_error_word) != cudaSuccess) return PHOTON_ERR_CUDA;
    p = static_cast<uint32_t*>(addr);
    g_err_ptr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return PHOTON_OK;
}

}  // namespace

extern "C" {

const char* photon_status_string(photon_status_t status) {
  switch (status) {
    case PHOTON_OK: return "ok";
    case PHOTON_ERR_INVALID_ARG: return "invalid argument";
    case PHOTON_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case PHOTON_ERR_MISALIGNED: return "buffer not 16-byte aligned";
    case PHOTON_ERR_WORKSPACE: return "workspace missing or too small";
    case PHOTON_ERR_CUDA: return "CUDA runtime error";
    case PHOTON_ERR_DEVICE_BOUNDS: return "device saw an out-of-range index";
  }
  return "unknown status";
}

photon_status_t photon_cache_write(const void* k, const void* v, const int64_t* slot_mapping,
                                   int32_t num_tokens, void* k_cache, void* v_cache,
                                   const photon_paged_shape_t* shape, photon_stream_t stream) {
  photon_status_t st = check_shape(shape);
  if (st != PHOTON_OK) return st;
  if (num_tokens < 0) return PHOTON_ERR_INVALID_ARG;
  if (num_tokens == 0) return PHOTON_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PHOTON_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PHOTON_ERR_MISALIGNED;
  uint32_t* err = nullptr;
  if ((st = error_word(&err)) != PHOTON_OK) return st;
  photon::CacheWriteArgs a{};
  a.k = k;
  a.v = v;
  a.slot_mapping = slot_mapping;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.err = err;
  a.T = num_tokens;
  a.Hkv = shape->num_kv_heads;
  a.row_bytes = (int)(shape->head_dim * elem_bytes(shape->dtype));
  a.block_size = shape->block_size;
  a.NB = shape->num_blocks;
  return photon::launch_cache_write(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PHOTON_OK
             : PHOTON_ERR_CUDA;
}

size_t photon_paged_decode_workspace_size(const photon_paged_shape_t* shape) {
  if (check_shape(shape) != PHOTON_OK) return 0;
  return layout_of(shape).total;
}

photon_status_t photon_cache_write_fp8(const void* k, const void* v,
                                       const int64_t* slot_mapping, int32_t num_tokens,
                                       void* k_cache, void* v_cache, float k_scale,
                                       float v_scale, const photon_paged_shape_t* shape,
                                       photon_stream_t stream) {
  photon_status_t st = check_shape(shape);
  if (st != PHOTON_OK) return st;
  if (shape->dtype != PHOTON_F16) return PHOTON_ERR_UNSUPPORTED;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return PHOTON_ERR_INVALID_ARG;
  if (num_tokens < 0) return PHOTON_ERR_INVALID_ARG;
  if (num_tokens == 0) return PHOTON_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PHOTON_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PHOTON_ERR_MISALIGNED;
  uint32_t* err = nullptr;
  if ((st = error_word(&err)) != PHOTON_OK) return st;
  photon::CacheWriteFp8Args a{};
  a.k = k;
  a.v = v;
  a.slot_mapping = slot_mapping;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.err = err;
  a.k_inv = 1.0f / k_scale;   // fp32 reciprocal, then an fp32 product per element
  a.v_inv = 1.0f / v_scale;
  a.T = num_tokens;
  a.Hkv = shape->num_kv_heads;
  a.D = shape->head_dim;
  a.block_size = shape->block_size;
  a.NB = shape->num_blocks;
  return photon::launch_cache_write_fp8(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PHOTON_OK
             : PHOTON_ERR_CUDA;
}

size_t photon_paged_decode_fp8_workspace_size(const photon_paged_shape_t* shape) {
  if (check_shape(shape) != PHOTON_OK || shape->dtype != PHOTON_F16) return 0;
  return layout_of(shape, -1, 1).total;
}

photon_status_t photon_paged_decode_plan(const photon_paged_shape_t* shape,
                                         int32_t* partition_size, int32_t* max_partitions,
                                         int32_t* attention_ctas, int32_t* kernels_per_call) {
  photon_status_t st = check_shape(shape);
  if (st != PHOTON_OK) return st;
  const int pmax = max_partitions_of(shape);
  if (partition_size) *partition_size = partition_of(shape);
  if (max_partitions) *max_partitions = pmax;
  if (kernels_per_call) *kernels_per_call = shape->num_seqs == 0 ? 0 : 2;
  if (attention_ctas) {
    // The persistent grid fills the device: two CTAs per SM of the current
    // device (0 when no device is visible).
    int sms = 0;
    *attention_ctas = num_sms(&sms) == PHOTON_OK ? 2 * sms : 0;
  }
  return PHOTON_OK;
}

}  // extern "C"

namespace {

// Shared body of photon_paged_decode and photon_paged_decode_step: checks the
// decode arguments, carves the workspace and launches.  k_new == nullptr means
// a plain decode.
photon_status_t decode_common(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, const int32_t* context_lens,
                              float scale, void* out, void* workspace, size_t workspace_bytes,
                              const photon_paged_shape_t* shape, photon_stream_t stream,
                              const void* k_new, const void* v_new,
                              const int64_t* slot_mapping, const void* rope_cos_sin,
                              int32_t rope_max_positions,
                              const int32_t* query_start = nullptr, int32_t num_tokens = 0,
                              int32_t max_query_len = 0, bool fp8 = false, float k_scale = 1.f,
                              float v_scale = 1.f) {
  photon_status_t st = check_shape(shape);
  if (st != PHOTON_OK) return st;
  if (!std::isfinite(scale)) return PHOTON_ERR_INVALID_ARG;
  if (fp8) {
    // e4m3 K/V, fp16 q and out; the scales turn codes into values
    if (shape->dtype != PHOTON_F16) return PHOTON_ERR_UNSUPPORTED;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) ||
        !std::isfinite(v_scale))
      return PHOTON_ERR_INVALID_ARG;
  }
  if (shape->num_seqs == 0) return PHOTON_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return PHOTON_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(block_tables) ||
      !aligned16(context_lens) || !aligned16(out))
    return PHOTON_ERR_MISALIGNED;
  const int kv_bytes = fp8 ? 1 : 0;
  const WorkspaceLayout wl = layout_of(shape, query_start ? (int64_t)num_tokens : -1, kv_bytes);
  if (wl.total > 0) {
    if (!workspace || workspace_bytes < wl.total) return PHOTON_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PHOTON_ERR_MISALIGNED;
  }
  uint32_t* err = nullptr;
  if ((st = error_word(&err)) != PHOTON_OK) return st;
  int sms = 0;
  if ((st = num_sms(&sms)) != PHOTON_OK) return st;

  photon::DecodeArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = out;
  char* ws = static_cast<char*>(workspace);
  a.ws_m = reinterpret_cast<float*>(ws + wl.off_m);
  a.ws_l = reinterpret_cast<float*>(ws + wl.off_l);
  a.ws_o = reinterpret_cast<float*>(ws + wl.off_o);
  a.ws_ctrl = reinterpret_cast<unsigned long long*>(ws + wl.off_ctrl);
  a.num_sms = sms;
  a.k_new = k_new;
  a.v_new = v_new;
  a.slot_mapping = slot_mapping;
  a.k_cache_w = k_new ? const_cast<void*>(k_cache) : nullptr;
  a.v_cache_w = k_new ? const_cast<void*>(v_cache) : nullptr;
  a.rope_cs = static_cast<const float2*>(rope_cos_sin);
  a.rope_max_pos = rope_cos_sin ? rope_max_positions : 0;
  a.err = err;
  // scale * log2(e) (times the K scale of an e4m3 cache)
  a.qscale = (float)((double)scale * (double)k_scale * 1.4426950408889634);
  a.v_scale = v_scale;
  a.B = shape->num_seqs;
  a.Hq = shape->num_q_heads;
  a.Hkv = shape->num_kv_heads;
  a.D = shape->head_dim;
  a.NB = shape->num_blocks;
  a.MBS = shape->max_blocks_per_seq;
  a.part = partition_of(shape, kv_bytes);
  a.pmax = max_partitions_of(shape, kv_bytes);
  a.query_start = query_start;
  a.num_tokens = num_tokens;
  a.max_q = max_query_len;
  a.ev_start = query_start ? nullptr : g_ev_start.load(std::memory_order_acquire);
  a.ev_stop = query_start ? nullptr : g_ev_stop.load(std::memory_order_acquire);
  if (!a.ev_start || !a.ev_stop) a.ev_start = a.ev_stop = nullptr;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (fp8) {
    e = photon::launch_paged_decode_fp8(a, s);
    return e == cudaSuccess ? PHOTON_OK : PHOTON_ERR_CUDA;
  }
  switch (shape->dtype) {
    case PHOTON_F32: e = photon::launch_paged_decode_f32(a, s); break;
    case PHOTON_F16: e = photon::launch_paged_decode_f16(a, s); break;
    default: e = photon::launch_paged_decode_bf16(a, s); break;
  }
  return e == cudaSuccess ? PHOTON_OK : PHOTON_ERR_CUDA;
}

}  // namespace

extern "C" {

photon_status_t photon_paged_decode(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, const int32_t* context_lens,
                                    float scale, void* out, void* workspace,
                                    size_t workspace_bytes, const photon_paged_shape_t* shape,
                                    photon_stream_t stream) {
  return decode_common(q, k_cache, v_cache, block_tables, context_lens, scale, out, workspace,
                       workspace_bytes, shape, stream, nullptr, nullptr, nullptr, nullptr, 0);
}

photon_status_t photon_paged_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_tables, const int32_t* context_lens,
                                        float scale, float k_scale, float v_scale, void* out,
                                        void* workspace, size_t workspace_bytes,
                                        const photon_paged_shape_t* shape,
                                        photon_stream_t stream) {
  return decode_common(q, k_cache, v_cache, block_tables, context_lens, scale, out, workspace,
                       workspace_bytes, shape, stream, nullptr, nullptr, nullptr, nullptr, 0,
                       nullptr, 0, 0, true, k_scale, v_scale);
}

photon_status_t photon_paged_decode_step(const void* k_new, const void* v_new,
                                         const int64_t* slot_mapping, const void* q,
                                         void* k_cache, void* v_cache,
                                         const int32_t* block_tables,
                                         const int32_t* context_lens, float scale, void* out,
                                         void* workspace, size_t workspace_bytes,
                                         const photon_paged_shape_t* shape,
                                         photon_stream_t stream) {
  photon_status_t st = check_shape(shape);
  if (st != PHOTON_OK) return st;
  if (shape->num_seqs == 0) return PHOTON_OK;
  if (!k_new || !v_new || !slot_mapping) return PHOTON_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PHOTON_ERR_MISALIGNED;
  return decode_common(q, k_cache, v_cache, block_tables, context_lens, scale, out, workspace,
                       workspace_bytes, shape, stream, k_new, v_new, slot_mapping, nullptr, 0);
}

photon_status_t photon_rope_cos_sin(double base, int32_t max_positions, int32_t head_dim,
                                    void* table, photon_stream_t stream) {
  if (!(base > 1.0) || !std::isfinite(base) || max_positions <= 0 || head_dim <= 0 ||
      head_dim % 2 != 0)
    return PHOTON_ERR_INVALID_ARG;
  if ((long long)max_positions * (head_dim / 2) > (1ll << 31)) return PHOTON_ERR_INVALID_ARG;
  if (!table) return PHOTON_ERR_INVALID_ARG;
  if (!aligned16(table)) return PHOTON_ERR_MISALIGNED;
  return photon::launch_rope_table(base, max_positions, head_dim, static_cast<float2*>(table),
                                   reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PHOTON_OK
             : PHOTON_ERR_CUDA;
}

photon_status_t photon_paged_decode_step_rope(
    const void* k_new, const void* v_new, const int64_t* slot_mapping, const void* q,
    void* k_cache, void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
    const void* rope_cos_sin, int32_t max_positions, float scale, void* out, void* workspace,
    size_t workspace_bytes, const photon_paged_shape_t* shape, photon_stream_t stream) {
  photon_status_t st = check_shape(shape);
  if (st != PHOTON_OK) return st;
  if (shape->num_seqs == 0) return PHOTON_OK;
  if (!k_new || !v_new || !slot_mapping || !rope_cos_sin || max_positions <= 0)
    return PHOTON_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) ||
      !aligned16(rope_cos_sin))
    return PHOTON_ERR_MISALIGNED;
  return decode_common(q, k_cache, v_cache, block_tables, context_lens, scale, out, workspace,
                       workspace_bytes, shape, stream, k_new, v_new, slot_mapping, rope_cos_sin,
                       max_positions);
}

}  // extern "C"

namespace {

// Split-KV plan of photon_paged_multi_query.  Without a split a launch has
// num_seqs x Hkv x ceil(max_query_len * G / 64) CTAs; when that is below
// about four waves of the device (2 CTAs per SM on 152 SMs) every tile's keys
// are cut into partitions (shape->partition_size rounded up to 64 keys, or
// 1024 by default, the best of 256..4096 measured on 64 x 4 draft tokens over
// long contexts) so that short query batches over long contexts still fill
// the SMs.  A fixed threshold keeps the plan, and so the workspace size, a
// function of the arguments alone.
struct MqPlan {
  int part, pmax;
  size_t off_l, off_o, total;
};

constexpr int kMqTileRows = 64;
constexpr int kMqSplitBelow = 4 * 2 * 152;

// Query batches whose every sequence fits the decode kernel's 8 query slots
// per KV head (max_query_len x G <= 8: speculative verification with a few
// draft tokens) can run as a decode over the same partitions: K/V streamed
// once per (sequence, KV head) for all of its tokens.
bool few_token(const photon_paged_shape_t* s, int32_t max_query_len) {
  return (int64_t)max_query_len * (s->num_q_heads / s->num_kv_heads) <= 8;
}

MqPlan mq_plan(const photon_paged_shape_t* s, int32_t num_tokens, int32_t max_query_len) {
  MqPlan p{};
  const int64_t G = s->num_q_heads / s->num_kv_heads;
  const int64_t tiles = ((int64_t)max_query_len * G + kMqTileRows - 1) / kMqTileRows;
  const int64_t ctas = (int64_t)s->num_seqs * s->num_kv_heads * tiles;
  const int64_t span = (int64_t)s->max_blocks_per_seq * s->block_size;
  int part = s->partition_size > 0 ? (s->partition_size + 63) / 64 * 64 : 1024;
  if (s->partition_size == 0 && ctas >= kMqSplitBelow) part = (int)((span + 63) / 64 * 64);
  if (part < 64) part = 64;
  p.part = part;
  p.pmax = (int)((span + part - 1) / part);
  if (p.pmax < 1) p.pmax = 1;
  if (p.pmax == 1) return p;
  const size_t rows = (size_t)num_tokens * s->num_q_heads * p.pmax;
  p.off_l = round_up(rows * sizeof(float), 256);
  p.off_o = p.off_l + round_up(rows * sizeof(float), 256);
  p.total = p.off_o + round_up(rows * (size_t)s->head_dim * sizeof(float), 256);
  return p;
}

}  // namespace

extern "C" {

size_t photon_paged_multi_query_workspace_size(const photon_paged_shape_t* shape,
                                               int32_t num_tokens, int32_t max_query_len) {
  if (check_shape(shape) != PHOTON_OK || shape->dtype == PHOTON_F32 || num_tokens <= 0 ||
      max_query_len <= 0)
    return 0;
  size_t total = mq_plan(shape, num_tokens, max_query_len).total;
  // enough for whichever kernel the call takes
  if (few_token(shape, max_query_len)) total = std::max(total, layout_of(shape, num_tokens).total);
  return total;
}

photon_status_t photon_paged_multi_query(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables,
                                         const int32_t* context_lens,
                                         const int32_t* query_start, int32_t num_tokens,
                                         int32_t max_query_len, float scale, void* out,
                                         void* workspace, size_t workspace_bytes,
                                         const photon_paged_shape_t* shape,
                                         photon_stream_t stream) {
  photon_status_t st = check_shape(shape);
  if (st != PHOTON_OK) return st;
  if (shape->dtype == PHOTON_F32) return PHOTON_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || num_tokens < 0 || max_query_len < 0) return PHOTON_ERR_INVALID_ARG;
  if (shape->num_seqs == 0 || num_tokens == 0 || max_query_len == 0) return PHOTON_OK;
  if (shape->num_seqs > 65535 || shape->num_kv_heads > 65535) return PHOTON_ERR_UNSUPPORTED;
  if ((int64_t)max_query_len * (shape->num_q_heads / shape->num_kv_heads) > INT_MAX / 2)
    return PHOTON_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start || !out)
    return PHOTON_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(block_tables) ||
      !aligned16(context_lens) || !aligned16(query_start) || !aligned16(out))
    return PHOTON_ERR_MISALIGNED;
  // Few draft tokens per sequence: the decode kernel in its few-token mode
  // (the default there; selector 3 asks for it, 1 and 2 for the others).
  const int choice = g_mq_kernel.load(std::memory_order_relaxed);
  if ((choice == 0 || choice == 3) && few_token(shape, max_query_len))
    return decode_common(q, k_cache, v_cache, block_tables, context_lens, scale, out, workspace,
                         workspace_bytes, shape, stream, nullptr, nullptr, nullptr, nullptr, 0,
                         query_start, num_tokens, max_query_len);
  const MqPlan plan = mq_plan(shape, num_tokens, max_query_len);
  {
    const int64_t G = shape->num_q_heads / shape->num_kv_heads;
    const int64_t tiles = ((int64_t)max_query_len * G + kMqTileRows - 1) / kMqTileRows;
    if (tiles * plan.pmax > INT_MAX || ((int64_t)max_query_len * shape->num_q_heads + 3) / 4 > INT_MAX)
      return PHOTON_ERR_UNSUPPORTED;
  }
  if (plan.total > 0) {
    if (!workspace || workspace_bytes < plan.total) return PHOTON_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PHOTON_ERR_MISALIGNED;
  }
  uint32_t* err = nullptr;
  if ((st = error_word(&err)) != PHOTON_OK) return st;
  photon::MultiQueryArgs a{};
  a.part = plan.part;
  a.pmax = plan.pmax;
  if (plan.total > 0) {
    char* ws = static_cast<char*>(workspace);
    a.ws_m = reinterpret_cast<float*>(ws);
    a.ws_l = reinterpret_cast<float*>(ws + plan.off_l);
    a.ws_o = reinterpret_cast<float*>(ws + plan.off_o);
  }
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.query_start = query_start;
  a.out = out;
  a.err = err;
  a.qscale = (float)((double)scale * 1.4426950408889634);  // scale * log2(e)
  a.B = shape->num_seqs;
  a.Hq = shape->num_q_heads;
  a.Hkv = shape->num_kv_heads;
  a.D = shape->head_dim;
  a.NB = shape->num_blocks;
  a.MBS = shape->max_blocks_per_seq;
  a.max_query_len = max_query_len;
  a.num_tokens = num_tokens;
  a.dtype = shape->dtype;
  // Query batches that fill the device without a key split (chunked prefill)
  // run on the tcgen05 kernel; split batches (a few tokens per sequence) on
  // the warp-level kernel and its merge.
  const bool tc = choice == 2 || ((choice == 0 || choice == 3) && plan.pmax == 1);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = tc ? photon::launch_multi_query_tc(a, s) : photon::launch_multi_query(a, s);
  return e == cudaSuccess ? PHOTON_OK : PHOTON_ERR_CUDA;
}

photon_status_t photon_debug_set_decode_consumer(int32_t which) {
  if (which < 0 || which > 2) return PHOTON_ERR_INVALID_ARG;
  photon::g_decode_consumer.store(which, std::memory_order_relaxed);
  return PHOTON_OK;
}

photon_status_t photon_debug_set_multi_query_kernel(int32_t which) {
  if (which < 0 || which > 3) return PHOTON_ERR_INVALID_ARG;
  g_mq_kernel.store(which, std::memory_order_relaxed);
  return PHOTON_OK;
}

photon_status_t photon_paged_gather(const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, const int32_t* context_lens,
                                    void* k_dense, void* v_dense,
                                    const photon_paged_shape_t* shape, photon_stream_t stream) {
  photon_status_t st = check_shape(shape);
  if (st != PHOTON_OK) return st;
  if (shape->num_seqs == 0) return PHOTON_OK;
  if (!k_cache || !v_cache || !block_tables || !context_lens || !k_dense || !v_dense)
    return PHOTON_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(block_tables) ||
      !aligned16(context_lens) || !aligned16(k_dense) || !aligned16(v_dense))
    return PHOTON_ERR_MISALIGNED;
  uint32_t* err = nullptr;
  if ((st = error_word(&err)) != PHOTON_OK) return st;
  photon::GatherArgs a{};
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.k_dense = k_dense;
  a.v_dense = v_dense;
  a.err = err;
  a.B = shape->num_seqs;
  a.Hkv = shape->num_kv_heads;
  a.row_bytes = (int)(shape->head_dim * elem_bytes(shape->dtype));
  a.block_size = shape->block_size;
  a.NB = shape->num_blocks;
  a.MBS = shape->max_blocks_per_seq;
  return photon::launch_gather(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PHOTON_OK
             : PHOTON_ERR_CUDA;
}

photon_status_t photon_get_last_device_error(photon_stream_t stream, uint32_t* bits) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PHOTON_ERR_CUDA;
  uint32_t word = 0;
  const uint32_t zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_photon_error_word, sizeof(word)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_photon_error_word, &zero, sizeof(zero)) != cudaSuccess)
    return PHOTON_ERR_CUDA;
  if (bits) *bits = word;
  return word ? PHOTON_ERR_DEVICE_BOUNDS : PHOTON_OK;
}

photon_status_t photon_debug_wait_probe(uint64_t limit_ns, photon_stream_t stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ull) return PHOTON_ERR_INVALID_ARG;
  uint32_t* err = nullptr;
  photon_status_t st = error_word(&err);
  if (st != PHOTON_OK) return st;
  return photon::launch_wait_probe(limit_ns, err, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? PHOTON_OK
             : PHOTON_ERR_CUDA;
}

photon_status_t photon_debug_read_probe(const void* k_cache, const void* v_cache,
                                       uint64_t pool_bytes, const int64_t* chunk_offsets,
                                       int64_t num_chunks, int32_t chunk_bytes,
                                       int32_t chunks_per_run, photon_stream_t stream) {
  if (num_chunks < 0 || chunk_bytes <= 0 || chunk_bytes > 4096 || chunk_bytes % 16 != 0 ||
      chunks_per_run <= 0)
    return PHOTON_ERR_INVALID_ARG;
  if (num_chunks == 0) return PHOTON_OK;
  if (!k_cache || !v_cache || !chunk_offsets) return PHOTON_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(chunk_offsets))
    return PHOTON_ERR_MISALIGNED;
  uint32_t* err = nullptr;
  photon_status_t st = error_word(&err);
  if (st != PHOTON_OK) return st;
  int sms = 0;
  if ((st = num_sms(&sms)) != PHOTON_OK) return st;
  return photon::launch_read_probe(k_cache, v_cache, chunk_offsets, num_chunks,
                                   (uint32_t)chunk_bytes, chunks_per_run, pool_bytes, sms, err,
                                   reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PHOTON_OK
             : PHOTON_ERR_CUDA;
}

photon_status_t photon_debug_set_attention_events(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr)) return PHOTON_ERR_INVALID_ARG;
  g_ev_start.store(static_cast<cudaEvent_t>(start_event), std::memory_order_release);
  g_ev_stop.store(static_cast<cudaEvent_t>(stop_event), std::memory_order_release);
  return PHOTON_OK;
}

}  // extern "C"
