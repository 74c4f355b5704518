/*
 * photon_paged.h -- C ABI of the GB300 paged decode-attention library
 * (libphoton_paged.so, CUDA kernels built for sm_103a).
 *
 * What the library computes comes from the PhotonInfer README
 * ("openaitx.github.io/projects/lumia431/photon_infer/README-ko.html"):
 *   - "Key features / GPU-optimized kernels": batched paged attention with a
 *     block-wise KV cache; softmax computed in a numerically stable way;
 *     vectorised 128-bit memory access;
 *   - "Technical details / Paged attention": block-wise KV cache without
 *     fragmentation, per-sequence cache offsets (block tables), and a single
 *     kernel that writes the new K/V rows of many sequences;
 *   - "Key features / Modern C++20 architecture": errors are returned as
 *     explicit values (a Result-style status), and buffers are passed without
 *     copies (the caller owns every buffer).
 * The page gives no formula.  The operation is scaled dot-product attention
 * of one new query row per sequence over that sequence's cached rows, with
 * grouped query heads:
 *     out[b][h] = sum_j softmax_j(scale * q[b][h] . K_j[kvh]) V_j[kvh],
 *     kvh = h / (num_q_heads / num_kv_heads),  j = 0 .. context_lens[b]-1,
 *     K_j, V_j found at cache[block_tables[b][j / block_size]][kvh][j % block_size].
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument named as a buffer is a DEVICE pointer on the
 *   current CUDA device, owned by the caller, and must be 16-byte aligned.
 *   The library allocates no memory, makes no host<->device copies and never
 *   synchronises on the decode/cache-write path; all work is enqueued on
 *   `stream` (NULL = the legacy default stream).
 * - Every entry point returns a photon_status_t.  Argument errors are found on
 *   the host before anything is launched and leave every buffer untouched.
 *   Nothing throws or aborts across this boundary.
 * - Index errors that only the device can see (a block id outside the pool,
 *   a slot outside the pool, a context length outside [0, max_blocks_per_seq *
 *   block_size]) never fault or trap: the offending row / block / sequence is
 *   skipped (a bad sequence is treated as empty, a bad block as absent) and a
 *   sticky device error word is set; photon_get_last_device_error() reads and
 *   clears it.
 *
 * Layouts (row-major, element type = shape->dtype)
 *   k, v (new rows)         [num_tokens][num_kv_heads][head_dim]
 *   q, out                  [num_seqs][num_q_heads][head_dim]
 *   k_cache, v_cache        [num_blocks][num_kv_heads][block_size][head_dim]
 *                           (head-major inside a block: the block_size rows of
 *                           one KV head are one contiguous chunk)
 *   slot_mapping            int64 [num_tokens]; slot = block * block_size +
 *                           offset; a negative slot marks a padding row
 *   block_tables            int32 [num_seqs][max_blocks_per_seq]; entries past
 *                           ceil(context_len / block_size) are never read
 *                           (padding -1 by convention)
 *   context_lens            int32 [num_seqs]; counts the new token
 */
#ifndef PHOTON_PAGED_H
#define PHOTON_PAGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same opaque type as CUDA's cudaStream_t, so a cudaStream_t passes as is. */
typedef struct CUstream_st* photon_stream_t;

typedef enum {
  PHOTON_OK = 0,
  PHOTON_ERR_INVALID_ARG = 1,   /* null pointer, negative size, Hq % Hkv != 0, ... */
  PHOTON_ERR_UNSUPPORTED = 2,   /* head_dim / block_size / dtype not built        */
  PHOTON_ERR_MISALIGNED = 3,    /* a buffer is not 16-byte aligned                */
  PHOTON_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required     */
  PHOTON_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed           */
  PHOTON_ERR_DEVICE_BOUNDS = 6  /* the device saw an out-of-range index (sticky)  */
} photon_status_t;

typedef enum { PHOTON_F32 = 0, PHOTON_F16 = 1, PHOTON_BF16 = 2 } photon_dtype_t;

/* Problem description shared by all calls.
 *   head_dim ∈ {64, 128}; block_size == 16; num_q_heads % num_kv_heads == 0
 *   with group size num_q_heads / num_kv_heads ∈ {1, 2, 4, 8};
 *   dtype ∈ {PHOTON_F32, PHOTON_F16, PHOTON_BF16}.
 *   partition_size: tokens per split-KV partition for photon_paged_decode, a
 *   multiple of block_size in [block_size, 4096]; 0 selects the library
 *   default.  Ignored by the other calls. */
typedef struct {
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t dtype;           /* photon_dtype_t */
  int32_t partition_size;  /* 0 = default */
} photon_paged_shape_t;

/* Batched cache write ("Technical details / Paged attention": one kernel for
 * the K/V writes of many sequences).  For every row t < num_tokens with
 * slot_mapping[t] >= 0 and every KV head h, copies k[t][h][:] and v[t][h][:]
 * bit for bit to k_cache / v_cache[slot / block_size][h][slot % block_size][:].
 * Rows with a negative slot are skipped.  A slot >= num_blocks * block_size is
 * skipped and sets the device error word.  Two rows with the same slot race
 * (the caller must not pass duplicates).  num_tokens == 0 is a no-op.
 * Uses shape: num_kv_heads, head_dim, block_size, num_blocks, dtype. */
photon_status_t photon_cache_write(const void* k, const void* v, const int64_t* slot_mapping,
                                   int32_t num_tokens, void* k_cache, void* v_cache,
                                   const photon_paged_shape_t* shape, photon_stream_t stream);

/* Bytes of device workspace photon_paged_decode needs for this shape (split-KV
 * partials and the work list).  Depends on num_seqs, num_q_heads,
 * num_kv_heads, head_dim, block_size, max_blocks_per_seq and partition_size.
 * Returns 0 for an invalid shape. */
size_t photon_paged_decode_workspace_size(const photon_paged_shape_t* shape);

/* Batched paged decode attention ("Key features / GPU-optimized kernels":
 * batched paged attention, numerically stable softmax).  Computes, for every
 * sequence b and q head h, the formula in this file's header, in fp32
 * arithmetic from the stored dtype, and stores out[b][h][:] rounded to the
 * stored dtype (round to nearest even).  A sequence with context 0 gets a
 * zero row.  The context of each sequence is cut into partitions of
 * partition_size tokens that are attended in parallel and then merged by
 * their log-sum-exp weights.  `workspace` (device, >= the size reported by
 * photon_paged_decode_workspace_size) is scratch owned by the caller; its
 * contents need no initialisation and are undefined afterwards; two calls
 * that may run at the same time must not share it.  scale must be finite. */
photon_status_t photon_paged_decode(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, const int32_t* context_lens,
                                    float scale, void* out, void* workspace,
                                    size_t workspace_bytes, const photon_paged_shape_t* shape,
                                    photon_stream_t stream);

/* One decode step in one call: the batched cache write of the step's new rows
 * followed by the paged decode, with exactly the result of
 * photon_cache_write(k_new, v_new, slot_mapping, num_seqs, ...) and then
 * photon_paged_decode(...) on the same stream (README "Technical details /
 * Paged attention": the per-step K/V write of many sequences, and the batched
 * attention over the block-wise cache).  Precondition of the fused form: one
 * new row per sequence -- row b of k_new / v_new ([num_seqs][Hkv][d]) is the
 * token at position context_lens[b] - 1 of sequence b, and slot_mapping[b]
 * (int64 [num_seqs]) is the slot the block table gives for that position.
 * The attention takes that row straight from k_new / v_new and the kernel that
 * consumes it also stores it into the cache, so no separate scatter pass runs.
 * A slot that disagrees with the block table is flagged (device error bit 2);
 * that row is then neither stored nor attended from k_new (the cache row is
 * used).  Rows of sequences with context 0 are ignored.  Workspace, layouts
 * and errors as photon_paged_decode. */
photon_status_t photon_paged_decode_step(const void* k_new, const void* v_new,
                                         const int64_t* slot_mapping, const void* q,
                                         void* k_cache, void* v_cache,
                                         const int32_t* block_tables,
                                         const int32_t* context_lens, float scale, void* out,
                                         void* workspace, size_t workspace_bytes,
                                         const photon_paged_shape_t* shape,
                                         photon_stream_t stream);

/* Rotary position embedding table for photon_paged_decode_step_rope (README
 * "Key features / GPU-optimized kernels": batched RoPE among the fused
 * kernels).  Writes table[pos][k] = (cos theta, sin theta) as two fp32 values,
 * theta = pos * base^(-2k / head_dim), for 0 <= pos < max_positions and
 * 0 <= k < head_dim / 2; angles are formed and evaluated in double and
 * rounded once to fp32.  `table` (device, 16-byte aligned, owned by the caller)
 * holds max_positions * head_dim / 2 float pairs = max_positions * head_dim * 4
 * bytes.  base must be finite and > 1, head_dim even and > 0, max_positions
 * > 0 with max_positions * head_dim / 2 <= 2^31; otherwise
 * PHOTON_ERR_INVALID_ARG.  Build it once per model; it is read-only to the
 * decode step. */
photon_status_t photon_rope_cos_sin(double base, int32_t max_positions, int32_t head_dim,
                                    void* table, photon_stream_t stream);

/* photon_paged_decode_step with the rotary embedding of the step's new token
 * fused in.  q and k_new arrive unrotated; for sequence b at position
 * pos = context_lens[b] - 1, every q head row and every k_new head row is
 * turned pairwise (rotate-half form): for k < d/2,
 *   y[k]       = x[k] cos(theta) - x[k + d/2] sin(theta)
 *   y[k + d/2] = x[k + d/2] cos(theta) + x[k] sin(theta)
 * with (cos, sin) = rope_cos_sin[pos][k] from photon_rope_cos_sin for the same
 * head_dim.  The cache is assumed to hold already-rotated keys (every earlier
 * step stored its key rotated); values are never rotated.  The rotated new key
 * row, rounded to the stored dtype, is what is attended and what is stored at
 * slot_mapping[b]; the rotated q row stays fp32 for the scores.  A position
 * >= max_positions (rows of the table) sets device error bit 16 and that
 * sequence is attended and stored unrotated.  Everything else -- layouts,
 * slot precondition, workspace, errors -- as photon_paged_decode_step;
 * rope_cos_sin must be 16-byte aligned and max_positions > 0. */
photon_status_t photon_paged_decode_step_rope(
    const void* k_new, const void* v_new, const int64_t* slot_mapping, const void* q,
    void* k_cache, void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
    const void* rope_cos_sin, int32_t max_positions, float scale, void* out, void* workspace,
    size_t workspace_bytes, const photon_paged_shape_t* shape, photon_stream_t stream);

/* Multi-query causal attention over the paged cache (README "Technical
 * details / Paged attention"; "Roadmap": FlashAttention-2 style attention for
 * long sequences): the chunked-prefill / speculative-verification form of
 * photon_paged_decode.  Sequence b has n_b = query_start[b+1] - query_start[b]
 * new query tokens, rows query_start[b] .. query_start[b+1]-1 of q; they are
 * the LAST n_b tokens of its context, so query token i sits at position
 * p_i = context_lens[b] - n_b + i, and its K/V rows must already be in the
 * cache (photon_cache_write first).  For every such token and q head h:
 *     out[query_start[b] + i][h] = sum_{j <= p_i} softmax_j(scale * q . K_j[kvh]) V_j[kvh]
 * (causal: keys 0 .. p_i of the sequence, kvh = h / G), in fp32 arithmetic
 * from fp16/bf16 operands on the tensor cores, out rounded to the stored
 * dtype.  n_b = 1 is exactly the decode row of photon_paged_decode.
 *   q, out        [num_tokens][num_q_heads][head_dim]
 *   query_start   int32 [num_seqs + 1], non-decreasing, query_start[0] >= 0,
 *                 query_start[num_seqs] <= num_tokens
 *   max_query_len host upper bound of every n_b (sizes the launch)
 * dtype must be PHOTON_F16 or PHOTON_BF16 (PHOTON_ERR_UNSUPPORTED for f32).
 * workspace: device scratch of at least
 * photon_paged_multi_query_workspace_size() bytes (may be NULL when that is
 * 0), owned by the caller, no initialisation needed, not shared by calls that
 * may overlap.  Device-side errors (never a fault): n_b < 0, n_b >
 * max_query_len or rows outside [0, num_tokens) set bit 32 and that sequence
 * is skipped (rows past max_query_len are zeroed when they are in range);
 * n_b > context_lens[b] or a context outside [0, max_blocks_per_seq *
 * block_size] sets bit 4 and zeroes the sequence's rows; a block id outside
 * the pool sets bit 1 and its keys read as zeros (that sequence's output is
 * then not meaningful).  num_seqs == 0, num_tokens == 0 or max_query_len == 0
 * is a no-op. */
photon_status_t photon_paged_multi_query(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables,
                                         const int32_t* context_lens,
                                         const int32_t* query_start, int32_t num_tokens,
                                         int32_t max_query_len, float scale, void* out,
                                         void* workspace, size_t workspace_bytes,
                                         const photon_paged_shape_t* shape,
                                         photon_stream_t stream);

/* Bytes of device workspace photon_paged_multi_query needs (0: none).  When
 * the query tiles alone (num_seqs x num_kv_heads x ceil(max_query_len * G /
 * 64)) give fewer than 1216 CTAs, each tile's keys are split into partitions
 * of shape->partition_size keys rounded up to a multiple of 64 (1024 when 0)
 * that run in parallel and are merged by their log-sum-exp weights; a nonzero
 * partition_size forces the split.  The workspace then holds the partials
 * (m, l, o) of num_tokens x num_q_heads rows x ceil(max_blocks_per_seq *
 * block_size / partition) partitions.  When max_query_len x G <= 8 the call
 * runs the decode kernel's few-token mode instead, with the decode's
 * partitions (as photon_paged_decode_workspace_size) per query token; the
 * size returned is the larger of the two, so a workspace of that size serves
 * whichever kernel runs.  0 for an invalid shape, f32, num_tokens <= 0 or
 * max_query_len <= 0. */
size_t photon_paged_multi_query_workspace_size(const photon_paged_shape_t* shape,
                                               int32_t num_tokens, int32_t max_query_len);

/* ---- fp8 (e4m3) KV cache: the further step of the bf16 variant (README
 * "Roadmap": lower-precision KV).  The pools hold OCP e4m3 codes, one byte per
 * element, in the same layout [num_blocks][Hkv][16][head_dim]; element value
 * = code value x scale, one scale for K and one for V (per tensor).  q, out
 * and the new rows stay fp16: shape->dtype must be PHOTON_F16
 * (PHOTON_ERR_UNSUPPORTED otherwise); k_scale and v_scale must be finite and
 * positive (PHOTON_ERR_INVALID_ARG).  Cache pointers 16-byte aligned. */

/* Quantising batched cache write: row t of k / v ([num_tokens][Hkv][d] fp16)
 * is stored at slot_mapping[t] as the e4m3 codes of x * (1 / scale) -- the
 * reciprocal rounded to fp32, the product in fp32, then rounded to the
 * nearest e4m3 value (ties to even), magnitudes beyond 448 saturating to 448.
 * Slots as photon_cache_write (negative = padding, out of range: device
 * error bit 2). */
photon_status_t photon_cache_write_fp8(const void* k, const void* v,
                                       const int64_t* slot_mapping, int32_t num_tokens,
                                       void* k_cache, void* v_cache, float k_scale,
                                       float v_scale, const photon_paged_shape_t* shape,
                                       photon_stream_t stream);

/* Workspace bytes of photon_paged_decode_fp8 (0 for an invalid shape or a
 * dtype other than PHOTON_F16).  Its partitions hold twice the tokens of the
 * fp16 decode's (the same bytes per work item). */
size_t photon_paged_decode_fp8_workspace_size(const photon_paged_shape_t* shape);

/* photon_paged_decode over an e4m3 cache: out = softmax(scale * q . K) V with
 * K = code value x k_scale and V = code value x v_scale, fp32 arithmetic on
 * the tensor cores (the codes widen exactly to fp16), out rounded to fp16.
 * Layouts, context lengths, block tables, errors and workspace rules as
 * photon_paged_decode. */
photon_status_t photon_paged_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_tables, const int32_t* context_lens,
                                        float scale, float k_scale, float v_scale, void* out,
                                        void* workspace, size_t workspace_bytes,
                                        const photon_paged_shape_t* shape,
                                        photon_stream_t stream);

/* Test and tuning hook: which consumer the decode attention kernel runs
 * (photon_paged_decode, _step, _step_rope, _noalloc).  0 (default) = by the group size: the tensor-core consumer
 * (mma.sync over tensor-map copies of the blocks) for fp16/bf16 storage and
 * 2 or more query heads per KV head, the CUDA-core consumer otherwise; 1 =
 * always the CUDA-core consumer; 2 = the tensor-core one wherever the storage
 * type is fp16 or bf16.  Results agree within the documented tolerance, not
 * bit for bit.  Process-wide; PHOTON_ERR_INVALID_ARG for another value. */
photon_status_t photon_debug_set_decode_consumer(int32_t which);

/* Test and tuning hook: which kernel photon_paged_multi_query runs.
 * 0 (default) = chosen by the plan: when max_query_len x G <= 8 (a few draft
 * tokens per sequence), the decode attention kernel in its few-token mode
 * (every (token, head) pair of a sequence's KV head is one of its 8 query
 * slots, with its own causal limit; decode partitions and merge); otherwise
 * the tcgen05/TMEM kernel (256-row tiles, no key split) when the query tiles
 * fill the device without a split, the warp-level mma.sync kernel with its
 * key split when they do not; 1 = always the warp-level kernel (with the
 * plan's split); 2 = always the tcgen05 kernel (no split, workspace unused);
 * 3 = the few-token mode where max_query_len x G <= 8, the plan elsewhere.
 * Results agree within the documented tolerance, not bit for bit.
 * Process-wide; PHOTON_ERR_INVALID_ARG for another value. */
photon_status_t photon_debug_set_multi_query_kernel(int32_t which);

/* Failure-detection self-test: launches one thread that waits on a barrier
 * phase nothing completes, bounded by limit_ns (1 .. 10^9 ns), exactly as
 * every wait inside this library's kernels is bounded.  The bound runs out,
 * the kernel sets device error bit 8 and returns: no fault, no hang, the
 * context stays usable.  Read the bit with photon_get_last_device_error.
 * PHOTON_ERR_INVALID_ARG for a limit outside the range. */
photon_status_t photon_debug_wait_probe(uint64_t limit_ns, photon_stream_t stream);

/* Measuring aid: the decode's K/V data movement with no arithmetic.  For each
 * byte offset in chunk_offsets[0 .. num_chunks) (device memory, int64), the
 * chunk_bytes bytes at that offset of k_cache and of v_cache are copied into
 * shared memory with the bulk copies the decode kernel uses, by a persistent
 * grid of two CTAs per SM that takes runs of chunks_per_run consecutive
 * offsets round robin; nothing reads the copies.  With the offsets of the
 * (block, KV head) runs a decode reads, in its order (README "Key features /
 * GPU-optimized kernels": the batched paged attention's block-table reads),
 * the call's time is the practical read ceiling of that decode.  chunk_bytes:
 * 16 .. 4096, a multiple of 16; offsets must be multiples of 16 with
 * offset + chunk_bytes <= pool_bytes, others are skipped and flagged (device
 * error bit 1); a bounded wait that runs out sets bit 8.  Nothing is written
 * to global memory. */
photon_status_t photon_debug_read_probe(const void* k_cache, const void* v_cache,
                                       uint64_t pool_bytes, const int64_t* chunk_offsets,
                                       int64_t num_chunks, int32_t chunk_bytes,
                                       int32_t chunks_per_run, photon_stream_t stream);

/* photon_paged_decode without a caller-provided workspace.  The pages have no
 * counterpart of this call; it exists for callers that cannot allocate device
 * memory for the decode: an engine that reserved nearly all of HBM for its KV
 * pool at start-up (a later cudaMalloc would fail or cut into that pool), a
 * plugin that is given no allocator by its host, or a decode path that must
 * not call cudaMalloc/cudaFree because those calls can synchronise the device.
 * Arguments, layouts, arithmetic and results are those of photon_paged_decode.
 * The split-KV scratch comes from one array built into the library:
 *   - its size is fixed at 32 MiB per GPU, held by every GPU that loads the
 *     library until the process exits; a problem whose
 *     photon_paged_decode_workspace_size() exceeds 32 MiB is rejected with
 *     PHOTON_ERR_WORKSPACE before anything is launched;
 *   - the first call made with a given device current looks up the array's
 *     device address for that device (cudaGetSymbolAddress) and keeps it for
 *     the life of the process; make that first call before starting any
 *     stream capture, and do not use this entry point on a device after a
 *     cudaDeviceReset of it (the kept address would then be stale);
 *   - every call on a device uses the same array and leaves its last contents
 *     there; nothing in it needs to be cleared between calls, but calls whose
 *     kernels may overlap on the GPU (different streams, no ordering) race on
 *     it and must not be issued.
 * No memory is allocated and nothing is copied between host and device. */
photon_status_t photon_paged_decode_noalloc(const void* q, const void* k_cache,
                                            const void* v_cache, const int32_t* block_tables,
                                            const int32_t* context_lens, float scale, void* out,
                                            const photon_paged_shape_t* shape,
                                            photon_stream_t stream);

/* Test / diagnostic export: the block-table gather the decode kernel performs,
 * materialised.  k_dense, v_dense are [num_seqs][num_kv_heads][max_blocks_per_seq
 * * block_size][head_dim]; row j of sequence b is a bit copy of the cached row
 * at logical position j for j < context_lens[b] and zero bytes after. */
photon_status_t photon_paged_gather(const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, const int32_t* context_lens,
                                    void* k_dense, void* v_dense,
                                    const photon_paged_shape_t* shape, photon_stream_t stream);

/* Synchronises `stream`, then reads and clears the current device's sticky
 * error word.  Returns PHOTON_ERR_DEVICE_BOUNDS if any kernel of this library
 * skipped an out-of-range index since the last call, PHOTON_ERR_CUDA if the
 * synchronisation itself failed, PHOTON_OK otherwise.  If `bits` is not NULL
 * it receives the word: 1 = block id out of range, 2 = slot out of range (or,
 * in the fused step, not the block table's slot for the new position),
 * 4 = context length out of range, 8 = a bounded wait inside a kernel ran out
 * (the call's output is then incomplete), 16 = a RoPE position outside the
 * cos/sin table, 32 = inconsistent query_start / max_query_len of
 * photon_paged_multi_query. */
photon_status_t photon_get_last_device_error(photon_stream_t stream, uint32_t* bits);

/* Static text for a status code (never NULL). */
const char* photon_status_string(photon_status_t status);

/* Diagnostic: launch geometry photon_paged_decode would use for `shape` on the
 * current device: the partition size in tokens, the largest number of
 * partitions a sequence can have, the number of CTAs of the attention kernel
 * and the number of kernels one call launches.  Any output pointer may be
 * NULL. */
photon_status_t photon_paged_decode_plan(const photon_paged_shape_t* shape,
                                         int32_t* partition_size, int32_t* max_partitions,
                                         int32_t* attention_ctas, int32_t* kernels_per_call);

/* Diagnostic timing hook: when both are non-NULL, photon_paged_decode records
 * start_event right before and stop_event right after its split-KV attention
 * kernel, on the call's stream (cudaEvent_t values passed as void*).  Pass
 * NULL, NULL to turn it off.  Process-wide; not for concurrent use. */
photon_status_t photon_debug_set_attention_events(void* start_event, void* stop_event);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif /* PHOTON_PAGED_H */
