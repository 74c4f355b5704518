/*
 * photon_scheduler.h -- host-side KV block manager and two-phase
 * continuous-batching scheduler of libphoton_paged.so (plain C++ on the CPU;
 * no CUDA call, no device memory).
 *
 * It produces, step by step, the integer inputs of the device calls in
 * photon_paged.h: which requests run, how many new tokens each one computes,
 * their block tables, context lengths and the cache slot of every new token.
 *
 * What it follows, from the PhotonInfer README
 * ("openaitx.github.io/projects/lumia431/photon_infer/README-ko.html"):
 *   - "Key features / vLLM-style continuous batching": token-level dynamic
 *     scheduling (new requests join in the middle of generation, without
 *     waiting for a batch to finish); a two-phase scheduler that keeps the
 *     running requests going while admitting new ones; per-request
 *     num_computed_tokens for exact resumption;
 *   - "Technical details / Continuous batching scheduler": phase 1 continues
 *     every RUNNING request, phase 2 admits WAITING requests into the capacity
 *     that is left; request states WAITING -> RUNNING -> FINISHED, with
 *     PREEMPTED;
 *   - "Technical details / Paged attention": a block-wise KV cache without
 *     fragmentation and per-sequence offsets (block tables).
 * The pages give the phases and states but no policy details; the ones taken
 * here are stated with each call below.
 *
 * Model of a request: prompt_len prompt tokens, then up to max_new_tokens
 * sampled tokens.  Its known tokens are the prompt plus the tokens sampled so
 * far; num_computed_tokens of them have their K/V rows in the cache.  A step
 * computes the next query_len known tokens of each scheduled request
 * (positions num_computed .. num_computed + query_len - 1).  When a step
 * brings num_computed up to the number of known tokens, the request samples
 * one token in that step (its last query row is the one the decode attention
 * serves); it finishes when it has sampled max_new_tokens tokens or the
 * caller flags it (e.g. an end-of-sequence token).  The last sampled token is
 * never computed, so a request holds at most prompt_len + max_new_tokens - 1
 * cached tokens.
 *
 * Objects are not thread-safe: one thread drives a scheduler at a time.  No
 * call allocates on the steady-state path except request admission
 * (add_request reserves the request's block-table capacity).
 */
#ifndef PHOTON_SCHEDULER_H
#define PHOTON_SCHEDULER_H

#include <stddef.h>
#include <stdint.h>

#include "photon_paged.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct photon_scheduler photon_scheduler_t;

typedef enum {
  PHOTON_REQ_WAITING = 0,    /* queued, never admitted                       */
  PHOTON_REQ_RUNNING = 1,    /* admitted, holds blocks                       */
  PHOTON_REQ_PREEMPTED = 2,  /* evicted for blocks; waits at the queue front */
  PHOTON_REQ_FINISHED = 3    /* done; its blocks are back in the free list   */
} photon_request_state_t;

/* Capacity of one scheduler.
 *   num_blocks          blocks of the KV pool it manages (ids 0 .. num_blocks-1)
 *   block_size          tokens per block (any value >= 1; the device calls
 *                       take 16)
 *   max_blocks_per_seq  width of a block-table row; a request whose
 *                       prompt_len + max_new_tokens - 1 tokens would need more
 *                       is rejected at add_request
 *   max_seqs            most requests in one step (rows of the outputs)
 *   max_step_tokens     token budget of one step (entries of slot_mapping)
 * All must be > 0, and max_step_tokens >= max_seqs. */
typedef struct {
  int32_t num_blocks;
  int32_t block_size;
  int32_t max_blocks_per_seq;
  int32_t max_seqs;
  int32_t max_step_tokens;
} photon_scheduler_config_t;

/* Result of one photon_scheduler_schedule call. */
typedef struct {
  int32_t num_rows;       /* requests scheduled in this step                  */
  int32_t num_tokens;     /* sum of query_lens: entries of slot_mapping       */
  int32_t num_decode;     /* rows with query_len == 1 (a decode-kernel row)   */
  int32_t num_admitted;   /* rows admitted from the queue in phase 2          */
  int32_t num_preempted;  /* RUNNING requests evicted in this step            */
  int32_t free_blocks;    /* free blocks after the step's allocations         */
} photon_schedule_t;

/* Creates a scheduler with every block free.  *out receives the handle
 * (release it with photon_scheduler_destroy).  PHOTON_ERR_INVALID_ARG for a
 * null pointer or a capacity that breaks the rules above. */
photon_status_t photon_scheduler_create(const photon_scheduler_config_t* config,
                                        photon_scheduler_t** out);

/* Frees the scheduler and everything it owns; NULL is a no-op. */
void photon_scheduler_destroy(photon_scheduler_t* sched);

/* Queues a request at the back of the WAITING queue (first come, first
 * served).  id must be unique among the requests this scheduler has seen;
 * prompt_len >= 1, max_new_tokens >= 1, and the request's
 * prompt_len + max_new_tokens - 1 tokens must fit one block-table row (see
 * max_blocks_per_seq) and the whole pool (so that a request running alone
 * always has the blocks it needs) -- otherwise PHOTON_ERR_INVALID_ARG and
 * nothing is queued. */
photon_status_t photon_scheduler_add_request(photon_scheduler_t* sched, int64_t id,
                                             int32_t prompt_len, int32_t max_new_tokens);

/* Plans one step and writes it into caller-owned HOST arrays:
 *   request_ids   int64 [max_seqs]                 row r's request
 *   query_lens    int32 [max_seqs]                 new tokens of row r
 *   context_lens  int32 [max_seqs]                 cached tokens of row r after
 *                                                  this step's writes (counts
 *                                                  its new tokens)
 *   block_tables  int32 [max_seqs][max_blocks_per_seq]  row r's blocks: the
 *                                                  first ceil(context_lens[r] /
 *                                                  block_size) entries are written,
 *                                                  the rest of the row is left as it
 *                                                  was (no kernel reads past them)
 *   slot_mapping  int64 [max_step_tokens]          slot of each new token, rows
 *                                                  in order, positions ascending
 * Only the first num_rows rows / num_tokens slots are written.  A row with
 * query_len == 1 is exactly what photon_paged_decode_step takes: one new token
 * at position context_len - 1, whose slot is the table's.
 *
 * Policy:
 *   phase 1 -- every RUNNING request, in admission order, gets
 *     min(known - num_computed, budget left) tokens (a decode request needs 1;
 *     a request still in its prompt takes a chunk); a request reached when the
 *     budget is spent is not run in this step (it stays RUNNING).  Blocks
 *     for the new tokens come from the free list; if too few are free, the
 *     most recently admitted RUNNING request is preempted (all of its blocks
 *     go back, num_computed = 0, it goes to the front of the queue as
 *     PREEMPTED and will recompute its known tokens), repeatedly, until the
 *     blocks suffice or the request being served was itself the one preempted;
 *   phase 2 -- skipped if phase 1 preempted; otherwise WAITING/PREEMPTED
 *     requests are admitted from the queue front, in order, while rows,
 *     budget and free blocks allow; admission stops at the first request
 *     whose first chunk does not fit the free blocks (no overtaking).
 * The free list is first in, first out: blocks are taken from its front and
 * returned to its back, in block-table order; at creation it holds
 * 0 .. num_blocks - 1 in order.
 * Every call must be followed by photon_scheduler_update before the next
 * schedule (PHOTON_ERR_INVALID_ARG otherwise).  Any output pointer may be
 * NULL if the caller does not need that array, except `out`. */
photon_status_t photon_scheduler_schedule(photon_scheduler_t* sched, int64_t* request_ids,
                                          int32_t* query_lens, int32_t* context_lens,
                                          int32_t* block_tables, int64_t* slot_mapping,
                                          photon_schedule_t* out);

/* Commits the step planned by the last schedule call: each row's
 * num_computed grows by its query_len; a row that reached its known tokens
 * samples one token; a request that has sampled max_new_tokens tokens, or
 * whose stop[r] is non-zero (stop may be NULL; stop[r] is only read for rows
 * that sampled), becomes FINISHED and its blocks return to the free list.
 * The ids of the requests finished by this call are written, in row order, to
 * finished_ids (host, >= max_seqs entries, may be NULL) and their count to
 * *num_finished (may be NULL).  PHOTON_ERR_INVALID_ARG if no schedule is
 * pending. */
photon_status_t photon_scheduler_update(photon_scheduler_t* sched, const uint8_t* stop,
                                        int64_t* finished_ids, int32_t* num_finished);

/* Counts: requests waiting (WAITING + PREEMPTED), running, finished, and the
 * free blocks.  Any pointer may be NULL. */
photon_status_t photon_scheduler_stats(const photon_scheduler_t* sched, int32_t* num_waiting,
                                       int32_t* num_running, int32_t* num_finished,
                                       int32_t* free_blocks);

/* State of one request: photon_request_state_t, num_computed_tokens, tokens
 * sampled so far and blocks held.  PHOTON_ERR_INVALID_ARG for an unknown id.
 * Any output pointer may be NULL. */
photon_status_t photon_scheduler_request_state(const photon_scheduler_t* sched, int64_t id,
                                               int32_t* state, int32_t* num_computed,
                                               int32_t* num_generated, int32_t* num_blocks);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif /* PHOTON_SCHEDULER_H */
