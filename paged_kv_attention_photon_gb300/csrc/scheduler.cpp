// scheduler.cpp -- host KV block manager and two-phase continuous-batching
// scheduler (the photon_scheduler_* calls of include/photon_scheduler.h).
//
// PhotonInfer README, "Technical details / Continuous batching scheduler":
// phase 1 keeps every RUNNING request going, phase 2 admits WAITING requests
// into what is left; states WAITING -> RUNNING -> FINISHED plus PREEMPTED;
// num_computed_tokens per request.  "Technical details / Paged attention":
// fixed-size blocks handed out from a pool, one block table per sequence.
//
// Plain host C++: requests live in a hash map; RUNNING is a vector in
// admission order (victims of preemption come off its back), the queue is a
// deque (preempted requests go back to its front), and the free list is a
// ring buffer of block ids, first in first out.
#include <algorithm>
#include <cstring>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/photon_scheduler.h"

namespace {

struct Request {
  int64_t id = 0;
  int32_t prompt_len = 0;
  int32_t max_new_tokens = 0;
  int32_t generated = 0;      // tokens sampled so far
  int32_t computed = 0;       // num_computed_tokens: known tokens with cached K/V
  int32_t state = PHOTON_REQ_WAITING;
  std::vector<int32_t> blocks;  // block table: blocks[i] holds positions [i*bs, (i+1)*bs)

  int32_t known() const { return prompt_len + generated; }
};

// First-in first-out free list of block ids over a fixed ring.
class FreeList {
 public:
  explicit FreeList(int32_t n) : ring_(n), head_(0), size_(n) {
    for (int32_t i = 0; i < n; ++i) ring_[i] = i;
  }
  int32_t size() const { return size_; }
  int32_t pop() {
    const int32_t b = ring_[head_];
    head_ = head_ + 1 == (int32_t)ring_.size() ? 0 : head_ + 1;
    --size_;
    return b;
  }
  void push(int32_t b) {
    int64_t tail = (int64_t)head_ + size_;
    if (tail >= (int64_t)ring_.size()) tail -= (int64_t)ring_.size();
    ring_[tail] = b;
    ++size_;
  }

 private:
  std::vector<int32_t> ring_;
  int32_t head_, size_;
};

struct Row {
  Request* req;
  int32_t query_len;
};

int32_t blocks_for(int64_t tokens, int32_t bs) { return (int32_t)((tokens + bs - 1) / bs); }

}  // namespace

struct photon_scheduler {
  photon_scheduler_config_t cfg;
  FreeList free_list;
  std::unordered_map<int64_t, Request> requests;
  std::vector<Request*> running;  // admission order
  std::deque<Request*> waiting;   // queue: front is next
  std::vector<Row> rows;          // the pending step
  bool pending = false;
  int32_t finished = 0;

  explicit photon_scheduler(const photon_scheduler_config_t& c)
      : cfg(c), free_list(c.num_blocks) {
    running.reserve(c.max_seqs);
    rows.reserve(c.max_seqs);
  }

  void release_blocks(Request* r) {
    for (int32_t b : r->blocks) free_list.push(b);
    r->blocks.clear();
  }

  // Gives r the blocks for `tokens` cached tokens; the caller checked the count.
  void grow(Request* r, int64_t tokens) {
    const int32_t need = blocks_for(tokens, cfg.block_size) - (int32_t)r->blocks.size();
    for (int32_t i = 0; i < need; ++i) r->blocks.push_back(free_list.pop());
  }

  int32_t blocks_missing(const Request* r, int64_t tokens) const {
    return blocks_for(tokens, cfg.block_size) - (int32_t)r->blocks.size();
  }

  // Evicts the most recently admitted RUNNING request (recompute on return).
  Request* preempt_last() {
    Request* v = running.back();
    running.pop_back();
    release_blocks(v);
    v->computed = 0;
    v->state = PHOTON_REQ_PREEMPTED;
    waiting.push_front(v);
    return v;
  }
};

extern "C" {

photon_status_t photon_scheduler_create(const photon_scheduler_config_t* c,
                                        photon_scheduler_t** out) {
  if (!c || !out) return PHOTON_ERR_INVALID_ARG;
  if (c->num_blocks <= 0 || c->block_size <= 0 || c->max_blocks_per_seq <= 0 ||
      c->max_seqs <= 0 || c->max_step_tokens <= 0 || c->max_step_tokens < c->max_seqs)
    return PHOTON_ERR_INVALID_ARG;
  if ((int64_t)c->max_blocks_per_seq * c->block_size > INT32_MAX) return PHOTON_ERR_INVALID_ARG;
  photon_scheduler_t* s = new (std::nothrow) photon_scheduler(*c);
  if (!s) return PHOTON_ERR_INVALID_ARG;
  *out = s;
  return PHOTON_OK;
}

void photon_scheduler_destroy(photon_scheduler_t* s) { delete s; }

photon_status_t photon_scheduler_add_request(photon_scheduler_t* s, int64_t id,
                                             int32_t prompt_len, int32_t max_new_tokens) {
  if (!s || prompt_len < 1 || max_new_tokens < 1) return PHOTON_ERR_INVALID_ARG;
  const int64_t most = (int64_t)prompt_len + max_new_tokens - 1;
  const int64_t need = (most + s->cfg.block_size - 1) / s->cfg.block_size;
  if (need > s->cfg.max_blocks_per_seq || need > s->cfg.num_blocks) return PHOTON_ERR_INVALID_ARG;
  if (s->requests.count(id)) return PHOTON_ERR_INVALID_ARG;
  Request& r = s->requests[id];
  r.id = id;
  r.prompt_len = prompt_len;
  r.max_new_tokens = max_new_tokens;
  r.blocks.reserve((size_t)need);
  s->waiting.push_back(&r);
  return PHOTON_OK;
}

photon_status_t photon_scheduler_schedule(photon_scheduler_t* s, int64_t* request_ids,
                                          int32_t* query_lens, int32_t* context_lens,
                                          int32_t* block_tables, int64_t* slot_mapping,
                                          photon_schedule_t* out) {
  if (!s || !out || s->pending) return PHOTON_ERR_INVALID_ARG;
  const int32_t bs = s->cfg.block_size;
  int32_t budget = s->cfg.max_step_tokens;
  int32_t preempted = 0, admitted = 0;
  s->rows.clear();

  // ---- phase 1: continue the RUNNING requests, oldest first
  for (size_t i = 0; i < s->running.size();) {
    Request* r = s->running[i];
    const int32_t n = std::min(r->known() - r->computed, budget);
    if (n <= 0) {
      ++i;
      continue;
    }
    bool self_evicted = false;
    while (s->free_list.size() < s->blocks_missing(r, (int64_t)r->computed + n)) {
      Request* v = s->preempt_last();
      ++preempted;
      if (v == r) {
        self_evicted = true;
        break;
      }
    }
    if (self_evicted) break;  // r was the last one: nothing after it remains
    s->grow(r, (int64_t)r->computed + n);
    s->rows.push_back({r, n});
    budget -= n;
    ++i;
  }

  // ---- phase 2: admit from the queue front while rows, budget and blocks allow
  if (preempted == 0) {
    while (!s->waiting.empty() && budget > 0 &&
           (int32_t)s->running.size() < s->cfg.max_seqs) {
      Request* r = s->waiting.front();
      const int32_t n = std::min(r->known() - r->computed, budget);
      if (s->free_list.size() < s->blocks_missing(r, (int64_t)r->computed + n)) break;
      s->waiting.pop_front();
      r->state = PHOTON_REQ_RUNNING;
      s->running.push_back(r);
      s->grow(r, (int64_t)r->computed + n);
      s->rows.push_back({r, n});
      budget -= n;
      ++admitted;
    }
  }

  // ---- outputs
  const int32_t mbs = s->cfg.max_blocks_per_seq;
  int32_t tok = 0, decode = 0;
  for (size_t i = 0; i < s->rows.size(); ++i) {
    const Request* r = s->rows[i].req;
    const int32_t n = s->rows[i].query_len;
    const int32_t ctx = r->computed + n;
    if (request_ids) request_ids[i] = r->id;
    if (query_lens) query_lens[i] = n;
    if (context_lens) context_lens[i] = ctx;
    if (block_tables) {
      // only the blocks the row holds: entries past them are never read
      int32_t* row = block_tables + i * (size_t)mbs;
      std::memcpy(row, r->blocks.data(), sizeof(int32_t) * r->blocks.size());
    }
    if (slot_mapping) {
      for (int32_t p = r->computed; p < ctx; ++p)
        slot_mapping[tok + (p - r->computed)] = (int64_t)r->blocks[p / bs] * bs + p % bs;
    }
    tok += n;
    decode += n == 1;
  }
  out->num_rows = (int32_t)s->rows.size();
  out->num_tokens = tok;
  out->num_decode = decode;
  out->num_admitted = admitted;
  out->num_preempted = preempted;
  out->free_blocks = s->free_list.size();
  s->pending = true;
  return PHOTON_OK;
}

photon_status_t photon_scheduler_update(photon_scheduler_t* s, const uint8_t* stop,
                                        int64_t* finished_ids, int32_t* num_finished) {
  if (!s || !s->pending) return PHOTON_ERR_INVALID_ARG;
  int32_t nf = 0;
  bool any_finished = false;
  for (size_t i = 0; i < s->rows.size(); ++i) {
    Request* r = s->rows[i].req;
    r->computed += s->rows[i].query_len;
    if (r->computed < r->known()) continue;  // a prompt chunk that samples nothing
    r->generated += 1;
    if (r->generated >= r->max_new_tokens || (stop && stop[i])) {
      r->state = PHOTON_REQ_FINISHED;
      s->release_blocks(r);
      if (finished_ids) finished_ids[nf] = r->id;
      ++nf;
      any_finished = true;
    }
  }
  if (any_finished) {
    s->running.erase(std::remove_if(s->running.begin(), s->running.end(),
                                     [](const Request* r) {
                                       return r->state == PHOTON_REQ_FINISHED;
                                     }),
                     s->running.end());
  }
  s->finished += nf;
  if (num_finished) *num_finished = nf;
  s->rows.clear();
  s->pending = false;
  return PHOTON_OK;
}

photon_status_t photon_scheduler_stats(const photon_scheduler_t* s, int32_t* num_waiting,
                                       int32_t* num_running, int32_t* num_finished,
                                       int32_t* free_blocks) {
  if (!s) return PHOTON_ERR_INVALID_ARG;
  if (num_waiting) *num_waiting = (int32_t)s->waiting.size();
  if (num_running) *num_running = (int32_t)s->running.size();
  if (num_finished) *num_finished = s->finished;
  if (free_blocks) *free_blocks = s->free_list.size();
  return PHOTON_OK;
}

photon_status_t photon_scheduler_request_state(const photon_scheduler_t* s, int64_t id,
                                               int32_t* state, int32_t* num_computed,
                                               int32_t* num_generated, int32_t* num_blocks) {
  if (!s) return PHOTON_ERR_INVALID_ARG;
  auto it = s->requests.find(id);
  if (it == s->requests.end()) return PHOTON_ERR_INVALID_ARG;
  const Request& r = it->second;
  if (state) *state = r.state;
  if (num_computed) *num_computed = r.computed;
  if (num_generated) *num_generated = r.generated;
  if (num_blocks) *num_blocks = (int32_t)r.blocks.size();
  return PHOTON_OK;
}

}  // extern "C"
