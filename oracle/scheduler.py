"""Plain-Python oracle of the two-phase continuous-batching scheduler and its
KV block manager.  TEST INFRASTRUCTURE ONLY: tests/, smoke() and bench.py's
CPU legs may use it; the library never does.

What it follows (PhotonInfer README, "Technical details / Continuous batching
scheduler" and "Key features / vLLM-style continuous batching"):
  * phase 1 continues every RUNNING request, phase 2 admits WAITING requests
    into the capacity left;
  * states WAITING -> RUNNING -> FINISHED, and PREEMPTED;
  * num_computed_tokens per request, so that a request resumes exactly where
    its cache stops;
and ("Technical details / Paged attention") fixed-size blocks from a pool, a
block table per sequence.

The pages state no policy beyond the two phases.  The readings taken (the
same ones the library documents for photon_scheduler_schedule):
  * a step has a token budget and a row limit; RUNNING requests are served
    oldest first, each with min(unfinished known tokens, budget left);
  * short of blocks, the newest RUNNING request is preempted (recompute: its
    blocks are freed, num_computed returns to 0, it waits at the queue front);
  * no admission in a step that preempted; admission is first come first
    served and stops at the first request that does not fit;
  * the free list is first in, first out, filled 0 .. num_blocks-1 at start,
    freed blocks appended in block-table order;
  * a step that completes a request's known tokens samples one token; the
    request finishes after max_new_tokens samples or when the caller stops it.

Written for clarity: lists and linear scans, nothing cached.
"""
from __future__ import annotations

from typing import Dict, List, Optional

WAITING, RUNNING, PREEMPTED, FINISHED = 0, 1, 2, 3


class OracleRequest:
    def __init__(self, rid: int, prompt_len: int, max_new_tokens: int):
        self.rid = rid
        self.prompt_len = prompt_len
        self.max_new_tokens = max_new_tokens
        self.generated = 0
        self.computed = 0
        self.state = WAITING
        self.table: List[int] = []

    def known(self) -> int:
        return self.prompt_len + self.generated


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


class OracleScheduler:
    def __init__(self, *, num_blocks: int, block_size: int, max_blocks_per_seq: int,
                 max_seqs: int, max_step_tokens: int):
        if min(num_blocks, block_size, max_blocks_per_seq, max_seqs, max_step_tokens) <= 0 \
                or max_step_tokens < max_seqs:
            raise ValueError("bad capacity")
        self.num_blocks = num_blocks
        self.bs = block_size
        self.mbs = max_blocks_per_seq
        self.max_seqs = max_seqs
        self.max_step_tokens = max_step_tokens
        self.free: List[int] = list(range(num_blocks))   # front = next block handed out
        self.requests: Dict[int, OracleRequest] = {}
        self.running: List[OracleRequest] = []          # admission order
        self.queue: List[OracleRequest] = []            # front = next admitted
        self.pending: Optional[List[tuple]] = None
        self.finished = 0

    # ---------------------------------------------------------------- requests
    def add_request(self, rid: int, prompt_len: int, max_new_tokens: int) -> None:
        if prompt_len < 1 or max_new_tokens < 1 or rid in self.requests:
            raise ValueError("bad request")
        blocks = _ceil_div(prompt_len + max_new_tokens - 1, self.bs)
        if blocks > self.mbs or blocks > self.num_blocks:
            raise ValueError("request does not fit")
        r = OracleRequest(rid, prompt_len, max_new_tokens)
        self.requests[rid] = r
        self.queue.append(r)

    # ---------------------------------------------------------------- blocks
    def _missing(self, r: OracleRequest, tokens: int) -> int:
        return _ceil_div(tokens, self.bs) - len(r.table)

    def _take(self, r: OracleRequest, tokens: int) -> None:
        for _ in range(self._missing(r, tokens)):
            r.table.append(self.free.pop(0))

    def _give_back(self, r: OracleRequest) -> None:
        self.free.extend(r.table)
        r.table = []

    # ---------------------------------------------------------------- a step
    def schedule(self) -> dict:
        if self.pending is not None:
            raise RuntimeError("update() the previous step first")
        budget = self.max_step_tokens
        rows = []              # (request, query_len, computed before the step)
        preempted = 0

        # Phase 1: every RUNNING request, oldest first.
        served = []
        i = 0
        while i < len(self.running):
            r = self.running[i]
            n = min(r.known() - r.computed, budget)
            if n == 0:
                i += 1
                continue
            gone = False
            while len(self.free) < self._missing(r, r.computed + n):
                victim = self.running.pop()          # newest admitted
                self._give_back(victim)
                victim.computed = 0
                victim.state = PREEMPTED
                self.queue.insert(0, victim)
                preempted += 1
                if victim is r:
                    gone = True
                    break
            if gone:
                break
            self._take(r, r.computed + n)
            rows.append((r, n, r.computed))
            served.append(r)
            budget -= n
            i += 1

        # Phase 2: admit from the queue front into what is left.
        admitted = 0
        if preempted == 0:
            while self.queue and budget > 0 and len(self.running) < self.max_seqs:
                r = self.queue[0]
                n = min(r.known() - r.computed, budget)
                if len(self.free) < self._missing(r, r.computed + n):
                    break
                self.queue.pop(0)
                r.state = RUNNING
                self.running.append(r)
                self._take(r, r.computed + n)
                rows.append((r, n, r.computed))
                budget -= n
                admitted += 1

        # Outputs: one row per scheduled request, the slot of each new token.
        ids, qlens, ctxs, tables, slots = [], [], [], [], []
        for r, n, c0 in rows:
            ids.append(r.rid)
            qlens.append(n)
            ctxs.append(c0 + n)
            tables.append(list(r.table) + [-1] * (self.mbs - len(r.table)))
            for pos in range(c0, c0 + n):
                slots.append(r.table[pos // self.bs] * self.bs + pos % self.bs)
        self.pending = [(r, n) for r, n, _ in rows]
        return {"request_ids": ids, "query_lens": qlens, "context_lens": ctxs,
                "block_tables": tables, "slot_mapping": slots, "num_rows": len(rows),
                "num_tokens": sum(qlens), "num_decode": sum(1 for q in qlens if q == 1),
                "num_admitted": admitted, "num_preempted": preempted,
                "free_blocks": len(self.free)}

    def update(self, stop: Optional[List[int]] = None) -> List[int]:
        if self.pending is None:
            raise RuntimeError("no step pending")
        done = []
        for row, (r, n) in enumerate(self.pending):
            r.computed += n
            if r.computed < r.known():
                continue
            r.generated += 1
            if r.generated >= r.max_new_tokens or (stop is not None and stop[row]):
                r.state = FINISHED
                self._give_back(r)
                done.append(r.rid)
        self.running = [r for r in self.running if r.state != FINISHED]
        self.finished += len(done)
        self.pending = None
        return done

    def stats(self) -> dict:
        return dict(waiting=len(self.queue), running=len(self.running),
                    finished=self.finished, free_blocks=len(self.free))

    def request_state(self, rid: int) -> dict:
        r = self.requests[rid]
        return dict(state=r.state, computed=r.computed, generated=r.generated,
                    blocks=len(r.table))
