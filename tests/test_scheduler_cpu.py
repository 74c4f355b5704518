"""The host scheduler (include/photon_scheduler.h, C++ in the library) and its
plain-Python oracle (oracle/scheduler.py), on the CPU.

* both reproduce two hand-derived traces (tests/golden/scheduler_*.json):
  chunked prefill + admission + block reuse, and preemption with recompute;
* on seeded random request traces (the batch-256 serving mix: 80 % short
  prompts, 20 % long ones, arrivals over time, random early stops, pools
  tight enough to preempt) the library's every output array equals the
  oracle's, step by step, bit for bit;
* invariants that neither side computes: no block held twice, held + free =
  pool, slots follow the block tables, budget and row limits, every request
  finishes and every block comes back.
"""
import json
import os

import numpy as np
import pytest

import paged_kv_attention_photon_gb300 as P
from oracle.scheduler import OracleScheduler
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
KEYS = ("request_ids", "query_lens", "context_lens", "block_tables", "slot_mapping",
        "num_admitted", "num_preempted", "free_blocks")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    P.build()


def _as_lists(step: dict, block_size: int) -> dict:
    """Plain lists; block-table rows cut to the blocks each row holds (the
    library leaves the rest of a row as it was)."""
    out = {k: (v.tolist() if isinstance(v, np.ndarray) else
               [list(r) for r in v] if k == "block_tables" else v) for k, v in step.items()}
    out["block_tables"] = [row[:-(-c // block_size)] for row, c in
                           zip(out["block_tables"], out["context_lens"])]
    return out


@pytest.mark.parametrize("name", ["scheduler_chunked_prefill", "scheduler_preemption"])
@pytest.mark.parametrize("impl", ["oracle", "library"])
def test_golden_trace(name, impl):
    g = json.load(open(os.path.join(GOLDEN, name + ".json")))
    cls = OracleScheduler if impl == "oracle" else P.Scheduler
    s = cls(**g["config"])
    for rid, prompt, new in g["requests"]:
        s.add_request(rid, prompt, new)
    for i, want in enumerate(g["steps"]):
        got = _as_lists(s.schedule(), g["config"]["block_size"])
        want = _as_lists(want, g["config"]["block_size"])
        for k in KEYS:
            assert got[k] == want[k], (name, impl, i, k, got[k], want[k])
        fin = s.update()
        assert list(fin) == want["finished"], (name, impl, i)
    st = s.stats()
    assert st["running"] == 0 and st["waiting"] == 0
    assert st["free_blocks"] == g["config"]["num_blocks"]


def _check_invariants(step: dict, sched_cfg: dict, held: dict) -> None:
    bs, mbs, nb = sched_cfg["block_size"], sched_cfg["max_blocks_per_seq"], \
        sched_cfg["num_blocks"]
    q, ctx, tabs, slots = (np.asarray(step[k]) for k in
                           ("query_lens", "context_lens", "block_tables", "slot_mapping"))
    assert step["num_rows"] <= sched_cfg["max_seqs"]
    assert q.sum() == step["num_tokens"] <= sched_cfg["max_step_tokens"]
    assert (q >= 1).all() and len(set(np.asarray(step["request_ids"]).tolist())) == len(q)
    tok = 0
    for r in range(len(q)):
        nblk = -(-int(ctx[r]) // bs)
        row = tabs[r].reshape(-1)
        assert (row[:nblk] >= 0).all() and (row[:nblk] < nb).all()
        for p in range(int(ctx[r]) - int(q[r]), int(ctx[r])):
            assert slots[tok] == row[p // bs] * bs + p % bs
            tok += 1
        held[int(step["request_ids"][r])] = row[:nblk].tolist()
    # blocks of all requests that hold some are pairwise disjoint
    allb = [b for blocks in held.values() for b in blocks]
    assert len(allb) == len(set(allb))
    assert len(allb) + step["free_blocks"] == nb


def _run_trace(seed: int, cfg: dict, n_req: int, steps: int, stop_p: float):
    trace = W.request_trace(seed, n_req, max_prompt=cfg["max_blocks_per_seq"] *
                            cfg["block_size"] // 2, max_new=cfg["max_blocks_per_seq"] *
                            cfg["block_size"] // 2, pool_tokens=cfg["num_blocks"] *
                            cfg["block_size"])
    lib, ora = P.Scheduler(**cfg), OracleScheduler(**cfg)
    rng = np.random.default_rng(seed + 1000)
    held, nxt, preempts = {}, 0, 0
    for t in range(steps):
        while nxt < len(trace) and trace[nxt][0] <= t:
            _, rid, prompt, new = trace[nxt]
            lib.add_request(rid, prompt, new)
            ora.add_request(rid, prompt, new)
            nxt += 1
        a, b = lib.schedule(), ora.schedule()
        la, lb = _as_lists(a, cfg["block_size"]), _as_lists(b, cfg["block_size"])
        for k in KEYS + ("num_rows", "num_tokens", "num_decode"):
            assert la[k] == lb[k], (seed, t, k)
        preempts += a["num_preempted"]
        for rid in list(held):
            if ora.request_state(rid)["blocks"] == 0:
                del held[rid]
        _check_invariants(a, cfg, held)
        stop = (rng.random(a["num_rows"]) < stop_p).astype(np.uint8)
        fa, fb = lib.update(stop), ora.update(stop.tolist())
        assert fa.tolist() == fb
        for rid in fb:
            held.pop(rid, None)
        assert lib.stats() == ora.stats()
        if nxt == len(trace) and lib.stats()["running"] == 0 and lib.stats()["waiting"] == 0:
            break
    st = lib.stats()
    assert st["finished"] == n_req and st["free_blocks"] == cfg["num_blocks"], st
    return preempts


@pytest.mark.parametrize("seed,cfg,n_req,stop_p", [
    (1, dict(num_blocks=64, block_size=4, max_blocks_per_seq=16, max_seqs=8,
             max_step_tokens=32), 40, 0.0),
    (2, dict(num_blocks=24, block_size=4, max_blocks_per_seq=12, max_seqs=6,
             max_step_tokens=16), 40, 0.05),
    (3, dict(num_blocks=400, block_size=16, max_blocks_per_seq=64, max_seqs=32,
             max_step_tokens=512), 120, 0.02),
    (4, dict(num_blocks=40, block_size=16, max_blocks_per_seq=32, max_seqs=16,
             max_step_tokens=64), 60, 0.0),
])
def test_library_equals_oracle_on_random_traces(seed, cfg, n_req, stop_p):
    _run_trace(seed, cfg, n_req, steps=20000, stop_p=stop_p)


@pytest.mark.parametrize("seed,cfg", [
    (2, dict(num_blocks=24, block_size=4, max_blocks_per_seq=12, max_seqs=6,
             max_step_tokens=16)),
    (5, dict(num_blocks=12, block_size=4, max_blocks_per_seq=10, max_seqs=4,
             max_step_tokens=6)),
])
def test_oracle_invariants_on_tight_random_traces(seed, cfg):
    """The oracle alone on traces tight enough to preempt: the invariants above,
    every request finishes and every block comes back, a step that preempts
    admits nobody (the second phase is skipped in such a step), and service is
    first come first served across preemptions: after every step each request
    that holds a running slot arrived before each request still waiting."""
    trace = W.request_trace(seed, 40, max_prompt=cfg["max_blocks_per_seq"] * cfg["block_size"]
                            // 2, max_new=cfg["max_blocks_per_seq"] * cfg["block_size"] // 2,
                            pool_tokens=cfg["num_blocks"] * cfg["block_size"])
    ora = OracleScheduler(**cfg)
    held, nxt, preempting_steps = {}, 0, 0
    for t in range(20000):
        while nxt < len(trace) and trace[nxt][0] <= t:
            ora.add_request(*trace[nxt][1:])
            nxt += 1
        st = ora.schedule()
        if st["num_preempted"]:
            preempting_steps += 1
            assert st["num_admitted"] == 0, (seed, t)
        for rid in list(held):
            if ora.request_state(rid)["blocks"] == 0:
                del held[rid]
        _check_invariants(st, cfg, held)
        order = [tr[1] for tr in trace[:nxt]]                  # arrival order of the ids
        states = [ora.request_state(rid)["state"] for rid in order]
        running = [i for i, x in enumerate(states) if x == 1]
        waiting = [i for i, x in enumerate(states) if x in (0, 2)]
        if running and waiting:
            assert max(running) < min(waiting), (seed, t)
        for rid in ora.update():
            held.pop(rid, None)
        s = ora.stats()
        if nxt == len(trace) and s["running"] == 0 and s["waiting"] == 0:
            break
    assert ora.stats() == dict(waiting=0, running=0, finished=40, free_blocks=cfg["num_blocks"])
    assert preempting_steps > 0


def test_tight_pool_preempts():
    cfg = dict(num_blocks=24, block_size=4, max_blocks_per_seq=12, max_seqs=6,
               max_step_tokens=16)
    assert _run_trace(2, cfg, 40, steps=20000, stop_p=0.0) > 0


def test_decode_rows_feed_the_decode_step():
    """Rows with query_len 1 are the decode step's input: the new token is
    position context_len - 1 and its slot is the table's."""
    s = P.Scheduler(num_blocks=100, block_size=16, max_blocks_per_seq=20, max_seqs=8,
                    max_step_tokens=512)
    for i in range(8):
        s.add_request(i, 17 + 9 * i, 5)
    s.schedule()
    s.update()
    st = s.schedule()
    assert st["num_decode"] == 8 and st["num_tokens"] == 8
    for r in range(8):
        pos = st["context_lens"][r] - 1
        assert st["slot_mapping"][r] == st["block_tables"][r][pos // 16] * 16 + pos % 16


def test_errors():
    with pytest.raises(P.PhotonError):
        P.Scheduler(num_blocks=0, block_size=16, max_blocks_per_seq=4, max_seqs=2,
                    max_step_tokens=8)
    with pytest.raises(P.PhotonError):
        P.Scheduler(num_blocks=8, block_size=16, max_blocks_per_seq=4, max_seqs=8,
                    max_step_tokens=4)                       # budget < rows
    s = P.Scheduler(num_blocks=8, block_size=4, max_blocks_per_seq=4, max_seqs=2,
                    max_step_tokens=8)
    s.add_request(1, 4, 4)
    for bad in [(1, 4, 4), (2, 0, 3), (3, 3, 0), (4, 16, 2), (5, -1, 1)]:
        with pytest.raises(P.PhotonError):
            s.add_request(*bad)                              # dup id, empty, too long
    with pytest.raises(P.PhotonError):
        s.update()                                           # nothing pending
    s.schedule()
    with pytest.raises(P.PhotonError):
        s.schedule()                                         # update first
    s.update()
    with pytest.raises(P.PhotonError):
        s.request_state(99)
    assert s.request_state(1) == dict(state=1, computed=4, generated=1, blocks=1)
