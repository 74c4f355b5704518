"""The host scheduler driving the device calls, step after step, against the
oracle on a host mirror of the pool.

A seeded request trace with the batch-256 serving mix (32 q / 8 KV heads,
d = 64, fp16, block 16) runs through photon_scheduler_*: every step's prompt
chunks are written with photon_cache_write at the scheduler's slots, and its
decode rows (query_len 1) run photon_paged_decode_step with the scheduler's
block tables, context lengths and slots.  The same writes go to a host copy
of the pool through the oracle's cache write, and each step's decode output is
compared with the oracle's decode on that copy.  Blocks freed by finished or
preempted requests are handed out again while still holding their old rows,
so a read past a context length would show.  At the end the device pool
equals the host mirror byte for byte.

The second test runs each whole step -- prompt chunks and decode rows alike --
as one cache write of every new row and one multi-query causal attention call
over all scheduled rows, each step against the oracle's multi-query.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_photon_gb300 as P
import workloads as W
from gpu_util import assert_close, dev, to_float64

pytestmark = pytest.mark.gpu

HQ, HKV, D, BS = 32, 8, 64, 16
DT = W.DTYPE_F16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    P.build()
    torch.cuda.init()


@pytest.mark.parametrize("seed,num_blocks,max_seqs,budget,n_req", [
    (5, 2048, 32, 1024, 48),     # roomy pool: admission, chunked prompts, reuse
    (6, 160, 16, 256, 40),       # tight pool: preemption and recompute
])
def test_scheduler_drives_decode_steps(seed, num_blocks, max_seqs, budget, n_req):
    max_prompt, max_new = 512, 48
    mbs = (max_prompt + max_new + BS - 1) // BS
    trace = W.request_trace(seed, n_req, max_prompt=max_prompt, max_new=max_new,
                            pool_tokens=num_blocks * BS, arrivals_per_step=2.0)
    rows = {rid: W.request_rows(seed, rid, prompt + new, HKV, D, DT)
            for _, rid, prompt, new in trace}
    sched = P.Scheduler(num_blocks=num_blocks, block_size=BS, max_blocks_per_seq=mbs,
                        max_seqs=max_seqs, max_step_tokens=budget)

    host_k = np.full((num_blocks, HKV, BS, D), np.nan, np.float16)
    host_v = np.full((num_blocks, HKV, BS, D), np.nan, np.float16)
    kc, vc = dev(host_k), dev(host_v)
    ws_cap = 0
    ws = None
    nxt, steps, decoded, preempted = 0, 0, 0, 0
    while steps < 4000:
        while nxt < len(trace) and trace[nxt][0] <= steps:
            _, rid, prompt, new = trace[nxt]
            sched.add_request(rid, prompt, new)
            nxt += 1
        st = sched.schedule()
        preempted += st["num_preempted"]
        q_lens, ctx, tabs, slots = (st["query_lens"], st["context_lens"], st["block_tables"],
                                    st["slot_mapping"])
        # ---- prompt chunks: K/V rows of their positions, written at their slots
        tok = 0
        ck, cv, cs = [], [], []
        dec = []
        for r in range(st["num_rows"]):
            rid, n, c = int(st["request_ids"][r]), int(q_lens[r]), int(ctx[r])
            if n == 1:
                dec.append(r)
            else:
                k_all, v_all = rows[rid]
                ck.append(k_all[c - n:c])
                cv.append(v_all[c - n:c])
                cs.append(slots[tok:tok + n])
            tok += n
        if ck:
            kk, vv, ss = np.concatenate(ck), np.concatenate(cv), np.concatenate(cs)
            shape = P.PagedShape.make(num_seqs=1, num_q_heads=HQ, num_kv_heads=HKV,
                                      head_dim=D, num_blocks=num_blocks,
                                      max_blocks_per_seq=mbs, dtype=DT)
            P.photon_cache_write(dev(kk), dev(vv), dev(ss), ss.shape[0], kc, vc, shape)
            oracle.cache_write(kk, vv, ss, host_k, host_v, block_size=BS, dtype=DT)
        # ---- decode rows: one fused step over all of them
        if dec:
            idx = np.asarray(dec)
            B = idx.shape[0]
            tok_of_row = np.concatenate([[0], np.cumsum(q_lens)[:-1]])
            d_ctx = ctx[idx].astype(np.int32)
            d_tab = np.ascontiguousarray(tabs[idx]).astype(np.int32)
            d_slot = slots[tok_of_row[idx]].astype(np.int64)
            ids = st["request_ids"][idx]
            q = np.stack([W.request_queries(seed, int(rid), int(c) - 1, HQ, D, DT)
                          for rid, c in zip(ids, d_ctx)])
            k_new = np.stack([rows[int(rid)][0][int(c) - 1] for rid, c in zip(ids, d_ctx)])
            v_new = np.stack([rows[int(rid)][1][int(c) - 1] for rid, c in zip(ids, d_ctx)])
            shape = P.PagedShape.make(num_seqs=B, num_q_heads=HQ, num_kv_heads=HKV, head_dim=D,
                                      num_blocks=num_blocks, max_blocks_per_seq=mbs, dtype=DT)
            need = P.photon_paged_decode_workspace_size(shape)
            if need > ws_cap:
                ws_cap = need
                ws = torch.empty(need, dtype=torch.uint8, device="cuda")
            out = torch.empty((B, HQ, D), dtype=torch.float16, device="cuda")
            P.photon_paged_decode_step(dev(k_new), dev(v_new), dev(d_slot), dev(q), kc, vc,
                                       dev(d_tab), dev(d_ctx), 0.125, out, ws, need, shape)
            oracle.cache_write(k_new, v_new, d_slot, host_k, host_v, block_size=BS, dtype=DT)
            want = oracle.paged_decode(q, host_k, host_v, d_tab, d_ctx, 0.125, dtype=DT,
                                       num_threads=8)
            torch.cuda.synchronize()
            s_, bits = P.photon_get_last_device_error()
            assert s_ == 0 and bits == 0, (steps, bits)
            assert_close(to_float64(out, DT), want, DT, f"step {steps}")
            decoded += B
        sched.update()
        steps += 1
        s = sched.stats()
        if nxt == len(trace) and s["running"] == 0 and s["waiting"] == 0:
            break
    torch.cuda.synchronize()
    assert sched.stats()["finished"] == n_req
    assert decoded > 0
    assert kc.cpu().numpy().tobytes() == host_k.tobytes()
    assert vc.cpu().numpy().tobytes() == host_v.tobytes()
    if num_blocks < 1000:
        assert preempted > 0


@pytest.mark.parametrize("seed,num_blocks,max_seqs,budget,n_req,max_new", [
    (7, 600, 16, 256, 24, 24),  # roomy: prompts chunked across steps
    (8, 32, 8, 128, 16, 48),    # tight: growing decodes force preemption and recompute
])
def test_scheduler_drives_multi_query_steps(seed, num_blocks, max_seqs, budget, n_req, max_new):
    """A whole serving step in one attention call: every scheduled row (prompt
    chunks and decode rows alike) writes its new K/V rows with one
    photon_cache_write and attends causally with one photon_paged_multi_query
    (query_start = the rows' cumulative query lengths); each step's output
    against the oracle's multi-query on the host mirror of the pool."""
    max_prompt = 200
    mbs = (max_prompt + max_new + BS - 1) // BS
    trace = W.request_trace(seed, n_req, max_prompt=max_prompt, max_new=max_new,
                            pool_tokens=num_blocks * BS, arrivals_per_step=2.0)
    rows = {rid: W.request_rows(seed, rid, prompt + new, HKV, D, DT)
            for _, rid, prompt, new in trace}
    sched = P.Scheduler(num_blocks=num_blocks, block_size=BS, max_blocks_per_seq=mbs,
                        max_seqs=max_seqs, max_step_tokens=budget)
    host_k = np.full((num_blocks, HKV, BS, D), np.nan, np.float16)
    host_v = np.full((num_blocks, HKV, BS, D), np.nan, np.float16)
    kc, vc = dev(host_k), dev(host_v)
    nxt, steps, rows_done, preempted = 0, 0, 0, 0
    while steps < 2000:
        while nxt < len(trace) and trace[nxt][0] <= steps:
            _, rid, prompt, new = trace[nxt]
            sched.add_request(rid, prompt, new)
            nxt += 1
        st = sched.schedule()
        preempted += st["num_preempted"]
        B, T = st["num_rows"], st["num_tokens"]
        if B:
            q_lens = st["query_lens"].astype(np.int32)
            ctx = st["context_lens"].astype(np.int32)
            tabs = np.ascontiguousarray(st["block_tables"]).astype(np.int32)
            slots = st["slot_mapping"].astype(np.int64).copy()
            ids = st["request_ids"].copy()
            kk, vv, qq = [], [], []
            for r in range(B):
                k_all, v_all = rows[int(ids[r])]
                c, n = int(ctx[r]), int(q_lens[r])
                kk.append(k_all[c - n:c])
                vv.append(v_all[c - n:c])
                qq.extend(W.request_queries(seed, int(ids[r]), pos, HQ, D, DT)
                          for pos in range(c - n, c))
            kk, vv, q = np.concatenate(kk), np.concatenate(vv), np.stack(qq)
            qs = np.zeros(B + 1, np.int32)
            qs[1:] = np.cumsum(q_lens)
            shape = P.PagedShape.make(num_seqs=B, num_q_heads=HQ, num_kv_heads=HKV, head_dim=D,
                                      num_blocks=num_blocks, max_blocks_per_seq=mbs, dtype=DT)
            P.photon_cache_write(dev(kk), dev(vv), dev(slots), T, kc, vc, shape)
            oracle.cache_write(kk, vv, slots, host_k, host_v, block_size=BS, dtype=DT)
            maxq = int(q_lens.max())
            nws = P.photon_paged_multi_query_workspace_size(shape, T, maxq)
            ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")
            out = torch.empty((T, HQ, D), dtype=torch.float16, device="cuda")
            P.photon_paged_multi_query(dev(q), kc, vc, dev(tabs), dev(ctx), dev(qs), T, maxq,
                                       0.125, out, ws, nws, shape)
            want = oracle.multi_query(q, host_k, host_v, tabs, ctx, qs, 0.125, dtype=DT,
                                      num_threads=8)
            torch.cuda.synchronize()
            s_, bits = P.photon_get_last_device_error()
            assert s_ == 0 and bits == 0, (steps, bits)
            assert_close(to_float64(out, DT), want, DT, f"step {steps}")
            rows_done += B
        sched.update()
        steps += 1
        s = sched.stats()
        if nxt == len(trace) and s["running"] == 0 and s["waiting"] == 0:
            break
    torch.cuda.synchronize()
    assert sched.stats()["finished"] == n_req and rows_done > 0
    assert kc.cpu().numpy().tobytes() == host_k.tobytes()
    if num_blocks < 100:
        assert preempted > 0
