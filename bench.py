#!/usr/bin/env python
"""Benchmark of the paged decode-attention step on GB300.

One step = the whole hot path over one batch: the batched cache write of the
new K/V rows, then split-KV paged decode attention with its partition merge,
through the library's C ABI (photon_paged_decode_step: the attention kernel
takes each sequence's new row from the step's inputs and stores it into its
cache slot, so no separate scatter pass runs).  Default workload: Qwen3-style
long context -- 64 sequences, 16 q / 8 KV heads, head_dim 128, 16-token
blocks, fp16, context lengths log-uniform in [128, 8192], a 40 000-block
pool in random order.

Prints one JSON line.  value = algorithmic HBM bytes of the step (every K/V
row inside the contexts, q, out, block-table entries used, context lengths,
plus the cache write's rows and slots) / device time per step, in GB/s.
L2 is flushed before every timed step, outside the timed events: a 512 MB
write, then a 256 MB read of another buffer so that the flush's dirty lines
are written back before the step starts (otherwise their write-back would land
inside the timed kernels).

--impl reference times the fp64 CPU oracle instead (the only reference this
method has), on a bounded sample of the same workload, on the host cores.
Multi-GPU (torchrun): every rank runs its own batch (sequences shard with no
exchange), value = all ranks' bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged-decode KV GB/s and fraction of GB300 HBM peak; decode tokens/s per layer"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 512 << 20
ROPE_BASE = 1.0e6          # rotary base of the Qwen family (the side measurement only)
L2_CLEAN_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen_b64", choices=sorted(W.NAMED))
    ap.add_argument("--partition", type=int, default=0, help="tokens per partition; 0 = default")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rope", action="store_true",
                    help="skip the side measurement of the step with RoPE fused in")
    ap.add_argument("--no-mq", action="store_true",
                    help="skip the side measurements of multi-query attention")
    ap.add_argument("--mq-case", default="", choices=["", "verify_b64x4", "prefill_b16x1024"],
                    help="profiling aid: run only this multi-query case (default kernel "
                         "choice, --steps calls) and print its timing")
    ap.add_argument("--no-fp8", action="store_true", help="skip the e4m3-cache decode line")
    ap.add_argument("--fp8-case", default="", choices=["", "qwen_b64", "qwen_b64_pool10k"],
                    help="profiling aid: run only the e4m3-cache decode on this workload")
    ap.add_argument("--no-bf16", action="store_true", help="skip the bf16-storage step line")
    ap.add_argument("--no-read-ceiling", action="store_true",
                    help="skip the read-only ceiling of the decode's copies")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the side measurements of the other decode configurations")
    ap.add_argument("--decode-consumer", type=int, default=0, choices=[0, 1, 2],
                    help="decode attention consumer: 0 by group size, 1 CUDA cores, 2 tensor cores")
    ap.add_argument("--json-out", default="")
    return ap.parse_args()


# ----------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def make_workload(name: str, rank: int) -> W.Workload:
    if rank == 0:
        return W.NAMED[name]()
    # weak scaling: every rank draws its own batch of the same recipe
    seeds = {"qwen_b64": 2, "mix_b256": 3, "llama_b16": 1, "tiny": 0}
    if name == "qwen_b64":
        return W.qwen_b64(seed=seeds[name] + 1000 * rank)
    if name == "mix_b256":
        return W.mix_b256(seed=seeds[name] + 1000 * rank)
    if name == "llama_b16":
        return W.llama_b16(seed=seeds[name] + 1000 * rank)
    return W.NAMED[name]()


def reduce_over_ranks(pg, ms, attn_ms, step_bytes, seqs, tokens):
    """Whole-job view of one rank's numbers: the slowest rank's step and decode
    times, and the bytes, sequences and tokens of all ranks summed.  `pg` is
    torch.distributed (already initialised) or None for a single process."""
    if pg is None:
        return ms, attn_ms, float(step_bytes), float(seqs), float(tokens)
    import torch
    t = torch.tensor([ms, attn_ms], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    tb = torch.tensor([float(step_bytes), float(seqs), float(tokens)], dtype=torch.float64)
    pg.all_reduce(tb)
    return float(t[0]), float(t[1]), float(tb[0]), float(tb[1]), float(tb[2])


def measured_bf16_tflops():
    """Dense bf16 tensor throughput (burst) from MEASURED_PEAKS.json, else the
    fallback figure; fp16 runs at the same rate."""
    try:
        v = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))).get("bf16_tflops")
        if isinstance(v, (int, float)):
            return float(v), "measured"
    except Exception:
        pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def multi_query_side(P, torch, stream, flush_l2, K, hbm_peak, only: str = "",
                     with_tc: bool = True):
    """Speculative-verify and chunked-prefill timings of photon_paged_multi_query."""
    rng = np.random.Generator(np.random.PCG64(2))
    ctx = W.qwen_context_lens(rng, 64)
    cases = {
        "verify_b64x4": (W.multi_query(311, query_lens=[4] * 64, prefix_lens=(ctx - 4).tolist(),
                                       num_q_heads=16, num_kv_heads=8, head_dim=128,
                                       dtype=W.DTYPE_F16), "hbm"),
        "prefill_b16x1024": (W.multi_query(320, query_lens=[1024] * 16,
                                           prefix_lens=[0] * 8 + [4096] * 8, num_q_heads=16,
                                           num_kv_heads=8, head_dim=128, dtype=W.DTYPE_F16),
                             "tensor"),
    }
    tpeak, tkind = measured_bf16_tflops()
    res = {}

    def dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    for name, (mq, bound) in cases.items():
        if only and name != only:
            continue
        p = mq.pool
        shape = P.PagedShape.make(**p.shape_dict())
        q, kc, vc = dev(mq.q), dev(p.k_cache), dev(p.v_cache)
        bt, cl, qs = dev(p.block_tables), dev(p.context_lens), dev(mq.query_start)
        out = torch.empty_like(q)
        nws = P.photon_paged_multi_query_workspace_size(shape, mq.num_tokens, mq.max_query_len)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")

        def call():
            P.photon_paged_multi_query(q, kc, vc, bt, cl, qs, mq.num_tokens, mq.max_query_len,
                                       p.scale, out, ws, nws, shape, stream)

        def timed(which):
            P.photon_debug_set_multi_query_kernel(which)
            for _ in range(3):
                flush_l2()
                call()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(K)]
            for i in range(K):
                flush_l2()
                ev[i][0].record(stream)
                call()
                ev[i][1].record(stream)
            torch.cuda.synchronize()
            P.photon_debug_set_multi_query_kernel(0)
            st, bits = P.photon_get_last_device_error(stream)
            if st != 0:
                raise RuntimeError(f"device error word {bits} in multi-query {name}")
            return sum(a.elapsed_time(b) for a, b in ev) / K

        ms = timed(0)
        g = p.num_q_heads // p.num_kv_heads
        default = ("decode kernel, few-token mode" if mq.max_query_len * g <= 8 else
                   "tcgen05" if nws == 0 else "warp-level mma.sync with key split")
        per_kernel = {}
        if with_tc:
            for which, key in ((1, "warp_level_mma_sync"), (2, "tcgen05"),
                               (3, "decode_few_token")):
                if which == 3 and mq.max_query_len * g > 8:
                    continue
                t = timed(which)
                per_kernel[key] = {"ms_per_call": round(t, 5),
                                   "TFLOPs": round(mq.flops() / (t / 1e3) / 1e12, 2),
                                   "kv_GBps": round(mq.kv_bytes() / (t / 1e3) / 1e9, 1)}
        gbs = mq.kv_bytes() / (ms / 1e3) / 1e9
        tfs = mq.flops() / (ms / 1e3) / 1e12
        achieved, peak, unit = (gbs, hbm_peak, "GB/s") if bound == "hbm" else \
            (tfs, tpeak, "TFLOP/s")
        res[name] = {"ms_per_call": round(ms, 5), "tokens": mq.num_tokens,
                     "kv_GBps": round(gbs, 1), "TFLOPs": round(tfs, 2),
                     "roofline": {"bound": bound, "achieved": round(achieved, 2),
                                  "peak": peak, "unit": unit,
                                  "frac": round(achieved / peak, 4),
                                  "peak_source": "measured" if bound == "hbm" else tkind},
                     "algorithmic_bytes": mq.kv_bytes(), "flops": mq.flops(),
                     "workspace_bytes": int(nws), "kernel": default,
                     "per_kernel": per_kernel}
        del q, kc, vc, bt, cl, qs, out, ws
    return res


def fp8_side(P, torch, stream, flush_l2, K, peak, workload: str = "qwen_b64"):
    """The same batch-64 long-context decode over an e4m3 K/V cache
    (photon_paged_decode_fp8): the codes of the synthetic fp8 pools, fp16 q
    and out.  Algorithmic bytes as the fp16 decode's with one byte per cached
    element."""
    wl = make_workload(workload, 0)
    k8, v8 = W.fp8_cache(wl, 2)
    shape = P.PagedShape.make(**wl.shape_dict())

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    q, kc, vc = dev(wl.q), dev(k8), dev(v8)
    bt, cl = dev(wl.block_tables), dev(wl.context_lens)
    out = torch.empty_like(q)
    nws = P.photon_paged_decode_fp8_workspace_size(shape)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")

    def call():
        P.photon_paged_decode_fp8(q, kc, vc, bt, cl, wl.scale, W.FP8_K_SCALE, W.FP8_V_SCALE,
                                  out, ws, nws, shape, stream)

    for _ in range(3):
        flush_l2()
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for i in range(K):
        flush_l2()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    st, bits = P.photon_get_last_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error word {bits} in the fp8 decode")
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    ctx = wl.context_lens.astype(np.int64)
    nbytes = (int(ctx.sum()) * wl.num_kv_heads * wl.head_dim * 2
              + 2 * wl.num_seqs * wl.num_q_heads * wl.head_dim * 2
              + 4 * int(((ctx + 15) // 16).sum()) + 4 * wl.num_seqs)
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"workload": f"{workload} with an e4m3 K/V cache (k_scale 0.5, v_scale 0.25)",
            "ms_per_call": round(ms, 5), "algorithmic_bytes": int(nbytes),
            "GBps": round(gbs, 1), "hbm_fraction": round(gbs / peak, 4),
            "tokens_attended_per_s": round(wl.tokens_attended() / (ms / 1e3), 1),
            "decode_tokens_per_s_per_layer": round(wl.num_seqs / (ms / 1e3), 1)}


def bf16_side(P, torch, stream, flush_l2, K, peak):
    """The headline step (cache write + decode, qwen_b64 shapes and contexts)
    with bf16 storage: the same sequences, K/V values drawn for bf16."""
    wl = W.qwen_b64(dtype=W.DTYPE_BF16)
    shape = P.PagedShape.make(**wl.shape_dict())

    def dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    q, kc, vc = dev(wl.q), dev(wl.k_cache), dev(wl.v_cache)
    bt, cl = dev(wl.block_tables), dev(wl.context_lens)
    kn, vn, sm = dev(wl.k_new), dev(wl.v_new), dev(wl.slot_mapping)
    out = torch.empty_like(q)
    nws = P.photon_paged_decode_workspace_size(shape)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")

    def step():
        P.photon_paged_decode_step(kn, vn, sm, q, kc, vc, bt, cl, wl.scale, out, ws, nws, shape,
                                   stream)

    for _ in range(3):
        flush_l2()
        step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for i in range(K):
        flush_l2()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    st, bits = P.photon_get_last_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error word {bits} in the bf16 step")
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    nbytes = wl.decode_bytes() + wl.cache_write_bytes()
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"workload": "qwen_b64 with bf16 storage (same contexts, tables and pool)",
            "dtype": "bf16", "ms_per_step": round(ms, 5), "algorithmic_bytes": int(nbytes),
            "GBps": round(gbs, 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(gbs / peak, 4),
                         "peak_source": "measured HBM copy bandwidth"},
            "decode_tokens_per_s_per_layer": round(wl.num_seqs / (ms / 1e3), 1),
            "tokens_attended_per_s": round(wl.tokens_attended() / (ms / 1e3), 1)}


def decode_chunk_offsets(wl: W.Workload, part: int) -> np.ndarray:
    """Byte offsets of the (block, KV head) runs the decode copies, in the
    order of its work items: sequence, partition, KV head, block."""
    bs, hkv = wl.block_size, wl.num_kv_heads
    run = wl.block_size * wl.head_dim * wl.elem_bytes
    out = []
    for b in range(wl.num_seqs):
        nblk = -(-int(wl.context_lens[b]) // bs)
        blocks = wl.block_tables[b, :nblk].astype(np.int64)
        for p0 in range(0, nblk, part // bs):
            pb = blocks[p0:p0 + part // bs]
            for h in range(hkv):
                out.append((pb * hkv + h) * run)
    return np.concatenate(out) if out else np.zeros(0, np.int64)


def read_ceiling_side(P, torch, stream, flush_l2, K, peak, wl, kc, vc, part: int):
    """The decode's K/V copies alone (photon_debug_read_probe: the same
    (block, KV head) runs in the same order, bulk copies into shared memory,
    no arithmetic), timed like the step: the practical ceiling of the
    decode's data movement on this device."""
    offs = decode_chunk_offsets(wl, part)
    doffs = torch.from_numpy(offs).cuda()
    run = wl.block_size * wl.head_dim * wl.elem_bytes
    pool_bytes = kc.numel() * kc.element_size()

    def call():
        P.photon_debug_read_probe(kc, vc, pool_bytes, doffs, offs.shape[0], run, part // 16,
                                  stream)

    for _ in range(3):
        flush_l2()
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for i in range(K):
        flush_l2()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    st, bits = P.photon_get_last_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error word {bits} in the read probe")
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    moved = 2 * run * offs.shape[0]
    gbs = moved / (ms / 1e3) / 1e9
    return {"what": "the decode's K/V (block, KV head) runs in its item order, bulk-copied "
                    "into shared memory by a persistent grid of 2 CTAs per SM, no arithmetic",
            "chunks": int(offs.shape[0]), "bytes_moved": int(moved), "ms_per_call": round(ms, 5),
            "GBps": round(gbs, 1), "frac_of_copy_peak": round(gbs / peak, 4)}


def consumer_name(choice: int, wl: W.Workload) -> str:
    """Which decode consumer a workload runs under a selector value (the
    library's rule: tensor cores for 16-bit storage with 2+ q heads per KV
    head by default)."""
    g = wl.num_q_heads // wl.num_kv_heads
    tc = wl.dtype != W.DTYPE_F32 and (choice == 2 or (choice == 0 and g >= 2))
    return "tensor cores (mma.sync)" if tc else "CUDA cores"


def configs_side(P, torch, stream, flush_l2, K, peak, choice=0):
    """The other decode configurations (Llama-3.2-1B-shaped batch 16, the
    batch sweep 4/8/16/32, the batch-256 serving mix): fused step per call,
    L2 flushed before each; for the mix also the cache write and the decode
    timed as separate calls."""
    def dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    def timed(fn, flush=True):
        for _ in range(3):
            if flush:
                flush_l2()
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        for i in range(K):
            if flush:
                flush_l2()
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / K

    res = {}
    for name in ("llama_b16", "sweep_b4", "sweep_b8", "sweep_b16", "sweep_b32", "mix_b256"):
        wl = W.NAMED[name]()
        shape = P.PagedShape.make(**wl.shape_dict())
        q, kc, vc = dev(wl.q), dev(wl.k_cache), dev(wl.v_cache)
        bt, cl = dev(wl.block_tables), dev(wl.context_lens)
        kn, vn, sm = dev(wl.k_new), dev(wl.v_new), dev(wl.slot_mapping)
        out = torch.empty_like(q)
        nws = P.photon_paged_decode_workspace_size(shape)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")
        T = wl.slot_mapping.shape[0]
        def fused():
            P.photon_paged_decode_step(kn, vn, sm, q, kc, vc, bt, cl, wl.scale, out, ws, nws,
                                       shape, stream)
        ms = timed(fused)
        # the same step on each consumer, for comparison
        per_consumer = {}
        for which, key in ((1, "cuda_cores"), (2, "tensor_cores")):
            P.photon_debug_set_decode_consumer(which)
            per_consumer[key] = round(timed(fused), 5)
        P.photon_debug_set_decode_consumer(choice)
        nbytes = wl.decode_bytes() + wl.cache_write_bytes()
        gbs = nbytes / (ms / 1e3) / 1e9
        r = {"ms_per_step": round(ms, 5), "GBps": round(gbs, 1),
             "hbm_fraction": round(gbs / peak, 4),
             "tokens_attended_per_s": round(wl.tokens_attended() / (ms / 1e3), 1),
             "decode_tokens_per_s_per_layer": round(wl.num_seqs / (ms / 1e3), 1),
             "algorithmic_bytes": int(nbytes), "consumer": consumer_name(choice, wl),
             "ms_per_consumer": per_consumer}
        if nbytes < 64 << 20:
            # small enough to stay in L2 (129 MB) between steps: also the warm
            # figure, steps back to back with no flush
            ms_warm = timed(fused, flush=False)
            r["warm"] = {"ms_per_step": round(ms_warm, 5),
                         "GBps": round(nbytes / (ms_warm / 1e3) / 1e9, 1),
                         "decode_tokens_per_s_per_layer": round(wl.num_seqs / (ms_warm / 1e3), 1),
                         "l2": "not flushed: the step's bytes stay in L2 between steps"}
        if name == "mix_b256":
            ms_w = timed(lambda: P.photon_cache_write(kn, vn, sm, T, kc, vc, shape, stream))
            ms_d = timed(lambda: P.photon_paged_decode(q, kc, vc, bt, cl, wl.scale, out, ws, nws,
                                                       shape, stream))
            r["separate_calls_ms"] = {"cache_write": round(ms_w, 5), "decode": round(ms_d, 5)}
        st, bits = P.photon_get_last_device_error(stream)
        if st != 0:
            raise RuntimeError(f"device error word {bits} in config {name}")
        res[name] = r
        del q, kc, vc, bt, cl, kn, vn, sm, out, ws
    return res


def scheduler_side(P, steps: int = 200):
    """Host cost of one continuous-batching step of the C++ scheduler (plan +
    commit, through the ctypes binding) with 256 running requests in the
    batch-256 serving mix, after a warm-up that fills the batch."""
    mbs = 1024
    sched = P.Scheduler(num_blocks=40000, block_size=16, max_blocks_per_seq=mbs, max_seqs=256,
                        max_step_tokens=8192)
    trace = W.request_trace(5, 2000, max_prompt=8192, max_new=2048, pool_tokens=40000 * 16,
                            arrivals_per_step=64.0)
    for _, rid, prompt, new in trace:
        sched.add_request(rid, prompt, new)
    for _ in range(100):              # fill the batch, get past the prompts
        sched.schedule()
        sched.update()
    t0 = time.perf_counter()
    rows = 0
    for _ in range(steps):
        r = sched.schedule()
        rows += r["num_rows"]
        sched.update()
    dt = (time.perf_counter() - t0) / steps
    sched.close()
    return {"us_per_step": round(dt * 1e6, 1), "rows_per_step": round(rows / steps, 1),
            "note": "schedule + update through the Python binding, host CPU"}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        data = json.load(open(path))
    except Exception:
        return None, "fallback"
    def find(d, keys):
        if isinstance(d, dict):
            for k in keys:
                if k in d and isinstance(d[k], (int, float)):
                    return float(d[k])
            for v in d.values():
                r = find(v, keys)
                if r is not None:
                    return r
        return None
    v = find(data, ["hbm_gbs", "hbm_gbs_burst", "hbm_copy_gbs", "hbm_GBps"])
    return (v, "measured") if v else (None, "fallback")


# The sources the decode attention kernel is compiled from.
ATTENTION_SOURCES = ("photon_common.cuh", "paged_decode.cuh", "paged_decode_f16.cu",
                     "paged_decode_bf16.cu", "paged_decode_f32.cu")


def _code_only(text: str) -> str:
    """A source file without its comments and blank lines: edits to comments
    leave the hash (and the recorded counters) valid."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln.strip())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_attention_photon_gb300", "csrc")
    for f in ATTENTION_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """Per-launch DRAM bytes of the attention kernel from a committed ncu summary,
    or None if the summary is missing or was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e or e.get("kernel_source_sha") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu_index = gpu_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is None:
            return False
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- CPU oracle timing
def oracle_sample(wl: W.Workload, max_tokens: int):
    """First sequences of the batch whose contexts sum to <= max_tokens (>= 1 seq)."""
    csum = np.cumsum(wl.context_lens.astype(np.int64))
    n = int(max(1, np.searchsorted(csum, max_tokens, side="right")))
    n = min(n, wl.num_seqs)
    return n, int(csum[n - 1])


def time_oracle_step(wl: W.Workload, n: int, threads: int):
    import oracle
    kc, vc = wl.k_cache, wl.v_cache
    t0 = time.perf_counter()
    oracle.cache_write(wl.k_new[:n], wl.v_new[:n], wl.slot_mapping[:n], kc, vc,
                       block_size=wl.block_size, dtype=wl.dtype)
    oracle.paged_decode(wl.q[:n], kc, vc, np.ascontiguousarray(wl.block_tables[:n]),
                        np.ascontiguousarray(wl.context_lens[:n]), wl.scale, dtype=wl.dtype,
                        num_threads=threads)
    return time.perf_counter() - t0


def sample_bytes(wl: W.Workload, n: int) -> int:
    sub = W.Workload(**{**wl.__dict__, "num_seqs": n, "context_lens": wl.context_lens[:n],
                        "block_tables": wl.block_tables[:n], "q": wl.q[:n],
                        "k_new": wl.k_new[:n], "v_new": wl.v_new[:n],
                        "slot_mapping": wl.slot_mapping[:n]})
    return sub.decode_bytes() + sub.cache_write_bytes()


def cpu_baseline(wl: W.Workload, budget_s: float = 20.0):
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    # calibrate on a small sample, then size the measured sample to the budget
    n0, tok0 = oracle_sample(wl, 4000)
    dt0 = time_oracle_step(wl, n0, threads)
    rate = tok0 / max(dt0, 1e-6)
    n, tok = oracle_sample(wl, int(rate * budget_s / 4))
    dt = time_oracle_step(wl, n, threads)
    gbs = sample_bytes(wl, n) / dt / 1e9
    # the same oracle on one thread, on a sample sized to about budget_s / 2
    rate1 = tok0 / max(time_oracle_step(wl, n0, 1), 1e-6)
    n1, tok1 = oracle_sample(wl, int(rate1 * budget_s / 2))
    dt1 = time_oracle_step(wl, n1, 1)
    gbs1 = sample_bytes(wl, n1) / dt1 / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"first {n} of {wl.num_seqs} sequences ({tok} tokens attended), "
                      f"cache write + decode, fp64, {threads} threads, one run of {dt:.2f} s",
            "single_thread": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"first {n1} of {wl.num_seqs} sequences ({tok1} tokens "
                                        f"attended), one run of {dt1:.2f} s"}}


def workload_config(wl: W.Workload) -> dict:
    """The keys naming the workload, shared by both arms' JSON lines."""
    return {"workload": wl.name, "batch": wl.num_seqs, "q_heads": wl.num_q_heads,
            "kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "block_size": wl.block_size,
            "num_blocks": wl.num_blocks, "tokens_attended": wl.tokens_attended()}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    wl = W.NAMED[args.workload]()
    threads = os.cpu_count() or 1
    total_budget = 150.0
    n0, tok0 = oracle_sample(wl, 4000)
    rate = tok0 / max(time_oracle_step(wl, n0, threads), 1e-6)
    per_step = total_budget / max(1, args.steps + args.warmup)
    n, tok = oracle_sample(wl, int(rate * per_step))
    for _ in range(args.warmup):
        time_oracle_step(wl, n, threads)
    times = [time_oracle_step(wl, n, threads) for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    gbs = sample_bytes(wl, n) / (ms / 1e3) / 1e9
    sample = (f"first {n} of {wl.num_seqs} sequences ({tok} tokens attended) per step, "
              f"cache write + decode, fp64 oracle, {threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(wl), sample_sequences=n,
                           parallelism="one host process (the oracle on all host cores)"),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- GPU arm
def run_ours(args):
    import torch
    import paged_kv_attention_photon_gb300 as P

    world, rank, local = dist_env()
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    torch.cuda.set_device(local)
    P.build()
    P.photon_debug_set_decode_consumer(args.decode_consumer)

    wl = make_workload(args.workload, rank)
    shape = P.PagedShape.make(partition_size=args.partition, **wl.shape_dict())
    plan = P.photon_paged_decode_plan(shape)

    def dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    kc, vc = dev(wl.k_cache), dev(wl.v_cache)
    # The per-step inputs (q, new K/V rows, slots, block tables, context
    # lengths) live in one packed device buffer, mirrored by one pinned host
    # buffer, so the end-to-end step moves them with a single copy.
    step_inputs = [wl.q, wl.k_new, wl.v_new, wl.slot_mapping, wl.block_tables, wl.context_lens]
    host_arrays = [np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)
                   for a in step_inputs]
    offsets, total = [], 0
    for a in host_arrays:
        offsets.append(total)
        total += (a.nbytes + 255) // 256 * 256
    packed_dev = torch.empty(total, dtype=torch.uint8, device="cuda")
    packed_host = torch.empty(total, dtype=torch.uint8).pin_memory()
    views = []
    for a, off in zip(host_arrays, offsets):
        t = torch.from_numpy(a)
        packed_host[off:off + a.nbytes].copy_(t.view(-1).view(torch.uint8))
        views.append(packed_dev[off:off + a.nbytes].view(t.dtype).view(t.shape))
    packed_dev.copy_(packed_host)
    q, kn, vn, sm, bt, cl = views
    out = torch.empty_like(q)
    ws_bytes = P.photon_paged_decode_workspace_size(shape)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush_r = torch.ones(L2_CLEAN_BYTES // 4, dtype=torch.float32, device="cuda")

    def flush_l2():
        flush_w.zero_()
        flush_r.sum()

    T = wl.slot_mapping.shape[0]
    stream = torch.cuda.current_stream()

    def step():
        # cache write of the new rows + decode, fused into one call
        P.photon_paged_decode_step(kn, vn, sm, q, kc, vc, bt, cl, wl.scale, out, ws, ws_bytes,
                                   shape, stream)

    for _ in range(max(3, args.warmup)):
        flush_l2()
        step()
    torch.cuda.synchronize()
    st, bits = P.photon_get_last_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error word {bits} during warm-up")

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    for a, b in kev:  # materialise the events so their raw handles exist
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()

    # Timed region: K steps, events around each step on the launching stream.
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    cvd = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    sampler = ClockSampler(cvd.split(",")[local] if cvd else str(local))
    with sampler:
        t_wall0 = time.perf_counter()
        for i in range(K):
            flush_l2()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    if pg:
        pg.barrier()

    # Same steps again with the library's timing hook: events recorded right
    # before the attention kernel and right after the merge kernel give the
    # decode kernels' own duration (kept out of the headline loop above).
    for i in range(K):
        flush_l2()
        P.photon_debug_set_attention_events(kev[i][0], kev[i][1])
        step()
    torch.cuda.synchronize()
    P.photon_debug_set_attention_events(None, None)
    st, bits = P.photon_get_last_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error word {bits} during the timed steps")

    step_ms = [a.elapsed_time(b) for a, b in ev]
    attn_ms = [a.elapsed_time(b) for a, b in kev]
    ms = sum(step_ms) / K
    attn_mean_ms = sum(attn_ms) / K

    step_bytes = wl.decode_bytes() + wl.cache_write_bytes()
    decode_bytes = wl.decode_bytes()

    # max over ranks of the step time, sum of bytes
    ms_max, attn_max, tot_bytes, tot_seqs, tot_tokens = reduce_over_ranks(
        pg, ms, attn_mean_ms, step_bytes, wl.num_seqs, wl.tokens_attended())
    value = tot_bytes / (ms_max / 1e3) / 1e9

    # ---- end to end through the public API, host buffers, copies inside the timing.
    # Every step copies its inputs (q, new K/V rows, slots, block tables,
    # context lengths: one packed pinned buffer) host -> device and its output
    # device -> host.  Pipelined as a serving loop would run it: two device
    # input/output sets, the copies on their own streams, so step i+1's input
    # copy and step i-1's output copy overlap step i's kernels.  The step's
    # working set (478 MB) exceeds L2, so no flush is needed inside this loop.
    e2e = None
    if not args.no_e2e:
        h_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        h2d = int(packed_host.numel())
        d2h = h_out[0].numel() * h_out[0].element_size()
        pdev = [packed_dev, torch.empty_like(packed_dev)]
        pviews = [views]
        v2 = []
        for a_, off in zip(host_arrays, offsets):
            t_ = torch.from_numpy(a_)
            v2.append(pdev[1][off:off + a_.nbytes].view(t_.dtype).view(t_.shape))
        pviews.append(v2)
        outs = [out, torch.empty_like(out)]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event(enable_timing=False)

        def run_pipelined(nsteps):
            in_ready = [ev(), ev()]
            done = [None, None]
            out_done = [None, None]
            t_start = torch.cuda.Event(enable_timing=True)
            t_end = torch.cuda.Event(enable_timing=True)
            t_start.record(s_in)
            for i in range(nsteps):
                j = i & 1
                if done[j] is not None:
                    s_in.wait_event(done[j])        # step i-2 has finished reading set j
                with torch.cuda.stream(s_in):
                    pdev[j].copy_(packed_host, non_blocking=True)
                in_ready[j].record(s_in)
                stream.wait_event(in_ready[j])
                if out_done[j] is not None:
                    stream.wait_event(out_done[j])  # step i-2's output has left set j
                qj, knj, vnj, smj, btj, clj = pviews[j]
                P.photon_paged_decode_step(knj, vnj, smj, qj, kc, vc, btj, clj, wl.scale,
                                           outs[j], ws, ws_bytes, shape, stream)
                done[j] = ev()
                done[j].record(stream)
                s_out.wait_event(done[j])
                with torch.cuda.stream(s_out):
                    h_out[j].copy_(outs[j], non_blocking=True)
                out_done[j] = ev()
                out_done[j].record(s_out)
            s_in.wait_stream(s_out)
            t_end.record(s_in)
            torch.cuda.synchronize()
            return t_start.elapsed_time(t_end)

        run_pipelined(max(3, args.warmup))
        e2e_ms = run_pipelined(K) / K
        # the same steps one at a time (copy in, step, copy out, no overlap)
        ee = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        for i in range(K):
            ee[i][0].record(stream)
            packed_dev.copy_(packed_host, non_blocking=True)
            step()
            h_out[0].copy_(out, non_blocking=True)
            ee[i][1].record(stream)
        torch.cuda.synchronize()
        serial_ms = sum(a.elapsed_time(b) for a, b in ee) / K
        if pg:
            t = torch.tensor([e2e_ms, serial_ms], dtype=torch.float64)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            e2e_ms, serial_ms = float(t[0]), float(t[1])
        e2e = {"value": round(tot_bytes / (e2e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h),
               "pipelining": "input copy of step i+1 and output copy of step i-1 overlap step i",
               "l2": "not flushed between the pipelined steps (each step reads 478 MB, "
                     "3.7x L2); the serial steps below are not flushed either",
               "serial_ms_per_step": round(serial_ms, 4),
               "serial_value": round(tot_bytes / (serial_ms / 1e3) / 1e9, 2)}
        st, bits = P.photon_get_last_device_error(stream)
        if st != 0:
            raise RuntimeError(f"device error word {bits} during the end-to-end steps")

    # ---- side measurement: the same step with the rotary embedding fused in
    rope = None
    if not args.no_rope:
        max_pos = wl.max_blocks_per_seq * wl.block_size
        table = torch.empty((max_pos, wl.head_dim // 2, 2), dtype=torch.float32, device="cuda")
        P.photon_rope_cos_sin(ROPE_BASE, max_pos, wl.head_dim, table, stream)

        def rope_step():
            P.photon_paged_decode_step_rope(kn, vn, sm, q, kc, vc, bt, cl, table, max_pos,
                                            wl.scale, out, ws, ws_bytes, shape, stream)

        for _ in range(3):
            flush_l2()
            rope_step()
        re = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        for i in range(K):
            flush_l2()
            re[i][0].record(stream)
            rope_step()
            re[i][1].record(stream)
        torch.cuda.synchronize()
        st, bits = P.photon_get_last_device_error(stream)
        if st != 0:
            raise RuntimeError(f"device error word {bits} during the RoPE steps")
        rope_ms = sum(a.elapsed_time(b) for a, b in re) / K
        rope = {"ms_per_step": round(rope_ms, 5),
                "value": round(step_bytes / (rope_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                "rope_base": ROPE_BASE, "table_positions": max_pos,
                "time_vs_plain_step": round(rope_ms / ms, 4)}

    peak, peak_kind = measured_peaks()
    if peak is None:
        peak = FALLBACK_HBM_GBS
    mq_side = None
    if not args.no_mq:
        mq_side = multi_query_side(P, torch, stream, flush_l2, K, peak)
    host_sched = scheduler_side(P) if rank == 0 and not args.no_mq else None
    fp8 = None
    if not args.no_fp8 and args.workload == "qwen_b64":
        fp8 = fp8_side(P, torch, stream, flush_l2, K, peak)
    bf16 = None
    if not args.no_bf16 and args.workload == "qwen_b64":
        bf16 = bf16_side(P, torch, stream, flush_l2, K, peak)
    read_ceiling = None
    if not args.no_read_ceiling:
        read_ceiling = read_ceiling_side(P, torch, stream, flush_l2, K, peak, wl, kc, vc,
                                         plan["partition_size"])
    other_configs = None
    if not args.no_configs:
        other_configs = configs_side(P, torch, stream, flush_l2, K, peak, args.decode_consumer)
    achieved = decode_bytes / (attn_mean_ms / 1e3) / 1e9
    roofline = {"bound": "hbm",
                "kernel": "paged_decode_attention_kernel + paged_decode_merge_kernel",
                "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} HBM copy bandwidth",
                "traffic": ncu_traffic(args.workload),
                "algorithmic_bytes_per_launch": int(decode_bytes),
                "ms_per_launch": round(attn_mean_ms, 5)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)

    if rank == 0:
        clocks = sampler.summary()
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": max(3, args.warmup), "ms_per_step": round(ms_max, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": W.DTYPE_NAMES[wl.dtype], "data": "synthetic",
            "config": {**workload_config(wl),
                       "partition_size": plan["partition_size"],
                       "decode_consumer": consumer_name(args.decode_consumer, wl),
                       "l2": "flushed before every step (512 MB write + 256 MB read of another buffer), outside the timed events; step working set 478 MB > L2",
                       "parallelism": f"dp{world} (independent batches per GPU)"},
            "hbm_fraction": round(value / peak, 4),
            "decode_tokens_per_s_per_layer": round(tot_seqs / (ms_max / 1e3), 1),
            "tokens_attended_per_s": round(tot_tokens / (ms_max / 1e3), 1),
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "rope_step": rope,
            "multi_query": mq_side,
            "host_scheduler": host_sched,
            "other_configs": other_configs,
            "fp8_kv_decode": fp8,
            "bf16_kv_decode": bf16,
            "read_ceiling": read_ceiling,
            "gpu_launches": K * plan["kernels_per_call"],
            "clocks": clocks,
            "wall_ms_per_step_incl_flush": round(1e3 * t_wall / K, 4),
            "step_ms_p10_p90": [round(float(np.percentile(step_ms, 10)), 5),
                                round(float(np.percentile(step_ms, 90)), 5)],
        }
        s = json.dumps(line)
        print(s, flush=True)
        if args.json_out:
            with open(args.json_out, "w") as f:
                f.write(s + "\n")
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    return 0


def run_mq_case(args):
    """Only one multi-query case (profiling aid)."""
    import torch
    import paged_kv_attention_photon_gb300 as P
    torch.cuda.set_device(0)
    P.build()
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def flush_l2():
        flush_w.zero_()

    peak, _ = measured_peaks()
    res = multi_query_side(P, torch, torch.cuda.current_stream(), flush_l2, args.steps,
                           peak or FALLBACK_HBM_GBS, only=args.mq_case, with_tc=False)
    print(json.dumps(res), flush=True)
    return 0


def run_fp8_case(args):
    """Only the e4m3-cache decode (profiling aid)."""
    import torch
    import paged_kv_attention_photon_gb300 as P
    torch.cuda.set_device(0)
    P.build()
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def flush_l2():
        flush_w.zero_()

    peak, _ = measured_peaks()
    res = fp8_side(P, torch, torch.cuda.current_stream(), flush_l2, args.steps,
                   peak or FALLBACK_HBM_GBS, workload=args.fp8_case)
    print(json.dumps(res), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.mq_case:
        return run_mq_case(args)
    if args.fp8_case:
        return run_fp8_case(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
