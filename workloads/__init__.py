"""Seeded synthetic inputs for the paged decode-attention path.

This module only *draws* inputs: context lengths, a fragmented physical block
pool with per-sequence block tables, query rows, new K/V rows and the slots
they go to.  It holds none of the attention arithmetic, so both the fp64 CPU
oracle and the CUDA library consume exactly the same host bytes.

Shapes follow the workloads the PhotonInfer README describes (Llama-3.2-1B and
Qwen3 decode, "Performance highlights" / "Technical details: paged attention"),
with every size that the page leaves open fixed here:

* KV pool layout ``[num_blocks][num_kv_heads][block_size][head_dim]`` (one
  contiguous chunk per physical block and KV head).
* ``block_tables`` is ``int32[B][max_blocks_per_seq]``, padded with -1.
* ``slot_mapping`` is ``int64[T]``: slot = physical_block * block_size + offset;
  a negative slot marks a padding row.
* Every pool element that no sequence owns -- unreferenced blocks and the
  unused tail of each sequence's last block -- holds NaN, so any stray read
  shows up in the result.
* Q and K/V values are N(0, 1) rounded once to the storage dtype.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Tuple, Dict, List, Optional

import numpy as np

DTYPE_F32 = 0
DTYPE_F16 = 1
DTYPE_BF16 = 2

_NP_STORAGE = {DTYPE_F32: np.float32, DTYPE_F16: np.float16, DTYPE_BF16: np.uint16}
ELEM_BYTES = {DTYPE_F32: 4, DTYPE_F16: 2, DTYPE_BF16: 2}
DTYPE_NAMES = {DTYPE_F32: "f32", DTYPE_F16: "f16", DTYPE_BF16: "bf16"}
_NAN_BITS = {DTYPE_F32: np.uint32(0x7FC00000), DTYPE_F16: np.uint16(0x7E00),
             DTYPE_BF16: np.uint16(0x7FC0)}


@dataclasses.dataclass
class Workload:
    """One batch of decode inputs, all host numpy arrays."""

    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    dtype: int
    scale: float
    context_lens: np.ndarray      # int32[B]
    block_tables: np.ndarray      # int32[B][MBS], -1 padded
    q: np.ndarray                 # dtype[B][Hq][d]
    k_cache: np.ndarray           # dtype[NB][Hkv][bs][d]
    v_cache: np.ndarray           # dtype[NB][Hkv][bs][d]
    k_new: np.ndarray             # dtype[T][Hkv][d]
    v_new: np.ndarray             # dtype[T][Hkv][d]
    slot_mapping: np.ndarray      # int64[T]
    seed: int = 0

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def shape_dict(self) -> Dict[str, int]:
        return dict(num_seqs=self.num_seqs, num_q_heads=self.num_q_heads,
                    num_kv_heads=self.num_kv_heads, head_dim=self.head_dim,
                    block_size=self.block_size, num_blocks=self.num_blocks,
                    max_blocks_per_seq=self.max_blocks_per_seq, dtype=self.dtype)

    # --- byte counts used by the benchmark (definitions, not arithmetic of the method)
    def decode_bytes(self) -> int:
        """Algorithmic HBM bytes of one decode call: every K and V row inside the
        contexts, q in, out written, the block-table entries used, context_lens."""
        ctx = self.context_lens.astype(np.int64)
        e = self.elem_bytes
        kv = int(ctx.sum()) * self.num_kv_heads * self.head_dim * e * 2
        qo = 2 * self.num_seqs * self.num_q_heads * self.head_dim * e
        tables = 4 * int(((ctx + self.block_size - 1) // self.block_size).sum())
        return kv + qo + tables + 4 * self.num_seqs

    def cache_write_bytes(self) -> int:
        t = int(self.slot_mapping.shape[0])
        row = self.num_kv_heads * self.head_dim * self.elem_bytes
        return 2 * t * row * 2 + 8 * t

    def tokens_attended(self) -> int:
        return int(self.context_lens.astype(np.int64).sum())


def _draw_values(rng: np.random.Generator, n: int, dtype: int) -> np.ndarray:
    x = rng.standard_normal(n, dtype=np.float32)
    if dtype == DTYPE_F32:
        return x
    if dtype == DTYPE_F16:
        return x.astype(np.float16)
    # bf16: round-to-nearest-even of the fp32 bit pattern, kept as raw uint16
    b = x.view(np.uint32)
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def _nan_pool(shape, dtype: int) -> np.ndarray:
    bits = _NAN_BITS[dtype]
    raw = np.full(shape, bits, dtype=bits.dtype)
    if dtype == DTYPE_F32:
        return raw.view(np.float32)
    if dtype == DTYPE_F16:
        return raw.view(np.float16)
    return raw


def build(name: str, *, num_q_heads: int, num_kv_heads: int, head_dim: int,
          context_lens: np.ndarray, num_blocks: int, dtype: int, scale: float,
          rng: np.random.Generator, block_size: int = 16,
          max_blocks_per_seq: Optional[int] = None, free_list_new_blocks: bool = False,
          seed: int = 0, shuffle_pool: bool = True) -> Workload:
    """Assemble a workload from sampled context lengths.

    The physical pool is handed out from one random permutation.  With
    ``free_list_new_blocks`` the blocks needed by the tokens *before* this step
    are handed out first, and a sequence whose new token opens a fresh block
    takes it from the remaining (randomly ordered) free list.
    """
    ctx = np.asarray(context_lens, dtype=np.int32)
    B = int(ctx.shape[0])
    bs = block_size
    nblk = (ctx.astype(np.int64) + bs - 1) // bs
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, int(nblk.max()) if B else 1)
    mbs = max_blocks_per_seq
    assert int(nblk.max(initial=0)) <= mbs
    assert int(nblk.sum()) <= num_blocks, "pool too small"

    perm = rng.permutation(num_blocks).astype(np.int32)
    if not shuffle_pool:   # contiguous pool: each sequence's blocks in order
        perm = np.arange(num_blocks, dtype=np.int32)
    tables = np.full((B, mbs), -1, dtype=np.int32)
    if free_list_new_blocks:
        prev = np.maximum(ctx.astype(np.int64) - 1, 0)
        prev_blk = (prev + bs - 1) // bs
        pos = 0
        for b in range(B):
            n = int(prev_blk[b])
            tables[b, :n] = perm[pos:pos + n]
            pos += n
        free = perm[pos:]
        fpos = 0
        for b in range(B):
            if int(nblk[b]) > int(prev_blk[b]):
                tables[b, int(prev_blk[b])] = free[fpos]
                fpos += 1
    else:
        pos = 0
        for b in range(B):
            n = int(nblk[b])
            tables[b, :n] = perm[pos:pos + n]
            pos += n

    H, d = num_kv_heads, head_dim
    k_cache = _nan_pool((num_blocks, H, bs, d), dtype)
    v_cache = _nan_pool((num_blocks, H, bs, d), dtype)
    for b in range(B):
        n = int(nblk[b])
        if n == 0:
            continue
        blocks = tables[b, :n]
        valid = int(ctx[b])
        cnt = n * H * bs * d
        kv = _draw_values(rng, cnt, dtype).reshape(n, H, bs, d)
        vv = _draw_values(rng, cnt, dtype).reshape(n, H, bs, d)
        tail = valid - (n - 1) * bs          # valid rows in the last block
        if tail < bs:
            kv[n - 1, :, tail:, :] = _nan_pool((H, bs - tail, d), dtype)
            vv[n - 1, :, tail:, :] = _nan_pool((H, bs - tail, d), dtype)
        k_cache[blocks] = kv
        v_cache[blocks] = vv

    q = _draw_values(rng, B * num_q_heads * d, dtype).reshape(B, num_q_heads, d)

    # One new K/V row per sequence: the token at position ctx-1 (context_lens
    # counts it).  Sequences with an empty context contribute a padding row.
    k_new = _draw_values(rng, B * H * d, dtype).reshape(B, H, d)
    v_new = _draw_values(rng, B * H * d, dtype).reshape(B, H, d)
    slots = np.full(B, -1, dtype=np.int64)
    for b in range(B):
        if ctx[b] > 0:
            j = int(ctx[b]) - 1
            slots[b] = int(tables[b, j // bs]) * bs + j % bs

    return Workload(name=name, num_seqs=B, num_q_heads=num_q_heads,
                    num_kv_heads=num_kv_heads, head_dim=d, block_size=bs,
                    num_blocks=num_blocks, max_blocks_per_seq=mbs, dtype=dtype,
                    scale=float(scale), context_lens=ctx, block_tables=tables, q=q,
                    k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
                    slot_mapping=slots, seed=seed)


# ---------------------------------------------------------------- named workloads

def tiny(seed: int = 0) -> Workload:
    """Batch 2, 4 q heads over 1 KV head, d=64, fp32, contexts {5, 37}, an
    8-block shuffled pool of which 4 blocks are unreferenced, scale 1/8."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return build("tiny", num_q_heads=4, num_kv_heads=1, head_dim=64,
                 context_lens=np.array([5, 37], np.int32), num_blocks=8,
                 dtype=DTYPE_F32, scale=1.0 / 8.0, rng=rng, max_blocks_per_seq=4,
                 seed=seed)


def llama_b16(seed: int = 1, dtype: int = DTYPE_F16) -> Workload:
    """Llama-3.2-1B attention layer: 16 sequences, 32q/8kv heads, d=64,
    contexts uniform in [100, 1124], pool of 16*71 blocks in random order."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = rng.integers(100, 1124, size=16, endpoint=True).astype(np.int32)
    return build("llama_b16", num_q_heads=32, num_kv_heads=8, head_dim=64,
                 context_lens=ctx, num_blocks=16 * 71, dtype=dtype,
                 scale=1.0 / 8.0, rng=rng, max_blocks_per_seq=71, seed=seed)


def sweep(batch: int, dtype: int = DTYPE_F16) -> Workload:
    """Llama-3.2-1B shape at batch 4/8/16/32, contexts uniform in [64, 2048]."""
    seed = 100 + batch
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = rng.integers(64, 2048, size=batch, endpoint=True).astype(np.int32)
    return build(f"sweep_b{batch}", num_q_heads=32, num_kv_heads=8, head_dim=64,
                 context_lens=ctx, num_blocks=batch * 128, dtype=dtype,
                 scale=1.0 / 8.0, rng=rng, max_blocks_per_seq=128, seed=seed)


def qwen_context_lens(rng: np.random.Generator, batch: int = 64) -> np.ndarray:
    u = rng.uniform(math.log(128.0), math.log(8192.0), size=batch)
    return np.clip(np.rint(np.exp(u)), 128, 8192).astype(np.int32)


def qwen_b64(seed: int = 2, batch: int = 64, num_blocks: int = 40000,
             dtype: int = DTYPE_F16, shuffle_pool: bool = True) -> Workload:
    """Qwen3-style long context: 64 sequences, 16q/8kv heads, d=128, contexts
    log-uniform in [128, 8192], a fragmented 40 000-block pool in random order."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = qwen_context_lens(rng, batch)
    return build("qwen_b64" if batch == 64 else f"qwen_b{batch}", num_q_heads=16,
                 num_kv_heads=8, head_dim=128, context_lens=ctx,
                 num_blocks=num_blocks, dtype=dtype, scale=1.0 / math.sqrt(128.0),
                 rng=rng, max_blocks_per_seq=512, seed=seed, shuffle_pool=shuffle_pool)


def mix_context_lens(rng: np.random.Generator, batch: int = 256) -> np.ndarray:
    long_mask = rng.uniform(size=batch) < 0.2
    short = rng.integers(32, 512, size=batch, endpoint=True)
    long_ = rng.integers(4096, 16384, size=batch, endpoint=True)
    return np.where(long_mask, long_, short).astype(np.int32)


def mix_b256(seed: int = 3, batch: int = 256, dtype: int = DTYPE_F16) -> Workload:
    """Continuous-batching step mix: 256 sequences, 32q/8kv heads, d=64,
    80% of contexts uniform in [32, 512] and 20% in [4096, 16384]; the new
    token of each sequence goes to a free-list slot."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = mix_context_lens(rng, batch)
    used = int(((ctx.astype(np.int64) + 15) // 16).sum())
    nb = int(math.ceil(1.3 * used))
    return build("mix_b256" if batch == 256 else f"mix_b{batch}", num_q_heads=32,
                 num_kv_heads=8, head_dim=64, context_lens=ctx, num_blocks=nb,
                 dtype=dtype, scale=1.0 / 8.0, rng=rng, max_blocks_per_seq=1024,
                 free_list_new_blocks=True, seed=seed)


def random_small(seed: int, *, batch: int, num_q_heads: int, num_kv_heads: int,
                 head_dim: int, max_ctx: int, dtype: int, block_size: int = 16,
                 extra_blocks: int = 3, context_lens: Optional[List[int]] = None,
                 scale: Optional[float] = None) -> Workload:
    """Small random workload for parity tests (ragged lengths, spare blocks)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if context_lens is None:
        ctx = rng.integers(0, max_ctx, size=batch, endpoint=True).astype(np.int32)
    else:
        ctx = np.asarray(context_lens, dtype=np.int32)
        batch = int(ctx.shape[0])
    mbs = max(1, (max(int(ctx.max(initial=0)), max_ctx) + block_size - 1) // block_size)
    nb = int(((ctx.astype(np.int64) + block_size - 1) // block_size).sum()) + extra_blocks
    return build(f"small_s{seed}", num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                 head_dim=head_dim, context_lens=ctx, num_blocks=max(nb, 1), dtype=dtype,
                 scale=(1.0 / math.sqrt(head_dim)) if scale is None else scale, rng=rng,
                 block_size=block_size, max_blocks_per_seq=mbs, seed=seed)


# e4m3 code of NaN: fills the unreferenced blocks of an fp8 pool (stray-read detector)
E4M3_NAN = 0x7F
# per-tensor scales of the synthetic fp8 caches
FP8_K_SCALE, FP8_V_SCALE = 0.5, 0.25


def fp8_cache(wl: Workload, seed: int):
    """e4m3 K and V pools for the sequences of `wl` (its tables and lengths):
    every block a table names gets random finite codes -- random sign,
    exponent field 5 .. 8, random mantissa, i.e. magnitudes 0.25 .. 3.75 --
    the other blocks the NaN code.  Bytes only; the scales are FP8_K_SCALE /
    FP8_V_SCALE.  Returns (k8, v8), uint8 [NB][Hkv][bs][d]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    pools = []
    used = np.unique(wl.block_tables[wl.block_tables >= 0])
    for _ in range(2):
        pool = np.full(shape, E4M3_NAN, dtype=np.uint8)
        n = used.shape[0] * int(np.prod(shape[1:]))
        sign = rng.integers(0, 2, size=n, dtype=np.uint8) << np.uint8(7)
        expo = rng.integers(5, 9, size=n, dtype=np.uint8) << np.uint8(3)
        mant = rng.integers(0, 8, size=n, dtype=np.uint8)
        pool[used] = (sign | expo | mant).reshape((used.shape[0],) + shape[1:])
        pools.append(pool)
    return pools[0], pools[1]


def request_trace(seed: int, num_requests: int, *, max_prompt: int, max_new: int,
                  pool_tokens: int, long_frac: float = 0.2,
                  arrivals_per_step: float = 1.0) -> List[tuple]:
    """Seeded serving trace for the scheduler: (arrival_step, request_id,
    prompt_len, max_new_tokens), arrival order.  The prompt mix follows the
    batch-256 serving step: long_frac of the prompts are long (uniform in
    [max_prompt/4, max_prompt]), the rest short (uniform in [1, max_prompt/8]);
    output lengths are uniform in [1, max_new]; arrivals are a Poisson stream
    of arrivals_per_step per step.  Every request fits max_prompt + max_new - 1
    tokens and the pool (pool_tokens)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out, t = [], 0.0
    for i in range(num_requests):
        t += rng.exponential(1.0 / arrivals_per_step)
        if rng.uniform() < long_frac:
            prompt = int(rng.integers(max(1, max_prompt // 4), max_prompt, endpoint=True))
        else:
            prompt = int(rng.integers(1, max(1, max_prompt // 8), endpoint=True))
        new = int(rng.integers(1, max_new, endpoint=True))
        new = max(1, min(new, pool_tokens - prompt + 1))
        out.append((int(t), 1000 + i, prompt, new))
    return out


def request_rows(seed: int, request_id: int, num_tokens: int, num_kv_heads: int,
                 head_dim: int, dtype: int) -> Tuple[np.ndarray, np.ndarray]:
    """The K and V rows of every position of one request, [num_tokens][Hkv][d],
    N(0,1) rounded to the storage dtype, a function of (seed, request_id) only:
    a request that is preempted and recomputed writes the same rows again."""
    rng = np.random.Generator(np.random.PCG64([seed, request_id]))
    n = num_tokens * num_kv_heads * head_dim
    k = _draw_values(rng, n, dtype).reshape(num_tokens, num_kv_heads, head_dim)
    v = _draw_values(rng, n, dtype).reshape(num_tokens, num_kv_heads, head_dim)
    return k, v


def request_queries(seed: int, request_id: int, position: int, num_q_heads: int,
                    head_dim: int, dtype: int) -> np.ndarray:
    """The query rows [Hq][d] of one request at one position."""
    rng = np.random.Generator(np.random.PCG64([seed, request_id, position, 7]))
    return _draw_values(rng, num_q_heads * head_dim, dtype).reshape(num_q_heads, head_dim)


@dataclasses.dataclass
class MultiQueryWorkload:
    """A paged pool whose sequences end in query_lens[b] new tokens (their K/V
    rows already in the pool) plus the query rows of those tokens."""
    pool: Workload            # pool, block tables, context lengths (= prefix + new)
    q: np.ndarray             # [T][Hq][d]
    query_start: np.ndarray   # int32 [B + 1]
    max_query_len: int

    @property
    def num_tokens(self) -> int:
        return int(self.query_start[-1])

    def flops(self) -> int:
        """Multiply-adds x 2 of QK^T and PV over the causal key ranges."""
        p = self.pool
        n = np.diff(self.query_start).astype(np.int64)
        first = p.context_lens.astype(np.int64) - n
        keys = (n * first + n * (n + 1) // 2).sum()          # sum over tokens of (pos + 1)
        return int(4 * keys * p.num_q_heads * p.head_dim)

    def kv_bytes(self) -> int:
        """K/V rows read once per (sequence, KV head), plus q and out."""
        p = self.pool
        kv = int(p.context_lens.astype(np.int64).sum()) * p.num_kv_heads * p.head_dim * \
            p.elem_bytes * 2
        return kv + 2 * self.q.nbytes


def multi_query(seed: int, *, query_lens, prefix_lens, num_q_heads: int, num_kv_heads: int,
                head_dim: int, dtype: int, extra_blocks: int = 3,
                scale: Optional[float] = None) -> MultiQueryWorkload:
    """Chunked-prefill / speculative-verify input: sequence b has prefix_lens[b]
    cached tokens followed by query_lens[b] new tokens whose K/V rows are
    already written; values N(0,1) in the storage dtype, blocks permuted."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n = np.asarray(query_lens, dtype=np.int32)
    ctx = (np.asarray(prefix_lens, dtype=np.int64) + n).astype(np.int32)
    bs = 16
    mbs = max(1, (int(ctx.max(initial=0)) + bs - 1) // bs)
    nb = int(((ctx.astype(np.int64) + bs - 1) // bs).sum()) + extra_blocks
    pool = build(f"mq_s{seed}", num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                 head_dim=head_dim, context_lens=ctx, num_blocks=max(nb, 1), dtype=dtype,
                 scale=(1.0 / math.sqrt(head_dim)) if scale is None else scale, rng=rng,
                 block_size=bs, max_blocks_per_seq=mbs, seed=seed)
    T = int(n.sum())
    q = _draw_values(rng, T * num_q_heads * head_dim, dtype).reshape(T, num_q_heads, head_dim)
    qs = np.zeros(n.shape[0] + 1, dtype=np.int32)
    qs[1:] = np.cumsum(n)
    return MultiQueryWorkload(pool=pool, q=q, query_start=qs,
                              max_query_len=int(n.max(initial=0)))


NAMED = {
    "tiny": tiny,
    "llama_b16": llama_b16,
    "qwen_b64": qwen_b64,
    "mix_b256": mix_b256,
    "qwen_b64_pool10k": lambda: qwen_b64(num_blocks=10000),
    "sweep_b4": lambda: sweep(4),
    "sweep_b8": lambda: sweep(8),
    "sweep_b16": lambda: sweep(16),
    "sweep_b32": lambda: sweep(32),
}
