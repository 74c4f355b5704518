"""GPU parity of the multi-query (causal) paged attention against the fp64
oracle, through the C ABI.

* ragged query lengths across the 64-row tile edges (1, 2, 7, 16, 17, 33, 64,
  65, 130 tokens x group size), prefixes from 0 to 2000 tokens, every group
  size, d = 64 and 128, fp16 and bf16: 2e-3 max-abs for fp16 (the decode
  bound); for bf16 the tensor-core product takes the softmax weights p_j
  rounded to bf16 (relative error <= 2^-9 each), which moves an output by up
  to 2^-9 sum_j p_j |V_j| / sum_j p_j on top of the output's own rounding, so
  the bound is 2^-8 |o| + 2^-8 a + 2e-4 with a = the oracle's attention over
  |V| (twice each rounding term);
* a chunked-prefill batch (4 sequences x 512 new tokens on up to 3.5k cached
  ones, 16q/8kv, d = 128) and a speculative-verify batch (64 sequences x 4
  draft tokens on the long-context batch-64 lengths), all rows;
* one token per sequence agrees with photon_paged_decode;
* inconsistent lengths are flagged (bits 4 / 32) and zero-filled, not faulted;
* every case runs on both kernels -- the warp-level mma.sync one (with and
  without key splits) and the tcgen05/TMEM one -- chosen through
  photon_debug_set_multi_query_kernel;
* the few-token mode (max_query_len x G <= 8: the decode kernel with one
  query slot per (token, head)): ragged token counts on every group size,
  partitions that cut through a sequence's query tokens (a token then sees
  none of the last partition's keys), the verify batch, and its error rules.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_photon_gb300 as P
import workloads as W
from gpu_util import BF16_ATOL, assert_close, dev, to_float64

pytestmark = pytest.mark.gpu
THREADS = max(1, min(32, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    P.build()
    torch.cuda.init()
    st, _ = P.photon_get_last_device_error()
    assert st == 0


@pytest.fixture(params=[1, 2, 3], ids=["mma_sync", "tcgen05", "few_token_else_plan"])
def kernel(request):
    P.photon_debug_set_multi_query_kernel(request.param)
    yield request.param
    P.photon_debug_set_multi_query_kernel(0)


def _workspace(shape, num_tokens, max_query_len):
    n = P.photon_paged_multi_query_workspace_size(shape, num_tokens, max_query_len)
    # no initialisation is needed: start from NaN bytes
    return torch.full((max(n, 16),), 0xFF, dtype=torch.uint8, device="cuda"), n


def _run(mq: W.MultiQueryWorkload, max_query_len=None, partition=0, context_lens=None,
         query_start=None):
    p = mq.pool
    shape = P.PagedShape.make(partition_size=partition, **p.shape_dict())
    mql = mq.max_query_len if max_query_len is None else max_query_len
    ws, nws = _workspace(shape, mq.num_tokens, mql)
    qd = dev(mq.q)
    out = torch.full(qd.shape, -1, dtype=qd.dtype, device="cuda")
    ctx = p.context_lens if context_lens is None else context_lens
    qs = mq.query_start if query_start is None else query_start
    P.photon_paged_multi_query(qd, dev(p.k_cache), dev(p.v_cache), dev(p.block_tables),
                               dev(ctx), dev(qs), mq.num_tokens, mql, p.scale, out,
                               ws, nws, shape)
    torch.cuda.synchronize()
    return out


def _want(mq: W.MultiQueryWorkload, abs_v: bool = False):
    p = mq.pool
    v = p.v_cache
    if abs_v:      # |V| in the storage type: clear the sign bit (NaN poison stays NaN)
        v = v.copy()
        v.view(np.uint32 if v.dtype == np.float32 else np.uint16)[...] &= \
            (0x7FFFFFFF if v.dtype == np.float32 else 0x7FFF)
    return oracle.multi_query(mq.q, p.k_cache, v, p.block_tables, p.context_lens,
                              mq.query_start, p.scale, dtype=p.dtype, num_threads=THREADS)


def _check(got: np.ndarray, mq: W.MultiQueryWorkload, what: str, rows=slice(None)) -> None:
    want = _want(mq)[rows]
    if mq.pool.dtype != W.DTYPE_BF16:
        assert_close(got, want, mq.pool.dtype, what)
        return
    assert np.isfinite(got).all(), what
    a = _want(mq, abs_v=True)[rows]
    bound = 2.0 ** -8 * (np.abs(want) + a) + BF16_ATOL
    worst = float((np.abs(got - want) - bound).max(initial=-1.0))
    assert worst <= 0, f"{what}: bf16 error exceeds bound by {worst}"


RAGGED_N = [1, 2, 7, 16, 17, 33, 64, 65, 130]
RAGGED_PREFIX = [0, 1, 15, 16, 100, 0, 511, 1000, 2000]


@pytest.mark.parametrize("dtype", [W.DTYPE_F16, W.DTYPE_BF16])
@pytest.mark.parametrize("Hq,Hkv,d", [(4, 4, 128), (16, 8, 128), (32, 8, 64), (16, 2, 64),
                                      (8, 2, 128), (8, 8, 64)])
def test_ragged_matches_oracle(dtype, Hq, Hkv, d, kernel):
    mq = W.multi_query(300 + Hq + d + dtype, query_lens=RAGGED_N, prefix_lens=RAGGED_PREFIX,
                       num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, dtype=dtype)
    out = _run(mq)
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0, bits
    _check(to_float64(out, dtype), mq, f"mq {Hq}/{Hkv}/{d}")


def test_chunked_prefill_batch(kernel):
    mq = W.multi_query(310, query_lens=[512] * 4, prefix_lens=[0, 512, 2048, 3584],
                       num_q_heads=16, num_kv_heads=8, head_dim=128, dtype=W.DTYPE_F16)
    out = _run(mq)
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0, bits
    assert_close(to_float64(out, W.DTYPE_F16), _want(mq), W.DTYPE_F16, "chunked prefill")


@pytest.mark.parametrize("which", [1, 2, 3], ids=["mma_sync", "tcgen05", "few_token"])
def test_speculative_verify_batch(which):
    P.photon_debug_set_multi_query_kernel(which)
    rng = np.random.Generator(np.random.PCG64(2))
    ctx = W.qwen_context_lens(rng, 64)
    mq = W.multi_query(311, query_lens=[4] * 64, prefix_lens=(ctx - 4).tolist(),
                       num_q_heads=16, num_kv_heads=8, head_dim=128, dtype=W.DTYPE_BF16)
    out = _run(mq)
    P.photon_debug_set_multi_query_kernel(0)
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0, bits
    _check(to_float64(out, W.DTYPE_BF16), mq, "verify")


def test_one_token_agrees_with_decode(kernel):
    mq = W.multi_query(312, query_lens=[1] * 9, prefix_lens=[0, 5, 15, 16, 63, 64, 200, 777, 0],
                       num_q_heads=16, num_kv_heads=8, head_dim=128, dtype=W.DTYPE_F16)
    got = to_float64(_run(mq), W.DTYPE_F16)
    p = mq.pool
    shape = P.PagedShape.make(**p.shape_dict())
    ws_bytes = P.photon_paged_decode_workspace_size(shape)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((9, 16, 128), dtype=torch.float16, device="cuda")
    P.photon_paged_decode(dev(mq.q), dev(p.k_cache), dev(p.v_cache), dev(p.block_tables),
                          dev(p.context_lens), p.scale, out, ws, ws_bytes, shape)
    torch.cuda.synchronize()
    dec = to_float64(out, W.DTYPE_F16)
    assert np.abs(got - dec).max() <= 2e-3
    assert_close(got, _want(mq), W.DTYPE_F16)


def test_inconsistent_lengths_are_flagged_and_zeroed(kernel):
    mq = W.multi_query(313, query_lens=[3, 40, 5], prefix_lens=[10, 10, 10], num_q_heads=8,
                       num_kv_heads=2, head_dim=64, dtype=W.DTYPE_F16)
    # max_query_len 8 < 40: sequence 1 is flagged (bit 32); its first 8 rows are zeroed
    out = _run(mq, max_query_len=8)
    st, bits = P.photon_get_last_device_error()
    assert st == 6 and bits == 32, bits
    got = to_float64(out, W.DTYPE_F16)
    want = _want(mq)
    qs = mq.query_start
    assert_close(got[qs[0]:qs[1]], want[qs[0]:qs[1]], W.DTYPE_F16)
    assert_close(got[qs[2]:qs[3]], want[qs[2]:qs[3]], W.DTYPE_F16)
    assert (got[qs[1]:qs[1] + 8] == 0).all()
    # a context shorter than the query count: bit 4, rows zeroed
    bad_ctx = mq.pool.context_lens.copy()
    bad_ctx[0] = 2
    out = _run(mq, context_lens=bad_ctx)
    st, bits = P.photon_get_last_device_error()
    assert st == 6 and bits == 4, bits
    got = to_float64(out, W.DTYPE_F16)
    assert (got[qs[0]:qs[1]] == 0).all()
    assert_close(got[qs[1]:], want[qs[1]:], W.DTYPE_F16)


@pytest.mark.parametrize("partition", [64, 128, 512, 4096])
def test_split_partitions_match_oracle(partition):
    """Forced split-KV: every tile's keys in partitions of `partition` keys,
    merged by the second kernel; rows whose position falls in an early
    partition and fully masked partitions included."""
    mq = W.multi_query(320 + partition, query_lens=[1, 4, 70, 3, 130, 9],
                       prefix_lens=[0, 60, 200, 1500, 700, 4000], num_q_heads=16,
                       num_kv_heads=4, head_dim=128, dtype=W.DTYPE_F16)
    out = _run(mq, partition=partition)
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0, bits
    assert_close(to_float64(out, W.DTYPE_F16), _want(mq), W.DTYPE_F16, f"part {partition}")




@pytest.mark.parametrize("which", [0, 1, 2], ids=["default", "mma_sync", "tcgen05"])
def test_prefill_without_split_matches(which):
    """A prefill batch big enough to skip the key split (no workspace), on
    every kernel: every row of four sequences against the oracle.  Unsplit,
    a sequence's keys (up to 5120) are one partition, longer than the
    warp-level kernel's 256-block table window."""
    P.photon_debug_set_multi_query_kernel(which)
    mq = W.multi_query(330, query_lens=[1024] * 16, prefix_lens=[0] * 8 + [4096] * 8,
                       num_q_heads=16, num_kv_heads=8, head_dim=128, dtype=W.DTYPE_F16)
    p = mq.pool
    shape = P.PagedShape.make(**p.shape_dict())
    assert P.photon_paged_multi_query_workspace_size(shape, mq.num_tokens, mq.max_query_len) == 0
    got = to_float64(_run(mq), W.DTYPE_F16)
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0, bits
    qs = mq.query_start
    for b in [0, 7, 8, 15]:
        want = oracle.multi_query(mq.q[qs[b]:qs[b + 1]], p.k_cache, p.v_cache,
                                  p.block_tables[b:b + 1], p.context_lens[b:b + 1],
                                  np.array([0, qs[b + 1] - qs[b]], np.int32), p.scale,
                                  dtype=p.dtype, num_threads=THREADS)
        assert_close(got[qs[b]:qs[b + 1]], want, W.DTYPE_F16, f"prefill seq {b}")
    P.photon_debug_set_multi_query_kernel(0)


@pytest.fixture
def few_token():
    P.photon_debug_set_multi_query_kernel(3)
    yield 3
    P.photon_debug_set_multi_query_kernel(0)


@pytest.mark.parametrize("partition", [0, 64])
@pytest.mark.parametrize("dtype", [W.DTYPE_F16, W.DTYPE_BF16])
@pytest.mark.parametrize("Hq,Hkv,d", [(8, 8, 64), (16, 8, 128), (32, 8, 64), (16, 2, 128)])
def test_few_token_matches_oracle(Hq, Hkv, d, dtype, partition, few_token):
    """Token counts 1 .. 8/G per sequence on prefixes around block and
    partition edges; with 64-key partitions the query tokens of several
    sequences straddle a partition edge, so an early token sees no key of
    the last partition."""
    g = Hq // Hkv
    nmax = 8 // g
    lens = [(i % nmax) + 1 for i in range(10)]
    prefix = [0, 1, 15, 16, 62, 63, 125, 200, 1000, 2000]
    mq = W.multi_query(340 + Hq + d + dtype + partition, query_lens=lens, prefix_lens=prefix,
                       num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, dtype=dtype)
    out = _run(mq, partition=partition)
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0, bits
    _check(to_float64(out, dtype), mq, f"few-token {Hq}/{Hkv}/{d} part {partition}")


def test_few_token_errors_are_flagged(few_token):
    """max_query_len 4 with 2 heads per KV head: the few-token mode.  A
    sequence with more tokens than that (bit 32, its first 4 rows zeroed), a
    context shorter than its token count (bit 4, rows zeroed), rows past
    num_tokens (bit 32, rows untouched); the other sequences exact."""
    mq = W.multi_query(350, query_lens=[3, 6, 2, 4], prefix_lens=[10, 10, 10, 30],
                       num_q_heads=16, num_kv_heads=8, head_dim=64, dtype=W.DTYPE_F16)
    qs = mq.query_start
    want = _want(mq)

    def good(got, seqs):
        for b in seqs:
            assert_close(got[qs[b]:qs[b + 1]], want[qs[b]:qs[b + 1]], W.DTYPE_F16, f"seq {b}")

    got = to_float64(_run(mq, max_query_len=4), W.DTYPE_F16)
    st, bits = P.photon_get_last_device_error()
    assert st == 6 and bits == 32, bits
    assert (got[qs[1]:qs[1] + 4] == 0).all()
    good(got, (0, 2, 3))
    bad_ctx = mq.pool.context_lens.copy()
    bad_ctx[2] = 1
    got = to_float64(_run(mq, max_query_len=4, context_lens=bad_ctx), W.DTYPE_F16)
    st, bits = P.photon_get_last_device_error()
    assert st == 6 and bits == 32 | 4, bits
    assert (got[qs[2]:qs[3]] == 0).all()
    good(got, (0, 3))
    bad_qs = qs.copy()
    bad_qs[4] = mq.num_tokens + 1
    got = to_float64(_run(mq, max_query_len=4, query_start=bad_qs), W.DTYPE_F16)
    st, bits = P.photon_get_last_device_error()
    assert st == 6 and bits == 32, bits
    assert (got[qs[3]:qs[4]] == -1).all()
    good(got, (0, 2))
