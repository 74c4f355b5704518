"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle on
the same seeded host bytes.

* cache write and block-table gather: bit-exact, whole pool / whole dense copy;
* decode: max-abs error <= 2e-3 for fp16 storage (fp32 accumulate), 1e-4 for
  fp32 storage, 2^-8 relative + 2e-4 for bf16 storage;
* edge cases: empty and one-token contexts, block and partition edges, every
  partition size, unreferenced NaN-filled blocks, device-side index errors;
* the full-size long-context batch-64 and batch-256 step workloads in the
  launch configuration the benchmark times.

The decode tests run under both attention consumers (photon_debug_set_decode_
consumer): the CUDA-core one and the tensor-core one (fp16/bf16 storage; fp32
cases take the CUDA-core path either way).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_photon_gb300 as P
import workloads as W
from gpu_util import DeviceWorkload, assert_close, dev, host

pytestmark = pytest.mark.gpu
THREADS = max(1, min(32, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    P.build()
    torch.cuda.init()
    st, _ = P.photon_get_last_device_error()
    assert st == 0


_ORACLE_CACHE = {}


def _oracle_step_cached(key: str, wl: W.Workload):
    """_oracle_step of a named workload, computed once per test session."""
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE[key] = _oracle_step(wl)
    return _ORACLE_CACHE[key]


def _oracle_step(wl: W.Workload, write: bool = True):
    """Oracle of one step: cache write of the new rows, then decode."""
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    if write:
        oracle.cache_write(wl.k_new, wl.v_new, wl.slot_mapping, kc, vc,
                           block_size=wl.block_size, dtype=wl.dtype)
    out = oracle.paged_decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale,
                              dtype=wl.dtype, num_threads=THREADS)
    return kc, vc, out


def _no_device_error():
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0, f"device error bits {bits}"


# ------------------------------------------------------------------ byte moves
@pytest.mark.parametrize("maker", [W.tiny, W.llama_b16,
                                   lambda: W.random_small(31, batch=9, num_q_heads=8,
                                                          num_kv_heads=2, head_dim=128,
                                                          max_ctx=70, dtype=W.DTYPE_BF16)])
def test_cache_write_bit_exact(maker):
    wl = maker()
    d = DeviceWorkload(wl)
    d.cache_write()
    torch.cuda.synchronize()
    _no_device_error()
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    oracle.cache_write(wl.k_new, wl.v_new, wl.slot_mapping, kc, vc, block_size=wl.block_size,
                       dtype=wl.dtype)
    assert host(d.k_cache, kc).tobytes() == kc.tobytes()
    assert host(d.v_cache, vc).tobytes() == vc.tobytes()


def test_cache_write_padding_and_bad_slot():
    wl = W.random_small(32, batch=6, num_q_heads=4, num_kv_heads=2, head_dim=64, max_ctx=40,
                        dtype=W.DTYPE_F16)
    slots = wl.slot_mapping.copy()
    slots[1] = -1
    slots[4] = wl.num_blocks * wl.block_size + 3            # out of the pool
    d = DeviceWorkload(wl)
    d.slot_mapping = dev(slots)
    d.cache_write()
    st, bits = P.photon_get_last_device_error()
    assert st == 6 and bits & 2
    good = slots.copy()
    good[4] = -1
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    oracle.cache_write(wl.k_new, wl.v_new, good, kc, vc, block_size=wl.block_size)
    assert host(d.k_cache, kc).tobytes() == kc.tobytes()
    assert host(d.v_cache, vc).tobytes() == vc.tobytes()
    _no_device_error()   # the word was cleared by the read above


@pytest.mark.parametrize("maker", [W.tiny, lambda: W.sweep(4),
                                   lambda: W.random_small(33, batch=5, num_q_heads=8,
                                                          num_kv_heads=8, head_dim=128,
                                                          max_ctx=65, dtype=W.DTYPE_F32,
                                                          context_lens=[0, 1, 16, 17, 65])])
def test_gather_bit_exact(maker):
    wl = maker()
    d = DeviceWorkload(wl)
    span = wl.max_blocks_per_seq * wl.block_size
    dense_shape = (wl.num_seqs, wl.num_kv_heads, span, wl.head_dim)
    kd = torch.full(dense_shape, 7, dtype=d.k_cache.dtype, device="cuda")
    vd = torch.full(dense_shape, 7, dtype=d.k_cache.dtype, device="cuda")
    P.photon_paged_gather(d.k_cache, d.v_cache, d.block_tables, d.context_lens, kd, vd, d.shape)
    torch.cuda.synchronize()
    _no_device_error()
    rk, rv = oracle.gather(wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                           dtype=wl.dtype)
    assert host(kd, rk).tobytes() == rk.tobytes()
    assert host(vd, rv).tobytes() == rv.tobytes()


# ------------------------------------------------------------------ decode
CASES = {
    "tiny": W.tiny,
    "llama_b16": W.llama_b16,
    "sweep_b4": lambda: W.sweep(4),
    "sweep_b8": lambda: W.sweep(8),
    "sweep_b16": lambda: W.sweep(16),
    "sweep_b32": lambda: W.sweep(32),
    "qwen_b8_small_pool": lambda: W.qwen_b64(seed=7, batch=8, num_blocks=3000),
    "edges_g1_d128_f16": lambda: W.random_small(41, batch=10, num_q_heads=4, num_kv_heads=4,
                                                head_dim=128, max_ctx=600, dtype=W.DTYPE_F16,
                                                context_lens=[0, 1, 15, 16, 17, 255, 256,
                                                              257, 513, 600]),
    "edges_g8_d64_f16": lambda: W.random_small(42, batch=6, num_q_heads=16, num_kv_heads=2,
                                               head_dim=64, max_ctx=1100, dtype=W.DTYPE_F16,
                                               context_lens=[1, 32, 48, 1024, 1025, 1100]),
    "g2_d128_bf16": lambda: W.random_small(43, batch=7, num_q_heads=16, num_kv_heads=8,
                                           head_dim=128, max_ctx=900, dtype=W.DTYPE_BF16),
    "g4_d64_bf16": lambda: W.random_small(44, batch=7, num_q_heads=8, num_kv_heads=2,
                                          head_dim=64, max_ctx=900, dtype=W.DTYPE_BF16),
    "g8_d128_f32": lambda: W.random_small(45, batch=4, num_q_heads=8, num_kv_heads=1,
                                          head_dim=128, max_ctx=700, dtype=W.DTYPE_F32),
    "g1_d64_f32": lambda: W.random_small(46, batch=5, num_q_heads=3, num_kv_heads=3,
                                         head_dim=64, max_ctx=300, dtype=W.DTYPE_F32),
    # more sequences than the producer caches (512): its walk reads the later
    # 32-sequence windows from global memory
    "b600_g4_d64_f16": lambda: W.random_small(47, batch=600, num_q_heads=8, num_kv_heads=2,
                                              head_dim=64, max_ctx=120, dtype=W.DTYPE_F16),
    "b1100_g2_d128_bf16": lambda: W.random_small(48, batch=1100, num_q_heads=4,
                                                 num_kv_heads=2, head_dim=128, max_ctx=90,
                                                 dtype=W.DTYPE_BF16),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_step_matches_oracle(name, consumer):
    """cache write + decode in one stream, against the oracle's step."""
    wl = CASES[name]()
    kc, vc, want = _oracle_step_cached(name, wl)
    d = DeviceWorkload(wl)
    d.cache_write()
    d.decode()
    torch.cuda.synchronize()
    _no_device_error()
    assert host(d.k_cache, kc).tobytes() == kc.tobytes()
    assert_close(d.out_f64(), want, wl.dtype, name)


@pytest.mark.parametrize("name", sorted(CASES) + ["qwen_b64", "mix_b256"])
def test_fused_step_matches_oracle_and_separate_calls(name, consumer):
    """photon_paged_decode_step == cache write then decode: output against the
    oracle, the written rows bit for bit, and bit-identical to the two
    separate calls."""
    wl = {"qwen_b64": W.qwen_b64, "mix_b256": W.mix_b256}.get(name, CASES.get(name))()
    kc, vc, want = _oracle_step_cached(name, wl)
    fused = DeviceWorkload(wl)
    fused.step()
    sep = DeviceWorkload(wl)
    sep.cache_write()
    sep.decode()
    torch.cuda.synchronize()
    _no_device_error()
    assert_close(fused.out_f64(), want, wl.dtype, name)
    assert fused.out.view(torch.int16).equal(sep.out.view(torch.int16))
    live = wl.slot_mapping >= 0
    blk = wl.slot_mapping[live] // wl.block_size
    off = wl.slot_mapping[live] % wl.block_size
    ib, io = torch.from_numpy(blk).cuda(), torch.from_numpy(off).cuda()
    for dev_pool, host_pool in ((fused.k_cache, kc), (fused.v_cache, vc)):
        got = dev_pool[ib, :, io].cpu().numpy()
        assert got.tobytes() == host_pool[blk, :, off].tobytes()
    if wl.k_cache.nbytes < (64 << 20):   # small pools: every other byte unchanged too
        assert host(fused.k_cache, kc).tobytes() == kc.tobytes()
        assert host(fused.v_cache, vc).tobytes() == vc.tobytes()


def test_fused_step_flags_a_slot_that_disagrees_with_the_table(consumer):
    wl = W.random_small(56, batch=4, num_q_heads=8, num_kv_heads=2, head_dim=64, max_ctx=70,
                        dtype=W.DTYPE_F16, context_lens=[20, 33, 64, 70], extra_blocks=4)
    slots = wl.slot_mapping.copy()
    slots[2] = slots[2] - 1                      # not the slot of position ctx-1
    d = DeviceWorkload(wl)
    d.slot_mapping = dev(slots)
    d.step()
    st, bits = P.photon_get_last_device_error()
    assert st == 6 and bits & 2
    # sequence 2 attends over the cache as it was; the others over their new rows
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    good = wl.slot_mapping.copy()
    good[2] = -1
    oracle.cache_write(wl.k_new, wl.v_new, good, kc, vc, block_size=wl.block_size)
    want = oracle.paged_decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale,
                               dtype=wl.dtype)
    assert_close(d.out_f64(), want, wl.dtype)
    assert host(d.k_cache, kc).tobytes() == kc.tobytes()


@pytest.mark.parametrize("part", [16, 32, 48, 128, 512, 4096])
def test_partition_size_invariance(part, consumer):
    wl = W.random_small(51, batch=6, num_q_heads=16, num_kv_heads=8, head_dim=128,
                        max_ctx=1500, dtype=W.DTYPE_F16,
                        context_lens=[1, 16, 100, 777, 1024, 1500])
    _, _, want = _oracle_step(wl, write=False)
    d = DeviceWorkload(wl, partition_size=part)
    d.decode()
    torch.cuda.synchronize()
    _no_device_error()
    assert_close(d.out_f64(), want, wl.dtype, f"part={part}")


@pytest.mark.parametrize("dtype", [W.DTYPE_F16, W.DTYPE_BF16, W.DTYPE_F32])
def test_one_token_context_is_v_exactly(dtype, consumer):
    wl = W.random_small(52, batch=4, num_q_heads=8, num_kv_heads=2, head_dim=64, max_ctx=1,
                        dtype=dtype, context_lens=[1, 1, 1, 1])
    d = DeviceWorkload(wl)
    d.decode()
    got = host(d.out, wl.q)
    for b in range(4):
        blk = wl.block_tables[b, 0]
        for h in range(8):
            assert got[b, h].tobytes() == wl.v_cache[blk, h // 4, 0].tobytes()


def test_zero_context_rows_are_zero_and_repeat_is_stable(consumer):
    wl = W.random_small(53, batch=5, num_q_heads=4, num_kv_heads=1, head_dim=64, max_ctx=300,
                        dtype=W.DTYPE_F16, context_lens=[0, 300, 0, 17, 0])
    _, _, want = _oracle_step(wl, write=False)
    d = DeviceWorkload(wl, partition_size=64)
    d.decode()
    first = d.out.clone()
    d.decode()                    # workspace reused, now holding the last call's data
    torch.cuda.synchronize()
    assert first.view(torch.int16).equal(d.out.view(torch.int16))
    got = d.out_f64()
    assert (got[[0, 2, 4]] == 0).all()
    assert_close(got, want, wl.dtype)


@pytest.mark.parametrize("maker", [W.qwen_b64, W.mix_b256])
def test_fresh_and_reused_workspace_agree_bitwise(maker, consumer):
    """A fresh workspace hands items out in a fixed order, a reused one through
    the work queue; every item is computed the same way, so the outputs must be
    identical bit for bit, call after call."""
    wl = maker()
    d = DeviceWorkload(wl)
    d.decode()
    first = d.out.clone()
    for _ in range(3):
        d.decode()
        assert first.view(torch.int16).equal(d.out.view(torch.int16))
    d.ws.fill_(0x5A)          # scribble over the workspace: back to the fixed order
    d.decode()
    assert first.view(torch.int16).equal(d.out.view(torch.int16))
    _no_device_error()


def test_uniform_scores_give_mean_of_v(consumer):
    wl = W.random_small(54, batch=3, num_q_heads=8, num_kv_heads=2, head_dim=128, max_ctx=700,
                        dtype=W.DTYPE_F16, context_lens=[5, 333, 700])
    d = DeviceWorkload(wl)
    d.decode(scale=0.0)
    dense_k, dense_v = oracle.gather(wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens)
    got = d.out_f64()
    for b, c in enumerate(wl.context_lens):
        for h in range(8):
            mean = dense_v[b, h // 4, :c].astype(np.float64).mean(axis=0)
            assert np.abs(got[b, h] - mean).max() <= 2e-3


def test_bad_block_and_context_are_flagged_not_faulted(consumer):
    wl = W.random_small(55, batch=4, num_q_heads=4, num_kv_heads=2, head_dim=64, max_ctx=90,
                        dtype=W.DTYPE_F16, context_lens=[40, 90, 33, 50])
    _, _, want = _oracle_step(wl, write=False)
    tables = wl.block_tables.copy()
    tables[1, 2] = wl.num_blocks + 5          # bad physical block in sequence 1
    ctx = wl.context_lens.copy()
    ctx[2] = wl.max_blocks_per_seq * wl.block_size + 1   # bad length in sequence 2
    d = DeviceWorkload(wl)
    d.block_tables = dev(tables)
    d.context_lens = dev(ctx)
    d.decode()
    st, bits = P.photon_get_last_device_error()
    assert st == 6 and bits & 1 and bits & 4
    got = d.out_f64()
    assert np.isfinite(got).all()
    assert (got[2] == 0).all()
    assert_close(got[[0, 3]], want[[0, 3]], wl.dtype)
    _no_device_error()


def test_nonzero_stream_and_unreferenced_blocks_untouched(consumer):
    wl = W.llama_b16()
    d = DeviceWorkload(wl)
    s = torch.cuda.Stream()
    k_before = d.k_cache.clone()
    with torch.cuda.stream(s):
        d.decode(stream=s)
    s.synchronize()
    assert k_before.view(torch.int16).equal(d.k_cache.view(torch.int16))   # bytes: NaN-safe
    _, _, want = _oracle_step(wl, write=False)
    assert_close(d.out_f64(), want, wl.dtype)


# ------------------------------------------------------------------ full-size workloads
def test_qwen_b64_full_size_step(consumer):
    """Batch 64, 16q/8kv, d=128, contexts log-uniform 128..8192, 40 000-block
    pool: the benchmark's workload and launch configuration, every output row
    against the oracle."""
    wl = W.qwen_b64()
    kc, vc, want = _oracle_step_cached("qwen_b64", wl)
    d = DeviceWorkload(wl)
    d.cache_write()
    d.decode()
    torch.cuda.synchronize()
    _no_device_error()
    err = assert_close(d.out_f64(), want, wl.dtype, "qwen_b64")
    assert err < 2e-3
    # the written rows, bit for bit (only the touched slots: the pool is 2.6 GB)
    slots = wl.slot_mapping
    blk, off = slots // wl.block_size, slots % wl.block_size
    got_k = d.k_cache[torch.from_numpy(blk).cuda(), :, torch.from_numpy(off).cuda()]
    assert got_k.cpu().numpy().tobytes() == kc[blk, :, off].tobytes()


def test_mix_b256_full_size_step(consumer):
    """Batch 256 continuous-batching step: 256 rows into free-list slots, then
    decode, one stream; all rows against the oracle."""
    wl = W.mix_b256()
    _, _, want = _oracle_step_cached("mix_b256", wl)
    d = DeviceWorkload(wl)
    d.cache_write()
    d.decode()
    torch.cuda.synchronize()
    _no_device_error()
    assert_close(d.out_f64(), want, wl.dtype, "mix_b256")
