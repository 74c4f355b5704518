"""The allocation-free decode entry point against the regular one.

photon_paged_decode_noalloc serves callers that cannot allocate device memory
for the decode (an engine that reserved nearly all of HBM for its KV pool, a
plugin with no allocator, a path that must not call cudaMalloc); it takes its
split-KV scratch from a 32 MiB array built into the library.  Its output must
match photon_paged_decode's, and the fp64 oracle's, within the tolerance the
other decode tests use, on two calls in a row (the second finds the scratch as
the first left it), on both attention consumers.  The first call of the file
finds the array as the process loaded it, zero and without the guard word the
merge kernel leaves, so it takes the fixed work order; the calls after it take
the dynamic queue.
This file is collected last so that a stop-at-first-failure run has already run
every other test when it gets here; it also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

import oracle
import paged_kv_attention_photon_gb300 as P
import workloads as W
from gpu_util import DeviceWorkload, assert_close, to_float64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    P.build()
    torch.cuda.init()


_ORACLE = {}


def _oracle_out(wl: W.Workload):
    """The fp64 oracle's decode after the workload's cache write (computed once
    per workload)."""
    if wl.name not in _ORACLE:
        kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
        oracle.cache_write(wl.k_new, wl.v_new, wl.slot_mapping, kc, vc,
                           block_size=wl.block_size, dtype=wl.dtype)
        _ORACLE[wl.name] = oracle.paged_decode(wl.q, kc, vc, wl.block_tables, wl.context_lens,
                                               wl.scale, dtype=wl.dtype, num_threads=16)
    return _ORACLE[wl.name]


@pytest.mark.parametrize("maker", [W.qwen_b64, W.llama_b16, W.tiny])
def test_noalloc_matches_workspace_entry_point_twice(maker, consumer):
    wl = maker()
    ref = _oracle_out(wl)
    d = DeviceWorkload(wl)
    d.cache_write()
    d.decode()                                   # regular entry point, caller workspace
    torch.cuda.synchronize()
    want = d.out_f64()
    assert_close(want, ref, wl.dtype, f"{wl.name} regular entry point vs oracle")
    lib = P._load()
    for call in range(2):
        out = torch.full_like(d.out, -7)
        st = lib.photon_paged_decode_noalloc(d.q.data_ptr(), d.k_cache.data_ptr(),
                                             d.v_cache.data_ptr(), d.block_tables.data_ptr(),
                                             d.context_lens.data_ptr(), wl.scale,
                                             out.data_ptr(), ctypes.byref(d.shape),
                                             torch.cuda.current_stream().cuda_stream)
        assert st == 0, P.photon_status_string(st)
        torch.cuda.synchronize()
        got = to_float64(out, wl.dtype)
        assert_close(got, want, wl.dtype, f"{wl.name} call {call} vs regular entry point")
        assert_close(got, ref, wl.dtype, f"{wl.name} call {call} vs oracle")
    status, bits = P.photon_get_last_device_error()
    assert status == 0 and bits == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 4096 sequences x 32 q heads x 16 partitions x (128 + 2) floats >> 32 MiB
    shape = P.PagedShape.make(num_seqs=4096, num_q_heads=32, num_kv_heads=8, head_dim=128,
                              num_blocks=1, max_blocks_per_seq=256, dtype=P.F16,
                              partition_size=256)
    assert P.photon_paged_decode_workspace_size(shape) > (32 << 20)
    fake = 1 << 20   # never dereferenced: the size check comes first
    st = P._load().photon_paged_decode_noalloc(fake, fake, fake, fake, fake, 0.1, fake,
                                                ctypes.byref(shape), None)
    assert st == 4   # PHOTON_ERR_WORKSPACE
