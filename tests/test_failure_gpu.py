"""Failure detection on the GPU without a GPU fault: a bounded wait is made to
run out on purpose (a barrier phase nothing completes), the kernel reports it
through device error bit 8 and returns, and the context keeps working."""
import time

import pytest
import torch

import oracle
import paged_kv_attention_photon_gb300 as P
import workloads as W
from gpu_util import DeviceWorkload, assert_close

pytestmark = pytest.mark.gpu


def test_expired_wait_sets_bit_8_and_the_context_survives():
    P.build()
    torch.cuda.init()
    st, _ = P.photon_get_last_device_error()
    assert st == 0
    t0 = time.perf_counter()
    P.photon_debug_wait_probe(20_000_000)           # 20 ms bound
    st, bits = P.photon_get_last_device_error()
    elapsed = time.perf_counter() - t0
    assert st == 6 and bits == 8, (st, bits)
    assert elapsed < 5.0
    # the error word was cleared by the read, and the library still computes
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0
    wl = W.tiny()
    d = DeviceWorkload(wl)
    d.cache_write()
    d.decode()
    torch.cuda.synchronize()
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    oracle.cache_write(wl.k_new, wl.v_new, wl.slot_mapping, kc, vc, block_size=wl.block_size,
                       dtype=wl.dtype)
    want = oracle.paged_decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale,
                               dtype=wl.dtype)
    assert_close(d.out_f64(), want, wl.dtype, "after the expired wait")
