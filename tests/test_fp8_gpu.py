"""GPU parity of the e4m3 (fp8) KV cache through the C ABI against the fp64
oracle.

* photon_cache_write_fp8: the stored codes bit for bit (round to nearest
  even of x * (1 / scale) in fp32, saturating at 448), padding and an
  out-of-range slot included, every other pool byte unchanged;
* photon_paged_decode_fp8: max-abs error <= 2e-3 against the oracle's
  decode over the dequantised values (codes widen exactly to fp16, scores and
  sums in fp32, out rounded to fp16) on every group size, d = 64 and 128,
  ragged and edge lengths, forced partitions, NaN codes in every unreferenced
  block, the full-size batch-64 long-context shape; a one-token context
  returns its V row exactly; bad blocks and lengths are flagged, not faulted.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_photon_gb300 as P
import workloads as W
from gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu
THREADS = max(1, min(32, os.cpu_count() or 1))
KS, VS = W.FP8_K_SCALE, W.FP8_V_SCALE


@pytest.fixture(scope="module", autouse=True)
def _lib():
    P.build()
    torch.cuda.init()
    st, _ = P.photon_get_last_device_error()
    assert st == 0


def _decode(wl, k8, v8, partition=0, context_lens=None, block_tables=None):
    shape = P.PagedShape.make(partition_size=partition, **wl.shape_dict())
    nws = P.photon_paged_decode_fp8_workspace_size(shape)
    ws = torch.full((max(nws, 16),), 0xFF, dtype=torch.uint8, device="cuda")
    q = dev(wl.q)
    out = torch.full(q.shape, -1, dtype=torch.float16, device="cuda")
    ctx = wl.context_lens if context_lens is None else context_lens
    bt = wl.block_tables if block_tables is None else block_tables
    P.photon_paged_decode_fp8(q, dev(k8), dev(v8), dev(bt), dev(ctx), wl.scale, KS, VS, out,
                              ws, nws, shape)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def _want(wl, k8, v8):
    return oracle.paged_decode_fp8(wl.q, k8, v8, wl.block_tables, wl.context_lens, wl.scale,
                                   KS, VS, num_threads=THREADS)


def test_cache_write_fp8_bit_exact():
    wl = W.random_small(71, batch=9, num_q_heads=16, num_kv_heads=8, head_dim=128,
                        max_ctx=200, dtype=W.DTYPE_F16, extra_blocks=6)
    k8, v8 = W.fp8_cache(wl, 1)
    # rows of several magnitudes, one beyond the saturation point after scaling
    k_new = (wl.k_new.astype(np.float32) * 3.0).astype(np.float16)
    k_new[0, 0, :4] = np.array([300.0, -250.0, 1e-4, 0.0], np.float16)
    slots = wl.slot_mapping.copy()
    slots[3] = -1                                      # padding row
    kd, vd = dev(k8), dev(v8)
    shape = P.PagedShape.make(**wl.shape_dict())
    P.photon_cache_write_fp8(dev(k_new), dev(wl.v_new), dev(slots), slots.shape[0], kd, vd,
                             KS, VS, shape)
    torch.cuda.synchronize()
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0, bits
    want_k, want_v = k8.copy(), v8.copy()
    oracle.cache_write_fp8(k_new, wl.v_new, slots, want_k, want_v, KS, VS, block_size=16)
    assert np.array_equal(kd.cpu().numpy(), want_k)
    assert np.array_equal(vd.cpu().numpy(), want_v)


def test_cache_write_fp8_flags_a_slot_past_the_pool():
    wl = W.random_small(72, batch=4, num_q_heads=8, num_kv_heads=2, head_dim=64, max_ctx=50,
                        dtype=W.DTYPE_F16)
    k8, v8 = W.fp8_cache(wl, 2)
    slots = wl.slot_mapping.copy()
    slots[1] = wl.num_blocks * 16 + 3
    kd, vd = dev(k8), dev(v8)
    shape = P.PagedShape.make(**wl.shape_dict())
    P.photon_cache_write_fp8(dev(wl.k_new), dev(wl.v_new), dev(slots), slots.shape[0], kd, vd,
                             KS, VS, shape)
    st, bits = P.photon_get_last_device_error()
    assert st == 6 and bits & 2
    want_k, want_v = k8.copy(), v8.copy()
    good = slots.copy()
    good[1] = -1
    oracle.cache_write_fp8(wl.k_new, wl.v_new, good, want_k, want_v, KS, VS, block_size=16)
    assert np.array_equal(kd.cpu().numpy(), want_k)


CASES = {
    "g1_d128": dict(seed=81, num_q_heads=4, num_kv_heads=4, head_dim=128, max_ctx=600,
                    context_lens=[0, 1, 15, 16, 17, 255, 256, 257, 513, 600]),
    "g2_d128": dict(seed=82, num_q_heads=16, num_kv_heads=8, head_dim=128, max_ctx=1500,
                    context_lens=[1, 16, 100, 777, 1024, 1500, 33]),
    "g4_d64": dict(seed=83, num_q_heads=32, num_kv_heads=8, head_dim=64, max_ctx=900,
                   context_lens=None, batch=11),
    "g8_d64": dict(seed=84, num_q_heads=16, num_kv_heads=2, head_dim=64, max_ctx=1100,
                   context_lens=[1, 32, 48, 1024, 1025, 1100]),
    "g8_d128": dict(seed=85, num_q_heads=64, num_kv_heads=8, head_dim=128, max_ctx=700,
                    context_lens=[5, 333, 700, 64]),
}


def _case(name):
    c = dict(CASES[name])
    seed = c.pop("seed")
    batch = c.pop("batch", None) or len(c["context_lens"])
    wl = W.random_small(seed, batch=batch, dtype=W.DTYPE_F16, **c)
    k8, v8 = W.fp8_cache(wl, seed)
    return wl, k8, v8


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("partition", [0, 64])
def test_decode_fp8_matches_oracle(name, partition):
    wl, k8, v8 = _case(name)
    got = _decode(wl, k8, v8, partition=partition)
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0, bits
    assert_close(got, _want(wl, k8, v8), W.DTYPE_F16, f"fp8 {name} part {partition}")
    assert (got[wl.context_lens == 0] == 0).all()


def test_one_token_context_is_v_exactly():
    wl = W.random_small(86, batch=4, num_q_heads=8, num_kv_heads=2, head_dim=64, max_ctx=1,
                        dtype=W.DTYPE_F16, context_lens=[1, 1, 1, 1])
    k8, v8 = W.fp8_cache(wl, 86)
    got = _decode(wl, k8, v8)
    for b in range(4):
        blk = wl.block_tables[b, 0]
        for h in range(8):
            want = (oracle.e4m3_decode(v8[blk, h // 4, 0]) * VS).astype(np.float16)
            assert np.array_equal(got[b, h].astype(np.float16), want)


def test_bad_block_and_context_are_flagged_not_faulted():
    wl = W.random_small(87, batch=4, num_q_heads=8, num_kv_heads=2, head_dim=128, max_ctx=90,
                        dtype=W.DTYPE_F16, context_lens=[40, 90, 33, 50])
    k8, v8 = W.fp8_cache(wl, 87)
    want = _want(wl, k8, v8)
    tables = wl.block_tables.copy()
    tables[1, 2] = wl.num_blocks + 5
    ctx = wl.context_lens.copy()
    ctx[2] = wl.max_blocks_per_seq * 16 + 1
    got = _decode(wl, k8, v8, context_lens=ctx, block_tables=tables)
    st, bits = P.photon_get_last_device_error()
    assert st == 6 and bits & 1 and bits & 4
    assert np.isfinite(got).all()
    assert (got[2] == 0).all()
    assert_close(got[[0, 3]], want[[0, 3]], W.DTYPE_F16)


def test_qwen_shaped_batch_full_size():
    """64 sequences, 16q/8kv, d = 128, contexts log-uniform 128..8192, a
    40 000-block e4m3 pool: every output row against the oracle."""
    wl = W.qwen_b64()
    k8, v8 = W.fp8_cache(wl, 2)
    got = _decode(wl, k8, v8)
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0, bits
    assert_close(got, _want(wl, k8, v8), W.DTYPE_F16, "fp8 qwen_b64")
