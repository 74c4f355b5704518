"""GPU parity of the decode step with the rotary embedding fused in
(photon_rope_cos_sin + photon_paged_decode_step_rope) against the fp64 oracle.

* the cos/sin table: each entry within one fp32 ulp of the double value;
* the output: the decode tolerances of the plain step (2e-3 fp16, 1e-4 fp32,
  2^-8 relative + 2e-4 bf16) against the oracle's RoPE step, whose rotated q
  rows stay in double;
* the stored K rows: within one storage ulp of the oracle's rotated-and-rounded
  rows plus the fp32 arithmetic error of the rotation (the kernel rotates in
  fp32, the oracle in double; both round to nearest even once); V rows and
  every other byte of the pool unchanged, bit for bit;
* a position beyond the table: flagged with device error bit 16, that
  sequence handled unrotated, the others rotated.

Each step test runs on both attention consumers (CUDA cores, tensor cores).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_photon_gb300 as P
import workloads as W
from gpu_util import DeviceWorkload, assert_close, rope_table

pytestmark = pytest.mark.gpu
THREADS = max(1, min(32, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    P.build()
    torch.cuda.init()
    st, _ = P.photon_get_last_device_error()
    assert st == 0


def _widen(a: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == W.DTYPE_BF16:
        return (a.view(np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(
            np.float64)
    return a.astype(np.float64)


def _storage_ulp(x: np.ndarray, dtype: int) -> np.ndarray:
    """Spacing of the storage type at |x| (bf16: fp32 spacing times 2^16)."""
    ax = np.abs(x)
    if dtype == W.DTYPE_F16:
        return np.spacing(ax.astype(np.float16)).astype(np.float64)
    sp = np.spacing(ax.astype(np.float32)).astype(np.float64)
    return sp * 65536.0 if dtype == W.DTYPE_BF16 else sp


def _assert_rotated_rows_close(got: np.ndarray, want: np.ndarray, k_in: np.ndarray,
                               dtype: int) -> None:
    """Each stored element y of a pair (x0, x1) may differ from the oracle's by
    one storage ulp (both round once, from fp32 vs double arithmetic) plus the
    fp32 arithmetic error of the rotation, at most a few 2^-24 (|x0| + |x1|)
    from the table's rounding, two products and one sum; 2^-21 (|x0| + |x1|)
    bounds it."""
    g, w, x = _widen(got, dtype), _widen(want, dtype), _widen(k_in, dtype)
    h = x.shape[-1] // 2
    pair = np.abs(x[..., :h]) + np.abs(x[..., h:])
    pair = np.concatenate([pair, pair], axis=-1)
    bound = _storage_ulp(w, dtype) + 2.0 ** -21 * pair
    excess = np.abs(g - w) - bound
    assert excess.max(initial=-1.0) <= 0, f"stored K row off by {excess.max()} beyond the bound"


@pytest.mark.parametrize("base,max_pos,d", [(1e4, 64, 64), (1e6, 8192, 128), (5e5, 300, 128)])
def test_cos_sin_table_within_one_fp32_ulp(base, max_pos, d):
    t = rope_table(base, max_pos, d).cpu().numpy().astype(np.float64)
    want = oracle.rope_cos_sin(base, max_pos, d)
    ulp = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
    assert (np.abs(t - want) <= ulp).all()


CASES = {
    "g2_d128_f16": lambda: W.random_small(81, batch=9, num_q_heads=16, num_kv_heads=8,
                                          head_dim=128, max_ctx=900, dtype=W.DTYPE_F16),
    "g4_d64_f16": lambda: W.random_small(82, batch=7, num_q_heads=8, num_kv_heads=2,
                                         head_dim=64, max_ctx=700, dtype=W.DTYPE_F16,
                                         context_lens=[1, 2, 16, 17, 385, 700, 699]),
    "g2_d128_bf16": lambda: W.random_small(83, batch=7, num_q_heads=16, num_kv_heads=8,
                                           head_dim=128, max_ctx=900, dtype=W.DTYPE_BF16),
    "g8_d64_bf16": lambda: W.random_small(84, batch=5, num_q_heads=16, num_kv_heads=2,
                                          head_dim=64, max_ctx=500, dtype=W.DTYPE_BF16),
    "g1_d128_f32": lambda: W.random_small(85, batch=5, num_q_heads=4, num_kv_heads=4,
                                          head_dim=128, max_ctx=400, dtype=W.DTYPE_F32),
    "g4_d64_f32": lambda: W.random_small(86, batch=5, num_q_heads=8, num_kv_heads=2,
                                         head_dim=64, max_ctx=400, dtype=W.DTYPE_F32,
                                         context_lens=[0, 1, 64, 65, 400]),
}


_ORACLE = {}


def _rope_oracle(key, wl: W.Workload, base: float):
    if key not in _ORACLE:
        _ORACLE[key] = oracle.rope_step(wl, base, THREADS)
    return _ORACLE[key]


def _check_rows(dwl: DeviceWorkload, kc: np.ndarray, vc: np.ndarray, wl: W.Workload,
                small_pool: bool) -> None:
    live = (wl.slot_mapping >= 0) & (wl.context_lens > 0)
    blk = wl.slot_mapping[live] // wl.block_size
    off = wl.slot_mapping[live] % wl.block_size
    ib, io = torch.from_numpy(blk).cuda(), torch.from_numpy(off).cuda()
    got_k = dwl.k_cache[ib, :, io].cpu().numpy().view(kc.dtype)
    got_v = dwl.v_cache[ib, :, io].cpu().numpy().view(vc.dtype)
    _assert_rotated_rows_close(got_k, kc[blk, :, off], wl.k_new[live], wl.dtype)
    assert got_v.tobytes() == vc[blk, :, off].tobytes()
    if small_pool:
        # every byte outside the new rows is the input pool's
        k_all = dwl.k_cache.cpu().numpy().view(kc.dtype).copy()
        k_all[blk, :, off] = kc[blk, :, off]
        assert k_all.tobytes() == kc.tobytes()
        assert dwl.v_cache.cpu().numpy().view(vc.dtype).tobytes() == vc.tobytes()


@pytest.mark.parametrize("base", [1e4, 1e6])
@pytest.mark.parametrize("name", sorted(CASES))
def test_rope_step_matches_oracle(name, base, consumer):
    wl = CASES[name]()
    kc, vc, want = _rope_oracle((name, base), wl, base)
    d = DeviceWorkload(wl)
    max_pos = int(wl.context_lens.max()) + 1
    table = rope_table(base, max_pos, wl.head_dim)
    d.step_rope(table, max_pos)
    torch.cuda.synchronize()
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0, bits
    assert_close(d.out_f64(), want, wl.dtype, name)
    _check_rows(d, kc, vc, wl, small_pool=True)


def test_rope_step_qwen_b64_full_size(consumer):
    """The benchmark's batch-64 workload (contexts up to 8192, 40 000-block
    pool) with a Qwen-style base of 10^6, every output row against the oracle."""
    wl = W.qwen_b64()
    kc, vc, want = _rope_oracle(("qwen_b64", 1e6), wl, 1e6)
    d = DeviceWorkload(wl)
    table = rope_table(1e6, 8192, wl.head_dim)
    d.step_rope(table, 8192)
    torch.cuda.synchronize()
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0, bits
    assert_close(d.out_f64(), want, wl.dtype, "qwen_b64 rope")
    _check_rows(d, kc, vc, wl, small_pool=False)


def test_position_beyond_the_table_is_flagged_and_left_unrotated(consumer):
    wl = W.random_small(87, batch=4, num_q_heads=8, num_kv_heads=2, head_dim=128, max_ctx=300,
                        dtype=W.DTYPE_F16, context_lens=[10, 100, 200, 300])
    max_pos = 150          # positions 199 and 299 are outside the table
    d = DeviceWorkload(wl)
    d.step_rope(rope_table(1e4, max_pos, 128), max_pos)
    st, bits = P.photon_get_last_device_error()
    assert st == 6 and bits == 16, bits
    _, _, rot = oracle.rope_step(wl, 1e4)
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    oracle.cache_write(wl.k_new, wl.v_new, wl.slot_mapping, kc, vc, block_size=wl.block_size,
                       dtype=wl.dtype)
    plain = oracle.paged_decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale,
                                dtype=wl.dtype)
    got = d.out_f64()
    assert_close(got[:2], rot[:2], wl.dtype, "rotated sequences")
    assert_close(got[2:], plain[2:], wl.dtype, "sequences past the table")
