"""Pins for the fp64 CPU oracle, checked against things other than itself.

Each test ties the oracle to mathematics the PhotonInfer README's paged
attention implies ("Key features: GPU-optimized kernels" -- batched paged
attention, numerically stable softmax; "Technical details: paged attention" --
block-wise KV cache, per-sequence offsets, batched cache write):

* a dense, unpaged attention computed with torch on CPU in float64 (a library
  softmax on a layout the test builds itself);
* closed-form golden fixtures (tests/golden/*.json);
* invariants: physical block permutation, one-token context, uniform scores,
  score shift, split/merge by log-sum-exp, threads;
* brute force for the byte moves (cache write, gather).

No GPU is needed.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------- test-side helpers
def _to_f64(a: np.ndarray, dtype: int) -> np.ndarray:
    """Widen stored values with numpy only (independent of the oracle's decoder)."""
    if dtype == W.DTYPE_BF16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _draw(rng, shape, dtype):
    x = rng.standard_normal(shape).astype(np.float32)
    if dtype == W.DTYPE_F32:
        return x
    if dtype == W.DTYPE_F16:
        return x.astype(np.float16)
    b = x.view(np.uint32)
    return ((b + np.uint32(0x7FFF) + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _page(dense_k, dense_v, ctx, bs, rng, spare=3, mbs=None, poison=True):
    """Scatter per-sequence dense K/V [B][Hkv][S][d] into a shuffled paged pool.

    Written independently of the oracle: a fresh random permutation hands out
    physical blocks; everything not owned is NaN (or zero if poison=False)."""
    B, Hkv, S, d = dense_k.shape
    nblk = [(int(c) + bs - 1) // bs for c in ctx]
    NB = sum(nblk) + spare
    mbs = mbs or max(1, max(nblk))
    perm = rng.permutation(NB)
    tables = np.full((B, mbs), -1, np.int32)
    fill = np.nan if poison else 0.0
    kc = np.full((NB, Hkv, bs, d), fill, dtype=dense_k.dtype) if dense_k.dtype != np.uint16 else \
        np.full((NB, Hkv, bs, d), 0x7FC0 if poison else 0, np.uint16)
    vc = kc.copy()
    pos = 0
    for b in range(B):
        for i in range(nblk[b]):
            blk = int(perm[pos]); pos += 1
            tables[b, i] = blk
            for off in range(bs):
                j = i * bs + off
                if j < ctx[b]:
                    kc[blk, :, off, :] = dense_k[b, :, j, :]
                    vc[blk, :, off, :] = dense_v[b, :, j, :]
    return kc, vc, tables


def _torch_dense_attention(q64, k64, v64, ctx, scale, G):
    """softmax(q K^T * scale) V with torch float64 on CPU; GQA by repeat_interleave."""
    B, Hq, d = q64.shape
    out = np.zeros((B, Hq, d))
    for b in range(B):
        c = int(ctx[b])
        if c == 0:
            continue
        K = torch.from_numpy(k64[b, :, :c, :]).repeat_interleave(G, dim=0)   # [Hq][c][d]
        V = torch.from_numpy(v64[b, :, :c, :]).repeat_interleave(G, dim=0)
        q = torch.from_numpy(q64[b]).unsqueeze(1)                          # [Hq][1][d]
        att = torch.softmax(torch.matmul(q, K.transpose(1, 2)) * scale, dim=-1)
        out[b] = torch.matmul(att, V).squeeze(1).numpy()
    return out


def _decode_wl(wl: W.Workload, **kw):
    return oracle.paged_decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                               wl.scale, dtype=wl.dtype, **kw)


# --------------------------------------------------------------- dense reference
@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_F16, W.DTYPE_BF16])
@pytest.mark.parametrize("Hq,Hkv,d,bs", [(4, 1, 64, 16), (8, 2, 16, 16), (6, 3, 8, 4),
                                         (16, 8, 32, 16), (2, 2, 8, 8)])
def test_decode_equals_dense_torch_attention(dtype, Hq, Hkv, d, bs):
    rng = np.random.default_rng(1000 + Hq * 7 + d + bs + dtype)
    ctx = np.array([1, bs - 1, bs, bs + 1, 3 * bs + 5, 0], np.int32)
    B, S = len(ctx), int(ctx.max())
    dk = _draw(rng, (B, Hkv, S, d), dtype)
    dv = _draw(rng, (B, Hkv, S, d), dtype)
    q = _draw(rng, (B, Hq, d), dtype)
    kc, vc, tables = _page(dk, dv, ctx, bs, rng)
    scale = 0.7 / math.sqrt(d)
    got = oracle.paged_decode(q, kc, vc, tables, ctx, scale, dtype=dtype)
    want = _torch_dense_attention(_to_f64(q, dtype), _to_f64(dk, dtype), _to_f64(dv, dtype),
                                  ctx, scale, Hq // Hkv)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


# --------------------------------------------------------------- golden fixtures
def _single_seq(q_row, k_rows, v_rows, bs, dtype=W.DTYPE_F32):
    """One sequence, one q head, one KV head; pool built by the test."""
    k = np.asarray(k_rows, np.float32)
    v = np.asarray(v_rows, np.float32)
    c, d = k.shape
    nb = (c + bs - 1) // bs
    kc = np.zeros((nb + 1, 1, bs, d), np.float32)
    vc = np.zeros_like(kc)
    # put the sequence in blocks 1..nb (block 0 unused, filled with NaN)
    kc[0] = np.nan
    vc[0] = np.nan
    for j in range(c):
        kc[1 + j // bs, 0, j % bs] = k[j]
        vc[1 + j // bs, 0, j % bs] = v[j]
    tables = np.arange(1, nb + 1, dtype=np.int32).reshape(1, nb)
    q = np.asarray(q_row, np.float32).reshape(1, 1, d)
    return q, kc, vc, tables, np.array([c], np.int32)


def test_golden_two_keys_closed_form():
    g = json.load(open(os.path.join(GOLDEN, "two_keys_closed_form.json")))
    q, kc, vc, t, ctx = _single_seq(g["q"], g["k_rows"], g["v_rows"], g["block_size"])
    out = oracle.paged_decode(q, kc, vc, t, ctx, math.log(3.0), dtype=W.DTYPE_F32)
    np.testing.assert_allclose(out[0, 0], g["expected_out"], rtol=0, atol=g["tolerance"])


def test_golden_large_logits_stable():
    g = json.load(open(os.path.join(GOLDEN, "stability_large_logits.json")))
    q, kc, vc, t, ctx = _single_seq(g["q"], g["k_rows"], g["v_rows"], g["block_size"])
    out = oracle.paged_decode(q, kc, vc, t, ctx, g["scale"], dtype=W.DTYPE_F32)
    assert np.all(np.isfinite(out))
    np.testing.assert_array_equal(out[0, 0], np.asarray(g["expected_out"], np.float64))


def test_golden_gqa_head_mapping():
    g = json.load(open(os.path.join(GOLDEN, "gqa_mapping.json")))
    Hq, Hkv, d, bs = g["num_q_heads"], g["num_kv_heads"], g["head_dim"], g["block_size"]
    kc = np.full((2, Hkv, bs, d), np.nan, np.float32)
    vc = np.full((2, Hkv, bs, d), np.nan, np.float32)
    kc[1, :, 0, :] = np.asarray(g["k_heads"], np.float32)
    vc[1, :, 0, :] = np.asarray(g["v_heads"], np.float32)
    q = np.ones((1, Hq, d), np.float32)
    out = oracle.paged_decode(q, kc, vc, np.array([[1]], np.int32), np.array([1], np.int32),
                              0.3, dtype=W.DTYPE_F32)
    np.testing.assert_array_equal(out[0], np.asarray(g["expected_out"], np.float64))


# --------------------------------------------------------------- invariants
@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_F16])
def test_block_permutation_invariance_bit_identical(dtype):
    wl = W.random_small(11, batch=5, num_q_heads=8, num_kv_heads=2, head_dim=64, max_ctx=80,
                        dtype=dtype, extra_blocks=6)
    base = _decode_wl(wl)
    rng = np.random.default_rng(5)
    perm = rng.permutation(wl.num_blocks)          # new position of each old block
    kc = np.empty_like(wl.k_cache)
    vc = np.empty_like(wl.v_cache)
    kc[perm] = wl.k_cache
    vc[perm] = wl.v_cache
    tables = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1)
    tables = tables.astype(np.int32)
    got = oracle.paged_decode(wl.q, kc, vc, tables, wl.context_lens, wl.scale, dtype=dtype)
    np.testing.assert_array_equal(got, base)


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_F16, W.DTYPE_BF16])
def test_one_token_context_returns_v_exactly(dtype):
    wl = W.random_small(12, batch=3, num_q_heads=4, num_kv_heads=2, head_dim=16, max_ctx=1,
                        dtype=dtype, context_lens=[1, 1, 1])
    out = _decode_wl(wl)
    G = wl.group
    for b in range(3):
        blk = wl.block_tables[b, 0]
        for h in range(wl.num_q_heads):
            v = _to_f64(wl.v_cache[blk, h // G, 0], dtype)
            np.testing.assert_array_equal(out[b, h], v)


def test_uniform_scores_give_mean_of_v():
    wl = W.random_small(13, batch=4, num_q_heads=4, num_kv_heads=1, head_dim=32, max_ctx=70,
                        dtype=W.DTYPE_F32, context_lens=[1, 17, 33, 70])
    dense_k, dense_v = oracle.gather(wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens)
    # (a) scale = 0
    out0 = oracle.paged_decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                               0.0, dtype=wl.dtype)
    # (b) q = 0
    qz = np.zeros_like(wl.q)
    outq = oracle.paged_decode(qz, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                               wl.scale, dtype=wl.dtype)
    # (c) every key identical
    kc = wl.k_cache.copy()
    kc[...] = np.float32(0.375)
    outk = oracle.paged_decode(wl.q, kc, wl.v_cache, wl.block_tables, wl.context_lens,
                               wl.scale, dtype=wl.dtype)
    for b, c in enumerate(wl.context_lens):
        mean = dense_v[b, 0, :c, :].astype(np.float64).mean(axis=0)
        for out in (out0, outq, outk):
            for h in range(4):
                np.testing.assert_allclose(out[b, h], mean, rtol=0, atol=1e-13)


def test_score_shift_invariance():
    wl = W.random_small(14, batch=3, num_q_heads=4, num_kv_heads=2, head_dim=32, max_ctx=50,
                        dtype=W.DTYPE_F16, context_lens=[9, 31, 50])
    # fp16 values widened to fp32 are exact, and so is the fp32 sum of two fp16
    # values of this size, so the shifted keys below are exactly K + u.
    q32 = wl.q.astype(np.float32)
    k32 = wl.k_cache.astype(np.float32)
    v32 = wl.v_cache.astype(np.float32)
    base = oracle.paged_decode(q32, k32, v32, wl.block_tables, wl.context_lens, wl.scale,
                               dtype=W.DTYPE_F32)
    # q is shared by a group; shift every key of KV head kvh by u, s_j moves by
    # scale*q.u for every j (constant within each (b, h)) -> output unchanged.
    rng = np.random.default_rng(2)
    u = rng.standard_normal((wl.num_kv_heads, 1, wl.head_dim)).astype(np.float16)
    kc = (k32 + u.astype(np.float32)[None]).astype(np.float32)
    got = oracle.paged_decode(q32, kc, v32, wl.block_tables, wl.context_lens,
                              wl.scale, dtype=W.DTYPE_F32)
    np.testing.assert_allclose(got, base, rtol=0, atol=1e-12)


def test_split_merge_equals_direct_sum():
    wl = W.random_small(15, batch=3, num_q_heads=4, num_kv_heads=2, head_dim=16, max_ctx=120,
                        dtype=W.DTYPE_F16, context_lens=[1, 47, 120])
    direct = _decode_wl(wl)
    for b, c in enumerate(wl.context_lens):
        c = int(c)
        for cuts in ([0, c], [0, 0, c], [0, 1, c], [0, c // 3, 2 * c // 3, c, c],
                     list(range(0, c, 16)) + [c]):
            for h in range(wl.num_q_heads):
                ms, ls, os_ = [], [], []
                for j0, j1 in zip(cuts[:-1], cuts[1:]):
                    m, l, o = oracle.attend_range(wl.q, wl.k_cache, wl.v_cache, wl.block_tables,
                                                  wl.context_lens, wl.scale, b, h, j0, j1,
                                                  dtype=wl.dtype)
                    ms.append(m); ls.append(l); os_.append(o)
                merged = oracle.merge(np.array(ms), np.array(ls), np.stack(os_))
                np.testing.assert_allclose(merged, direct[b, h], rtol=0, atol=1e-12)


def test_merge_closed_form_two_partials():
    # Two partials with maxima 0 and ln 2: weights e^-ln2 and 1 on (l, o).
    m = np.array([0.0, math.log(2.0)])
    l = np.array([1.0, 1.0])
    o = np.array([[2.0, 0.0], [0.0, 4.0]])
    out = oracle.merge(m, l, o)
    # num = 0.5*(2,0) + 1*(0,4) = (1,4); den = 0.5 + 1 = 1.5
    np.testing.assert_allclose(out, [1.0 / 1.5, 4.0 / 1.5], rtol=0, atol=1e-15)
    # an empty partial (l = 0, m = -inf) changes nothing
    out2 = oracle.merge(np.append(m, -np.inf), np.append(l, 0.0), np.vstack([o, [0.0, 0.0]]))
    np.testing.assert_array_equal(out2, out)
    # all empty -> zero
    np.testing.assert_array_equal(oracle.merge([-np.inf], [0.0], [[0.0, 0.0]]), [0.0, 0.0])


def test_zero_context_gives_zeros_and_poison_is_never_read():
    wl = W.random_small(16, batch=4, num_q_heads=4, num_kv_heads=2, head_dim=16, max_ctx=40,
                        dtype=W.DTYPE_F16, context_lens=[0, 5, 0, 40], extra_blocks=4)
    out = _decode_wl(wl)
    assert np.all(np.isfinite(out))           # NaN pool slack never enters
    np.testing.assert_array_equal(out[0], 0.0)
    np.testing.assert_array_equal(out[2], 0.0)
    # sanity: poisoning an owned row does show up, only in that sequence
    kc = wl.k_cache.copy()
    kc[wl.block_tables[1, 0], 0, 2, 3] = np.nan
    bad = oracle.paged_decode(wl.q, kc, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                              dtype=wl.dtype)
    assert np.isnan(bad[1, :2]).all() and np.isfinite(bad[1, 2:]).all()
    np.testing.assert_array_equal(bad[3], out[3])


def test_threads_bit_identical():
    wl = W.random_small(17, batch=7, num_q_heads=8, num_kv_heads=2, head_dim=64, max_ctx=300,
                        dtype=W.DTYPE_F16)
    np.testing.assert_array_equal(_decode_wl(wl, num_threads=1), _decode_wl(wl, num_threads=5))


def test_decode_row_matches_full():
    wl = W.random_small(18, batch=3, num_q_heads=4, num_kv_heads=2, head_dim=32, max_ctx=90,
                        dtype=W.DTYPE_F16)
    full = _decode_wl(wl)
    for b in range(3):
        for h in range(4):
            row = oracle.paged_decode_row(wl.q, wl.k_cache, wl.v_cache, wl.block_tables,
                                          wl.context_lens, wl.scale, b, h, dtype=wl.dtype)
            np.testing.assert_array_equal(row, full[b, h])


def test_widen_matches_numpy():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(4096) * 1000).astype(np.float16)
    x[:4] = [np.float16(6e-8), np.float16(-0.0), np.float16(65504), np.float16(np.inf)]
    np.testing.assert_array_equal(oracle.widen(x), x.astype(np.float64))
    y = rng.standard_normal(512).astype(np.float32)
    bf = (y.view(np.uint32) >> 16).astype(np.uint16)
    np.testing.assert_array_equal(oracle.widen(bf, W.DTYPE_BF16), _to_f64(bf, W.DTYPE_BF16))


def test_bad_inputs_rejected():
    wl = W.random_small(19, batch=2, num_q_heads=4, num_kv_heads=2, head_dim=16, max_ctx=20,
                        dtype=W.DTYPE_F32, context_lens=[20, 3])
    ctx = wl.context_lens.copy()
    ctx[0] = wl.max_blocks_per_seq * wl.block_size + 1
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, ctx, wl.scale)
    tables = wl.block_tables.copy()
    tables[0, 0] = wl.num_blocks
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(wl.q, wl.k_cache, wl.v_cache, tables, wl.context_lens, wl.scale)


# --------------------------------------------------------------- byte moves
@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_F16, W.DTYPE_BF16])
def test_cache_write_brute_force(dtype):
    rng = np.random.default_rng(21 + dtype)
    NB, Hkv, bs, d, T = 9, 3, 8, 16, 12
    kc = _draw(rng, (NB, Hkv, bs, d), dtype)
    vc = _draw(rng, (NB, Hkv, bs, d), dtype)
    kn = _draw(rng, (T, Hkv, d), dtype)
    vn = _draw(rng, (T, Hkv, d), dtype)
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int64)
    slots[[2, 7]] = -1                                        # padding rows
    k0, v0 = kc.copy(), vc.copy()
    oracle.cache_write(kn, vn, slots, kc, vc, block_size=bs, dtype=dtype)
    written = {int(s): t for t, s in enumerate(slots) if s >= 0}
    for blk in range(NB):
        for off in range(bs):
            s = blk * bs + off
            if s in written:
                t = written[s]
                assert kc[blk, :, off].tobytes() == kn[t].tobytes()
                assert vc[blk, :, off].tobytes() == vn[t].tobytes()
            else:
                assert kc[blk, :, off].tobytes() == k0[blk, :, off].tobytes()
                assert vc[blk, :, off].tobytes() == v0[blk, :, off].tobytes()


def test_cache_write_rejects_bad_slots_without_writing():
    rng = np.random.default_rng(22)
    NB, Hkv, bs, d = 4, 2, 16, 8
    kc = _draw(rng, (NB, Hkv, bs, d), W.DTYPE_F16)
    vc = kc.copy()
    k0 = kc.copy()
    kn = _draw(rng, (2, Hkv, d), W.DTYPE_F16)
    for slots in ([0, NB * bs], [5, 5]):
        with pytest.raises(oracle.OracleError):
            oracle.cache_write(kn, kn, np.array(slots, np.int64), kc, vc, block_size=bs)
        np.testing.assert_array_equal(kc.view(np.uint16), k0.view(np.uint16))


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_F16])
def test_gather_closed_form_and_permutation(dtype):
    wl = W.random_small(23, batch=4, num_q_heads=4, num_kv_heads=2, head_dim=16, max_ctx=50,
                        dtype=dtype, extra_blocks=5, context_lens=[0, 16, 17, 50])
    kd, vd = oracle.gather(wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens)
    bs = wl.block_size
    span = wl.max_blocks_per_seq * bs
    for b in range(4):
        c = int(wl.context_lens[b])
        for j in range(span):
            if j < c:
                blk = wl.block_tables[b, j // bs]
                assert kd[b, :, j].tobytes() == wl.k_cache[blk, :, j % bs].tobytes()
                assert vd[b, :, j].tobytes() == wl.v_cache[blk, :, j % bs].tobytes()
            else:
                assert not kd[b, :, j].view(np.uint8).any()
                assert not vd[b, :, j].view(np.uint8).any()
    assert np.isfinite(kd.astype(np.float64)).all() and np.isfinite(vd.astype(np.float64)).all()
    perm = np.random.default_rng(1).permutation(wl.num_blocks)
    kc = np.empty_like(wl.k_cache); kc[perm] = wl.k_cache
    vc = np.empty_like(wl.v_cache); vc[perm] = wl.v_cache
    tables = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1)
    kd2, vd2 = oracle.gather(kc, vc, tables.astype(np.int32), wl.context_lens)
    assert kd2.tobytes() == kd.tobytes() and vd2.tobytes() == vd.tobytes()


# --------------------------------------------------------------- the named workloads
def test_tiny_workload_shape_and_finite():
    wl = W.tiny()
    assert wl.block_tables.tolist()[0][1:] == [-1, -1, -1]
    assert (wl.block_tables >= 0).sum() == 4 and wl.num_blocks == 8
    out = _decode_wl(wl)
    assert out.shape == (2, 4, 64) and np.isfinite(out).all()


def test_step_order_cache_write_then_decode():
    """The step writes each sequence's new row at position ctx-1, then attends
    over [0, ctx): the new row must take part (its V appears when its key
    dominates)."""
    wl = W.random_small(24, batch=3, num_q_heads=2, num_kv_heads=1, head_dim=16, max_ctx=40,
                        dtype=W.DTYPE_F32, context_lens=[1, 16, 33])
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    kn = (wl.q[:, :1, :] * 50.0).astype(np.float32)       # key aligned with q head 0
    oracle.cache_write(kn, wl.v_new, wl.slot_mapping, kc, vc, block_size=wl.block_size)
    out = oracle.paged_decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, 1.0)
    for b in range(3):
        np.testing.assert_allclose(out[b, 0], wl.v_new[b, 0].astype(np.float64), atol=1e-6)


# --------------------------------------------------------------- rotary embedding
# The README lists batched RoPE among the fused operations and names no
# variant; the oracle takes the rotate-half form with theta_k = pos *
# base^(-2k/d).  The pins below fix that reading against closed forms and the
# algebra of rotations, not against the oracle's own formula.

def test_rope_position_zero_is_identity():
    x = np.random.default_rng(70).standard_normal((3, 128))
    assert oracle.rope(x, 0, 1e6).tobytes() == x.tobytes()


@pytest.mark.parametrize("pos", [1, 3])
def test_rope_closed_form_base_10000_d8(pos):
    """base 10000, d = 8: base^(-2k/8) = 10^(-k), so the unit vector e_k turns
    into cos(pos 10^-k) e_k + sin(pos 10^-k) e_(k+4) and e_(k+4) into
    -sin(pos 10^-k) e_k + cos(pos 10^-k) e_(k+4).  Pins the pairing (k with
    k + d/2, not 2k with 2k+1), the exponent 2k/d, the base and the sign."""
    for k in range(4):
        ang = pos * 10.0 ** (-k)
        c, s = math.cos(ang), math.sin(ang)
        e = np.zeros(8)
        e[k] = 1.0
        want = np.zeros(8)
        want[k], want[k + 4] = c, s
        np.testing.assert_allclose(oracle.rope(e, pos, 10000.0), want, rtol=0, atol=1e-15)
        e = np.zeros(8)
        e[k + 4] = 1.0
        want = np.zeros(8)
        want[k], want[k + 4] = -s, c
        np.testing.assert_allclose(oracle.rope(e, pos, 10000.0), want, rtol=0, atol=1e-15)


def test_rope_preserves_every_pair_norm():
    x = np.random.default_rng(71).standard_normal((5, 64))
    y = oracle.rope(x, 4321, 5e5)
    nx = x[:, :32] ** 2 + x[:, 32:] ** 2
    ny = y[:, :32] ** 2 + y[:, 32:] ** 2
    np.testing.assert_allclose(ny, nx, rtol=1e-13)


def test_rope_scores_depend_only_on_relative_position():
    """<R(m) q, R(n) k> = <R(m - n) q, k>: the property RoPE exists for."""
    rng = np.random.default_rng(72)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for m, n in [(5000, 1234), (17, 17), (8191, 0), (300, 301)]:
        lhs = oracle.rope(q, m, 1e6) @ oracle.rope(k, n, 1e6)
        rhs = oracle.rope(q, m - n, 1e6) @ k
        assert abs(lhs - rhs) <= 1e-11 * (np.abs(q).sum() * np.abs(k).sum()), (m, n)


def test_rope_composes_additively():
    x = np.random.default_rng(73).standard_normal(128)
    a = oracle.rope(oracle.rope(x, 700, 1e4), 900, 1e4)
    np.testing.assert_allclose(a, oracle.rope(x, 1600, 1e4), rtol=0, atol=1e-11)


def test_rope_d2_is_complex_rotation_by_pos():
    """d = 2: one pair with frequency 1 whatever the base, i.e. multiplication
    of x0 + i x1 by e^(i pos)."""
    for pos in (1, 2, 100):
        z = complex(0.3, -1.7) * complex(math.cos(pos), math.sin(pos))
        y = oracle.rope(np.array([0.3, -1.7]), pos, 123.0)
        np.testing.assert_allclose(y, [z.real, z.imag], rtol=0, atol=1e-14)


def test_rope_cos_sin_table_rows():
    t = oracle.rope_cos_sin(10000.0, 4, 8)
    assert t.shape == (4, 4, 2)
    np.testing.assert_array_equal(t[0], np.stack([np.ones(4), np.zeros(4)], -1))
    for pos in range(4):
        for k in range(4):
            ang = pos * 10.0 ** (-k)
            assert abs(t[pos, k, 0] - math.cos(ang)) <= 1e-15
            assert abs(t[pos, k, 1] - math.sin(ang)) <= 1e-15


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_F16, W.DTYPE_BF16])
def test_narrow_rounds_to_nearest_even_like_torch(dtype):
    x = np.random.default_rng(74).standard_normal(4096) * 3.0
    x[:4] = [1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8]  # ties
    got = oracle.narrow(x, dtype)
    t = torch.from_numpy(x)
    if dtype == W.DTYPE_BF16:
        want = t.to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    else:
        want = t.to(torch.float32 if dtype == W.DTYPE_F32 else torch.float16).numpy()
    assert got.tobytes() == want.tobytes()


@pytest.mark.parametrize("dtype", [W.DTYPE_F16, W.DTYPE_BF16])
def test_decode_with_widened_q_equals_decode(dtype):
    wl = W.random_small(75, batch=5, num_q_heads=8, num_kv_heads=2, head_dim=64, max_ctx=90,
                        dtype=dtype)
    a = oracle.paged_decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                            wl.scale, dtype=dtype)
    b = oracle.paged_decode_q64(_to_f64(wl.q, dtype), wl.k_cache, wl.v_cache, wl.block_tables,
                                wl.context_lens, wl.scale, dtype=dtype)
    assert a.tobytes() == b.tobytes()


def test_rope_step_at_position_zero_is_the_plain_step():
    """Every context 1: the new token sits at position 0, where RoPE is the
    identity, so the RoPE step equals cache write + decode bit for bit (a step
    that turned by context_len instead of context_len - 1 would not)."""
    wl = W.random_small(76, batch=6, num_q_heads=4, num_kv_heads=2, head_dim=64, max_ctx=1,
                        dtype=W.DTYPE_F16, context_lens=[1] * 6)
    kc, vc, out = oracle.rope_step(wl, 1e4)
    kc2, vc2 = wl.k_cache.copy(), wl.v_cache.copy()
    oracle.cache_write(wl.k_new, wl.v_new, wl.slot_mapping, kc2, vc2,
                       block_size=wl.block_size, dtype=wl.dtype)
    out2 = oracle.paged_decode(wl.q, kc2, vc2, wl.block_tables, wl.context_lens, wl.scale,
                               dtype=wl.dtype)
    assert kc.tobytes() == kc2.tobytes() and vc.tobytes() == vc2.tobytes()
    assert out.tobytes() == out2.tobytes()


def test_rope_step_stores_rotated_keys_and_plain_values():
    """The stored K row of each sequence keeps the pair norms of k_new (a
    rotation), differs from k_new (it did turn: positions > 0), and the V row
    is stored unchanged."""
    wl = W.random_small(77, batch=4, num_q_heads=4, num_kv_heads=2, head_dim=64, max_ctx=64,
                        dtype=W.DTYPE_F32, context_lens=[5, 17, 33, 64])
    kc, vc, _ = oracle.rope_step(wl, 1e4)
    blk, off = wl.slot_mapping // wl.block_size, wl.slot_mapping % wl.block_size
    k_st = kc[blk, :, off].astype(np.float64)
    k_in = wl.k_new.astype(np.float64)
    norm = lambda x: x[..., :32] ** 2 + x[..., 32:] ** 2
    np.testing.assert_allclose(norm(k_st), norm(k_in), rtol=1e-6, atol=1e-6)
    assert not np.allclose(k_st, k_in)
    assert vc[blk, :, off].tobytes() == wl.v_new.tobytes()


# --------------------------------------------------------------- multi-query (causal)
@pytest.mark.parametrize("dtype", [W.DTYPE_F16, W.DTYPE_BF16, W.DTYPE_F32])
def test_multi_query_equals_dense_causal_torch(dtype):
    """A torch float64 causal attention on dense K/V the test pages itself:
    query token i of sequence b (position first_b + i) sees keys 0..first_b+i,
    through an explicit upper-triangular -inf mask on the full score matrix."""
    rng = np.random.default_rng(900 + dtype)
    Hq, Hkv, d, bs = 8, 2, 16, 16
    n = np.array([1, 5, 16, 3, 0, 20], np.int32)          # new tokens per sequence
    prefix = np.array([0, 11, 16, 40, 7, 1], np.int32)
    ctx = prefix + n
    B, S = len(ctx), int(ctx.max())
    dk = _draw(rng, (B, Hkv, S, d), dtype)
    dv = _draw(rng, (B, Hkv, S, d), dtype)
    T = int(n.sum())
    q = _draw(rng, (T, Hq, d), dtype)
    qs = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    kc, vc, tables = _page(dk, dv, ctx, bs, rng)
    scale = 0.9 / math.sqrt(d)
    got = oracle.multi_query(q, kc, vc, tables, ctx, qs, scale, dtype=dtype)
    q64, k64, v64 = _to_f64(q, dtype), _to_f64(dk, dtype), _to_f64(dv, dtype)
    G = Hq // Hkv
    for b in range(B):
        if n[b] == 0:
            continue
        c = int(ctx[b])
        K = torch.from_numpy(k64[b, :, :c]).repeat_interleave(G, dim=0)     # [Hq][c][d]
        V = torch.from_numpy(v64[b, :, :c]).repeat_interleave(G, dim=0)
        Q = torch.from_numpy(q64[qs[b]:qs[b + 1]]).transpose(0, 1)          # [Hq][n][d]
        s = torch.matmul(Q, K.transpose(1, 2)) * scale                      # [Hq][n][c]
        i = torch.arange(int(n[b])).unsqueeze(1) + int(prefix[b])
        j = torch.arange(c).unsqueeze(0)
        s = s.masked_fill(j > i, float("-inf"))
        want = torch.matmul(torch.softmax(s, dim=-1), V).transpose(0, 1).numpy()
        np.testing.assert_allclose(got[qs[b]:qs[b + 1]], want, rtol=0, atol=1e-12)


def test_multi_query_with_one_token_is_the_decode():
    wl = W.random_small(78, batch=6, num_q_heads=8, num_kv_heads=2, head_dim=64, max_ctx=200,
                        dtype=W.DTYPE_F16, context_lens=[1, 17, 64, 100, 150, 200])
    qs = np.arange(7, dtype=np.int32)
    a = oracle.multi_query(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, qs,
                           wl.scale, dtype=wl.dtype)
    assert a.tobytes() == _decode_wl(wl).tobytes()


def test_multi_query_first_token_of_a_fresh_prompt_returns_its_v():
    """A prompt with no prefix: its first token sees only itself, so its output
    is its own V row exactly, whatever q and K are."""
    mq = W.multi_query(79, query_lens=[4, 9], prefix_lens=[0, 0], num_q_heads=4, num_kv_heads=2,
                       head_dim=64, dtype=W.DTYPE_F32)
    p = mq.pool
    out = oracle.multi_query(mq.q, p.k_cache, p.v_cache, p.block_tables, p.context_lens,
                             mq.query_start, p.scale, dtype=p.dtype)
    for b in range(2):
        blk = p.block_tables[b, 0]
        v0 = p.v_cache[blk, :, 0].astype(np.float64)              # [Hkv][d], position 0
        np.testing.assert_array_equal(out[mq.query_start[b]], np.repeat(v0, 2, axis=0))


# ------------------------------------------------------------------ fp8 (e4m3) cache
def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    # closed forms: largest finite, smallest subnormal, one, the NaN codes
    assert oracle.e4m3_decode([0x7E, 0x01, 0x38, 0xB8])[:4].tolist() == [448.0, 2.0 ** -9,
                                                                      1.0, -1.0]
    assert np.isnan(oracle.e4m3_decode([0x7F, 0xFF])).all()


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-12, 6, 100000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), want)


def test_e4m3_encode_ties_saturation_and_round_trip():
    # halfway between 1.0 and 1.125 -> the even code (1.0); between 1.125 and 1.25 -> 1.25
    assert oracle.e4m3_encode([1.0625, 1.1875, -1.0625]).tolist() == [0x38, 0x3A, 0xB8]
    # beyond the largest finite value: saturates to +-448; NaN stays NaN
    assert oracle.e4m3_encode([449.0, 500.0, 1e30, -1e30]).tolist() == [0x7E, 0x7E, 0x7E, 0xFE]
    assert oracle.e4m3_encode([np.nan]).tolist() == [0x7F]
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = oracle.e4m3_encode(oracle.e4m3_decode(finite))
    assert np.array_equal(back[finite != 0x80], finite[finite != 0x80])   # -0 may become +0


def test_fp8_cache_write_quantises_each_row_at_its_slot():
    wl = W.random_small(61, batch=3, num_q_heads=4, num_kv_heads=2, head_dim=64, max_ctx=40,
                        dtype=W.DTYPE_F16)
    k8, v8 = W.fp8_cache(wl, 5)
    k0, v0 = k8.copy(), v8.copy()
    # K and V take different scales (0.5 and 0.25), so a swapped or shared
    # scale, or rows written to the other pool, fails below.  The expected
    # codes come from torch's float8_e4m3fn conversion (a library routine, not
    # the oracle's encoder): the scaled fp16 N(0,1) rows stay far inside +-448,
    # where that conversion rounds to nearest even like the e4m3 definition.
    oracle.cache_write_fp8(wl.k_new, wl.v_new, wl.slot_mapping, k8, v8, 0.5, 0.25,
                           block_size=16)

    def codes(rows, inv_scale):
        x = torch.from_numpy(rows.astype(np.float32)) * inv_scale
        assert float(x.abs().max()) < 448
        return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()

    for t, slot in enumerate(wl.slot_mapping):
        blk, off = slot // 16, slot % 16
        assert np.array_equal(k8[blk, :, off], codes(wl.k_new[t], 2.0))
        assert np.array_equal(v8[blk, :, off], codes(wl.v_new[t], 4.0))
        k0[blk, :, off] = k8[blk, :, off]
        v0[blk, :, off] = v8[blk, :, off]
    assert np.array_equal(k0, k8) and np.array_equal(v0, v8)   # nothing else changed


def test_fp8_decode_equals_brute_force_on_dequantised_values():
    """The definition written out: dequantise every cached K/V element
    (code value x scale) and take softmax(scale q.K) V per head in numpy."""
    wl = W.random_small(62, batch=3, num_q_heads=8, num_kv_heads=2, head_dim=64, max_ctx=70,
                        dtype=W.DTYPE_F16, context_lens=[1, 33, 70])
    k8, v8 = W.fp8_cache(wl, 6)
    ks, vs = 0.5, 0.25
    got = oracle.paged_decode_fp8(wl.q, k8, v8, wl.block_tables, wl.context_lens, wl.scale,
                                  ks, vs)
    G = wl.num_q_heads // wl.num_kv_heads
    for b in range(3):
        c = int(wl.context_lens[b])
        blocks = wl.block_tables[b, :(c + 15) // 16]
        for h in range(wl.num_q_heads):
            kv = h // G
            K = np.concatenate([oracle.e4m3_decode(k8[p, kv]) for p in blocks])[:c] * ks
            V = np.concatenate([oracle.e4m3_decode(v8[p, kv]) for p in blocks])[:c] * vs
            s_ = wl.scale * (K @ wl.q[b, h].astype(np.float64))
            w = np.exp(s_ - s_.max())
            want = (w[:, None] * V).sum(0) / w.sum()
            assert np.abs(got[b, h] - want).max() <= 1e-12


def test_fp8_pools_hold_finite_codes_only_where_tables_point():
    wl = W.random_small(63, batch=5, num_q_heads=8, num_kv_heads=2, head_dim=64, max_ctx=90,
                        dtype=W.DTYPE_F16, extra_blocks=4)
    k8, v8 = W.fp8_cache(wl, 9)
    used = np.zeros(wl.num_blocks, bool)
    used[wl.block_tables[wl.block_tables >= 0]] = True
    for pool in (k8, v8):
        assert (pool[~used] == W.E4M3_NAN).all()                  # the stray-read detector
        vals = np.abs(oracle.e4m3_decode(pool[used]))
        assert np.isfinite(vals).all() and vals.min() >= 0.25 and vals.max() <= 3.75
    assert not np.array_equal(k8, v8)
