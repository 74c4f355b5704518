"""Host-side checks of the C-ABI library: it builds, loads, exports every
symbol the header declares, and rejects bad arguments with the documented
status before touching CUDA.  Needs no GPU."""
import ctypes
import math

import pytest

import paged_kv_attention_photon_gb300 as P


@pytest.fixture(scope="module")
def lib():
    P.build()
    return P._load()


def _shape(**over):
    base = dict(num_seqs=4, num_q_heads=16, num_kv_heads=8, head_dim=128, block_size=16,
                num_blocks=100, max_blocks_per_seq=8, dtype=P.F16, partition_size=0)
    base.update(over)
    return P.PagedShape.make(**base)


FAKE = 0x10000          # aligned non-null "device" addresses: never dereferenced,
FAKE2 = 0x20000         # every case below fails validation before any launch


def test_exports_every_declared_symbol(lib):
    names = P.exported_symbols()
    assert {"photon_cache_write", "photon_paged_decode", "photon_paged_decode_workspace_size",
            "photon_paged_gather", "photon_get_last_device_error",
            "photon_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(7):
        assert P.photon_status_string(code) not in ("", "unknown status")
    assert P.photon_status_string(99) == "unknown status"


def _decode_status(shape, *, q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, cl=FAKE, out=FAKE2,
                   ws=FAKE2, ws_bytes=1 << 40, scale=0.1):
    return P._load().photon_paged_decode(q, kc, vc, bt, cl, scale, out, ws, ws_bytes,
                                         ctypes.byref(shape), None)


def test_decode_validation(lib):
    ok = _shape()
    assert _decode_status(_shape(num_q_heads=12)) == 1          # Hq % Hkv != 0
    assert _decode_status(_shape(num_q_heads=24, num_kv_heads=8)) == 2   # group 3
    assert _decode_status(_shape(head_dim=96)) == 2
    assert _decode_status(_shape(block_size=32)) == 2
    assert _decode_status(_shape(dtype=7)) == 2
    assert _decode_status(_shape(partition_size=24)) == 1
    assert _decode_status(_shape(partition_size=8192)) == 1
    assert _decode_status(_shape(num_seqs=-1)) == 1
    assert _decode_status(ok, q=None) == 1
    assert _decode_status(ok, out=None) == 1
    assert _decode_status(ok, q=FAKE + 8) == 3
    assert _decode_status(ok, bt=FAKE + 4) == 3
    assert _decode_status(ok, ws=None) == 4
    assert _decode_status(ok, ws_bytes=16) == 4
    assert _decode_status(ok, scale=math.nan) == 1
    assert _decode_status(ok, scale=math.inf) == 1
    assert lib.photon_paged_decode(None, None, None, None, None, 0.1, None, None, 0, None,
                                   None) == 1
    # an empty batch is a no-op, whatever the pointers
    assert _decode_status(_shape(num_seqs=0), q=None, out=None, ws=None, ws_bytes=0) == 0


def test_cache_write_validation(lib):
    s = _shape()
    f = lib.photon_cache_write
    assert f(FAKE, FAKE, FAKE, 0, FAKE, FAKE, ctypes.byref(s), None) == 0     # no rows: no-op
    assert f(FAKE, FAKE, FAKE, -1, FAKE, FAKE, ctypes.byref(s), None) == 1
    assert f(None, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(s), None) == 1
    assert f(FAKE, FAKE, FAKE + 4, 4, FAKE, FAKE, ctypes.byref(s), None) == 3
    assert f(FAKE, FAKE + 8, FAKE, 4, FAKE, FAKE, ctypes.byref(s), None) == 3
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(_shape(head_dim=80)), None) == 2


def test_fp8_validation(lib):
    s = _shape()
    w = lib.photon_cache_write_fp8
    assert w(FAKE, FAKE, FAKE, 0, FAKE, FAKE, 0.5, 0.5, ctypes.byref(s), None) == 0   # no rows
    assert w(FAKE, FAKE, FAKE, -1, FAKE, FAKE, 0.5, 0.5, ctypes.byref(s), None) == 1
    assert w(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 0.0, 0.5, ctypes.byref(s), None) == 1
    assert w(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 0.5, math.nan, ctypes.byref(s), None) == 1
    assert w(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 0.5, -1.0, ctypes.byref(s), None) == 1
    assert w(FAKE, FAKE, FAKE, 4, FAKE + 8, FAKE, 0.5, 0.5, ctypes.byref(s), None) == 3
    assert w(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 0.5, 0.5,
             ctypes.byref(_shape(dtype=P.BF16)), None) == 2          # fp16 rows only
    d = lib.photon_paged_decode_fp8

    def dec(shape, *, q=FAKE, ks=0.5, vs=0.5, ws_bytes=1 << 40, scale=0.1):
        return d(q, FAKE, FAKE, FAKE, FAKE, scale, ks, vs, FAKE2, FAKE2, ws_bytes,
                 ctypes.byref(shape), None)
    assert dec(_shape(dtype=P.F32)) == 2
    assert dec(_shape(dtype=P.BF16)) == 2
    assert dec(s, ks=0.0) == 1
    assert dec(s, vs=math.inf) == 1
    assert dec(s, scale=math.nan) == 1
    assert dec(s, q=None) == 1
    assert dec(s, ws_bytes=16) == 4
    assert dec(_shape(num_seqs=0)) == 0
    # fp8 partitions hold twice the tokens: about half the fp16 decode's
    # partials (each has one more for the halved last full partition)
    big = _shape(num_seqs=64, max_blocks_per_seq=512)
    assert 2 * lib.photon_paged_decode_fp8_workspace_size(ctypes.byref(big)) \
        <= 1.1 * lib.photon_paged_decode_workspace_size(ctypes.byref(big))
    assert lib.photon_paged_decode_fp8_workspace_size(ctypes.byref(_shape(dtype=P.BF16))) == 0


def test_gather_validation(lib):
    s = _shape()
    f = lib.photon_paged_gather
    assert f(FAKE, FAKE, FAKE, FAKE, None, FAKE, ctypes.byref(s), None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE + 2, FAKE, ctypes.byref(s), None) == 3
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(_shape(num_seqs=0)), None) == 0


def test_default_partition_sizes(lib):
    """The default partition: 192 KB of K+V per (partition, KV head) item,
    and for a batch whose worst case (num_seqs x max_blocks_per_seq x 16 x
    Hkv tokens) would give fewer than about two items per resident CTA (608
    items), that worst case / 608 rounded to the nearest whole stage of 64
    tokens (one 16-token block per consumer warp), at least 64 tokens."""
    def part(**over):
        return P.photon_paged_decode_plan(_shape(**over))["partition_size"]
    d64 = dict(num_q_heads=32, num_kv_heads=8, head_dim=64, num_blocks=40000)
    # the item cap: 192 KB / (2 x d x 2 bytes)
    assert part(num_seqs=64, max_blocks_per_seq=512) == 384
    assert part(num_seqs=256, max_blocks_per_seq=1024, **d64) == 768
    # small batches of the d = 64 sweep shape (contexts up to 2048 tokens):
    # 4 x 128 x 16 x 8 / 608 = 107.8 -> 128; 8 x ... = 215.6 -> 192;
    # 16 x ... = 431.2 -> 448; 32 x ... = 862.3 -> the cap, 768
    assert part(num_seqs=4, max_blocks_per_seq=128, **d64) == 128
    assert part(num_seqs=8, max_blocks_per_seq=128, **d64) == 192
    assert part(num_seqs=16, max_blocks_per_seq=128, **d64) == 448
    assert part(num_seqs=32, max_blocks_per_seq=128, **d64) == 768
    # 16 x 71 x 16 x 8 / 608 = 239.2 -> 256 (round to nearest, not down)
    assert part(num_seqs=16, max_blocks_per_seq=71, **d64) == 256
    # tiny: 64 at the least
    assert part(num_seqs=2, max_blocks_per_seq=4, num_q_heads=4, num_kv_heads=1,
                head_dim=64) == 64
    # every shrunk partition is whole stages
    for b in (1, 2, 3, 5, 6, 7, 9, 12, 20, 24):
        assert part(num_seqs=b, max_blocks_per_seq=128, **d64) % 64 == 0


def test_workspace_size_and_plan(lib):
    s = _shape(num_seqs=64, max_blocks_per_seq=512, partition_size=256)
    pl = P.photon_paged_decode_plan(s)
    # 8192 tokens: 32 full partitions of 256, the last one cut in two halves
    assert pl["partition_size"] == 256 and pl["max_partitions"] == 33
    ws = P.photon_paged_decode_workspace_size(s)
    rows = 64 * 16 * 33
    assert ws >= rows * (128 + 2) * 4
    assert ws % 256 == 0
    assert P.photon_paged_decode_workspace_size(_shape(head_dim=96)) == 0
    assert P.photon_paged_decode_workspace_size(_shape(num_seqs=0)) == 0
    d = P.photon_paged_decode_plan(_shape())
    assert d["partition_size"] > 0 and d["partition_size"] % 16 == 0
    assert d["kernels_per_call"] in (2, 3)
    with pytest.raises(P.PhotonError):
        P.photon_paged_decode_plan(_shape(num_q_heads=3))


def test_events_hook_argument_check(lib):
    assert lib.photon_debug_set_attention_events(FAKE, None) == 1
    assert lib.photon_debug_set_attention_events(None, None) == 0


def test_rope_entry_points_validation(lib):
    f = lib.photon_rope_cos_sin
    assert f(1e4, 16, 128, None, None) == 1
    assert f(1.0, 16, 128, FAKE, None) == 1              # base must be > 1
    assert f(math.nan, 16, 128, FAKE, None) == 1
    assert f(math.inf, 16, 128, FAKE, None) == 1
    assert f(1e4, 0, 128, FAKE, None) == 1
    assert f(1e4, 16, 127, FAKE, None) == 1              # odd head_dim
    assert f(1e4, 1 << 30, 128, FAKE, None) == 1         # table too large
    assert f(1e4, 16, 128, FAKE + 4, None) == 3          # 16-byte alignment
    assert f(1e4, 16, 128, FAKE + 8, None) == 3
    g = lib.photon_paged_decode_step_rope
    s = _shape()
    args = lambda **o: [o.get("kn", FAKE), o.get("vn", FAKE), o.get("sm", FAKE), FAKE, FAKE,
                        FAKE, FAKE, FAKE, o.get("cs", FAKE), o.get("mp", 4096), 0.1, FAKE2,
                        FAKE2, 1 << 40, ctypes.byref(o.get("shape", s)), None]
    assert g(*args(cs=None)) == 1
    assert g(*args(mp=0)) == 1
    assert g(*args(kn=None)) == 1
    assert g(*args(cs=FAKE + 4)) == 3
    assert g(*args(cs=FAKE + 8)) == 3
    assert g(*args(sm=FAKE + 4)) == 3
    assert g(*args(shape=_shape(head_dim=96))) == 2
    assert g(*args(shape=_shape(num_seqs=0), cs=None)) == 0    # empty batch: no-op


def test_multi_query_validation(lib):
    f = lib.photon_paged_multi_query
    s = _shape()
    args = lambda **o: [o.get("q", FAKE), FAKE, FAKE, FAKE, FAKE, o.get("qs", FAKE),
                        o.get("T", 64), o.get("maxq", 16), o.get("scale", 0.1), o.get("out", FAKE2),
                        o.get("ws", FAKE2), o.get("wsb", 1 << 40),
                        ctypes.byref(o.get("shape", s)), None]
    assert f(*args(shape=_shape(dtype=P.F32))) == 2            # tensor-core path: 16-bit only
    assert f(*args(shape=_shape(head_dim=96))) == 2
    assert f(*args(qs=None)) == 1
    assert f(*args(q=None)) == 1
    assert f(*args(T=-1)) == 1
    assert f(*args(maxq=-1)) == 1
    assert f(*args(scale=math.nan)) == 1
    assert f(*args(qs=FAKE + 4)) == 3
    assert f(*args(out=FAKE2 + 2)) == 3
    assert f(*args(T=0, q=None, qs=None, out=None)) == 0        # no tokens: no-op
    assert f(*args(maxq=0, q=None)) == 0
    assert f(*args(shape=_shape(num_seqs=0), q=None)) == 0
    # a small batch over long contexts splits its keys: it needs a workspace
    long_ctx = _shape(max_blocks_per_seq=512)
    need = P.photon_paged_multi_query_workspace_size(long_ctx, 64, 16)
    assert need > 0 and need % 256 == 0
    assert f(*args(ws=None, shape=long_ctx)) == 4
    assert f(*args(wsb=need - 1, shape=long_ctx)) == 4
    assert f(*args(ws=FAKE2 + 8, shape=long_ctx)) == 3
    assert P.photon_paged_multi_query_workspace_size(_shape(dtype=P.F32), 64, 16) == 0
    assert P.photon_paged_multi_query_workspace_size(s, 0, 16) == 0


def test_multi_query_plan_splits_small_batches_only(lib):
    s = _shape(num_seqs=64, max_blocks_per_seq=512)
    # 64 sequences x 8 KV heads x 1 tile (4 tokens x group 2 rows): split
    assert P.photon_paged_multi_query_workspace_size(s, 256, 4) > 0
    # 1024 tokens each: 64 x 8 x 32 tiles fill the device without a split
    assert P.photon_paged_multi_query_workspace_size(s, 64 * 1024, 1024) == 0
    # a nonzero partition_size forces the split
    s2 = _shape(num_seqs=64, max_blocks_per_seq=512, partition_size=1024)
    assert P.photon_paged_multi_query_workspace_size(s2, 64 * 1024, 1024) > 0


def test_multi_query_workspace_covers_the_few_token_path():
    # 608 sequences x 2 KV heads x one 64-row tile fill the device without a
    # key split (the warp-level and tcgen05 plans need no workspace), but
    # max_query_len x G = 4 x 2 <= 8 runs the decode kernel's few-token mode,
    # whose split-KV partials are per query token
    s = _shape(num_seqs=608, num_q_heads=4, num_kv_heads=2, max_blocks_per_seq=64)
    need = P.photon_paged_multi_query_workspace_size(s, 608 * 4, 4)
    assert need >= 608 * 4 * 4 * (128 + 2) * 4     # (m, l, o) per token, head, partition >= 1
    # 5 tokens x 2 heads > 8 slots: the plans without a split need none
    assert P.photon_paged_multi_query_workspace_size(s, 608 * 5, 5) == 0


def test_multi_query_kernel_hook(lib):
    assert lib.photon_debug_set_multi_query_kernel(4) == 1
    assert lib.photon_debug_set_multi_query_kernel(-1) == 1
    for k in (1, 2, 3, 0):
        assert lib.photon_debug_set_multi_query_kernel(k) == 0


def test_decode_consumer_hook(lib):
    assert lib.photon_debug_set_decode_consumer(3) == 1
    assert lib.photon_debug_set_decode_consumer(-1) == 1
    for k in (1, 2, 0):
        assert lib.photon_debug_set_decode_consumer(k) == 0


def test_wait_probe_argument_check(lib):
    assert lib.photon_debug_wait_probe(0, None) == 1
    assert lib.photon_debug_wait_probe(2_000_000_000, None) == 1
