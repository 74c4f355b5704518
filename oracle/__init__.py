"""fp64 CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product path (the CUDA library and
its Python binding) never touches it and shares no code with it.

The arithmetic lives in ``paged_ref.c`` (plain loops in double); this module
builds it with gcc and wraps it with ctypes and numpy.  ``scheduler.py`` holds
the plain-Python oracle of the host scheduler (integer bookkeeping only).  Every function states
which passage of the PhotonInfer README it restates; see the C file's header
for the formula and the layouts.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_ref.c")
_LIB_PATH = os.path.join(_HERE, "libphoton_oracle.so")
_lib = None

ERRORS = {0: "ok", -1: "bad argument", -2: "slot out of range", -3: "duplicate slot",
          -4: "block id out of range", -5: "context length out of range"}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile paged_ref.c into libphoton_oracle.so (plain -O2, no SIMD flags)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.ref_cache_write.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, i32]
    lib.ref_gather.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32]
    lib.ref_paged_decode.argtypes = [P, P, P, P, P, f64, P] + [i32] * 9
    lib.ref_paged_decode_row.argtypes = [P, P, P, P, P, f64, i32, i32, P] + [i32] * 8
    lib.ref_attend_range.argtypes = [P, P, P, P, P, f64, i32, i32, i64, i64, P, P, P] + [i32] * 8
    lib.ref_merge.argtypes = [i32, P, P, P, i32, P]
    lib.ref_merge.restype = None
    lib.ref_widen.argtypes = [P, ctypes.c_size_t, i32, P]
    lib.ref_widen.restype = None
    lib.ref_rope.argtypes = [P, i32, i64, f64, P]
    lib.ref_rope.restype = None
    lib.ref_paged_decode_q64.argtypes = [P, P, P, P, P, f64, P] + [i32] * 9
    lib.ref_paged_decode_q64.restype = ctypes.c_int
    for fn in (lib.ref_cache_write, lib.ref_gather, lib.ref_paged_decode,
               lib.ref_paged_decode_row, lib.ref_attend_range):
        fn.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _check(rc: int) -> None:
    if rc != 0:
        raise OracleError(ERRORS.get(rc, f"error {rc}"))


def _dtype_code(a: np.ndarray, dtype: Optional[int]) -> int:
    if dtype is not None:
        return dtype
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.float16:
        return 1
    raise ValueError("pass dtype explicitly for raw 16-bit storage (bf16)")


def cache_write(k_new, v_new, slot_mapping, k_cache, v_cache, *, block_size: int,
                dtype: Optional[int] = None) -> None:
    """Batched cache write (README "Technical details: paged attention", the
    single kernel for multi-sequence K/V writes): bit-copies row t to slot_t,
    in place on the numpy pools."""
    lib = _load()
    T = int(slot_mapping.shape[0])
    NB, Hkv, bs, d = k_cache.shape
    assert bs == block_size
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    _check(lib.ref_cache_write(_ptr(k_new), _ptr(v_new), _ptr(sm), T, _ptr(k_cache),
                               _ptr(v_cache), Hkv, d, bs, NB, _dtype_code(k_cache, dtype)))


def gather(k_cache, v_cache, block_tables, context_lens, *, dtype: Optional[int] = None
           ) -> Tuple[np.ndarray, np.ndarray]:
    """Block-table gather (README "Technical details: paged attention",
    per-sequence cache offsets): dense [B][Hkv][MBS*bs][d], zero past ctx."""
    lib = _load()
    NB, Hkv, bs, d = k_cache.shape
    B, MBS = block_tables.shape
    kd = np.empty((B, Hkv, MBS * bs, d), dtype=k_cache.dtype)
    vd = np.empty_like(kd)
    _check(lib.ref_gather(_ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
                          _ptr(kd), _ptr(vd), B, Hkv, d, bs, NB, MBS,
                          _dtype_code(k_cache, dtype)))
    return kd, vd


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, *,
                 dtype: Optional[int] = None, num_threads: int = 1) -> np.ndarray:
    """Batched paged decode attention in fp64 (README "Key features: GPU
    kernels", batched paged attention with numerically stable softmax).
    Returns float64 [B][Hq][d]."""
    lib = _load()
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    MBS = block_tables.shape[1]
    out = np.empty((B, Hq, d), dtype=np.float64)
    _check(lib.ref_paged_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                _ptr(context_lens), float(scale), _ptr(out), B, Hq, Hkv, d, bs,
                                NB, MBS, _dtype_code(q, dtype), int(num_threads)))
    return out


def paged_decode_row(q, k_cache, v_cache, block_tables, context_lens, scale: float, b: int,
                     h: int, *, dtype: Optional[int] = None) -> np.ndarray:
    """One (sequence, q head) output row of paged_decode, float64 [d]."""
    lib = _load()
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    MBS = block_tables.shape[1]
    out = np.empty(d, dtype=np.float64)
    _check(lib.ref_paged_decode_row(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                    _ptr(context_lens), float(scale), int(b), int(h), _ptr(out),
                                    B, Hq, Hkv, d, bs, NB, MBS, _dtype_code(q, dtype)))
    return out


def attend_range(q, k_cache, v_cache, block_tables, context_lens, scale: float, b: int, h: int,
                 j0: int, j1: int, *, dtype: Optional[int] = None):
    """Partial (m, l, unnormalised o) over logical positions [j0, j1)."""
    lib = _load()
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    MBS = block_tables.shape[1]
    m = np.zeros(1, np.float64)
    l = np.zeros(1, np.float64)
    o = np.zeros(d, np.float64)
    _check(lib.ref_attend_range(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                _ptr(context_lens), float(scale), int(b), int(h), int(j0),
                                int(j1), _ptr(m), _ptr(l), _ptr(o), B, Hq, Hkv, d, bs, NB, MBS,
                                _dtype_code(q, dtype)))
    return float(m[0]), float(l[0]), o


def merge(m, l, o) -> np.ndarray:
    """Partition merge by log-sum-exp weights (the split-KV combination step)."""
    lib = _load()
    m = np.ascontiguousarray(m, np.float64)
    l = np.ascontiguousarray(l, np.float64)
    o = np.ascontiguousarray(o, np.float64)
    P, d = o.shape
    out = np.empty(d, np.float64)
    lib.ref_merge(P, _ptr(m), _ptr(l), _ptr(o), d, _ptr(out))
    return out


def widen(a: np.ndarray, dtype: Optional[int] = None) -> np.ndarray:
    """Exact widening of stored fp32/fp16/bf16 elements to float64."""
    lib = _load()
    a = np.ascontiguousarray(a)
    out = np.empty(a.shape, np.float64)
    lib.ref_widen(_ptr(a), a.size, _dtype_code(a, dtype), _ptr(out))
    return out


def rope(x, pos: int, base: float) -> np.ndarray:
    """Rotate-half rotary position embedding of the last axis of x (float64),
    every row at position pos (the README lists batched RoPE among its fused
    operations)."""
    lib = _load()
    x = np.ascontiguousarray(x, np.float64)
    d = x.shape[-1]
    flat = x.reshape(-1, d)
    out = np.empty_like(flat)
    for r in range(flat.shape[0]):
        lib.ref_rope(_ptr(flat[r]), d, int(pos), float(base), out[r].ctypes.data)
    return out.reshape(x.shape)


def rope_cos_sin(base: float, max_positions: int, head_dim: int) -> np.ndarray:
    """(cos, sin) of every position and pair, float64 [max_positions][d/2][2]:
    the rotation of the vector with ones in its lower half and zeros in its
    upper half has cos theta_k at k and sin theta_k at k + d/2."""
    half = head_dim // 2
    x = np.concatenate([np.ones(half), np.zeros(half)])
    out = np.empty((max_positions, half, 2))
    for pos in range(max_positions):
        y = rope(x, pos, base)
        out[pos, :, 0] = y[:half]
        out[pos, :, 1] = y[half:]
    return out


def rope_step(wl, base: float, num_threads: int = 1):
    """Oracle of the decode step with RoPE: the q rows and the new K rows are
    rotated (rope) by the new token's position, context_len - 1; the rotated K
    rows are stored in the storage dtype (round to nearest even) by the cache
    write; the decode then attends with the rotated q rows, kept in double.
    Returns (k_cache, v_cache, out float64 [B][Hq][d])."""
    B = wl.num_seqs
    q64 = widen(wl.q, wl.dtype)
    k64 = widen(wl.k_new, wl.dtype)
    q_rot = np.empty_like(q64)
    k_rot = np.empty_like(k64)
    for b in range(B):
        pos = max(int(wl.context_lens[b]) - 1, 0)
        q_rot[b] = rope(q64[b], pos, base)
        k_rot[b] = rope(k64[b], pos, base)
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    cache_write(narrow(k_rot, wl.dtype), wl.v_new, wl.slot_mapping, kc, vc,
                block_size=wl.block_size, dtype=wl.dtype)
    out = paged_decode_q64(q_rot, kc, vc, wl.block_tables, wl.context_lens, wl.scale,
                           dtype=wl.dtype, num_threads=num_threads)
    return kc, vc, out


def multi_query(q, k_cache, v_cache, block_tables, context_lens, query_start, scale: float, *,
                dtype: int, num_threads: int = 1) -> np.ndarray:
    """Causal multi-query attention (chunked prefill / verification), float64
    [T][Hq][d].  Sequence b's query rows query_start[b] .. query_start[b+1]-1
    are its last n_b tokens; token i sits at position context_lens[b] - n_b + i
    and attends to the keys at positions 0 .. that position.  Written as what
    it is: one decode row per query token, over the same block table with the
    context cut at the token's own position."""
    qs = np.asarray(query_start, dtype=np.int64)
    B = qs.shape[0] - 1
    rows_b, rows_ctx = [], []
    for b in range(B):
        n = int(qs[b + 1] - qs[b])
        first = int(context_lens[b]) - n
        for i in range(n):
            rows_b.append(b)
            rows_ctx.append(first + i + 1)
    if not rows_b:
        return np.zeros((0,) + tuple(q.shape[1:]))
    tables = np.ascontiguousarray(np.asarray(block_tables)[rows_b])
    ctx = np.asarray(rows_ctx, dtype=np.int32)
    qq = np.ascontiguousarray(q[int(qs[0]):int(qs[-1])])
    return paged_decode(qq, k_cache, v_cache, tables, ctx, scale, dtype=dtype,
                        num_threads=num_threads)


# ------------------------------------------------------------------ fp8 (e4m3) KV cache
# The further step of the bf16 row (README "Roadmap": lower-precision KV):
# K and V stored as OCP e4m3 codes -- 1 sign bit, 4 exponent bits (bias 7),
# 3 mantissa bits; exponent field 0 is subnormal (m * 2^-9); exponent 15 with
# mantissa 7 is NaN; no infinities; the largest finite value is 448 -- each
# with one per-tensor scale: value = decode(code) * scale.

def e4m3_decode(codes) -> np.ndarray:
    """float64 values of e4m3 codes (NaN for 0x7F / 0xFF), read off the bit
    fields as defined above."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.power(2.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


_E4M3_POS = e4m3_decode(np.arange(0x7F, dtype=np.uint8))   # codes 0x00 .. 0x7E, increasing


def e4m3_encode(x) -> np.ndarray:
    """e4m3 codes of float values: round to the nearest finite e4m3 value,
    ties to the even code (even mantissa), magnitudes beyond 448 saturate to
    448 (the finite-saturating conversion), NaN -> 0x7F.  A brute-force search
    over the 127 non-negative finite values."""
    v = np.asarray(x, dtype=np.float64)
    a = np.abs(v)
    i = np.clip(np.searchsorted(_E4M3_POS, a), 1, len(_E4M3_POS) - 1)   # a in (pos[i-1], pos[i]]
    lo, hi = _E4M3_POS[i - 1], _E4M3_POS[i]
    pick_hi = (hi - a < a - lo) | ((hi - a == a - lo) & (i % 2 == 0))
    code = np.where(pick_hi, i, i - 1)
    code = np.where(a >= _E4M3_POS[-1], 0x7E, code)                  # saturate
    code = np.where(a == 0, 0, code)
    code = code.astype(np.int64) | np.where(np.signbit(v), 0x80, 0)
    code = np.where(np.isnan(v), 0x7F, code)
    return code.astype(np.uint8)


def cache_write_fp8(k_new, v_new, slot_mapping, k_cache8, v_cache8, k_scale: float,
                    v_scale: float, *, block_size: int) -> None:
    """Quantising cache write: row t of k_new / v_new (fp16) goes to slot_t as
    e4m3 codes of x * (1 / scale), the product taken in fp32 (the reciprocal
    rounded to fp32 first), in place on the uint8 pools.  Negative slots are
    padding."""
    NB, Hkv, bs, d = k_cache8.shape
    assert bs == block_size
    for src, dst, scale in ((k_new, k_cache8, k_scale), (v_new, v_cache8, v_scale)):
        inv = np.float32(1.0) / np.float32(scale)
        for t, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
            if slot < 0:
                continue
            if slot >= NB * bs:
                raise OracleError("slot out of range")
            x = np.asarray(src[t], dtype=np.float16).astype(np.float32) * inv
            dst[slot // bs, :, slot % bs, :] = e4m3_encode(x)


def paged_decode_fp8(q, k_cache8, v_cache8, block_tables, context_lens, scale: float,
                     k_scale: float, v_scale: float, *, num_threads: int = 1) -> np.ndarray:
    """Paged decode over an e4m3 cache: attention over K = decode(code) *
    k_scale and V = decode(code) * v_scale, in fp64.  Written through the
    identity softmax(scale q.(s_k K)) (s_v V) = s_v softmax((scale s_k) q.K) V
    so that the fp64 decode above reads the codes' values exactly (as fp32
    pools); float64 [B][Hq][d]."""
    k32 = e4m3_decode(k_cache8).astype(np.float32)
    v32 = e4m3_decode(v_cache8).astype(np.float32)
    q32 = np.asarray(q, dtype=np.float16).astype(np.float32)
    out = paged_decode(q32, k32, v32, block_tables, context_lens, float(scale) * float(k_scale),
                       dtype=0, num_threads=num_threads)
    return out * float(v_scale)


def narrow(x64: np.ndarray, dtype: int) -> np.ndarray:
    """float64 -> storage dtype, round to nearest even (bf16 through fp32)."""
    if dtype == 0:
        return x64.astype(np.float32)
    if dtype == 1:
        return x64.astype(np.float16)
    b = x64.astype(np.float32).view(np.uint32)
    return ((b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
            ).astype(np.uint16)


def paged_decode_q64(q64, k_cache, v_cache, block_tables, context_lens, scale: float, *,
                     dtype: int, num_threads: int = 1) -> np.ndarray:
    """paged_decode with the query rows given in float64 (already widened)."""
    lib = _load()
    q64 = np.ascontiguousarray(q64, np.float64)
    B, Hq, d = q64.shape
    NB, Hkv, bs, _ = k_cache.shape
    MBS = block_tables.shape[1]
    out = np.empty((B, Hq, d), dtype=np.float64)
    _check(lib.ref_paged_decode_q64(_ptr(q64), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                    _ptr(context_lens), float(scale), _ptr(out), B, Hq, Hkv, d,
                                    bs, NB, MBS, int(dtype), int(num_threads)))
    return out
