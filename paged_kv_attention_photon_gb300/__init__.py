"""Python binding of libphoton_paged.so (GB300 paged decode attention).

Argument marshalling only: every step of the cache write, the block-table
gather, the split-KV attention and the partition merge runs in the CUDA
kernels of the shared library.  There is no Python or CPU fallback: if the
library is missing, importing this package fails.

Buffers may be given as torch CUDA tensors (their ``data_ptr()`` is passed) or
as raw integer device addresses.  ``stream`` is a ``torch.cuda.Stream``, a raw
``cudaStream_t`` integer, or None for torch's current stream.

Functions carry the names of the C entry points declared in
``include/photon_paged.h`` and raise :class:`PhotonError` on a non-OK status.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Tuple

from . import _build

__all__ = [
    "PhotonError", "PagedShape", "build", "library_path", "exported_symbols",
    "photon_cache_write", "photon_paged_decode_workspace_size", "photon_paged_decode",
    "photon_paged_gather", "photon_get_last_device_error", "photon_status_string",
    "photon_paged_decode_plan", "photon_debug_set_attention_events",
    "photon_paged_decode_noalloc", "photon_paged_decode_step",
    "photon_rope_cos_sin", "photon_paged_decode_step_rope", "photon_paged_multi_query",
    "photon_paged_multi_query_workspace_size", "photon_debug_set_multi_query_kernel",
    "photon_debug_set_decode_consumer", "photon_cache_write_fp8",
    "photon_paged_decode_fp8_workspace_size", "photon_paged_decode_fp8",
    "photon_debug_wait_probe", "photon_debug_read_probe", "Scheduler",
    "F32", "F16", "BF16", "STATUS",
]

F32, F16, BF16 = 0, 1, 2
STATUS = {0: "PHOTON_OK", 1: "PHOTON_ERR_INVALID_ARG", 2: "PHOTON_ERR_UNSUPPORTED",
          3: "PHOTON_ERR_MISALIGNED", 4: "PHOTON_ERR_WORKSPACE", 5: "PHOTON_ERR_CUDA",
          6: "PHOTON_ERR_DEVICE_BOUNDS"}


class PhotonError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} "
                         f"({_string(status)})")


class PagedShape(ctypes.Structure):
    """Mirror of photon_paged_shape_t."""

    _fields_ = [("num_seqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("partition_size", ctypes.c_int32)]

    @classmethod
    def make(cls, *, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size=16,
             num_blocks, max_blocks_per_seq, dtype, partition_size=0) -> "PagedShape":
        return cls(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                   max_blocks_per_seq, dtype, partition_size)


def library_path() -> str:
    return _build.LIB_PATH


def build(force: bool = False) -> str:
    """Compile the CUDA sources for sm_103a (in-tree) and return the .so path."""
    return _build.build(force=force)


_lib = None


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "paged_kv_attention_photon_gb300.build() (needs nvcc)")
    lib = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    SP = ctypes.POINTER(PagedShape)
    lib.photon_cache_write.argtypes = [P, P, P, I32, P, P, SP, P]
    lib.photon_paged_decode_workspace_size.argtypes = [SP]
    lib.photon_paged_decode_workspace_size.restype = SZ
    lib.photon_paged_decode.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, SZ, SP, P]
    lib.photon_paged_gather.argtypes = [P, P, P, P, P, P, SP, P]
    lib.photon_get_last_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    lib.photon_status_string.argtypes = [ctypes.c_int]
    lib.photon_status_string.restype = ctypes.c_char_p
    lib.photon_paged_decode_plan.argtypes = [SP] + [ctypes.POINTER(I32)] * 4
    lib.photon_debug_set_attention_events.argtypes = [P, P]
    lib.photon_paged_decode_noalloc.argtypes = [P, P, P, P, P, ctypes.c_float, P, SP, P]
    lib.photon_paged_decode_step.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_float, P, P, SZ,
                                             SP, P]
    lib.photon_rope_cos_sin.argtypes = [ctypes.c_double, I32, I32, P, P]
    lib.photon_paged_decode_step_rope.argtypes = [P, P, P, P, P, P, P, P, P, I32,
                                                  ctypes.c_float, P, P, SZ, SP, P]
    lib.photon_paged_multi_query.argtypes = [P, P, P, P, P, P, I32, I32, ctypes.c_float, P, P,
                                             SZ, SP, P]
    lib.photon_paged_multi_query_workspace_size.argtypes = [SP, I32, I32]
    lib.photon_paged_multi_query_workspace_size.restype = SZ
    lib.photon_debug_wait_probe.argtypes = [ctypes.c_uint64, P]
    lib.photon_debug_wait_probe.restype = ctypes.c_int
    lib.photon_debug_read_probe.argtypes = [P, P, ctypes.c_uint64, P, ctypes.c_int64, I32, I32, P]
    lib.photon_debug_read_probe.restype = ctypes.c_int
    lib.photon_debug_set_multi_query_kernel.argtypes = [I32]
    lib.photon_debug_set_multi_query_kernel.restype = ctypes.c_int
    lib.photon_debug_set_decode_consumer.argtypes = [I32]
    lib.photon_debug_set_decode_consumer.restype = ctypes.c_int
    F32 = ctypes.c_float
    lib.photon_cache_write_fp8.argtypes = [P, P, P, I32, P, P, F32, F32,
                                           ctypes.POINTER(PagedShape), P]
    lib.photon_cache_write_fp8.restype = ctypes.c_int
    lib.photon_paged_decode_fp8_workspace_size.argtypes = [ctypes.POINTER(PagedShape)]
    lib.photon_paged_decode_fp8_workspace_size.restype = SZ
    lib.photon_paged_decode_fp8.argtypes = [P, P, P, P, P, F32, F32, F32, P, P, SZ,
                                            ctypes.POINTER(PagedShape), P]
    lib.photon_paged_decode_fp8.restype = ctypes.c_int
    lib.photon_paged_multi_query.restype = ctypes.c_int
    # host scheduler (include/photon_scheduler.h)
    lib.photon_scheduler_create.argtypes = [P, ctypes.POINTER(P)]
    lib.photon_scheduler_destroy.argtypes = [P]
    lib.photon_scheduler_destroy.restype = None
    lib.photon_scheduler_add_request.argtypes = [P, ctypes.c_int64, I32, I32]
    lib.photon_scheduler_schedule.argtypes = [P, P, P, P, P, P, P]
    lib.photon_scheduler_update.argtypes = [P, P, P, P]
    lib.photon_scheduler_stats.argtypes = [P, P, P, P, P]
    lib.photon_scheduler_request_state.argtypes = [P, ctypes.c_int64, P, P, P, P]
    for fn in ("photon_scheduler_create", "photon_scheduler_add_request",
               "photon_scheduler_schedule", "photon_scheduler_update",
               "photon_scheduler_stats", "photon_scheduler_request_state"):
        getattr(lib, fn).restype = ctypes.c_int
    for fn in ("photon_cache_write", "photon_paged_decode", "photon_paged_gather",
               "photon_get_last_device_error", "photon_paged_decode_plan",
               "photon_debug_set_attention_events", "photon_paged_decode_noalloc",
               "photon_paged_decode_step", "photon_rope_cos_sin",
               "photon_paged_decode_step_rope"):
        getattr(lib, fn).restype = ctypes.c_int
    _lib = lib
    return lib


HEADERS = ("photon_paged.h", "photon_scheduler.h")


def exported_symbols() -> Tuple[str, ...]:
    """Names of the functions declared in the library's public headers."""
    names = set()
    for h in HEADERS:
        text = open(os.path.join(_build.INCLUDE, h)).read()
        names.update(re.findall(r"^\S.*?\b(photon_\w+)\(", text, re.M))
    return tuple(sorted(names))


def _string(status: int) -> str:
    try:
        return _load().photon_status_string(int(status)).decode()
    except Exception:  # pragma: no cover - only used inside error messages
        return "?"


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != 0:
        raise PhotonError(status, where)


# ------------------------------------------------------------------ entry points
def photon_status_string(status: int) -> str:
    return _string(status)


def photon_cache_write(k, v, slot_mapping, num_tokens: int, k_cache, v_cache,
                       shape: PagedShape, stream=None) -> None:
    _check(_load().photon_cache_write(_ptr(k), _ptr(v), _ptr(slot_mapping), int(num_tokens),
                                      _ptr(k_cache), _ptr(v_cache), ctypes.byref(shape),
                                      _stream(stream)), "photon_cache_write")


def photon_paged_decode_workspace_size(shape: PagedShape) -> int:
    return int(_load().photon_paged_decode_workspace_size(ctypes.byref(shape)))


def photon_paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, out,
                        workspace, workspace_bytes: int, shape: PagedShape, stream=None) -> None:
    _check(_load().photon_paged_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(block_tables), _ptr(context_lens),
                                       float(scale), _ptr(out), _ptr(workspace),
                                       int(workspace_bytes), ctypes.byref(shape),
                                       _stream(stream)), "photon_paged_decode")


def photon_paged_decode_step(k_new, v_new, slot_mapping, q, k_cache, v_cache, block_tables,
                             context_lens, scale: float, out, workspace, workspace_bytes: int,
                             shape: PagedShape, stream=None) -> None:
    """Cache write of each sequence's new row + paged decode in one call."""
    _check(_load().photon_paged_decode_step(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                            _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                            _ptr(block_tables), _ptr(context_lens),
                                            float(scale), _ptr(out), _ptr(workspace),
                                            int(workspace_bytes), ctypes.byref(shape),
                                            _stream(stream)), "photon_paged_decode_step")


def photon_rope_cos_sin(base: float, max_positions: int, head_dim: int, table,
                        stream=None) -> None:
    """Fills table ([max_positions][head_dim/2] pairs of fp32) with the rotary
    embedding's (cos, sin) for every position and pair."""
    _check(_load().photon_rope_cos_sin(float(base), int(max_positions), int(head_dim),
                                       _ptr(table), _stream(stream)), "photon_rope_cos_sin")


def photon_paged_decode_step_rope(k_new, v_new, slot_mapping, q, k_cache, v_cache,
                                  block_tables, context_lens, rope_cos_sin, max_positions: int,
                                  scale: float, out, workspace, workspace_bytes: int,
                                  shape: PagedShape, stream=None) -> None:
    """photon_paged_decode_step with q and the new K rows rotated by RoPE at
    position context_len - 1."""
    _check(_load().photon_paged_decode_step_rope(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), _ptr(context_lens), _ptr(rope_cos_sin), int(max_positions),
        float(scale), _ptr(out), _ptr(workspace), int(workspace_bytes), ctypes.byref(shape),
        _stream(stream)), "photon_paged_decode_step_rope")


def photon_paged_multi_query_workspace_size(shape: PagedShape, num_tokens: int,
                                            max_query_len: int) -> int:
    return int(_load().photon_paged_multi_query_workspace_size(
        ctypes.byref(shape), int(num_tokens), int(max_query_len)))


def photon_paged_multi_query(q, k_cache, v_cache, block_tables, context_lens, query_start,
                             num_tokens: int, max_query_len: int, scale: float, out,
                             workspace, workspace_bytes: int, shape: PagedShape,
                             stream=None) -> None:
    """Causal attention of the last n_b tokens of each sequence over its cache."""
    _check(_load().photon_paged_multi_query(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(query_start), int(num_tokens), int(max_query_len), float(scale), _ptr(out),
        _ptr(workspace), int(workspace_bytes), ctypes.byref(shape), _stream(stream)),
        "photon_paged_multi_query")


def photon_debug_wait_probe(limit_ns: int, stream=None) -> None:
    """Runs the bounded-wait self-test kernel (sets device error bit 8)."""
    _check(_load().photon_debug_wait_probe(int(limit_ns), _stream(stream)),
           "photon_debug_wait_probe")


def photon_debug_read_probe(k_cache, v_cache, pool_bytes: int, chunk_offsets, num_chunks: int,
                            chunk_bytes: int, chunks_per_run: int, stream=None) -> None:
    """Copies the K and V chunks at chunk_offsets (device int64 byte offsets)
    into shared memory and nothing else: the decode's read pattern alone."""
    _check(_load().photon_debug_read_probe(
        _ptr(k_cache), _ptr(v_cache), int(pool_bytes), _ptr(chunk_offsets), int(num_chunks),
        int(chunk_bytes), int(chunks_per_run), _stream(stream)), "photon_debug_read_probe")


def photon_debug_set_multi_query_kernel(which: int) -> None:
    """0 = by the plan, 1 = warp-level mma.sync kernel, 2 = tcgen05 kernel."""
    _check(_load().photon_debug_set_multi_query_kernel(int(which)),
           "photon_debug_set_multi_query_kernel")


def photon_debug_set_decode_consumer(which: int) -> None:
    """Decode attention consumer: 0 = by group size, 1 = CUDA cores, 2 = tensor
    cores (fp16/bf16 storage)."""
    _check(_load().photon_debug_set_decode_consumer(int(which)),
           "photon_debug_set_decode_consumer")


def photon_cache_write_fp8(k, v, slot_mapping, num_tokens: int, k_cache, v_cache,
                           k_scale: float, v_scale: float, shape: PagedShape,
                           stream=None) -> None:
    """Quantising cache write into e4m3 pools (uint8 tensors)."""
    _check(_load().photon_cache_write_fp8(_ptr(k), _ptr(v), _ptr(slot_mapping), int(num_tokens),
                                          _ptr(k_cache), _ptr(v_cache), float(k_scale),
                                          float(v_scale), ctypes.byref(shape),
                                          _stream(stream)),
           "photon_cache_write_fp8")


def photon_paged_decode_fp8_workspace_size(shape: PagedShape) -> int:
    return int(_load().photon_paged_decode_fp8_workspace_size(ctypes.byref(shape)))


def photon_paged_decode_fp8(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                            k_scale: float, v_scale: float, out, workspace,
                            workspace_bytes: int, shape: PagedShape, stream=None) -> None:
    """Paged decode over e4m3 K/V pools (uint8 tensors) with fp16 q and out."""
    _check(_load().photon_paged_decode_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                           _ptr(block_tables), _ptr(context_lens),
                                           float(scale), float(k_scale), float(v_scale),
                                           _ptr(out), _ptr(workspace), int(workspace_bytes),
                                           ctypes.byref(shape), _stream(stream)),
           "photon_paged_decode_fp8")


def photon_paged_decode_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                                out, shape: PagedShape, stream=None) -> None:
    """photon_paged_decode with the library's built-in 32 MiB scratch instead of a
    caller-allocated workspace, for callers that cannot allocate device memory."""
    _check(_load().photon_paged_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                               _ptr(block_tables), _ptr(context_lens),
                                               float(scale), _ptr(out), ctypes.byref(shape),
                                               _stream(stream)), "photon_paged_decode_noalloc")


def photon_paged_gather(k_cache, v_cache, block_tables, context_lens, k_dense, v_dense,
                        shape: PagedShape, stream=None) -> None:
    _check(_load().photon_paged_gather(_ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                       _ptr(context_lens), _ptr(k_dense), _ptr(v_dense),
                                       ctypes.byref(shape), _stream(stream)),
           "photon_paged_gather")


def photon_get_last_device_error(stream=None) -> Tuple[int, int]:
    """Returns (status, bits); does not raise for PHOTON_ERR_DEVICE_BOUNDS."""
    bits = ctypes.c_uint32(0)
    st = _load().photon_get_last_device_error(_stream(stream), ctypes.byref(bits))
    if st not in (0, 6):
        raise PhotonError(st, "photon_get_last_device_error")
    return int(st), int(bits.value)


def photon_paged_decode_plan(shape: PagedShape) -> dict:
    vals = [ctypes.c_int32(0) for _ in range(4)]
    _check(_load().photon_paged_decode_plan(ctypes.byref(shape), *[ctypes.byref(v) for v in vals]),
           "photon_paged_decode_plan")
    return dict(partition_size=vals[0].value, max_partitions=vals[1].value,
                attention_ctas=vals[2].value, kernels_per_call=vals[3].value)


def photon_debug_set_attention_events(start_event=None, stop_event=None) -> None:
    def raw(ev):
        if ev is None:
            return None
        return ev.cuda_event if hasattr(ev, "cuda_event") else int(ev)
    _check(_load().photon_debug_set_attention_events(raw(start_event), raw(stop_event)),
           "photon_debug_set_attention_events")


from .scheduler import Scheduler  # noqa: E402  (needs _load and PhotonError above)
