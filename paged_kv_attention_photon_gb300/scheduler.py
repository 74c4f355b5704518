"""ctypes marshalling of the host scheduler (include/photon_scheduler.h).

Every decision is taken by the library's C++ scheduler; this class only owns
the handle and the host output arrays and turns them into numpy views.
"""
from __future__ import annotations

import ctypes
from typing import Dict, Optional

import numpy as np

WAITING, RUNNING, PREEMPTED, FINISHED = 0, 1, 2, 3


class SchedulerConfig(ctypes.Structure):
    """Mirror of photon_scheduler_config_t."""

    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("max_seqs", ctypes.c_int32),
                ("max_step_tokens", ctypes.c_int32)]


class ScheduleResult(ctypes.Structure):
    """Mirror of photon_schedule_t."""

    _fields_ = [("num_rows", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
                ("num_decode", ctypes.c_int32), ("num_admitted", ctypes.c_int32),
                ("num_preempted", ctypes.c_int32), ("free_blocks", ctypes.c_int32)]


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


class Scheduler:
    """One photon_scheduler_t.  schedule() returns a dict of numpy views of the
    first num_rows rows / num_tokens slots of this object's output buffers
    (valid until the next schedule(); copy them to keep them) plus the counts.
    Block-table rows hold the row's blocks first; entries past them are
    stale (no kernel reads them)."""

    def __init__(self, *, num_blocks: int, block_size: int, max_blocks_per_seq: int,
                 max_seqs: int, max_step_tokens: int):
        from . import PhotonError, _load
        self._lib = _load()
        self._err = PhotonError
        self.cfg = SchedulerConfig(num_blocks, block_size, max_blocks_per_seq, max_seqs,
                                   max_step_tokens)
        h = ctypes.c_void_p(None)
        st = self._lib.photon_scheduler_create(ctypes.byref(self.cfg), ctypes.byref(h))
        if st != 0:
            raise PhotonError(st, "photon_scheduler_create")
        self._h = h
        self._ids = np.zeros(max_seqs, np.int64)
        self._qlen = np.zeros(max_seqs, np.int32)
        self._ctx = np.zeros(max_seqs, np.int32)
        self._tables = np.full((max_seqs, max_blocks_per_seq), -1, np.int32)
        self._slots = np.zeros(max_step_tokens, np.int64)
        self._fin = np.zeros(max_seqs, np.int64)
        # the buffers never move: their addresses, and the result structs, once
        self._out_ptrs = tuple(_p(a) for a in (self._ids, self._qlen, self._ctx, self._tables,
                                               self._slots))
        self._fin_ptr = _p(self._fin)
        self._res = ScheduleResult()
        self._res_ref = ctypes.byref(self._res)
        self._nf = ctypes.c_int32(0)
        self._nf_ref = ctypes.byref(self._nf)

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.photon_scheduler_destroy(self._h)
            self._h = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.close()
        except Exception:  # pragma: no cover - interpreter shutdown
            pass

    def _check(self, st: int, where: str) -> None:
        if st != 0:
            raise self._err(st, where)

    def add_request(self, request_id: int, prompt_len: int, max_new_tokens: int) -> None:
        self._check(self._lib.photon_scheduler_add_request(self._h, int(request_id),
                                                           int(prompt_len),
                                                           int(max_new_tokens)),
                    "photon_scheduler_add_request")

    def schedule(self) -> Dict[str, object]:
        res = self._res
        self._check(self._lib.photon_scheduler_schedule(self._h, *self._out_ptrs, self._res_ref),
                    "photon_scheduler_schedule")
        n, t = res.num_rows, res.num_tokens
        return {"request_ids": self._ids[:n], "query_lens": self._qlen[:n],
                "context_lens": self._ctx[:n], "block_tables": self._tables[:n],
                "slot_mapping": self._slots[:t], "num_rows": n, "num_tokens": t,
                "num_decode": res.num_decode, "num_admitted": res.num_admitted,
                "num_preempted": res.num_preempted, "free_blocks": res.free_blocks}

    def update(self, stop: Optional[np.ndarray] = None) -> np.ndarray:
        stop_arr = None if stop is None else np.ascontiguousarray(stop, np.uint8)
        self._check(self._lib.photon_scheduler_update(
            self._h, None if stop_arr is None else _p(stop_arr), self._fin_ptr, self._nf_ref),
            "photon_scheduler_update")
        return self._fin[:self._nf.value].copy()

    def stats(self) -> Dict[str, int]:
        v = [ctypes.c_int32(0) for _ in range(4)]
        self._check(self._lib.photon_scheduler_stats(self._h, *[ctypes.addressof(x) for x in v]),
                    "photon_scheduler_stats")
        return dict(waiting=v[0].value, running=v[1].value, finished=v[2].value,
                    free_blocks=v[3].value)

    def request_state(self, request_id: int) -> Dict[str, int]:
        v = [ctypes.c_int32(0) for _ in range(4)]
        self._check(self._lib.photon_scheduler_request_state(
            self._h, int(request_id), *[ctypes.addressof(x) for x in v]),
            "photon_scheduler_request_state")
        return dict(state=v[0].value, computed=v[1].value, generated=v[2].value,
                    blocks=v[3].value)
