"""Shared helpers for the GPU tests: move a workload's host bytes to the device
and run the library's calls on them.  The oracle is called by the tests
themselves, never from here."""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_attention_photon_gb300 as P
import workloads as W

TOL = {W.DTYPE_F16: 2e-3, W.DTYPE_F32: 1e-4}
# bf16 output keeps 8 significant bits: rounding alone can move |o| by 2^-9 |o|.
BF16_RTOL, BF16_ATOL = 2.0 ** -8, 2e-4


def dev(a: np.ndarray) -> torch.Tensor:
    """Raw-byte copy of a host array to the GPU (bf16 travels as int16 bits)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def host(t: torch.Tensor, like: np.ndarray) -> np.ndarray:
    arr = t.cpu().numpy()
    return arr.view(like.dtype).reshape(like.shape) if arr.dtype != like.dtype else arr


def shape_of(wl: W.Workload, partition_size: int = 0) -> P.PagedShape:
    return P.PagedShape.make(partition_size=partition_size, **wl.shape_dict())


def to_float64(out: torch.Tensor, dtype: int) -> np.ndarray:
    if dtype == W.DTYPE_BF16:
        bits = out.cpu().numpy().view(np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    return out.cpu().numpy().astype(np.float64)


class DeviceWorkload:
    """Device copies of one workload plus an output and a garbage-filled workspace."""

    def __init__(self, wl: W.Workload, partition_size: int = 0):
        self.wl = wl
        self.shape = shape_of(wl, partition_size)
        self.q = dev(wl.q)
        self.k_cache = dev(wl.k_cache)
        self.v_cache = dev(wl.v_cache)
        self.block_tables = dev(wl.block_tables)
        self.context_lens = dev(wl.context_lens)
        self.k_new = dev(wl.k_new)
        self.v_new = dev(wl.v_new)
        self.slot_mapping = dev(wl.slot_mapping)
        self.out = torch.full(wl.q.shape, -1, dtype=self.q.dtype, device="cuda")
        self.ws_bytes = P.photon_paged_decode_workspace_size(self.shape)
        # the workspace needs no initialisation: start from NaN bytes
        self.ws = torch.full((max(self.ws_bytes, 16),), 0xFF, dtype=torch.uint8, device="cuda")

    def set_partition(self, partition_size: int) -> None:
        self.shape = shape_of(self.wl, partition_size)
        need = P.photon_paged_decode_workspace_size(self.shape)
        if need > self.ws.numel():
            self.ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
        self.ws_bytes = need

    def cache_write(self, stream=None) -> None:
        P.photon_cache_write(self.k_new, self.v_new, self.slot_mapping,
                             self.wl.slot_mapping.shape[0], self.k_cache, self.v_cache,
                             self.shape, stream)

    def step(self, stream=None) -> None:
        """Fused cache write + decode (photon_paged_decode_step)."""
        P.photon_paged_decode_step(self.k_new, self.v_new, self.slot_mapping, self.q,
                                   self.k_cache, self.v_cache, self.block_tables,
                                   self.context_lens, self.wl.scale, self.out, self.ws,
                                   self.ws_bytes, self.shape, stream)

    def step_rope(self, table: torch.Tensor, max_positions: int, stream=None) -> None:
        """Fused cache write + decode with RoPE (photon_paged_decode_step_rope)."""
        P.photon_paged_decode_step_rope(self.k_new, self.v_new, self.slot_mapping, self.q,
                                        self.k_cache, self.v_cache, self.block_tables,
                                        self.context_lens, table, max_positions,
                                        self.wl.scale, self.out, self.ws, self.ws_bytes,
                                        self.shape, stream)

    def decode(self, scale=None, stream=None) -> None:
        P.photon_paged_decode(self.q, self.k_cache, self.v_cache, self.block_tables,
                              self.context_lens, self.wl.scale if scale is None else scale,
                              self.out, self.ws, self.ws_bytes, self.shape, stream)

    def out_f64(self) -> np.ndarray:
        return to_float64(self.out, self.wl.dtype)


def rope_table(base: float, max_positions: int, head_dim: int) -> torch.Tensor:
    """Device (cos, sin) table from photon_rope_cos_sin, fp32 [max_positions][d/2][2]."""
    t = torch.empty((max_positions, head_dim // 2, 2), dtype=torch.float32, device="cuda")
    P.photon_rope_cos_sin(base, max_positions, head_dim, t)
    return t


def assert_close(got: np.ndarray, want: np.ndarray, dtype: int, what: str = "") -> float:
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - want)
    if dtype == W.DTYPE_BF16:
        bound = BF16_ATOL + BF16_RTOL * np.abs(want)
        worst = float((err - bound).max(initial=-1.0))
        assert worst <= 0, f"{what}: bf16 error exceeds bound by {worst}"
        return float(err.max(initial=0.0))
    tol = TOL[dtype]
    m = float(err.max(initial=0.0))
    assert m <= tol, f"{what}: max abs error {m} > {tol}"
    return m
