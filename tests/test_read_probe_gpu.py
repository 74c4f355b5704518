"""The read probe (photon_debug_read_probe), the measuring aid that moves the
decode's K/V runs with the decode's bulk copies and computes nothing: it runs
through a real decode's offsets without raising an error bit, and offsets it
cannot copy (misaligned, past the pool, negative) are skipped and flagged with
bit 1, not followed."""
import numpy as np
import pytest
import torch

import paged_kv_attention_photon_gb300 as P
import workloads as W

pytestmark = pytest.mark.gpu


def _offsets(wl, part):
    bs, hkv = wl.block_size, wl.num_kv_heads
    run = bs * wl.head_dim * wl.elem_bytes
    out = []
    for b in range(wl.num_seqs):
        nblk = -(-int(wl.context_lens[b]) // bs)
        for h in range(hkv):
            out.append((wl.block_tables[b, :nblk].astype(np.int64) * hkv + h) * run)
    return np.concatenate(out), run


def test_read_probe_runs_clean_on_decode_offsets():
    P.build()
    wl = W.llama_b16()
    offs, run = _offsets(wl, 256)
    kc = torch.from_numpy(wl.k_cache.view(np.int16)).cuda()
    vc = torch.from_numpy(wl.v_cache.view(np.int16)).cuda()
    d = torch.from_numpy(offs).cuda()
    P.photon_debug_read_probe(kc, vc, kc.numel() * 2, d, offs.shape[0], run, 16)
    P.photon_debug_read_probe(kc, vc, kc.numel() * 2, d, offs.shape[0], run, 5)
    st, bits = P.photon_get_last_device_error()
    assert st == 0 and bits == 0


def test_read_probe_skips_and_flags_bad_offsets():
    P.build()
    wl = W.tiny()
    kc = torch.from_numpy(wl.k_cache).cuda()
    vc = torch.from_numpy(wl.v_cache).cuda()
    pool = kc.numel() * 4
    run = 16 * 64 * 4
    offs = np.array([0, run, 8, pool - run + 16, pool, -run, 2 * run], np.int64)
    d = torch.from_numpy(offs).cuda()
    P.photon_debug_read_probe(kc, vc, pool, d, offs.shape[0], run, 2)
    st, bits = P.photon_get_last_device_error()
    assert st == 6 and bits == 1, (st, bits)
    # host-side checks launch nothing
    with pytest.raises(P.PhotonError):
        P.photon_debug_read_probe(kc, vc, pool, d, offs.shape[0], 24, 2)      # not x16
    with pytest.raises(P.PhotonError):
        P.photon_debug_read_probe(kc, vc, pool, d, offs.shape[0], 8192, 2)    # > 4096
