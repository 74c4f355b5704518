"""The benchmark's multi-GPU host path on CPU: two gloo ranks, no GPU.

Sequences shard across ranks with no exchange on the data path: every rank
draws its own batch of the same recipe (rank 0 the canonical one), and the
only collectives are the timing reductions -- the slowest rank's time and the
summed bytes, sequences and tokens."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo")
    wl = bench.make_workload("llama_b16", rank)
    ms = 1.0 + rank            # rank 1 is the slower one
    res = bench.reduce_over_ranks(dist, ms, 0.5 + rank, wl.decode_bytes(), wl.num_seqs,
                                  wl.tokens_attended())
    out[rank] = (res, wl.decode_bytes(), wl.tokens_attended(), int(wl.context_lens.sum()),
                 wl.seed)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_weak_scaling_reduction():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    r0, r1 = out[0], out[1]
    assert r0[0] == r1[0]                        # every rank sees the same totals
    ms_max, attn_max, tot_bytes, tot_seqs, tot_tokens = r0[0]
    assert ms_max == 2.0 and attn_max == 1.5     # the slowest rank's times
    assert tot_bytes == r0[1] + r1[1]            # work of both ranks
    assert tot_seqs == 32 and tot_tokens == r0[2] + r1[2]
    assert r0[4] != r1[4] and r0[3] != r1[3]     # each rank its own batch


def test_single_process_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(None, 2.0, 1.0, 100, 4, 50) == (2.0, 1.0, 100.0, 4.0, 50.0)
    import workloads as W
    assert bench.make_workload("llama_b16", 0).seed == W.llama_b16().seed


def test_reference_arm_prints_one_json_line():
    """bench.py --impl reference times the fp64 oracle on the host cores."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    import json
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
