"""Multi-rank host logic on the CPU with two gloo ranks (no GPU).

1. Data parallel (what `bench.py --gpus N` does): sequences are independent,
   so ranks take disjoint sets and need no exchange; the gathered per-rank
   results equal the single-process result.
2. Context parallel for one long sequence: each rank attends over its own
   range of blocks and returns (o, lse); one all-gather of those partials
   and the log-sum-exp merge ("split-KV merge", "vLLM Fork with focus on
   GB10 Homelabs", "Acknowledgments") give the unsplit result.

The arithmetic on each rank is the fp64 oracle; what is under test is the
sharding, the exchange and the merge plan.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from paged_kv_decode_07_gb300 import workloads as W

WORLD = 2
NAME = "int8_b32_l1k_32k_d256"
LENS = [300, 17, 1024, 1, 64, 500]


def shard(B, world, rank):
    """Sequences of one rank: a contiguous, balanced range."""
    lo = B * rank // world
    hi = B * (rank + 1) // world
    return list(range(lo, hi))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        wl = W.make_workload(NAME, seq_lens=LENS)
        h = W.host_arrays(wl)
        cache = oracle.HostCache.from_host_arrays(h, wl.dtype, wl.k_global, wl.v_global)

        # 1. data parallel over sequences
        mine = shard(wl.B, WORLD, rank)
        o, _ = oracle.attend(cache, h["q"][mine], h["block_tables"][mine], h["seq_lens"][mine],
                             wl.softmax_scale, nthreads=1)
        got = [None] * WORLD
        dist.all_gather_object(got, (mine, o))
        dp = np.zeros((wl.B,) + o.shape[1:])
        for ids, oo in got:
            dp[ids] = oo

        # 2. context parallel: rank r takes blocks [r*n/2, (r+1)*n/2) of every sequence
        nblk = [(L + 15) // 16 for L in LENS]
        kb = np.array([16 * (n * rank // WORLD) for n in nblk], np.int32)
        ke = np.array([min(L, 16 * (n * (rank + 1) // WORLD)) for n, L in zip(nblk, LENS)],
                      np.int32)
        po, pl = oracle.attend(cache, h["q"], h["block_tables"], h["seq_lens"], wl.softmax_scale,
                               key_begin=kb, key_end=ke, nthreads=1)
        ten_o = torch.from_numpy(po.reshape(-1, wl.D).copy())
        ten_l = torch.from_numpy(pl.reshape(-1).copy())
        go = [torch.empty_like(ten_o) for _ in range(WORLD)]
        gl = [torch.empty_like(ten_l) for _ in range(WORLD)]
        dist.all_gather(go, ten_o)
        dist.all_gather(gl, ten_l)
        cp, _ = oracle.merge(torch.stack(go).numpy(), torch.stack(gl).numpy())
        if rank == 0:
            q.put((dp, cp.reshape(o.shape[:0] + (wl.B,) + o.shape[1:])))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_data_and_context_parallel():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    dp, cp = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl = W.make_workload(NAME, seq_lens=LENS)
    full, _ = oracle.attend_workload(wl, nthreads=1)
    assert np.array_equal(dp, full)                     # disjoint sequences: identical
    np.testing.assert_allclose(cp, full, atol=1e-12, rtol=0)


def test_shard_covers_every_sequence_once():
    for B in (1, 2, 5, 32, 257):
        for world in (1, 2, 3, 8):
            ids = [i for r in range(world) for i in shard(B, world, r)]
            assert sorted(ids) == list(range(B))
