"""Multi-rank split of the forward, on CPU with the gloo backend (world size 2).

Each rank computes its shard with the oracle; the gathered shards must equal
the single-process output exactly (the rows are independent), and the
benchmark's max-over-ranks reduction must return the slowest rank's value.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from differential_attention_diffattn_gb300 import shard
from differential_attention_diffattn_gb300 import workloads as W


def test_sequence_shards_cover_in_order():
    lens = [700, 130, 4096, 128, 2000, 17, 999]
    for world in (1, 2, 3, 4, 7, 9):
        sh = shard.sequence_shards(lens, world)
        assert len(sh) == world
        assert sh[0][0] == 0 and sh[-1][1] == len(lens)
        for (a, b), (c, _) in zip(sh, sh[1:]):
            assert b == c and a <= b


def test_sequence_shards_balance():
    lens = [1000] * 8
    assert shard.sequence_shards(lens, 4) == [(0, 2), (2, 4), (4, 6), (6, 8)]


def test_head_shard():
    hs, ks = shard.head_shard(16, 4, 1, 2)
    assert list(hs) == list(range(8, 16)) and list(ks) == [2, 3]
    with pytest.raises(ValueError):
        shard.head_shard(16, 4, 0, 3)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    from oracle import oracle as orc
    from differential_attention_diffattn_gb300 import shard as sh
    from differential_attention_diffattn_gb300 import workloads as WW

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        wl = WW.Workload("s", "f32", num_heads=8, num_kv_heads=4, d=8, dv=16, depth=5, batch=1, seqlen=1,
                         random_subln=True)
        inp = WW.generate(wl, seed=3, seq_lens=[40, 7, 63, 1, 25])
        li = orc.lambda_init(wl.depth)
        lam = orc.lambda_values(inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2, li)
        cu = inp.cu_seqlens.tolist()
        # by sequences
        s0, s1 = sh.sequence_shards(inp.seq_lens, world)[rank]
        t0, t1 = sh.token_range(cu, (s0, s1))
        sub_cu = [c - t0 for c in cu[s0:s1 + 1]]
        part = orc.forward_rows(sub_cu, inp.q[t0:t1], inp.k[t0:t1], inp.v[t0:t1], lam, li, inp.subln_w,
                                wl.eps, True)
        # by kv head groups
        hs, ks = sh.head_shard(wl.num_heads, wl.num_kv_heads, rank, world)
        hpart = orc.forward_rows(cu, inp.q[:, hs.start:hs.stop], inp.k[:, ks.start:ks.stop],
                                 inp.v[:, ks.start:ks.stop], lam, li, inp.subln_w, wl.eps, True)
        parts = [None] * world
        hparts = [None] * world
        dist.all_gather_object(parts, part)
        dist.all_gather_object(hparts, hpart)
        slowest = sh.max_over_ranks(10.0 * (rank + 1))
        if rank == 0:
            np.save(os.path.join(outdir, "seq.npy"), np.concatenate(parts, axis=0))
            np.save(os.path.join(outdir, "head.npy"), np.concatenate(hparts, axis=1))
            np.save(os.path.join(outdir, "max.npy"), np.array([slowest]))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_split_equals_single(tmp_path):
    from oracle import oracle as orc
    orc.build()
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    wl = W.Workload("s", "f32", num_heads=8, num_kv_heads=4, d=8, dv=16, depth=5, batch=1, seqlen=1,
                    random_subln=True)
    inp = W.generate(wl, seed=3, seq_lens=[40, 7, 63, 1, 25])
    full = orc.forward(inp)
    np.testing.assert_array_equal(np.load(tmp_path / "seq.npy"), full)
    np.testing.assert_array_equal(np.load(tmp_path / "head.npy"), full)
    assert float(np.load(tmp_path / "max.npy")[0]) == 20.0


def test_max_over_ranks_single_process():
    assert shard.max_over_ranks(3.5) == 3.5
