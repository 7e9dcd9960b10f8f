"""Context-parallel split on CPU: the zigzag assignment, and the ring exchange
with world sizes 2 and 3 over gloo. The ring's arithmetic is stood in for by
the partial / merge oracle (oracle/partial.py) so that the test checks the
exchange and the schedule: every rank must receive every key chunk it needs
exactly once, and the merged outputs, gathered, must equal the independent C
oracle's forward of the whole sequence."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from differential_attention_diffattn_gb300 import context_parallel as cp


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_zigzag_covers_every_chunk_once_with_equal_work(world):
    owned = [c for r in range(world) for c in cp.zigzag_chunk_ids(world, r)]
    assert sorted(owned) == list(range(2 * world))
    work = {sum(cp.causal_blocks(c) for c in cp.zigzag_chunk_ids(world, r)) for r in range(world)}
    assert work == {2 * world + 1}


def test_split_zigzag_views():
    x = torch.arange(24).view(12, 2)
    ch = cp.split_zigzag(x, 3, 1)
    assert sorted(ch) == [1, 4]
    assert torch.equal(ch[1], x[2:4]) and torch.equal(ch[4], x[8:10])
    with pytest.raises(ValueError):
        cp.split_zigzag(torch.zeros(10, 2), 3, 0)


class OracleKernels:
    """Stand-in arithmetic for the CPU test: the fp64 partial / merge oracle."""

    def __init__(self, lam, li, w, eps, chunk, calls):
        self.lam, self.li, self.w, self.eps, self.chunk, self.calls = lam, li, w, eps, chunk, calls

    def alloc_parts(self, q, n, dv):
        return [None] * n

    def partial(self, q, k, v, causal, parts, j):
        from oracle import partial as op
        pos = np.arange(q.shape[0])
        parts[j] = op.partial(q.numpy(), k.numpy(), v.numpy(), pos, pos, causal)
        self.calls.append(causal)

    def merge(self, parts, n):
        from oracle import partial as op
        assert all(p is not None for p in parts[:n])
        return op.merge([p[0] for p in parts[:n]], [p[1] for p in parts[:n]], [p[2] for p in parts[:n]],
                        self.lam, self.li, self.w, self.eps)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    sys.path.insert(0, os.path.join(root, "tests"))
    from oracle import oracle as orc
    from differential_attention_diffattn_gb300 import context_parallel as cpp
    from differential_attention_diffattn_gb300 import workloads as WW
    from test_context_parallel import OracleKernels

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        wl = WW.Workload("cp", "f32", num_heads=4, num_kv_heads=2, d=8, dv=16, depth=3, batch=1, seqlen=1,
                         random_subln=True)
        T = 2 * world * 9
        inp = WW.generate(wl, seed=17, seq_lens=[T])
        li = orc.lambda_init(wl.depth)
        lam = orc.lambda_values(inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2, li)
        q, k, v = inp.q.double(), inp.k.double(), inp.v.double()
        calls = []
        kern = OracleKernels(lam, li, inp.subln_w.double().numpy(), wl.eps, T // (2 * world), calls)
        outs = cpp.ring_forward(cpp.split_zigzag(q, world, rank), cpp.split_zigzag(k, world, rank),
                                cpp.split_zigzag(v, world, rank), kern)
        gathered = [None] * world
        dist.all_gather_object(gathered, (outs, len(calls), sum(calls)))
        if rank == 0:
            c = T // (2 * world)
            full = np.zeros((T, wl.num_heads, wl.dv))
            for o, _, _ in gathered:
                for a, y in o.items():
                    full[a * c:(a + 1) * c] = y
            np.save(os.path.join(outdir, "cp.npy"), full)
            want = orc.forward_rows(inp.cu_seqlens, q, k, v, lam, li, inp.subln_w, wl.eps, True)
            np.save(os.path.join(outdir, "want.npy"), want)
            np.save(os.path.join(outdir, "calls.npy"), np.array([(n, d) for _, n, d in gathered]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ring_forward_gloo(tmp_path, world):
    port = _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True, start_method="spawn")
    got, want = np.load(tmp_path / "cp.npy"), np.load(tmp_path / "want.npy")
    np.testing.assert_allclose(got, want, atol=1e-11)
    calls = np.load(tmp_path / "calls.npy")
    # every rank: 2N + 1 blocks, two of them diagonal (causal)
    assert (calls[:, 0] == 2 * world + 1).all() and (calls[:, 1] == 2).all()
