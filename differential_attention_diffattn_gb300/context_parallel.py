"""Context-parallel split of one long sequence across ranks.

The sequence (T tokens) is cut into 2N equal chunks; rank r holds chunks r and
2N - 1 - r (the zigzag assignment: under the causal mask chunk a attends to
chunks 0..a, so pairing an early chunk with a late one gives every rank the
same number of (query chunk, key chunk) blocks, 2N + 1).

Per query chunk a and key chunk b <= a, the training forward (diffattn_fwd_train)
yields a partial: per component the log2-sum-exp and the output normalised over
that key chunk (causal mask on the diagonal block a == b, none below it). The
merge (diffattn_merge_partials) combines the partials of a query chunk per
component, weighted by their sums of exponentials, and only then applies the
combine with lambda and the RMSNorm ("DiffTransformer.py",
MultiHeadDifferentialAttention.forward; the RMSNorm is not linear, so it cannot
run per block).

Exchange: the K/V chunks travel around a ring of ranks (N - 1 steps of one
send to the next rank and one receive from the previous one); a rank computes
the partials of the chunks it holds while the next pair is in flight. Nothing
else crosses ranks: the outputs stay with the rank that owns the query chunk.
"""
from __future__ import annotations

from typing import Callable, Dict, List, Optional, Tuple


def zigzag_chunk_ids(world: int, rank: int) -> Tuple[int, int]:
    """The two chunk indices (of 2 * world) that `rank` owns."""
    if not 0 <= rank < world:
        raise ValueError("rank outside the group")
    return rank, 2 * world - 1 - rank


def causal_blocks(chunk: int) -> int:
    """(query chunk, key chunk) blocks chunk `chunk` needs under the causal mask."""
    return chunk + 1


def split_zigzag(x, world: int, rank: int):
    """This rank's two chunks of x (tokens along dim 0), as a dict id -> view."""
    n = 2 * world
    if x.shape[0] % n != 0:
        raise ValueError(f"{x.shape[0]} tokens do not split into {n} equal chunks")
    c = x.shape[0] // n
    return {i: x[i * c:(i + 1) * c] for i in zigzag_chunk_ids(world, rank)}


class GpuKernels:
    """The library's kernels for one rank: partials by diffattn_fwd_train, the
    merge by diffattn_merge_partials. lam: device fp32 [1] or [H]."""

    def __init__(self, lam, lambda_init: float, subln_w, eps: float = 1e-5, stream=None):
        self.lam, self.lambda_init, self.subln_w, self.eps, self.stream = lam, lambda_init, subln_w, eps, stream

    def alloc_parts(self, q, n: int, dv: int):
        import torch
        T, H = q.shape[0], q.shape[1]
        return (torch.empty(n, T, H, 2, dtype=torch.float32, device=q.device),
                torch.empty(n, T, H, dv, dtype=torch.float32, device=q.device),
                torch.empty(n, T, H, dv, dtype=torch.float32, device=q.device))

    def partial(self, q, k, v, causal: bool, parts, j: int, scratch=None):
        from . import _lib
        lse, o1, o2 = parts
        _lib.diffattn_fwd_train(q, k, v, self.lam, self.lambda_init, self.subln_w, causal=causal, eps=self.eps,
                                out=scratch, lse=lse[j], o1=o1[j], o2=o2[j], stream=self.stream)

    def merge(self, parts, n: int):
        from . import _lib
        lse, o1, o2 = parts
        return _lib.diffattn_merge_partials(lse[:n], o1[:n], o2[:n], self.lam, self.lambda_init, self.subln_w,
                                            eps=self.eps, stream=self.stream)


def local_forward(q_chunks: Dict[int, object], kv_chunks: Dict[int, Tuple[object, object]], kernels) -> Dict:
    """Outputs of the query chunks from key/value chunks that are all present
    (one GPU, or after the exchange): every block b <= a, then one merge per a."""
    outs = {}
    for a, q in sorted(q_chunks.items()):
        dv = kv_chunks[a][1].shape[-1]
        parts = kernels.alloc_parts(q, causal_blocks(a), dv)
        for j, b in enumerate(range(causal_blocks(a))):
            k, v = kv_chunks[b]
            kernels.partial(q, k, v, a == b, parts, j)
        outs[a] = kernels.merge(parts, causal_blocks(a))
    return outs


def ring_forward(q_chunks: Dict[int, object], k_chunks: Dict[int, object], v_chunks: Dict[int, object], kernels,
                 group=None, wait_hook: Optional[Callable[[], None]] = None) -> Dict:
    """Context-parallel forward of this rank's query chunks. k_chunks / v_chunks
    hold this rank's own two chunks (same ids as q_chunks). The K/V chunk pairs
    go around the ring; partials are computed for every held chunk b <= a as the
    pairs arrive, and each query chunk is merged once all its blocks are in."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    ids = sorted(q_chunks)
    dv = next(iter(v_chunks.values())).shape[-1]
    parts = {a: kernels.alloc_parts(q_chunks[a], causal_blocks(a), dv) for a in ids}
    filled = {a: 0 for a in ids}

    def consume(held: Dict[int, Tuple[object, object]]):
        for a in ids:
            for b, (k, v) in sorted(held.items()):
                if b <= a:
                    kernels.partial(q_chunks[a], k, v, a == b, parts[a], filled[a])
                    filled[a] += 1

    own = sorted(k_chunks)
    cur_k = torch.stack([k_chunks[i] for i in own])
    cur_v = torch.stack([v_chunks[i] for i in own])
    cur_ids = own
    nxt, prv = (rank + 1) % world, (rank - 1) % world
    for step in range(world):
        reqs: List = []
        if step < world - 1:
            recv_k, recv_v = torch.empty_like(cur_k), torch.empty_like(cur_v)
            ops = [dist.P2POp(dist.isend, cur_k, nxt, group), dist.P2POp(dist.isend, cur_v, nxt, group),
                   dist.P2POp(dist.irecv, recv_k, prv, group), dist.P2POp(dist.irecv, recv_v, prv, group)]
            reqs = dist.batch_isend_irecv(ops)
        consume({i: (cur_k[n], cur_v[n]) for n, i in enumerate(cur_ids)})
        if reqs:
            for r in reqs:
                r.wait()
            if wait_hook is not None:
                wait_hook()
            cur_k, cur_v = recv_k, recv_v
            cur_ids = list(zigzag_chunk_ids(world, (rank - step - 1) % world))
    for a in ids:
        if filled[a] != causal_blocks(a):
            raise RuntimeError(f"query chunk {a}: {filled[a]} of {causal_blocks(a)} key blocks arrived")
    return {a: kernels.merge(parts[a], causal_blocks(a)) for a in ids}
