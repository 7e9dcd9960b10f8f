"""Splitting one differential-attention forward across ranks (one GPU each).

Every (sequence, diff head) of the forward is independent, so the work splits
with no data exchange. Two ways are provided:

* by sequences: each rank takes a contiguous run of packed sequences, chosen
  so that the causal work (sum of L (L + 1) / 2) is balanced;
* by key/value head groups: each rank takes Hkv / world kv heads and the
  H / world diff heads that read them (tensor-parallel style).

Outputs of the ranks concatenate (along tokens, or along heads) into the
single-device output. `max_over_ranks` is the one collective the benchmark
uses: the slowest rank's time.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple


def sequence_shards(seq_lens: Sequence[int], world: int, causal: bool = True) -> List[Tuple[int, int]]:
    """[start, end) ranges of sequence indices, one per rank, contiguous and
    in order, balancing the per-rank attention work greedily."""
    if world < 1:
        raise ValueError("world must be >= 1")
    cost = [(n * (n + 1) // 2) if causal else n * n for n in seq_lens]
    total = sum(cost)
    bounds = []
    start, acc = 0, 0
    for r in range(world - 1):
        target = total * (r + 1) / world
        end = start
        while end < len(cost) and acc + cost[end] / 2 <= target:
            acc += cost[end]
            end += 1
        bounds.append((start, end))
        start = end
    bounds.append((start, len(cost)))
    return bounds


def token_range(cu_seqlens: Sequence[int], seq_range: Tuple[int, int]) -> Tuple[int, int]:
    """Packed-token range [t0, t1) covered by a range of sequences."""
    return int(cu_seqlens[seq_range[0]]), int(cu_seqlens[seq_range[1]])


def head_shard(num_heads: int, num_kv_heads: int, rank: int, world: int) -> Tuple[range, range]:
    """(diff heads, kv heads) owned by `rank` when kv heads are split evenly.
    Diff head h reads kv head h // (H / Hkv), so a rank owning kv heads
    [g0, g1) owns diff heads [g0 * G, g1 * G)."""
    if num_kv_heads % world != 0:
        raise ValueError("num_kv_heads must be divisible by the world size")
    group = num_heads // num_kv_heads
    per = num_kv_heads // world
    g0, g1 = rank * per, (rank + 1) * per
    return range(g0 * group, g1 * group), range(g0, g1)


def max_over_ranks(value: float) -> float:
    """Maximum of a per-rank scalar (e.g. elapsed milliseconds) over the
    default process group; the value itself when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
