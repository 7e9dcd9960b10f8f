"""Seeded synthetic workloads for the causal differential-attention forward.

This module is shared by the tests, the benchmark and the smoke check. It only
draws random numbers and fixes shapes; it holds none of the method's arithmetic
(no lambda_init, no softmax, no normalisation), so that the CUDA path and the
CPU oracle can both consume its output without sharing any computation.

Shapes follow the pages:
  * q  [tokens, H,   2d]  -- per diff head the two query components Q1 | Q2
    ("Differential Transformer" PyTorch module, forward: Q.chunk(2, dim=-1)),
  * k  [tokens, Hkv, 2d]  -- K1 | K2 of each key/value head,
  * v  [tokens, Hkv, dv]  -- one shared value of width dv = 2d,
  * lambda vectors of length d (shared by all heads, as in the Llama gist's
    lambda_q1 ... lambda_k2 parameters, N(0, 0.1)), optionally per head [H, d]
    (as in the PyTorch module's per-head parameters),
  * the sub-layer RMSNorm weight [dv] (ones at initialisation).

Draw order per workload (one CPU torch.Generator seeded with `seed`):
varlen lengths -> q -> k -> v -> lambda_q1 -> lambda_k1 -> lambda_q2 -> lambda_k2
(-> subln weight, only when a random weight is requested).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and generation recipe of one synthetic forward call."""

    name: str
    dtype: str               # "f32" or "bf16": the element type of q, k, v and out
    num_heads: int           # H diff heads
    num_kv_heads: int        # Hkv key/value diff heads (H % Hkv == 0)
    d: int                   # component dim of Q1, Q2, K1, K2
    dv: int                  # value dim per diff head (2d on every page)
    depth: int               # layer index l >= 1 that fixes lambda_init
    causal: bool = True
    batch: int = 0           # dense mode: batch x seqlen tokens
    seqlen: int = 0
    varlen_total: int = 0    # varlen mode: total packed tokens
    varlen_min: int = 0      # lengths drawn uniformly from [varlen_min, varlen_max]
    varlen_max: int = 0
    lambda_per_head: bool = False
    random_subln: bool = False
    eps: float = 1e-5

    @property
    def varlen(self) -> bool:
        return self.varlen_total > 0


# The five workloads of the benchmark table: shapes from the pages (the
# Llama-3.2-1B gist, the FlashDiffAttention pull request test) regrouped as
# diff heads of component dim 64 and value dim 128.
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", "f32", num_heads=2, num_kv_heads=2, d=16, dv=32,
                         depth=1, batch=1, seqlen=64),
    "b2_t512_gqa": Workload("b2_t512_gqa", "bf16", num_heads=16, num_kv_heads=4, d=64, dv=128,
                            depth=12, batch=2, seqlen=512),
    "llama1b_b4_t2048": Workload("llama1b_b4_t2048", "bf16", num_heads=16, num_kv_heads=4, d=64,
                                 dv=128, depth=8, batch=4, seqlen=2048),
    "long_t16384": Workload("long_t16384", "bf16", num_heads=16, num_kv_heads=16, d=64, dv=128,
                            depth=12, batch=1, seqlen=16384),
    "varlen_32k": Workload("varlen_32k", "bf16", num_heads=16, num_kv_heads=4, d=64, dv=128,
                           depth=24, varlen_total=32768, varlen_min=128, varlen_max=4096),
}
WORKLOAD_ORDER = ["tiny_f32", "b2_t512_gqa", "llama1b_b4_t2048", "long_t16384", "varlen_32k"]


@dataclasses.dataclass
class Inputs:
    """One generated call: CPU tensors plus the packed-sequence table."""

    wl: Workload
    seq_lens: List[int]        # length of every sequence, in packing order
    cu_seqlens: torch.Tensor   # int32 [num_seqs + 1], prefix sums of seq_lens
    q: torch.Tensor            # [tokens, H, 2d]   (f32 or bf16)
    k: torch.Tensor            # [tokens, Hkv, 2d]
    v: torch.Tensor            # [tokens, Hkv, dv]
    lambda_q1: torch.Tensor    # f32 [d] or [H, d]
    lambda_k1: torch.Tensor
    lambda_q2: torch.Tensor
    lambda_k2: torch.Tensor
    subln_w: torch.Tensor      # f32 [dv]

    @property
    def tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def max_seqlen(self) -> int:
        return max(self.seq_lens) if self.seq_lens else 0


def draw_varlen_lengths(gen: torch.Generator, total: int, lo: int, hi: int) -> List[int]:
    """Lengths uniform on {lo..hi}, appended while the running sum is below
    `total`; the last sequence takes whatever remains (it may be shorter than lo)."""
    lens: List[int] = []
    acc = 0
    while acc < total:
        n = int(torch.randint(lo, hi + 1, (1,), generator=gen).item())
        n = min(n, total - acc)
        lens.append(n)
        acc += n
    return lens


def generate(wl: Workload, seed: int = 0, seq_lens: Optional[List[int]] = None) -> Inputs:
    """Draw one seeded set of inputs for `wl` on the CPU.

    q, k, v are N(0, 1) in fp32, then rounded to bf16 for bf16 workloads; the
    lambda vectors are N(0, 0.1^2) in fp32 and stay fp32; the sub-layer norm
    weight is ones unless `wl.random_subln` (then U(0.5, 1.5)). `seq_lens`
    overrides the dense / drawn sequence lengths (used by edge-case tests).
    """
    gen = torch.Generator().manual_seed(seed)
    if seq_lens is None:
        if wl.varlen:
            seq_lens = draw_varlen_lengths(gen, wl.varlen_total, wl.varlen_min, wl.varlen_max)
        else:
            seq_lens = [wl.seqlen] * wl.batch
    seq_lens = [int(n) for n in seq_lens]
    cu = torch.zeros(len(seq_lens) + 1, dtype=torch.int32)
    if seq_lens:
        cu[1:] = torch.cumsum(torch.tensor(seq_lens, dtype=torch.int64), 0).to(torch.int32)
    tokens = int(cu[-1])
    H, Hkv, d, dv = wl.num_heads, wl.num_kv_heads, wl.d, wl.dv
    q = torch.randn(tokens, H, 2 * d, generator=gen, dtype=torch.float32)
    k = torch.randn(tokens, Hkv, 2 * d, generator=gen, dtype=torch.float32)
    v = torch.randn(tokens, Hkv, dv, generator=gen, dtype=torch.float32)
    if wl.dtype == "bf16":
        q, k, v = q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
    lshape = (H, d) if wl.lambda_per_head else (d,)
    lam = [torch.randn(lshape, generator=gen, dtype=torch.float32) * 0.1 for _ in range(4)]
    if wl.random_subln:
        w = torch.rand(dv, generator=gen, dtype=torch.float32) + 0.5
    else:
        w = torch.ones(dv, dtype=torch.float32)
    return Inputs(wl, seq_lens, cu, q, k, v, lam[0], lam[1], lam[2], lam[3], w)


def with_overrides(wl: Workload, **kw) -> Workload:
    """A copy of `wl` with some fields replaced (edge-case shapes in tests)."""
    return dataclasses.replace(wl, **kw)


# ----------------------------------------------------------------- cache ---

@dataclasses.dataclass(frozen=True)
class KvWorkload:
    """New queries against a key/value cache (decode or a short query block)."""

    name: str
    num_heads: int
    num_kv_heads: int
    d: int
    dv: int
    depth: int
    batch: int
    q_len: int            # new query tokens per sequence
    capacity: int         # cache rows per sequence
    len_min: int = 0      # valid cache lengths drawn uniformly from [len_min, capacity];
                          # 0: every sequence holds `capacity` keys
    causal: bool = True
    lambda_per_head: bool = False
    random_subln: bool = False
    eps: float = 1e-5


KV_WORKLOADS = {
    # one decoded token per sequence, Llama-3.2-1B-shaped heads (16 diff heads
    # over 4 kv heads), 16k-token caches
    "decode_b8_c16384": KvWorkload("decode_b8_c16384", num_heads=16, num_kv_heads=4, d=64, dv=128, depth=12,
                                   batch=8, q_len=1, capacity=16384),
    # ragged caches, 4 new tokens per sequence (a short speculative block)
    "decode_b16_q4_ragged": KvWorkload("decode_b16_q4_ragged", num_heads=16, num_kv_heads=4, d=64, dv=128,
                                       depth=12, batch=16, q_len=4, capacity=8192, len_min=512),
}


@dataclasses.dataclass
class KvInputs:
    wl: KvWorkload
    cache_seqlens: torch.Tensor   # int32 [batch]
    q: torch.Tensor               # bf16 [batch, q_len, H, 2d]
    k_cache: torch.Tensor         # bf16 [batch, capacity, Hkv, 2d]
    v_cache: torch.Tensor         # bf16 [batch, capacity, Hkv, dv]
    lambda_q1: torch.Tensor
    lambda_k1: torch.Tensor
    lambda_q2: torch.Tensor
    lambda_k2: torch.Tensor
    subln_w: torch.Tensor


def generate_kv(wl: KvWorkload, seed: int = 0, lengths: Optional[List[int]] = None) -> KvInputs:
    """Seeded cache inputs. Draw order: cache lengths -> q -> k_cache -> v_cache
    -> lambda_q1, lambda_k1, lambda_q2, lambda_k2 (-> subln weight). Cache rows
    beyond a sequence's length hold random values too: they must not matter."""
    gen = torch.Generator().manual_seed(seed)
    B, H, Hkv, d, dv = wl.batch, wl.num_heads, wl.num_kv_heads, wl.d, wl.dv
    if lengths is None:
        if wl.len_min > 0:
            lengths = [int(torch.randint(max(wl.len_min, wl.q_len), wl.capacity + 1, (1,), generator=gen))
                       for _ in range(B)]
        else:
            lengths = [wl.capacity] * B
    lens = torch.tensor(lengths, dtype=torch.int32)
    q = torch.randn(B, wl.q_len, H, 2 * d, generator=gen).to(torch.bfloat16)
    k = torch.randn(B, wl.capacity, Hkv, 2 * d, generator=gen).to(torch.bfloat16)
    v = torch.randn(B, wl.capacity, Hkv, dv, generator=gen).to(torch.bfloat16)
    lshape = (H, d) if wl.lambda_per_head else (d,)
    lam = [torch.randn(lshape, generator=gen, dtype=torch.float32) * 0.1 for _ in range(4)]
    w = (torch.rand(dv, generator=gen) + 0.5) if wl.random_subln else torch.ones(dv)
    return KvInputs(wl, lens, q, k, v, lam[0], lam[1], lam[2], lam[3], w.float())
