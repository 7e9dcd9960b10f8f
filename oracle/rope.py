"""Oracle for the rotary position embedding applied to q and k before the
differential attention.

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark baseline); never used
by the product path, and it shares no code with the CUDA library.

Two placements appear on the pages:
  * "LlamaDiffSdpaAttention.py", forward ("Apply RoPE before splitting"): the
    whole head row of width 2d is rotated with the half-split pairing of
    `apply_rotary_pos_emb` (coordinate i with i + d), and only then chunked into
    q1 | q2. Rotary width R = 2d, so the pairs cross the two components.
  * "Add an isolated implementation of FlashDiffAttention" (test script,
    `apply_rotary_emb(..., interleaved=True)` on the doubled heads): every
    d-wide component is rotated on its own with interleaved pairs (2i, 2i+1).
    Rotary width R = d.
Both are one rule: split the head row into segments of R coordinates; in each
segment, pair i (i < R/2) is (i, i + R/2) ("half") or (2i, 2i+1)
("interleaved"), and is rotated by the angle pos * theta^(-2i/R):
    a' = a cos - b sin,   b' = b cos + a sin.
cos and sin are computed here in fp64 from theta (the pages' modules cache them
and cast them to bf16; the GPU path keeps them in fp32).
"""
from __future__ import annotations

import numpy as np


def tables(theta: float, n_pos: int, rot_dim: int):
    """cos, sin [n_pos, rot_dim/2] in fp64: angle(p, i) = p * theta^(-2i/rot_dim)."""
    i = np.arange(rot_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / rot_dim)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang), np.sin(ang)


def pair_index(rot_dim: int, interleaved: bool):
    """(first, second) coordinate of each pair inside one segment."""
    i = np.arange(rot_dim // 2)
    if interleaved:
        return 2 * i, 2 * i + 1
    return i, i + rot_dim // 2


def apply(x, positions, cos, sin, rot_dim: int, interleaved: bool):
    """Rotate x [tokens, rows, width] (width a multiple of rot_dim) in fp64.
    positions: int [tokens]; cos, sin: [n_pos, rot_dim/2]."""
    x = np.asarray(x, dtype=np.float64)
    tokens, rows, width = x.shape
    assert width % rot_dim == 0 and rot_dim % 2 == 0
    pos = np.asarray(positions, dtype=np.int64)
    c = np.asarray(cos, dtype=np.float64)[pos][:, None, None, :]   # [tokens, 1, 1, R/2]
    s = np.asarray(sin, dtype=np.float64)[pos][:, None, None, :]
    seg = x.reshape(tokens, rows, width // rot_dim, rot_dim)
    first, second = pair_index(rot_dim, interleaved)
    a, b = seg[..., first], seg[..., second]
    out = np.empty_like(seg)
    out[..., first] = a * c - b * s
    out[..., second] = b * c + a * s
    return out.reshape(tokens, rows, width)


def positions_from_cu_seqlens(cu_seqlens):
    """Position of every packed token inside its own sequence (from 0)."""
    cu = [int(v) for v in cu_seqlens]
    return np.concatenate([np.arange(cu[i + 1] - cu[i]) for i in range(len(cu) - 1)] or [np.zeros(0, int)])
