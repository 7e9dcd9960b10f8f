"""Oracle for the context-parallel split of the differential attention: the
partial attention of a block of queries against a block of keys, and the merge
of such partials into the final output.

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark baseline); never used
by the product path, and it shares no code with the CUDA library.

The pages give no context-parallel scheme. The split follows from the
definition of the forward ("DiffTransformer.py", MultiHeadDifferentialAttention
.forward): each component's softmax over all visible keys is the weighted
combination of softmaxes over disjoint key blocks, weighted by each block's
sum of exponentials. So per query row and component c a key block j yields
    lse_c^j = log2 sum_{visible keys k in j} 2^(s log2(e) <q_c, k_c>)
    O_c^j   = softmax over those keys of s <q_c, k_c>, times V
and the merge is, per component, with L = max_j lse_c^j,
    O_c = sum_j 2^(lse_c^j - L) O_c^j / sum_j 2^(lse_c^j - L),
after which the two components are combined with lambda and normalised as in
the forward (the RMSNorm is not linear, so it runs only after both merges).
"""
from __future__ import annotations

import numpy as np


def partial(q, k, v, q_pos, k_pos, causal: bool):
    """q [Tq, H, 2d], k [Tk, Hkv, 2d], v [Tk, Hkv, dv] (fp64); positions of the
    rows in the whole sequence. Returns lse [Tq, H, 2] (log2 units, -inf for a
    row with no visible key) and O1, O2 [Tq, H, dv] (zero for such a row)."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    Tq, H, two_d = q.shape
    Hkv, dv = k.shape[1], v.shape[2]
    d, G = two_d // 2, H // k.shape[1]
    qp, kp = np.asarray(q_pos), np.asarray(k_pos)
    visible = (kp[None, :] <= qp[:, None]) if causal else np.ones((Tq, len(kp)), dtype=bool)
    lse = np.full((Tq, H, 2), -np.inf)
    outs = [np.zeros((Tq, H, dv)), np.zeros((Tq, H, dv))]
    for h in range(H):
        g = h // G
        for c in range(2):
            s = q[:, h, c * d:(c + 1) * d] @ k[:, g, c * d:(c + 1) * d].T * d ** -0.5
            s = np.where(visible, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            has = np.isfinite(m[:, 0])
            e = np.where(visible, np.exp(s - np.where(np.isfinite(m), m, 0.0)), 0.0)
            z = e.sum(axis=1, keepdims=True)
            lse[has, h, c] = (m[has, 0] + np.log(z[has, 0])) / np.log(2.0)
            outs[c][has, h] = (e[has] / z[has]) @ v[:, g]
    return lse, outs[0], outs[1]


def merge(lse_parts, o1_parts, o2_parts, lam, lambda_init: float, w, eps: float):
    """Merge partials [n][T, H, ...] into the forward output [T, H, dv]."""
    lse = np.asarray(lse_parts, dtype=np.float64)
    o = [np.asarray(o1_parts, dtype=np.float64), np.asarray(o2_parts, dtype=np.float64)]
    H = lse.shape[2]
    lam_h = np.broadcast_to(np.asarray(lam, dtype=np.float64).reshape(-1), (H,))
    merged = []
    for c in range(2):
        L = lse[..., c].max(axis=0)                                   # [T, H]
        wt = np.where(np.isfinite(lse[..., c]), np.exp2(lse[..., c] - np.where(np.isfinite(L), L, 0.0)), 0.0)
        merged.append((wt[..., None] * o[c]).sum(axis=0) / wt.sum(axis=0)[..., None])
    D = merged[0] - lam_h[None, :, None] * merged[1]
    r = np.sqrt((D * D).mean(axis=-1, keepdims=True) + eps)
    return D / r * np.asarray(w, dtype=np.float64) * (1.0 - lambda_init)

