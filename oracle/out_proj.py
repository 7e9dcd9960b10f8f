"""Oracle for the output projection after the differential attention.

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark baseline); never used
by the product path, and it shares no code with the CUDA library.

"LlamaDiffSdpaAttention.py", forward: the attention output [tokens, H, dv] is
reshaped to [tokens, H * dv] and passed through o_proj, an nn.Linear(H * dv,
hidden_size, bias=False); "DiffTransformer.py" has the same W_o without bias.
nn.Linear computes y = x W^T with W stored [out_features, in_features]. The
oracle is that product in fp64 (a library matmul).
"""
from __future__ import annotations

import numpy as np


def out_proj(x, w):
    """x [tokens, K] (or [tokens, H, dv] with K = H * dv), w [N, K] -> [tokens, N] in fp64."""
    x = np.asarray(x, dtype=np.float64)
    x = x.reshape(x.shape[0], -1)
    return x @ np.asarray(w, dtype=np.float64).T
