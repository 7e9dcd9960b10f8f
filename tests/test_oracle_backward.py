"""Pins for the gradient oracle (CPU only).

The autograd gradients of the fp64 restatement are checked against central
finite differences of the independent C oracle (a different implementation of
the forward), element by element for every input, and against the closed-form
fact that with eps = 0 the output does not change along V (y(cV) = y(V)), so
the directional derivative <dV, V> vanishes.
"""
import numpy as np
import pytest
import torch

from oracle import backward as ob
from oracle import oracle as orc
from differential_attention_diffattn_gb300 import workloads as W


def _case(seed, causal=True, lens=(5, 9), H=4, Hkv=2, d=8, per_head=False):
    wl = W.Workload("g", "f32", num_heads=H, num_kv_heads=Hkv, d=d, dv=2 * d, depth=4, causal=causal,
                    batch=1, seqlen=1, random_subln=True, lambda_per_head=per_head)
    inp = W.generate(wl, seed=seed, seq_lens=list(lens))
    g = torch.Generator().manual_seed(seed + 100)
    dy = torch.randn(inp.tokens, H, 2 * d, generator=g, dtype=torch.float64)
    return inp, dy


def _c_objective(inp, dy, **over):
    """sum(y * dy) with the C oracle; `over` replaces inputs (fp64 arrays)."""
    t = {n: over.get(n, getattr(inp, n)) for n in ("q", "k", "v", "lambda_q1", "lambda_k1", "lambda_q2",
                                                   "lambda_k2", "subln_w")}
    li = orc.lambda_init(inp.wl.depth)
    lam = orc.lambda_values(t["lambda_q1"], t["lambda_k1"], t["lambda_q2"], t["lambda_k2"], li)
    y = orc.forward_rows(inp.cu_seqlens, t["q"], t["k"], t["v"], lam, li, t["subln_w"], inp.wl.eps, inp.wl.causal)
    return float((y * dy.numpy()).sum())


def _grads(inp, dy, eps=None):
    li = orc.lambda_init(inp.wl.depth)
    return ob.gradients(inp.cu_seqlens.tolist(), inp.q.double(), inp.k.double(), inp.v.double(),
                        inp.lambda_q1.double(), inp.lambda_k1.double(), inp.lambda_q2.double(),
                        inp.lambda_k2.double(), inp.subln_w.double(), li,
                        inp.wl.eps if eps is None else eps, inp.wl.causal, dy)


def test_torch_forward_equals_c_oracle():
    inp, _ = _case(1)
    li = orc.lambda_init(inp.wl.depth)
    y = ob.forward(inp.cu_seqlens.tolist(), inp.q.double(), inp.k.double(), inp.v.double(),
                   inp.lambda_q1.double(), inp.lambda_k1.double(), inp.lambda_q2.double(), inp.lambda_k2.double(),
                   inp.subln_w.double(), li, inp.wl.eps, inp.wl.causal)
    np.testing.assert_allclose(y.numpy(), orc.forward(inp), atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal,per_head", [(True, False), (False, False), (True, True)])
def test_gradients_match_finite_differences(causal, per_head):
    inp, dy = _case(2 + causal + 2 * per_head, causal=causal, per_head=per_head)
    grads = _grads(inp, dy)
    names = {"q": "q", "k": "k", "v": "v", "lambda_q1": "lq1", "lambda_k1": "lk1", "lambda_q2": "lq2",
             "lambda_k2": "lk2", "subln_w": "w"}
    rng = np.random.default_rng(5)
    h = 1e-5
    for name, gname in names.items():
        base = getattr(inp, name).double().numpy()
        flat = base.reshape(-1)
        for idx in rng.choice(flat.size, size=min(6, flat.size), replace=False):
            plus, minus = flat.copy(), flat.copy()
            plus[idx] += h
            minus[idx] -= h
            fd = (_c_objective(inp, dy, **{name: plus.reshape(base.shape)}) -
                  _c_objective(inp, dy, **{name: minus.reshape(base.shape)})) / (2 * h)
            ag = float(grads[gname].reshape(-1)[idx])
            assert abs(fd - ag) <= 1e-6 * max(1.0, abs(ag)), (name, idx, fd, ag)


def test_value_scale_direction_is_flat():
    """With eps = 0, y(cV) = y(V): the gradient has no component along V."""
    inp, dy = _case(9)
    grads = _grads(inp, dy, eps=0.0)
    dot = float((grads["v"] * inp.v.double()).sum())
    assert abs(dot) < 1e-9 * float(grads["v"].abs().sum())
