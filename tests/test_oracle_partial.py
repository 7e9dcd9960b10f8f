"""Pins for the context-parallel oracle (CPU only): partials over a partition of
the keys, merged, equal the independent C oracle's forward; a partial's
components equal the C oracle's attention outputs (read through lambda = 0 and
a huge eps); the log-sum-exp of disjoint key blocks adds in the exponent; the
merge ignores part order and parts with no visible key; planted mistakes in
the merge are caught."""
import numpy as np
import pytest
import torch

from differential_attention_diffattn_gb300 import workloads as W
from oracle import oracle as orc
from oracle import partial as op


def _case(seed, lens, H=4, Hkv=2, d=8, causal=True, per_head=False):
    wl = W.Workload("p", "f32", num_heads=H, num_kv_heads=Hkv, d=d, dv=2 * d, depth=5, causal=causal, batch=1,
                    seqlen=1, random_subln=True, lambda_per_head=per_head)
    inp = W.generate(wl, seed=seed, seq_lens=lens)
    li = orc.lambda_init(wl.depth)
    lam = orc.lambda_values(inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2, li)
    return inp, lam, li


def _split_merge(inp, lam, li, bounds, causal):
    q, k, v = inp.q.double().numpy(), inp.k.double().numpy(), inp.v.double().numpy()
    T = q.shape[0]
    pos = np.arange(T)
    parts = [op.partial(q, k[a:b], v[a:b], pos, pos[a:b], causal) for a, b in zip(bounds[:-1], bounds[1:])]
    return parts, op.merge([p[0] for p in parts], [p[1] for p in parts], [p[2] for p in parts], lam, li,
                           inp.subln_w.double().numpy(), inp.wl.eps)


@pytest.mark.parametrize("causal,per_head,bounds", [
    (True, False, [0, 37]),
    (True, False, [0, 10, 11, 30, 37]),
    (False, True, [0, 20, 37]),
    (True, True, [0, 1, 2, 36, 37]),
])
def test_merged_partials_equal_full_forward(causal, per_head, bounds):
    inp, lam, li = _case(3, [37], causal=causal, per_head=per_head)
    _, y = _split_merge(inp, lam, li, bounds, causal)
    want = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, lam, li, inp.subln_w, inp.wl.eps, causal)
    np.testing.assert_allclose(y, want, atol=1e-11)


def test_partial_components_equal_c_oracle_attention():
    inp, _, _ = _case(4, [29])
    q, k, v = inp.q.double().numpy(), inp.k.double().numpy(), inp.v.double().numpy()
    pos = np.arange(29)
    _, o1, o2 = op.partial(q, k, v, pos, pos, True)
    E, d = 1e12, inp.wl.d
    ones = np.ones(inp.wl.dv)
    want1 = orc.forward_rows(inp.cu_seqlens, q, k, v, 0.0, 0.0, ones, E, True) * np.sqrt(E)
    sw = lambda x: np.concatenate([x[..., d:], x[..., :d]], -1)  # noqa: E731
    want2 = orc.forward_rows(inp.cu_seqlens, sw(q), sw(k), v, 0.0, 0.0, ones, E, True) * np.sqrt(E)
    np.testing.assert_allclose(o1, want1, atol=1e-9)
    np.testing.assert_allclose(o2, want2, atol=1e-9)


def test_lse_single_key_and_additivity():
    inp, _, _ = _case(5, [16], H=2, Hkv=2)
    q, k, v = inp.q.double().numpy(), inp.k.double().numpy(), inp.v.double().numpy()
    d = inp.wl.d
    pos = np.arange(16)
    lse1, *_ = op.partial(q[3:4], k[5:6], v[5:6], [3], [5], False)
    want = float(q[3, 1, d:] @ k[5, 1, d:]) * d ** -0.5 / np.log(2.0)
    assert abs(lse1[0, 1, 1] - want) < 1e-12
    la, *_ = op.partial(q, k[:6], v[:6], pos, pos[:6], False)
    lb, *_ = op.partial(q, k[6:], v[6:], pos, pos[6:], False)
    lab, *_ = op.partial(q, k, v, pos, pos, False)
    np.testing.assert_allclose(np.exp2(lab), np.exp2(la) + np.exp2(lb), rtol=1e-12)


def test_merge_ignores_order_and_empty_parts():
    inp, lam, li = _case(6, [24])
    parts, y = _split_merge(inp, lam, li, [0, 8, 24], True)
    w = inp.subln_w.double().numpy()
    rev = op.merge([p[0] for p in parts[::-1]], [p[1] for p in parts[::-1]], [p[2] for p in parts[::-1]], lam, li,
                   w, inp.wl.eps)
    np.testing.assert_allclose(rev, y, atol=1e-13)
    # the first query rows see no key of [8, 24): those parts have lse = -inf and must not count
    assert np.isneginf(parts[1][0][:8]).all()
    empty = (np.full_like(parts[0][0], -np.inf), np.full_like(parts[0][1], 7.0), np.full_like(parts[0][2], -3.0))
    plus = op.merge([p[0] for p in parts] + [empty[0]], [p[1] for p in parts] + [empty[1]],
                    [p[2] for p in parts] + [empty[2]], lam, li, w, inp.wl.eps)
    np.testing.assert_allclose(plus, y, atol=1e-13)


def _mutant_merges():
    def natural_exp(lse, o1, o2, lam, li, w, eps):
        lse = np.asarray(lse)
        return op.merge(lse * np.log(2.0) / np.log(2.0) * np.log2(np.e), o1, o2, lam, li, w, eps)

    def norm_then_merge(lse, o1, o2, lam, li, w, eps):
        ys = [op.merge([l], [a], [b], lam, li, w, eps) for l, a, b in zip(lse, o1, o2)]
        return np.mean(ys, axis=0)

    def shared_weights(lse, o1, o2, lam, li, w, eps):
        lse = np.asarray(lse).copy()
        lse[..., 1] = lse[..., 0]
        return op.merge(lse, o1, o2, lam, li, w, eps)

    def plain_average(lse, o1, o2, lam, li, w, eps):
        return op.merge(np.zeros_like(np.asarray(lse)), o1, o2, lam, li, w, eps)
    return [natural_exp, norm_then_merge, shared_weights, plain_average]


@pytest.mark.parametrize("mutant", _mutant_merges())
def test_merge_mutants_are_caught(mutant):
    inp, lam, li = _case(7, [30])
    parts, _ = _split_merge(inp, lam, li, [0, 12, 30], True)
    parts = [(np.where(np.isneginf(p[0]), -1e300, p[0]), p[1], p[2]) for p in parts]
    y = mutant([p[0] for p in parts], [p[1] for p in parts], [p[2] for p in parts], lam, li,
               inp.subln_w.double().numpy(), inp.wl.eps)
    want = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, lam, li, inp.subln_w, inp.wl.eps, True)
    assert not np.allclose(y, want, atol=1e-6)
