"""GPU parity of the context-parallel split: the merge kernel against the merge
oracle on partials the oracle computes, and the whole split (every rank's
blocks, emulated one rank after another on one GPU, no exchange needed) against
the C oracle's forward of the whole sequence."""
import numpy as np
import pytest
import torch

import differential_attention_diffattn_gb300 as da
from differential_attention_diffattn_gb300 import context_parallel as cp
from differential_attention_diffattn_gb300 import workloads as W
from oracle import oracle as orc
from oracle import partial as op

from gpu_util import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    da.build()
    da.load_library()
    torch.cuda.set_device(0)


# more than two parts: the merge kernel takes them two at a time and rescales
@pytest.mark.parametrize("bounds,per_head", [([0, 96], False), ([0, 30, 31, 96], True), ([0, 48, 96], False),
                                             ([0, 5, 9, 13, 17, 21, 96], True),
                                             ([0, 10, 20, 30, 40, 50, 60, 70, 96], False)])
def test_merge_kernel_matches_oracle(bounds, per_head):
    wl = W.Workload("m", "bf16", num_heads=4, num_kv_heads=2, d=64, dv=128, depth=6, causal=True, batch=1,
                    seqlen=1, random_subln=True, lambda_per_head=per_head)
    inp = W.generate(wl, seed=31, seq_lens=[96])
    q, k, v = inp.q.double().numpy(), inp.k.double().numpy(), inp.v.double().numpy()
    pos = np.arange(96)
    parts = [op.partial(q, k[a:b], v[a:b], pos, pos[a:b], True) for a, b in zip(bounds[:-1], bounds[1:])]
    li = orc.lambda_init(wl.depth)
    lam = orc.lambda_values(inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2, li)
    want = op.merge([p[0] for p in parts], [p[1] for p in parts], [p[2] for p in parts], lam, li,
                    inp.subln_w.double().numpy(), wl.eps)
    st = lambda i: torch.tensor(np.stack([p[i] for p in parts]), dtype=torch.float32).cuda()  # noqa: E731
    lam_d = torch.tensor(np.atleast_1d(lam), dtype=torch.float32).cuda()
    got = da.diffattn_merge_partials(st(0), st(1), st(2), lam_d, li, inp.subln_w.cuda(), eps=wl.eps,
                                     out_dtype=torch.float32)
    assert da.diffattn_get_device_status() == 0
    # fp32 arithmetic on fp32-rounded partials; the norm divides by rms(D), so the
    # bound scales with each row's condition rms(O1) / rms(D)
    kappa = np.sqrt((parts[0][1] ** 2).mean(-1) + 1e-30) / np.sqrt(
        ((want / (inp.subln_w.double().numpy() * (1 - li))) ** 2).mean(-1) + 1e-30)
    err = np.abs(got.double().cpu().numpy() - want).max(-1)
    assert (err <= 2e-5 * np.maximum(1.0, kappa) * np.abs(want).max()).all(), float(err.max())


# every kernel shape (rows of up to 64, 128, 256 and 512 values; row counts that
# leave the last block part-filled; one to seven parts) on random partials. Parts
# a row does not see (lse = -inf) carry NaN outputs, which must be dropped; every
# row sees at least one part per component.
@pytest.mark.parametrize("n,T,H,dv", [(1, 37, 3, 36), (2, 37, 3, 64), (3, 29, 5, 128), (5, 23, 3, 200),
                                      (2, 19, 3, 512), (7, 11, 2, 256)])
def test_merge_kernel_shapes(n, T, H, dv):
    rng = np.random.default_rng(1000 + 10 * dv + n)
    f32 = lambda a: np.asarray(a, dtype=np.float32).astype(np.float64)  # noqa: E731
    lse = f32(rng.normal(0.0, 3.0, (n, T, H, 2)))
    hide = rng.random((n, T, H, 2)) < 0.3
    keep = rng.integers(0, n, (T, H, 2))
    hide[keep, np.arange(T)[:, None, None], np.arange(H)[None, :, None], np.arange(2)[None, None, :]] = False
    lse[hide] = -np.inf
    o1, o2 = f32(rng.normal(size=(n, T, H, dv))), f32(rng.normal(size=(n, T, H, dv)))
    lam, w, li, eps = f32(rng.normal(0.0, 0.3, H)), f32(rng.normal(size=dv)), 0.35, 1e-5
    want = op.merge(lse, np.where(hide[..., :1], 0.0, o1), np.where(hide[..., 1:], 0.0, o2), lam, li, w, eps)
    dev = lambda a: torch.tensor(a, dtype=torch.float32).cuda()  # noqa: E731
    got = da.diffattn_merge_partials(dev(lse), dev(np.where(hide[..., :1], np.nan, o1)),
                                     dev(np.where(hide[..., 1:], np.nan, o2)), dev(lam), li, dev(w), eps=eps,
                                     out_dtype=torch.float32)
    assert da.diffattn_get_device_status() == 0
    got = got.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - want).max(-1)
    assert (err <= 1e-4 * np.abs(want).max(-1)).all(), float(err.max())


@pytest.mark.parametrize("world,chunk,H,Hkv", [(1, 256, 16, 4), (2, 256, 16, 4), (4, 128, 8, 8), (3, 200, 4, 1)])
def test_split_forward_matches_full_forward(world, chunk, H, Hkv):
    wl = W.with_overrides(W.WORKLOADS["b2_t512_gqa"], num_heads=H, num_kv_heads=Hkv, random_subln=True)
    T = 2 * world * chunk
    inp = W.generate(wl, seed=40 + world, seq_lens=[T])
    li = da.diffattn_lambda_init(wl.depth)
    lam = da.diffattn_lambda(*(x.cuda() for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)), li)
    q, k, v, w = inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.subln_w.cuda()
    kern = cp.GpuKernels(lam, li, w, wl.eps)
    kv = {b: (k[b * chunk:(b + 1) * chunk], v[b * chunk:(b + 1) * chunk]) for b in range(2 * world)}
    y = torch.empty(T, H, wl.dv, dtype=torch.bfloat16, device="cuda")
    for r in range(world):
        for a, out in cp.local_forward(cp.split_zigzag(q, world, r), kv, kern).items():
            y[a * chunk:(a + 1) * chunk] = out
    assert da.diffattn_get_device_status() == 0
    rows = (np.arange(0, T, 3).repeat(2), np.tile([0, H - 1], len(range(0, T, 3))))
    oli = orc.lambda_init(wl.depth)
    olam = orc.lambda_values(inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2, oli)
    want = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, olam, oli, inp.subln_w, wl.eps, True, rows)
    compare(y[rows[0], rows[1]], want, "bf16")
