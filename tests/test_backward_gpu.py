"""GPU parity of the training forward outputs and the backward pass against
the fp64 gradient oracle (autograd of the plain forward, itself pinned by
finite differences of the C oracle)."""
import numpy as np
import pytest
import torch

import differential_attention_diffattn_gb300 as da
from differential_attention_diffattn_gb300 import workloads as W
from oracle import backward as ob
from oracle import oracle as orc

from gpu_util import compare, oracle_out

pytestmark = pytest.mark.gpu

# bf16 operands (P, dS, dD and the inputs) bound the gradient accuracy: each
# gradient tensor must match the fp64 oracle to a normalised L1 of 2e-2 and a
# max-abs error of 5e-2 of its largest magnitude.
TOL_REL_L1 = 2e-2
TOL_MAX_REL = 5e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    da.build()
    da.load_library()
    torch.cuda.set_device(0)


def grad_close(got, want, name):
    g = got.detach().double().cpu().numpy()
    w = want.detach().double().cpu().numpy()
    assert np.isfinite(g).all(), name
    err = np.abs(g - w)
    rel = err.sum() / max(np.abs(w).sum(), 1e-30)
    mx = err.max() / max(np.abs(w).max(), 1e-30)
    assert rel <= TOL_REL_L1 and mx <= TOL_MAX_REL, (name, rel, mx)


def run_case(wl, lens, seed, one_lambda_set=False):
    inp = W.generate(wl, seed=seed, seq_lens=lens)
    if one_lambda_set:  # per-head layout, every head given head 0's vectors
        for n in ("lambda_q1", "lambda_k1", "lambda_q2", "lambda_k2"):
            t = getattr(inp, n)
            setattr(inp, n, t[:1].expand_as(t).contiguous())
    dev = "cuda"
    li = da.diffattn_lambda_init(wl.depth)
    lv = [x.to(dev) for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)]
    lam = da.diffattn_lambda(*lv, li)
    q, k, v, w = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.subln_w.to(dev)
    cu = inp.cu_seqlens.to(dev)
    out, lse, o1, o2 = da.diffattn_fwd_train(q, k, v, lam, li, w, causal=wl.causal, cu_seqlens=cu,
                                             max_seqlen=inp.max_seqlen, eps=wl.eps)
    g = torch.Generator().manual_seed(seed + 1)
    dy = torch.randn(out.shape, generator=g).to(torch.bfloat16)
    dq, dk, dv, dlam, dw = da.diffattn_bwd(q, k, v, lam, li, w, dy.to(dev), lse, o1, o2, causal=wl.causal,
                                           cu_seqlens=cu, max_seqlen=inp.max_seqlen, eps=wl.eps)
    dl = da.diffattn_lambda_bwd(*lv, dlam)
    assert da.diffattn_get_device_status() == 0
    return inp, dy, out, lse, o1, o2, dq, dk, dv, dlam, dw, dl


BF = W.WORKLOADS["b2_t512_gqa"]


# two packed sequences: the one-item-per-CTA kernel; eight (384 items of up to
# three key tiles): the persistent kernel, whose epilogue warpgroup writes O1, O2
@pytest.mark.parametrize("lens,kernel", [([300, 129], "diffattn_fwd_bf16_sm103a_kernel"),
                                         ([300, 129, 200, 1, 256, 77, 300, 150],
                                          "diffattn_fwd_bf16_persistent_kernel")])
def test_training_outputs_match_oracle(lens, kernel):
    chk = W.generate(BF, seed=81, seq_lens=lens)
    lam1 = torch.ones(1, dtype=torch.float32, device="cuda")
    assert da.diffattn_fwd_kernel(chk.q.cuda(), chk.k.cuda(), chk.v.cuda(), lam1, chk.subln_w.cuda(),
                                  cu_seqlens=chk.cu_seqlens.cuda(), max_seqlen=chk.max_seqlen) == kernel
    inp, dy, out, lse, o1, o2, *_ = run_case(BF, lens, 81)
    compare(out, oracle_out(inp), "bf16")
    # normalised attention outputs: the oracle with lambda = 0, lambda_init = 0,
    # w = 1 and a huge eps returns O1 / sqrt(eps); swapping components gives O2
    E = 1e12
    G = inp.wl.num_heads // inp.wl.num_kv_heads
    ones = np.ones(inp.wl.dv)
    want1 = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, 0.0, 0.0, ones, E, True) * np.sqrt(E)
    d = inp.wl.d
    q_sw = torch.cat([inp.q[..., d:], inp.q[..., :d]], -1)
    k_sw = torch.cat([inp.k[..., d:], inp.k[..., :d]], -1)
    want2 = orc.forward_rows(inp.cu_seqlens, q_sw, k_sw, inp.v, 0.0, 0.0, ones, E, True) * np.sqrt(E)
    for got, want in ((o1, want1), (o2, want2)):
        err = np.abs(got.float().cpu().numpy() - want)
        assert err.max() <= 2e-2 and err.sum() / np.abs(want).sum() <= 5e-3
        # the first query of a causal sequence sees one key: its probability is
        # exactly 1, so the normalised output is that key's value (to fp32 rounding
        # of the exponential of a zero argument)
        for t in inp.cu_seqlens[:-1].tolist():
            row = got[t].double().cpu()
            v0 = inp.v[t].double().repeat_interleave(G, dim=0)
            assert (row - v0).abs().max() <= 1e-6 * v0.abs().max(), t
    # lse: log2 sum over visible keys of 2^(s log2(e) <q_c, k_c>), per component
    qf, kf = inp.q.double(), inp.k.double()
    cu = inp.cu_seqlens.tolist()
    for t in (0, 1, 150, 299, 300, 428):
        sq = max(i for i in range(len(cu) - 1) if cu[i] <= t)
        a = cu[sq]
        for h in (0, 5, 15):
            for c in range(2):
                sc = (kf[a:t + 1, h // G, c * d:(c + 1) * d] @ qf[t, h, c * d:(c + 1) * d]) * d ** -0.5 / np.log(2)
                want = float(torch.logsumexp(sc * np.log(2), 0) / np.log(2))
                assert abs(float(lse[t, h, c]) - want) < 1e-3


# the last case's training forward runs on the persistent kernel (384 items)
@pytest.mark.parametrize("lens,H,Hkv,causal,per_head", [
    ([256], 16, 4, True, False),
    ([300, 129, 1], 8, 2, True, True),
    ([200], 4, 4, False, False),
    ([513], 16, 16, True, False),
    ([300, 129, 200, 1, 256, 77, 300, 150], 16, 4, True, False),
    # 16 query blocks per key tile and 8 key tiles per query tile: the rings of both
    # kernels wrap several times, and the last blocks run past the sequences' ends
    ([1000], 16, 4, True, True),
    ([777, 1000], 8, 8, True, False),
    # token x head rows not a multiple of the preprocessing kernel's 4-row chunks (a last
    # chunk of 3 rows; per-head and shared lambda)
    ([333], 3, 1, True, True),
    ([301, 2], 5, 5, True, False),
])
def test_backward_matches_oracle(lens, H, Hkv, causal, per_head):
    wl = W.with_overrides(BF, num_heads=H, num_kv_heads=Hkv, causal=causal, lambda_per_head=per_head,
                          random_subln=True)
    inp, dy, out, lse, o1, o2, dq, dk, dv, dlam, dw, dl = run_case(wl, lens, 90 + H + len(lens))
    li = orc.lambda_init(wl.depth)
    want = ob.gradients(inp.cu_seqlens.tolist(), inp.q.double(), inp.k.double(), inp.v.double(),
                        inp.lambda_q1.double(), inp.lambda_k1.double(), inp.lambda_q2.double(),
                        inp.lambda_k2.double(), inp.subln_w.double(), li, wl.eps, causal, dy.double())
    grad_close(dq, want["q"], "dq")
    grad_close(dk, want["k"], "dk")
    grad_close(dv, want["v"], "dv")
    grad_close(dw, want["w"], "dw")
    for got, name in zip(dl, ("lq1", "lk1", "lq2", "lk2")):
        grad_close(got, want[name], name)


# More heads than the preprocessing kernel sums per head in shared memory (1024): the
# per-head lambda gradients accumulate in global memory instead. Every head gets the same
# lambda vectors (random ones per head would, over a thousand heads, include heads whose
# two maps nearly cancel, where the bf16 bound of the forward itself does not hold).
def test_backward_many_heads_per_head_lambda():
    wl = W.with_overrides(BF, num_heads=1030, num_kv_heads=1030, causal=True, lambda_per_head=True,
                          random_subln=True)
    lens = [200, 7]
    inp, dy, out, lse, o1, o2, dq, dk, dv, dlam, dw, dl = run_case(wl, lens, 97, one_lambda_set=True)
    li = orc.lambda_init(wl.depth)
    want = ob.gradients(inp.cu_seqlens.tolist(), inp.q.double(), inp.k.double(), inp.v.double(),
                        inp.lambda_q1.double(), inp.lambda_k1.double(), inp.lambda_q2.double(),
                        inp.lambda_k2.double(), inp.subln_w.double(), li, wl.eps, True, dy.double())
    grad_close(dq, want["q"], "dq")
    grad_close(dk, want["k"], "dk")
    grad_close(dv, want["v"], "dv")
    grad_close(dw, want["w"], "dw")
    for got, name in zip(dl, ("lq1", "lk1", "lq2", "lk2")):
        grad_close(got, want[name], name)


# Full-size batches against the same sequences one call each: dQ, dK and dV of a
# token depend only on its own sequence, so the bits must agree. The two shapes
# take the two launch orders of the backward kernels: 2 x 8192 tokens with 16 kv
# heads launches sequence-major (many waves, no tail); 4 x 2048 tokens with 4 kv
# heads puts the key tiles outermost (a dK/dV grid of 256 CTAs); a single
# sequence is the same grid either way.
@pytest.mark.parametrize("lens,H,Hkv", [([8192] * 2, 16, 16), ([2048] * 4, 16, 4)])
def test_backward_batch_equals_separate_calls_bitwise(lens, H, Hkv):
    wl = W.with_overrides(BF, num_heads=H, num_kv_heads=Hkv, random_subln=True)
    inp = W.generate(wl, seed=131, seq_lens=lens)
    B, T = len(lens), lens[0]
    dev = "cuda"
    li = da.diffattn_lambda_init(wl.depth)
    lam = da.diffattn_lambda(*(x.to(dev) for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)), li)
    q, k, v = (x.to(dev).view(B, T, *x.shape[1:]) for x in (inp.q, inp.k, inp.v))
    w = inp.subln_w.to(dev)
    out, lse, o1, o2 = da.diffattn_fwd_train(q, k, v, lam, li, w, causal=True, eps=wl.eps)
    dy = (torch.randn(out.shape, generator=torch.Generator().manual_seed(132)) * 0.1).to(torch.bfloat16).to(dev)
    batch = da.diffattn_bwd(q, k, v, lam, li, w, dy, lse, o1, o2, causal=True, eps=wl.eps)[:3]
    for b in range(B):
        one = da.diffattn_bwd(q[b:b + 1], k[b:b + 1], v[b:b + 1], lam, li, w, dy[b:b + 1], lse[b:b + 1],
                              o1[b:b + 1], o2[b:b + 1], causal=True, eps=wl.eps)[:3]
        for got, want, name in zip(batch, one, ("dq", "dk", "dv")):
            assert torch.equal(got[b:b + 1], want), (name, b)
    assert da.diffattn_get_device_status() == 0
