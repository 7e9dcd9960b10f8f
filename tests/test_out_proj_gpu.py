"""GPU parity of the output projection (tcgen05 GEMM y = x W^T) against the
fp64 oracle, on shapes with ragged row, column and K tails, and the attention
followed by the projection against the oracle attention followed by the oracle
projection."""
import numpy as np
import pytest
import torch

import differential_attention_diffattn_gb300 as da
from differential_attention_diffattn_gb300 import workloads as W
from oracle import oracle as orc
from oracle import out_proj as oo

from gpu_util import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    da.build()
    da.load_library()
    torch.cuda.set_device(0)


def _check(y, x, w):
    xd, wd = x.double().cpu().numpy(), w.double().cpu().numpy()
    want = oo.out_proj(xd, wd)
    mag = oo.out_proj(np.abs(xd), np.abs(wd))  # sum_k |x_k w_k|: scale of fp32 accumulation error
    err = np.abs(y.double().cpu().numpy() - want)
    bound = 2.0 ** -8 * np.abs(want) + 1e-5 * mag + 1e-6
    assert (err <= bound).all(), (float((err - bound).max()), np.unravel_index(np.argmax(err - bound), err.shape))


@pytest.mark.parametrize("M,K,N", [(1, 64, 8), (333, 200, 136), (1000, 2048, 2048), (129, 4096, 520), (2048, 2048, 256)])
def test_out_proj_matches_oracle(M, K, N):
    g = torch.Generator().manual_seed(M + K + N)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(N, K, generator=g) * K ** -0.5).to(torch.bfloat16).cuda()
    y = da.diffattn_out_proj(x, w)
    assert da.diffattn_get_device_status() == 0
    _check(y, x, w)


def test_out_proj_reuses_persistent_tiles():
    """More tiles than SMs: every CTA walks several tiles and both accumulators."""
    g = torch.Generator().manual_seed(5)
    M, K, N = 8192, 512, 2048       # 64 x 8 = 512 tiles
    x = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(N, K, generator=g) * K ** -0.5).to(torch.bfloat16).cuda()
    y = da.diffattn_out_proj(x, w)
    assert da.diffattn_get_device_status() == 0
    rows = np.r_[0:64, 4000:4064, M - 64:M]
    _check(y[rows], x[rows], w)


def test_attention_then_out_proj_matches_oracle():
    wl = W.with_overrides(W.WORKLOADS["b2_t512_gqa"], random_subln=True)
    inp = W.generate(wl, seed=8, seq_lens=[300, 129])
    li = da.diffattn_lambda_init(wl.depth)
    lam = da.diffattn_lambda(*(x.cuda() for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)), li)
    cu = inp.cu_seqlens.cuda()
    attn = da.diffattn_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), lam, li, inp.subln_w.cuda(), causal=True,
                           cu_seqlens=cu, max_seqlen=inp.max_seqlen, eps=wl.eps)
    hidden = 1024
    wo = (torch.randn(hidden, wl.num_heads * wl.dv, generator=torch.Generator().manual_seed(9)) *
          (wl.num_heads * wl.dv) ** -0.5).to(torch.bfloat16)
    y = da.diffattn_out_proj(attn, wo.cuda())
    assert da.diffattn_get_device_status() == 0
    oli = orc.lambda_init(wl.depth)
    olam = orc.lambda_values(inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2, oli)
    a64 = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, olam, oli, inp.subln_w, wl.eps, True)
    compare(y, oo.out_proj(a64, wo.double().numpy()), "bf16")
